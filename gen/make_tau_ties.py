"""Write gen/tau_ties/<workload>.json: per request, the token the oracle ranks
K-th (score descending, token ascending) after the hot plants, and a digest of
its key bytes so that the generator can tell a stale table.

    python gen/make_tau_ties.py [workload ...]    (default: b64_ctx16k_128k_ties)

Calls only the generator (with the tie planting switched off) and the oracle's
indexer scores; the stored values come from nothing else.
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import gen  # noqa: E402
from oracle import dsa as O  # noqa: E402


def tau_table(name: str) -> list:
    inp = gen.make_workload(name, tau_ties=None)
    out = []
    for b in range(inp.batch):
        sc = O.indexer_scores(inp, b, 0)
        order = np.lexsort((np.arange(len(sc)), -sc.astype(np.float64)))
        s_tau = int(order[min(inp.topk, len(sc)) - 1])
        pg, sl = inp.block_table[b, s_tau // inp.page_size], s_tau % inp.page_size
        kb = inp.key_pool[pg, sl * gen.IDX_DIM:(sl + 1) * gen.IDX_DIM]
        off = inp.page_size * gen.IDX_DIM + 4 * sl
        out.append({"s_tau": s_tau, "score": float(sc[s_tau]),
                    "key_digest": gen._key_digest(kb, inp.key_pool[pg, off:off + 4])})
    return out


def main(names):
    for name in names:
        table = tau_table(name)
        path = os.path.join(gen.TAU_DIR, name + ".json")
        with open(path, "w") as f:
            json.dump({"workload": name, "rank": gen.WORKLOADS[name].get("topk", gen.TOPK),
                       "written_by": "gen/make_tau_ties.py (oracle indexer scores)", "requests": table}, f, indent=0)
        print(path, len(table))


if __name__ == "__main__":
    main(sys.argv[1:] or ["b64_ctx16k_128k_ties"])
