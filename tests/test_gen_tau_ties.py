"""The tie workload's tau ties (CPU): the stored table still matches the
generator, and the planted copies tie with the oracle's K-th token exactly
(16 positions) or within one fp32 ulp of its scale (16 more), so the selection
boundary falls inside a cluster of ties."""
import numpy as np

import gen
from oracle import dsa as O


def test_tau_ties_straddle_the_kth_score():
    inp = gen.make_workload("b64_ctx16k_128k_ties")  # raises if the table is stale
    table = gen.load_tau_table("b64_ctx16k_128k_ties")
    assert len(inp.meta["tau_exact"]) == inp.batch
    for b in (0, 17, 63):
        sc = O.indexer_scores(inp, b, 0)
        s_tau = table[b]["s_tau"]
        tau = sc[s_tau]
        assert tau == np.float32(table[b]["score"])
        ex, nr = inp.meta["tau_exact"][b], inp.meta["tau_near"][b]
        assert len(ex) == 16 and len(nr) == 16
        assert (sc[ex] == tau).all()
        # one ulp of the scale moves the fp64 score by ~6e-8 relative: fp32 scores may round back to tau
        assert (np.abs(sc[nr] - tau) <= 1e-6 * abs(tau)).all()
        kth = np.sort(sc)[::-1][inp.topk - 1]
        assert abs(kth - tau) <= 1e-6 * abs(tau)
        # the hot tokens are still planted and untouched
        assert not (set(ex.tolist()) | set(nr.tolist())) & set(inp.meta["hot_positions"][b].tolist())
