"""Device copies of generated inputs, for the tests and the benchmark.

``Dev`` uploads one ``gen.DSAInputs`` to the GPU (pools, block table, queries,
a zeroed workspace sized by ``dsa_workspace_size``) and calls libdsa's entry
points on it. It holds no arithmetic of the method: every stage runs in the
library's kernels.
"""
from __future__ import annotations

import numpy as np

import dsa_sparse_mla_paged_gb300 as dsa

KEY_FMT = {"fp8": dsa.DSA_KEY_FP8_132, "mxfp4": dsa.DSA_KEY_MXFP4_68}
LAT_FMT = {"fp8": dsa.DSA_LAT_FP8_576, "nvfp4": dsa.DSA_LAT_NVFP4_352}


def params_for(inp, flags=0):
    return dsa.make_params(
        batch=inp.batch, n_q=inp.n_q, max_pages_per_req=inp.max_pages, num_pages=inp.num_pages,
        key_page_stride=inp.key_page_stride, lat_page_stride=inp.lat_page_stride, topk=inp.topk,
        page_size=inp.page_size, key_fmt=KEY_FMT[inp.key_fmt], lat_fmt=LAT_FMT[inp.lat_fmt],
        softmax_scale=inp.softmax_scale, latent_scale=inp.latent_scale, flags=flags)


class Dev:
    """Device copies of one DSAInputs plus a zeroed workspace."""

    def __init__(self, inp, flags=0, device="cuda"):
        import torch

        self.inp = inp
        self.p = params_for(inp, flags)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
        self.q_idx = t(inp.q_idx.view(np.int16)).view(torch.bfloat16)
        self.w = t(inp.w)
        self.key_pool = t(inp.key_pool)
        self.q = t(inp.q.view(np.int16)).view(torch.bfloat16)
        self.lat_pool = t(inp.lat_pool)
        self.block_table = t(inp.block_table)
        self.ctx = t(inp.ctx)
        self.rows = inp.batch * inp.n_q
        self.cap = inp.max_pages * inp.page_size
        self.ws = torch.zeros(dsa.workspace_size(self.p), dtype=torch.uint8, device=device)

    def scores(self, stride=None):
        import torch

        stride = stride or (self.cap + 3) // 4 * 4
        sc = torch.full((self.rows, stride), float("nan"), dtype=torch.float32, device="cuda")
        dsa.indexer_scores(self.p, self.q_idx, self.w, self.key_pool, self.block_table, self.ctx, sc, stride,
                           self.ws)
        return sc

    def topk(self, scores_np=None, scores_dev=None, phys=False):
        import torch

        if scores_dev is None:
            stride = (scores_np.shape[1] + 3) // 4 * 4
            scores_dev = torch.zeros((self.rows, stride), dtype=torch.float32, device="cuda")
            scores_dev[:, :scores_np.shape[1]] = torch.from_numpy(scores_np)
        idx = torch.full((self.rows, self.inp.topk), -7, dtype=torch.int32, device="cuda")
        pr = torch.full_like(idx, -7) if phys else None
        dsa.topk(self.p, scores_dev, scores_dev.shape[1], self.ctx, self.block_table, idx, pr, self.ws)
        return idx, pr

    def mla(self, topk_idx):
        import torch

        out = torch.empty((self.rows, 96, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((self.rows, 96), dtype=torch.float32, device="cuda")
        dsa.sparse_mla_decode(self.p, self.q, self.lat_pool, self.block_table, self.ctx, topk_idx, out, lse,
                              self.ws)
        return out, lse

    def decode(self):
        import torch

        out = torch.empty((self.rows, 96, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((self.rows, 96), dtype=torch.float32, device="cuda")
        idx = torch.empty((self.rows, self.inp.topk), dtype=torch.int32, device="cuda")
        dsa.decode(self.p, self.q_idx, self.w, self.key_pool, self.q, self.lat_pool, self.block_table, self.ctx,
                   out, lse, idx, self.ws)
        return out, lse, idx
