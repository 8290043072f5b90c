"""Device-side plumbing for tests, the benchmark and the smoke run: moves a
seeded Workload to the GPU and calls the C ABI through the binding.  No part of
the computation happens here."""
import numpy as np
import torch

from . import (alloc_workspace, dsa_indexer_score, dsa_layer_step, dsa_sparse_mla, dsa_topk, make_batch,
               make_layout)


class DeviceWorkload:
    def __init__(self, wl, device="cuda", topk=None, flags=0):
        self.wl = wl
        self.device = device
        self.topk = int(wl.topk if topk is None else topk)
        self.pool = torch.from_numpy(wl.pool).to(device)
        self.bt = torch.from_numpy(np.ascontiguousarray(wl.block_table)).to(device)
        self.ctx = torch.from_numpy(wl.ctx_lens).to(device)
        self.q_req = torch.from_numpy(wl.q_req).to(device)
        self.q_pos = torch.from_numpy(wl.q_pos).to(device)
        self.q_idx = torch.from_numpy(wl.q_idx).to(device)
        self.w = torch.from_numpy(wl.w).to(device)
        self.q = torch.from_numpy(wl.q.view(np.int16)).to(device).view(torch.bfloat16)
        self.layout = make_layout(self.pool, wl.num_rows, wl.row_stride, wl.idx_page_offset, wl.lat_page_offset,
                                  wl.block_size, wl.idx_fmt, wl.lat_fmt)
        self.batch = make_batch(self.q_req, self.q_pos, self.ctx, self.bt, wl.max_ctx_len, flags)
        self.ws = alloc_workspace(self.layout, self.batch, self.topk, device)
        T = wl.num_tokens
        self.ld = (wl.max_ctx_len + 3) // 4 * 4
        self.out = torch.empty(T, 96, 512, dtype=torch.bfloat16, device=device)
        self.lse = torch.empty(T, 96, dtype=torch.float32, device=device)
        self.idx = torch.empty(T, self.topk, dtype=torch.int32, device=device)

    def pool_copy_layout(self, pool):
        """Layout over another device copy of the pool (same rows, other addresses)."""
        wl = self.wl
        return make_layout(pool, wl.num_rows, wl.row_stride, wl.idx_page_offset, wl.lat_page_offset, wl.block_size,
                           wl.idx_fmt, wl.lat_fmt)

    def layer_step(self, stream=None, layout=None):
        dsa_layer_step(self.layout if layout is None else layout, self.batch, self.q_idx, self.w, self.q, self.topk,
                       self.wl.sm_scale, self.out, idx_out=self.idx, lse=self.lse, ws=self.ws, stream=stream)
        return self.idx, self.out, self.lse

    def indexer_scores(self, stream=None):
        scores = torch.full((self.wl.num_tokens, self.ld), float("nan"), dtype=torch.float32, device=self.device)
        dsa_indexer_score(self.layout, self.batch, self.q_idx, self.w, scores, self.ld, self.ws, stream=stream)
        return scores

    def topk_of(self, scores, with_phys=False, stream=None):
        idx = torch.empty(self.wl.num_tokens, self.topk, dtype=torch.int32, device=self.device)
        phys = torch.empty_like(idx) if with_phys else None
        dsa_topk(self.layout, self.batch, scores, scores.shape[1], self.topk, idx, phys, ws=self.ws, stream=stream)
        return (idx, phys) if with_phys else idx

    def sparse_mla_of(self, idx, stream=None):
        out = torch.empty(self.wl.num_tokens, 96, 512, dtype=torch.bfloat16, device=self.device)
        lse = torch.empty(self.wl.num_tokens, 96, dtype=torch.float32, device=self.device)
        dsa_sparse_mla(self.layout, self.batch, self.q, idx, self.topk, self.wl.sm_scale, out, lse, ws=self.ws,
                       stream=stream)
        return out, lse
