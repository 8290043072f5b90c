"""Device-side plumbing for tests, the benchmark and the smoke run: moves a
seeded Workload to the GPU and calls the C ABI through the binding.  No part of
the computation happens here."""
import numpy as np
import torch

from . import (alloc_workspace, dsa_indexer_score, dsa_layer_step, dsa_sparse_mla, dsa_topk, make_batch,
               make_host_io, make_layout, prepare_layer_step_host)


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
        if getattr(wl, "q_fmt", 0) == 1:   # MXFP4 index queries in q_idx
            flags |= 2
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


class HostStep:
    """Page-locked host copies of a device workload's per-step inputs and outputs,
    the device buffers dsa_layer_step_host copies them into, and that call.

    packed=True lays the inputs out back to back, in the order DSA_HOST_PACKED
    names, in one host buffer and one device buffer, and sets that flag (the call
    moves them with one copy); packed=False gives every input its own allocation
    on both sides and one copy each.  pinned=False keeps the host side in pageable
    memory; misalign > 0 (a multiple of 4) starts every host array that many bytes
    into its allocation."""

    def __init__(self, dw, packed=True, with_lse=True, with_idx=True, pinned=True, misalign=0):
        self.dw = dw
        src = [dw.q.view(torch.uint8), dw.q_idx, dw.w, dw.q_req, dw.q_pos, dw.ctx, dw.bt]
        sizes = [t.numel() * t.element_size() for t in src]
        def host_empty(shape, dtype):
            n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
            buf = torch.empty(n + misalign, dtype=torch.uint8)
            buf = buf.pin_memory() if pinned else buf
            return buf[misalign:].view(dtype).view(shape)

        if packed:
            dev_all = torch.empty(sum(sizes), dtype=torch.uint8, device=dw.device)
            host_all = host_empty((sum(sizes),), torch.uint8)
            dev, host, off = [], [], 0
            for t, n in zip(src, sizes):
                dev.append(dev_all[off:off + n].view(t.dtype).view(t.shape))
                host.append(host_all[off:off + n].view(t.dtype).view(t.shape))
                off += n
            self._keep = (dev_all, host_all)
        else:
            dev = [torch.empty_like(t) for t in src]
            host = [host_empty(t.shape, t.dtype) for t in src]
        for h, t in zip(host, src):
            h.copy_(t.cpu())
        self.dev, self.host = dev, host
        q, q_idx, w, q_req, q_pos, ctx, bt = dev
        self.q, self.q_idx, self.w = q.view(torch.bfloat16), q_idx, w
        self.batch = make_batch(q_req, q_pos, ctx, bt, dw.wl.max_ctx_len, dw.batch.flags)
        T = dw.wl.num_tokens
        self.out = torch.empty(T, 96, 512, dtype=torch.bfloat16, device=dw.device)
        self.lse = torch.empty(T, 96, dtype=torch.float32, device=dw.device) if with_lse else None
        self.idx = torch.empty(T, dw.topk, dtype=torch.int32, device=dw.device) if with_idx else None
        self.out_host = host_empty(self.out.shape, self.out.dtype)
        self.lse_host = host_empty((T, 96), torch.float32) if with_lse else None
        self.idx_host = host_empty((T, dw.topk), torch.int32) if with_idx else None
        self.io = make_host_io(host[1], host[2], host[0], host[3], host[4], host[5], host[6], self.out_host,
                               self.lse_host, self.idx_host, packed=packed)
        self._calls = {}
        self.h2d_bytes = sum(sizes)
        self.d2h_bytes = sum(t.numel() * t.element_size() for t in (self.out_host, self.lse_host, self.idx_host)
                             if t is not None)

    def step(self, stream=None, layout=None):
        """One dsa_layer_step_host call (arguments marshalled once per layout and stream)."""
        dw = self.dw
        layout = dw.layout if layout is None else layout
        if stream is None:
            stream = torch.cuda.current_stream()
        key = (id(layout), stream.cuda_stream)
        entry = self._calls.get(key)
        if entry is None:
            call = prepare_layer_step_host(layout, self.batch, self.q_idx, self.w, self.q, dw.topk, dw.wl.sm_scale,
                                           self.out, self.io, idx_out=self.idx, lse=self.lse, ws=dw.ws,
                                           stream=stream)
            entry = self._calls[key] = (call, layout, stream)   # the layout and stream outlive the call
        entry[0]()
