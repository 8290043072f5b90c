"""Python binding of the GB300 DSA layer-step library (include/dsa.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``_lib/libdsa_gb300.so``.  The first call loads that library and
raises ImportError if it is missing (build it with
``dsa_sparse_attention_gb300.build``); there is no fallback path.  Tensors are torch tensors on the current CUDA device
(host tensors are accepted only where a call documents it); PyTorch supplies
device memory and streams.

Names mirror the C ABI: dsa_workspace_size, dsa_indexer_score, dsa_topk,
dsa_sparse_mla, dsa_layer_step, dsa_layer_step_host (and
prepare_layer_step_host, the same call with its arguments marshalled once),
dsa_topk_noalloc, dsa_indexer_front, dsa_write_latent, dsa_selftest_wait_timeout,
dsa_check, dsa_status_string, dsa_abi_version.
"""
import ctypes
import os

import torch

from .build import LIB as _LIB_PATH

DSA_OK = 0
DSA_IDX_FP8, DSA_IDX_MXFP4 = 0, 1
DSA_LAT_FP8, DSA_LAT_NVFP4 = 0, 1
DSA_MAX_TOPK = 2048
DSA_BATCH_INVARIANT = 1
DSA_BATCH_QIDX_MXFP4 = 2
DSA_HOST_PACKED = 1
STATUS_NAMES = {0: "DSA_OK", -1: "DSA_ERR_INVALID_ARG", -2: "DSA_ERR_UNSUPPORTED", -3: "DSA_ERR_CUDA",
                -4: "DSA_ERR_WORKSPACE", -5: "DSA_ERR_TIMEOUT", -6: "DSA_ERR_DEVICE_CHECK"}


class DSAError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class dsa_kv_layout(ctypes.Structure):
    _fields_ = [("pool", ctypes.c_void_p), ("num_rows", ctypes.c_int64), ("row_stride_bytes", ctypes.c_int64),
                ("idx_page_offset", ctypes.c_int64), ("lat_page_offset", ctypes.c_int64),
                ("block_size", ctypes.c_int32), ("idx_fmt", ctypes.c_int32), ("lat_fmt", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class dsa_batch(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int32), ("num_reqs", ctypes.c_int32), ("q_req", ctypes.c_void_p),
                ("q_pos", ctypes.c_void_p), ("ctx_lens", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("bt_stride", ctypes.c_int32), ("flags", ctypes.c_int32), ("max_ctx_len", ctypes.c_int64)]


class dsa_host_io(ctypes.Structure):
    _fields_ = [("q_idx", ctypes.c_void_p), ("w", ctypes.c_void_p), ("q", ctypes.c_void_p), ("q_req", ctypes.c_void_p),
                ("q_pos", ctypes.c_void_p), ("ctx_lens", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("idx", ctypes.c_void_p), ("flags", ctypes.c_int32)]


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"DSA CUDA library not built ({_LIB_PATH}); run dsa_sparse_attention_gb300.build.build()")
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.POINTER
    L, B = P(dsa_kv_layout), P(dsa_batch)
    vp, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    sig = {
        "dsa_abi_version": (i32, []),
        "dsa_status_string": (ctypes.c_char_p, [i32]),
        "dsa_workspace_size": (sz, [L, B, i32]),
        "dsa_indexer_score": (i32, [L, B, vp, vp, vp, i64, vp, sz, vp]),
        "dsa_topk": (i32, [L, B, vp, i64, i32, vp, vp, vp, sz, vp]),
        "dsa_sparse_mla": (i32, [L, B, vp, vp, i32, f32, vp, vp, vp, sz, vp]),
        "dsa_layer_step": (i32, [L, B, vp, vp, vp, i32, f32, vp, vp, vp, vp, sz, vp]),
        "dsa_layer_step_host": (i32, [L, B, vp, vp, vp, i32, f32, vp, vp, vp, P(dsa_host_io), vp, sz, vp]),
        "dsa_check": (i32, [vp, sz, vp]),
        "dsa_last_cuda_error": (i32, [P(ctypes.c_char_p)]),
        "dsa_topk_noalloc": (i32, [L, B, vp, i64, i32, vp, vp, vp]),
        "dsa_selftest_wait_timeout": (i32, [vp, sz, i64, vp]),
        "dsa_indexer_front": (i32, [L, B, vp, i32, vp, f32, vp, vp, vp, vp, vp, vp, sz, vp]),
        "dsa_write_latent": (i32, [L, B, vp, vp, sz, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_LIB = None


def library():
    """The loaded ctypes library (loaded on first use; raises if not built)."""
    global _LIB
    if _LIB is None:
        _LIB = _load()
    return _LIB


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def dsa_last_cuda_error():
    """(code, name) of the CUDA error behind the last DSA_ERR_CUDA on this thread."""
    name = ctypes.c_char_p()
    code = library().dsa_last_cuda_error(ctypes.byref(name))
    return int(code), name.value.decode()


def _check(status, where):
    if status != DSA_OK:
        if status == -3:   # DSA_ERR_CUDA
            code, name = dsa_last_cuda_error()
            where = f"{where} (CUDA error {code}: {name})"
        raise DSAError(status, where)


def make_layout(pool, num_rows, row_stride, idx_page_offset, lat_page_offset, block_size=64,
                idx_fmt=DSA_IDX_FP8, lat_fmt=DSA_LAT_FP8):
    """Layout descriptor over a device uint8 pool tensor (kept alive by the caller)."""
    return dsa_kv_layout(_ptr(pool), int(num_rows), int(row_stride), int(idx_page_offset), int(lat_page_offset),
                         int(block_size), int(idx_fmt), int(lat_fmt), 0)


def make_batch(q_req, q_pos, ctx_lens, block_table, max_ctx_len, flags=0):
    """Batch descriptor over device int32 tensors (kept alive by the caller).  flags:
    DSA_BATCH_INVARIANT and/or DSA_BATCH_QIDX_MXFP4 (q_idx holds MXFP4 index
    queries: T x 32 x 64 code bytes, then T x 32 x 4 E8M0 bytes)."""
    return dsa_batch(int(q_req.shape[0]), int(ctx_lens.shape[0]), _ptr(q_req), _ptr(q_pos), _ptr(ctx_lens),
                     _ptr(block_table), int(block_table.shape[1]), int(flags), int(max_ctx_len))


def dsa_abi_version():
    return library().dsa_abi_version()


def dsa_status_string(status):
    return library().dsa_status_string(int(status)).decode()


def dsa_workspace_size(layout, batch, topk):
    return int(library().dsa_workspace_size(ctypes.byref(layout), ctypes.byref(batch), int(topk)))


def alloc_workspace(layout, batch, topk, device="cuda"):
    """A zeroed workspace of the required size (256-byte aligned by the allocator)."""
    n = dsa_workspace_size(layout, batch, topk)
    if n == 0:
        raise DSAError(-1, "dsa_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def dsa_indexer_score(layout, batch, q_idx, w, scores, ld, ws, stream=None):
    _check(library().dsa_indexer_score(ctypes.byref(layout), ctypes.byref(batch), _ptr(q_idx), _ptr(w), _ptr(scores),
                                 int(ld), _ptr(ws), ws.numel(), _stream(stream)), "dsa_indexer_score")


def dsa_topk(layout, batch, scores, ld, topk, idx, phys_slots=None, ws=None, stream=None):
    lay = ctypes.byref(layout) if layout is not None else None
    _check(library().dsa_topk(lay, ctypes.byref(batch), _ptr(scores), int(ld), int(topk), _ptr(idx), _ptr(phys_slots),
                        _ptr(ws), ws.numel(), _stream(stream)), "dsa_topk")


def dsa_sparse_mla(layout, batch, q, idx, topk, sm_scale, out, lse=None, ws=None, stream=None):
    _check(library().dsa_sparse_mla(ctypes.byref(layout), ctypes.byref(batch), _ptr(q), _ptr(idx), int(topk),
                              float(sm_scale), _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)),
           "dsa_sparse_mla")


def dsa_layer_step(layout, batch, q_idx, w, q, topk, sm_scale, out, idx_out=None, lse=None, ws=None, stream=None):
    _check(library().dsa_layer_step(ctypes.byref(layout), ctypes.byref(batch), _ptr(q_idx), _ptr(w), _ptr(q), int(topk),
                              float(sm_scale), _ptr(idx_out), _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                              _stream(stream)), "dsa_layer_step")


def make_host_io(q_idx, w, q, q_req, q_pos, ctx_lens, block_table, out, lse=None, idx=None, packed=False):
    """Host-buffer descriptor over CPU tensors (page-locked for asynchronous copies;
    kept alive by the caller until the stream has passed the call).  packed: the
    inputs, and their device buffers, lie back to back in one allocation each in
    the order q, q_idx, w, q_req, q_pos, ctx_lens, block_table (DSA_HOST_PACKED)."""
    for t in (q_idx, w, q, q_req, q_pos, ctx_lens, block_table, out, lse, idx):
        if t is not None and t.is_cuda:
            raise ValueError("dsa_host_io takes host tensors")
    return dsa_host_io(*(_ptr(t) for t in (q_idx, w, q, q_req, q_pos, ctx_lens, block_table, out, lse, idx)),
                       DSA_HOST_PACKED if packed else 0)


def dsa_layer_step_host(layout, batch, q_idx, w, q, topk, sm_scale, out, host, idx_out=None, lse=None, ws=None,
                        stream=None):
    """dsa_layer_step with the inputs copied from, and the results copied to, the
    host buffers of `host` (make_host_io) on the same stream."""
    _check(library().dsa_layer_step_host(ctypes.byref(layout), ctypes.byref(batch), _ptr(q_idx), _ptr(w), _ptr(q),
                                   int(topk), float(sm_scale), _ptr(idx_out), _ptr(out), _ptr(lse),
                                   ctypes.byref(host), _ptr(ws), ws.numel(), _stream(stream)), "dsa_layer_step_host")


def prepare_layer_step_host(layout, batch, q_idx, w, q, topk, sm_scale, out, host, idx_out=None, lse=None, ws=None,
                            stream=None):
    """dsa_layer_step_host with its arguments marshalled once: returns a function
    of no arguments that makes the call, for loops that repeat the same call.  The
    descriptors, tensors and stream passed here must outlive it."""
    fn = library().dsa_layer_step_host
    args = (ctypes.byref(layout), ctypes.byref(batch), _ptr(q_idx), _ptr(w), _ptr(q), int(topk), float(sm_scale),
            _ptr(idx_out), _ptr(out), _ptr(lse), ctypes.byref(host), _ptr(ws), ws.numel(), _stream(stream))

    def call():
        status = fn(*args)
        if status != DSA_OK:
            _check(status, "dsa_layer_step_host")

    return call


def dsa_topk_noalloc(layout, batch, scores, ld, topk, idx, phys_slots=None, stream=None):
    """dsa_topk with the library's own fixed scratch instead of a workspace."""
    lay = ctypes.byref(layout) if layout is not None else None
    _check(library().dsa_topk_noalloc(lay, ctypes.byref(batch), _ptr(scores), int(ld), int(topk), _ptr(idx),
                                      _ptr(phys_slots), _stream(stream)), "dsa_topk_noalloc")


def dsa_selftest_wait_timeout(ws, limit_cycles, stream=None):
    """Runs a bounded wait that nothing completes (the failure path); dsa_check
    then reports DSA_ERR_TIMEOUT."""
    _check(library().dsa_selftest_wait_timeout(_ptr(ws), ws.numel(), int(limit_cycles), _stream(stream)),
           "dsa_selftest_wait_timeout")


def dsa_indexer_front(layout, batch, c_q, norm_weight, eps, w_qi, head_w, q_idx, w_out, k_new=None, ws=None,
                      stream=None):
    """The fused indexer front: q_idx / w_out for the scorer (e4m3 with folded head
    weights, or MXFP4 when the batch has DSA_BATCH_QIDX_MXFP4) and, with k_new, the
    new tokens' index keys written into the pool (FP8 or MXFP4 pages)."""
    _check(library().dsa_indexer_front(ctypes.byref(layout), ctypes.byref(batch), _ptr(c_q), int(c_q.shape[1]),
                                       _ptr(norm_weight), float(eps), _ptr(w_qi), _ptr(head_w), _ptr(k_new),
                                       _ptr(q_idx), _ptr(w_out), _ptr(ws), ws.numel(), _stream(stream)),
           "dsa_indexer_front")


def dsa_write_latent(layout, batch, latent, ws=None, stream=None):
    """The new tokens' latents (bf16 [T, 576]) into their cache slots, in the pool's format."""
    _check(library().dsa_write_latent(ctypes.byref(layout), ctypes.byref(batch), _ptr(latent), _ptr(ws), ws.numel(),
                                      _stream(stream)), "dsa_write_latent")


def dsa_check(ws, stream=None):
    """Synchronise, read and clear the workspace status word; returns the status code."""
    return int(library().dsa_check(_ptr(ws), ws.numel(), _stream(stream)))
