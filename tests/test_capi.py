"""The C-ABI library: it loads, exports every symbol include/dsa.h declares,
and rejects invalid arguments on the host (no kernel is launched)."""
import ctypes
import os
import re

import pytest

import dsa_sparse_attention_gb300 as dsa
from dsa_sparse_attention_gb300.build import build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "dsa.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return dsa.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"dsa_layer_step", "dsa_indexer_score", "dsa_topk", "dsa_sparse_mla"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert dsa.dsa_abi_version() == 1
    assert dsa.dsa_status_string(-6) == "DSA_ERR_DEVICE_CHECK"
    assert dsa.dsa_last_cuda_error() == (0, "no error")


def _layout(**kw):
    args = dict(pool=0x10000, num_rows=100, row_stride=45312, idx_page_offset=0, lat_page_offset=8448)
    args.update(kw)
    return dsa.make_layout(args.pop("pool"), **args)


def _batch(T=2, B=2, max_ctx=1000, bt_stride=16, flags=0):
    b = dsa.dsa_batch(T, B, 0x20000, 0x30000, 0x40000, 0x50000, bt_stride, flags, max_ctx)
    return b


def test_workspace_size_and_validation(lib):
    n = dsa.dsa_workspace_size(_layout(), _batch(), 2048)
    assert n > 0 and n % 256 == 0
    assert dsa.dsa_workspace_size(_layout(), _batch(), 0) == 0
    assert dsa.dsa_workspace_size(_layout(), _batch(), 4096) == 0
    assert dsa.dsa_workspace_size(_layout(block_size=48), _batch(), 2048) == 0
    assert dsa.dsa_workspace_size(_layout(row_stride=45300), _batch(), 2048) == 0
    assert dsa.dsa_workspace_size(_layout(), _batch(max_ctx=16 * 64 + 1), 2048) == 0
    assert dsa.dsa_workspace_size(_layout(), _batch(flags=2), 2048) == 0
    inv = dsa.dsa_workspace_size(_layout(), _batch(T=64, flags=dsa.DSA_BATCH_INVARIANT), 2048)
    dflt = dsa.dsa_workspace_size(_layout(), _batch(T=64), 2048)
    assert inv > dflt


def _call_step(lay, bat, ws_ptr=0x100000, ws_bytes=1 << 30, q=0x60000):
    L = dsa.library()
    return L.dsa_layer_step(ctypes.byref(lay), ctypes.byref(bat), 0x70000, 0x80000, q, 2048, 1 / 24, None,
                            0x90000, None, ws_ptr, ws_bytes, None)


def test_host_validation_errors(lib):
    assert _call_step(_layout(), _batch(), ws_bytes=16) == -4          # workspace too small
    assert _call_step(_layout(), _batch(), ws_ptr=0x100010) == -4      # misaligned workspace
    assert _call_step(_layout(pool=0x10008), _batch()) == -1           # misaligned pool
    assert _call_step(_layout(), _batch(), q=0x60008) == -1            # misaligned q
    assert _call_step(_layout(idx_fmt=7), _batch()) == -1
    assert _call_step(_layout(block_size=512), _batch()) == -2
    L = dsa.library()
    assert L.dsa_layer_step(None, ctypes.byref(_batch()), 0, 0, 0, 2048, 1.0, None, 0, None, 0, 0, None) == -1
    assert L.dsa_topk(None, ctypes.byref(_batch()), 0x1000, 1000, 0, 0x2000, None, 0x100000, 1 << 30, None) == -1
    assert L.dsa_check(None, 0, None) == -4


def _call_step_host(host, lse=None, idx=None):
    L = dsa.library()
    return L.dsa_layer_step_host(ctypes.byref(_layout()), ctypes.byref(_batch()), 0x70000, 0x80000, 0x60000, 2048,
                                 1 / 24, idx, 0x90000, lse, host, 0x100000, 1 << 30, None)


def test_host_step_validation_errors(lib):
    full = dict(q_idx=0x1000, w=0x2000, q=0x3000, q_req=0x4000, q_pos=0x5000, ctx_lens=0x6000, block_table=0x7000,
                out=0x8000)
    assert _call_step_host(None) == -1                                          # no host descriptor
    for missing in full:                                                        # each required host pointer
        h = dsa.dsa_host_io(**{k: (0 if k == missing else v) for k, v in full.items()})
        assert _call_step_host(ctypes.byref(h)) == -1, missing
    h = dsa.dsa_host_io(**full, lse=0x9000)
    assert _call_step_host(ctypes.byref(h)) == -1                               # host lse without device lse
    h = dsa.dsa_host_io(**full, idx=0xa000)
    assert _call_step_host(ctypes.byref(h)) == -1                               # host idx without idx_out
    h = dsa.dsa_host_io(**full, flags=2)
    assert _call_step_host(ctypes.byref(h)) == -1                               # unknown flag
    h = dsa.dsa_host_io(**full, flags=dsa.DSA_HOST_PACKED)
    assert _call_step_host(ctypes.byref(h)) == -1                               # packed, but not back to back
    L = dsa.library()
    h = dsa.dsa_host_io(**full)
    assert L.dsa_layer_step_host(ctypes.byref(_layout()), ctypes.byref(_batch()), 0x70000, 0x80000, 0x60000, 2048,
                                 1 / 24, None, 0x90000, None, ctypes.byref(h), 0x100000, 16, None) == -4
    import torch
    ts = [torch.zeros(4, dtype=torch.int32) for _ in range(8)]
    h = dsa.make_host_io(*ts)
    assert [h.q_idx, h.w, h.q, h.q_req, h.q_pos, h.ctx_lens, h.block_table, h.out] == [t.data_ptr() for t in ts]
    assert h.lse is None and h.idx is None and h.flags == 0
    assert dsa.make_host_io(*ts, packed=True).flags == dsa.DSA_HOST_PACKED
