"""The C-ABI library: it loads, exports every symbol include/dsa.h declares,
rejects invalid arguments on the host (no kernel is launched), links into a
plain C99 program, and the binding's structures have the C compiler's layout."""
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
    assert dsa.dsa_workspace_size(_layout(), _batch(flags=4), 2048) == 0
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
    # MXFP4 index pages (read by a packed 4-bit tensor copy) need 32-byte alignment of
    # the pool, the row stride and the index page; FP8 ones only 16
    mx = dict(idx_fmt=1, row_stride=4352 + 36864, lat_page_offset=4352)
    assert dsa.dsa_workspace_size(_layout(**mx), _batch(), 2048) > 0
    assert dsa.dsa_workspace_size(_layout(**dict(mx, row_stride=4352 + 36864 + 16)), _batch(), 2048) == 0
    assert dsa.dsa_workspace_size(_layout(**dict(mx, idx_page_offset=16, lat_page_offset=4368,
                                                 row_stride=4352 + 36864 + 32)), _batch(), 2048) == 0
    assert dsa.dsa_workspace_size(_layout(row_stride=45312 + 16), _batch(), 2048) > 0
    assert _call_step(_layout(pool=0x10010, **mx), _batch()) == -1
    # MXFP4 index queries: only with MXFP4 keys, and q_idx 32-byte aligned
    qmx = _batch(flags=dsa.DSA_BATCH_QIDX_MXFP4)
    assert _call_step(_layout(), qmx) == -2
    L = dsa.library()
    call = lambda q_idx: L.dsa_layer_step(ctypes.byref(_layout(**mx)), ctypes.byref(qmx), q_idx, 0x80000, 0x60000,
                                          2048, 1 / 24, None, 0x90000, None, 0x100000, 1 << 30, None)
    assert call(0x70010) == -1
    assert dsa.dsa_workspace_size(_layout(**mx), qmx, 2048) > 0
    assert dsa.dsa_workspace_size(_layout(**mx), _batch(flags=4), 2048) == 0
    L = dsa.library()
    assert L.dsa_layer_step(None, ctypes.byref(_batch()), 0, 0, 0, 2048, 1.0, None, 0, None, 0, 0, None) == -1
    assert L.dsa_topk(None, ctypes.byref(_batch()), 0x1000, 1000, 0, 0x2000, None, 0x100000, 1 << 30, None) == -1
    assert L.dsa_check(None, 0, None) == -4


def test_noalloc_topk_validation(lib):
    # the same argument checks as dsa_topk, all on the host before any launch
    f = dsa.library().dsa_topk_noalloc
    b = ctypes.byref(_batch())
    assert f(None, None, 0x1000, 1000, 2048, 0x2000, None, None) == -1           # no batch
    assert f(None, b, 0x1000, 1000, 0, 0x2000, None, None) == -1                 # topk 0
    assert f(None, b, 0x1000, 1000, 4096, 0x2000, None, None) == -1              # topk above 2048
    assert f(None, b, 0x1000, 999, 2048, 0x2000, None, None) == -1               # ld below max_ctx_len
    assert f(None, b, 0x1000, 1002, 2048, 0x2000, None, None) == -1              # ld not a multiple of 4
    assert f(None, b, 0x1008, 1000, 2048, 0x2000, None, None) == -1              # misaligned scores
    assert f(None, b, 0x1000, 1000, 2048, None, None, None) == -1                # no index output
    assert f(None, b, 0x1000, 1000, 2048, 0x2000, 0x3000, None) == -1            # slots need a layout
    assert f(ctypes.byref(_layout(block_size=48)), b, 0x1000, 1000, 2048, 0x2000, 0x3000, None) == -2
    bad = _layout()
    bad.reserved = 1
    assert f(ctypes.byref(bad), b, 0x1000, 1000, 2048, 0x2000, 0x3000, None) == -1
    assert f(ctypes.byref(_layout(idx_fmt=9)), b, 0x1000, 1000, 2048, 0x2000, 0x3000, None) == -1
    assert f(None, ctypes.byref(_batch(flags=4)), 0x1000, 1000, 2048, 0x2000, None, None) == -1
    # rows over 65,536 scores use the fixed array: 98 tokens at 1M context do not fit
    big = _batch(T=98, max_ctx=1 << 20, bt_stride=(1 << 20) // 64)
    assert f(None, ctypes.byref(big), 0x1000, 1 << 20, 2048, 0x2000, None, None) == -4


def test_front_and_latent_write_validation(lib):
    # every check runs on the host before a launch
    L = dsa.library()
    b = ctypes.byref(_batch())
    front = lambda lay, d_q=1536, eps=1e-6, ws=0x100000, ws_bytes=4096, k=0x6000: L.dsa_indexer_front(
        ctypes.byref(lay), b, 0x1000, d_q, 0x2000, eps, 0x3000, 0x4000, k, 0x7000, 0x8000, ws, ws_bytes, None)
    assert front(_layout(), d_q=7) == -1                       # not a multiple of 8
    assert front(_layout(), d_q=8192) == -1                    # wider than 4096
    assert front(_layout(), d_q=56) == -1                      # narrower than 64
    assert front(_layout(), eps=-1.0) == -1
    assert front(_layout(), eps=float("nan")) == -1
    assert front(_layout(), ws_bytes=16) == -4
    assert front(_layout(), ws=0x100010) == -4
    # MXFP4 index queries need MXFP4 index pages and a 32-byte aligned q_idx
    bq = ctypes.byref(_batch(flags=dsa.DSA_BATCH_QIDX_MXFP4))
    mx = _layout(idx_fmt=1, row_stride=4352 + 36864, lat_page_offset=4352)
    frontq = lambda lay, q_idx: L.dsa_indexer_front(ctypes.byref(lay), bq, 0x1000, 1536, 0x2000, 1e-6, 0x3000, 0x4000,
                                                    None, q_idx, 0x8000, 0x100000, 4096, None)
    assert frontq(_layout(), 0x7000) == -2
    assert frontq(mx, 0x7010) == -1
    assert L.dsa_indexer_front(ctypes.byref(_layout()), b, 0x1008, 1536, 0x2000, 1e-6, 0x3000, 0x4000, None, 0x7000,
                               0x8000, 0x100000, 4096, None) == -1   # misaligned query
    assert L.dsa_write_latent(ctypes.byref(_layout()), b, None, 0x100000, 4096, None) == -1
    assert L.dsa_write_latent(ctypes.byref(_layout()), b, 0x1000, 0x100000, 16, None) == -4
    assert L.dsa_write_latent(None, b, 0x1000, 0x100000, 4096, None) == -1


def test_selftest_validation(lib):
    f = dsa.library().dsa_selftest_wait_timeout
    assert f(None, 4096, 100000, None) == -4            # no workspace
    assert f(0x100010, 4096, 100000, None) == -4        # misaligned
    assert f(0x100000, 128, 100000, None) == -4         # no room for the status word
    assert f(0x100000, 4096, 10, None) == -1            # limit too short
    assert f(0x100000, 4096, 10 ** 10, None) == -1      # limit longer than any wait of the kernels


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


C_PROBE = r"""
#include <stddef.h>
#include <stdio.h>
#include "dsa.h"
#define F(S, m) printf(#S " " #m " %zu %zu\n", offsetof(S, m), sizeof(((S *)0)->m))
int main(void) {
  printf("dsa_kv_layout size %zu\n", sizeof(dsa_kv_layout));
  F(dsa_kv_layout, pool); F(dsa_kv_layout, num_rows); F(dsa_kv_layout, row_stride_bytes);
  F(dsa_kv_layout, idx_page_offset); F(dsa_kv_layout, lat_page_offset); F(dsa_kv_layout, block_size);
  F(dsa_kv_layout, idx_fmt); F(dsa_kv_layout, lat_fmt); F(dsa_kv_layout, reserved);
  printf("dsa_batch size %zu\n", sizeof(dsa_batch));
  F(dsa_batch, num_tokens); F(dsa_batch, num_reqs); F(dsa_batch, q_req); F(dsa_batch, q_pos);
  F(dsa_batch, ctx_lens); F(dsa_batch, block_table); F(dsa_batch, bt_stride); F(dsa_batch, flags);
  F(dsa_batch, max_ctx_len);
  printf("dsa_host_io size %zu\n", sizeof(dsa_host_io));
  F(dsa_host_io, q_idx); F(dsa_host_io, w); F(dsa_host_io, q); F(dsa_host_io, q_req); F(dsa_host_io, q_pos);
  F(dsa_host_io, ctx_lens); F(dsa_host_io, block_table); F(dsa_host_io, out); F(dsa_host_io, lse);
  F(dsa_host_io, idx); F(dsa_host_io, flags);
  /* the library is usable from plain C: version, and a workspace size with no device */
  dsa_kv_layout l = {(const void *)0x10000, 100, 45312, 0, 8448, 64, DSA_IDX_FP8, DSA_LAT_FP8, 0};
  dsa_batch b = {2, 2, (const int32_t *)0x20000, (const int32_t *)0x30000, (const int32_t *)0x40000,
                 (const int32_t *)0x50000, 16, 0, 1000};
  printf("abi %d ws %zu\n", (int)dsa_abi_version(), dsa_workspace_size(&l, &b, 2048));
  return 0;
}
"""


def test_c_program_links_and_struct_layouts_match(lib, tmp_path):
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    from dsa_sparse_attention_gb300.build import LIB
    src = tmp_path / "probe.c"
    src.write_text(C_PROBE)
    exe = tmp_path / "probe"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe),
                    LIB, "-Wl,-rpath," + os.path.dirname(LIB)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    structs = {"dsa_kv_layout": dsa.dsa_kv_layout, "dsa_batch": dsa.dsa_batch, "dsa_host_io": dsa.dsa_host_io}
    seen = set()
    for line in out:
        f = line.split()
        if f[:1] == ["abi"]:
            assert int(f[1]) == 1
            assert int(f[3]) == dsa.dsa_workspace_size(_layout(), _batch(), 2048) > 0
            seen.add("abi")
        elif len(f) == 3 and f[1] == "size":
            assert ctypes.sizeof(structs[f[0]]) == int(f[2]), line
        elif len(f) == 4:
            field = getattr(structs[f[0]], f[1])
            assert (field.offset, field.size) == (int(f[2]), int(f[3])), line
            seen.add((f[0], f[1]))
    assert "abi" in seen
    for name, st in structs.items():   # every ctypes field was compared
        assert {(name, fn) for fn, _ in st._fields_} <= seen


def test_prepared_host_step_passes_the_same_arguments(monkeypatch):
    # the prepared call marshals once and then passes exactly what the plain call
    # passes (checked against a recording stand-in for the library: no CUDA)
    import torch

    calls = []

    class Rec:
        def dsa_layer_step_host(self, *args):
            norm = []
            for a in args:
                if type(a).__name__ == "CArgObject":
                    norm.append(("byref", id(a._obj)))
                elif isinstance(a, ctypes.c_void_p):
                    norm.append(("stream", a.value))
                else:
                    norm.append(a)
            calls.append(tuple(norm))
            return 0

    monkeypatch.setattr(dsa, "library", lambda: Rec())
    stream = type("S", (), {"cuda_stream": 0x1234})()
    t = [torch.zeros(16, dtype=torch.int32) for _ in range(7)]
    lay, bat = _layout(), _batch()
    h = dsa.make_host_io(*t[:7], t[0])
    kw = dict(idx_out=t[4], lse=t[5], ws=t[6], stream=stream)
    dsa.dsa_layer_step_host(lay, bat, t[0], t[1], t[2], 2048, 1 / 24, t[3], h, **kw)
    prepared = dsa.prepare_layer_step_host(lay, bat, t[0], t[1], t[2], 2048, 1 / 24, t[3], h, **kw)
    prepared()
    prepared()
    assert len(calls) == 3 and calls[0] == calls[1] == calls[2]
    assert calls[0][-1] == ("stream", 0x1234) and calls[0][2] == t[0].data_ptr()


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    # no fallback: without the built CUDA library every call raises, none computes
    import torch
    monkeypatch.setattr(dsa, "_LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(dsa, "_LIB", None)
    with pytest.raises(ImportError):
        dsa.library()
    t = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(ImportError):
        dsa.dsa_layer_step(_layout(), _batch(), t, t, t, 2048, 1 / 24, t, ws=t)
    with pytest.raises(ImportError):
        dsa.dsa_workspace_size(_layout(), _batch(), 2048)
