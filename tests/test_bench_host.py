"""The benchmark's host-side logic, on the CPU: the algorithmic byte model behind
`achieved` and `achieved_hbm_tbs_step`, the lookup of the scorer's captured DRAM
traffic (keyed on the scorer's code), the clock record that decides whether a
run is kept, and the reference arm (the oracle timed on the host cores: its JSON
line, and no work on ranks other than 0)."""
import os
import shutil
import types

import numpy as np

import bench

KEY_FP8, KEY_MXFP4, LAT_FP8, LAT_NVFP4 = 132, 68, 576, 352
Q_AND_OUT = 4096 + 128 + 96 * 576 * 2 + 96 * 512 * 2   # q_idx, w, q, out per query token


def _wl(ctx, q_req, idx_fmt=0, lat_fmt=0):
    return types.SimpleNamespace(idx_fmt=idx_fmt, lat_fmt=lat_fmt, num_reqs=len(ctx),
                                 ctx_lens=np.asarray(ctx, np.int32), q_req=np.asarray(q_req, np.int32),
                                 num_tokens=len(q_req))


def test_decode_b8_64k_step_bytes():
    # one query per request, 2048 distinct selections each: L*132 + 2048*576 per
    # query plus its q/out tensors (80.35 MB for the batch)
    wl = _wl([65536] * 8, list(range(8)))
    rng = np.random.default_rng(0)
    idx = np.stack([np.sort(rng.choice(65536, 2048, replace=False)) for _ in range(8)]).astype(np.int32)
    per_query = 65536 * KEY_FP8 + 2048 * LAT_FP8 + Q_AND_OUT
    assert bench.algorithmic_bytes(wl, idx) == 8 * per_query == 80_348_160
    assert bench.scorer_bytes(wl) == 8 * (65536 * KEY_FP8 + 4096 + 128) == 69_239_808


def test_latents_counted_once_per_request_and_padding_skipped():
    # two queries of request 0 share three selections; request 1 has a short
    # context padded with -1; keys are read once per request
    wl = _wl([100, 3], [0, 0, 1])
    idx = np.array([[1, 2, 3, 4], [3, 4, 5, 6], [0, 1, 2, -1]], np.int32)
    want = (100 + 3) * KEY_FP8 + (6 + 3) * LAT_FP8 + 3 * Q_AND_OUT
    assert bench.algorithmic_bytes(wl, idx) == want


def test_fp4_widths():
    wl = _wl([1000], [0], idx_fmt=1, lat_fmt=1)
    idx = np.arange(8, dtype=np.int32)[None]
    assert bench.algorithmic_bytes(wl, idx) == 1000 * KEY_MXFP4 + 8 * LAT_NVFP4 + Q_AND_OUT
    assert bench.scorer_bytes(wl) == 1000 * KEY_MXFP4 + 4096 + 128
    wq = _wl([1000], [0], idx_fmt=1, lat_fmt=1)
    wq.q_fmt = 1                                                  # MXFP4 index queries: 68 B per head
    assert bench.scorer_bytes(wq) == 1000 * KEY_MXFP4 + 32 * 68 + 128


def _copy_sources(tmp_path):
    src = os.path.join(bench.ROOT, "dsa_sparse_attention_gb300", "csrc")
    dst = tmp_path / "dsa_sparse_attention_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in bench.SCORER_SOURCES:
        shutil.copy(os.path.join(src, f), dst / f)
    return dst


def test_scorer_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    base = bench.scorer_code_hash()
    dst = _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.scorer_code_hash() == base
    f = dst / "indexer.cu"
    f.write_text("// a new comment line\n/* and a block\n   comment */\n" + f.read_text() + "\n\n   \n")
    assert bench.scorer_code_hash() == base
    f.write_text(f.read_text() + "\nstatic int unused_symbol_for_the_test;\n")
    assert bench.scorer_code_hash() != base


def test_scorer_traffic_only_for_the_captured_code(tmp_path, monkeypatch):
    prof = tmp_path / "scorer.md"
    prof.write_text(f"scorer_code_sha256: {bench.scorer_code_hash()}\ndram_bytes_per_launch: 123456\n")
    monkeypatch.setattr(bench, "SCORER_PROFILE", str(prof))
    assert bench.scorer_traffic() == 123456
    prof.write_text("scorer_code_sha256: " + "0" * 64 + "\ndram_bytes_per_launch: 123456\n")
    assert bench.scorer_traffic() is None
    monkeypatch.setattr(bench, "SCORER_PROFILE", str(tmp_path / "missing.md"))
    assert bench.scorer_traffic() is None


class _DoneProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _clock_record(tmp_path, lines):
    path = tmp_path / "clocks.csv"
    path.write_text("\n".join(lines) + "\n")
    cs = bench.ClockSampler(0)
    cs.path, cs.proc, cs.f = str(path), _DoneProc(), open(path, "a")
    return cs.stop()


def test_clock_record_median_max_and_reasons(tmp_path):
    idle = "Not Active"
    rec = _clock_record(tmp_path, [
        f"0, 2070, 2070, 900.1, 0x0, {idle}, {idle}, {idle}, {idle}",
        f"0, 1980, 2070, 1390.0, 0x4, {idle}, {idle}, {idle}, Active",
        f"0, 2055, 2070, 1100.0, 0x0, {idle}, {idle}, {idle}, {idle}",
        "0, [N/A], 2070, 0, 0x0, a, b, c, d",      # unreadable sample: skipped
        "garbage",
    ])
    assert rec == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "samples": 3, "reasons": ["sw_power_cap"]}
    rec = _clock_record(tmp_path, [f"0, 1500, 2070, 1000, 0x8, {idle}, Active, {idle}, {idle}"])
    assert rec["reasons"] == ["hw_thermal_slowdown"]
    assert _clock_record(tmp_path, ["nothing here"]) is None


def _run_bench(extra_env, *args, expect_rc=0, wall=None):
    import json
    import subprocess
    import sys
    import time
    env = dict(os.environ, **extra_env)
    t0 = time.perf_counter()
    r = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), *args], capture_output=True, text=True,
                       env=env, timeout=600)
    if wall is not None:
        wall.append(time.perf_counter() - t0)
    assert r.returncode == expect_rc, r.stderr[-2000:]
    if expect_rc:
        return r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    return [json.loads(ln) for ln in lines]


def test_reference_arm_line():
    # the oracle timed as the reference arm: one JSON line with the contract's keys;
    # each timed step is a whole layer step, so K steps fit inside the run's wall time
    wall = []
    (line,) = _run_bench({}, "--impl", "reference", "--steps", "2", "--warmup", "0", wall=wall)
    assert line["ms_per_step"] * line["steps"] / 1000.0 < wall[0]
    assert line["impl"] == "reference" and line["unit"] == "layer-steps/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["steps"] == 2 and line["warmup"] == 0 and line["n_gpus"] == 1
    assert abs(line["value"] * line["ms_per_step"] - 1000.0) < 1e-6
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "layer-steps/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["metric"].startswith("DSA decode layer-steps/s") and line["config"]["workload"] == bench.WORKLOAD


def test_reference_arm_other_ranks_exit_without_work():
    assert _run_bench({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, "--impl", "reference", "--gpus",
                      "2") == []


def test_gpus_must_match_the_launch():
    # --gpus N runs N replicas only when launched as N ranks; anything else is refused
    args = lambda n: types.SimpleNamespace(gpus=n)
    assert bench.check_world(args(1), 1) is None and bench.check_world(args(4), 4) is None
    assert "torch.distributed.run" in bench.check_world(args(8), 1)
    assert "WORLD_SIZE=2" in bench.check_world(args(4), 2)
    assert bench.check_world(args(0), 1) is not None
    err = _run_bench({"WORLD_SIZE": "1"}, "--gpus", "2", "--impl", "reference", expect_rc=2)
    assert "--gpus 2 does not match 1 rank" in err


def test_call_rooflines_decode_b8_64k():
    # 8 queries at position 65,535, 2048 selections each; times of 1e-2 ms per call
    wl = _wl([65536] * 8, list(range(8)))
    wl.q_pos = np.full(8, 65535, np.int32)
    idx = np.tile(np.arange(2048, dtype=np.int32), (8, 1))
    r = bench.call_rooflines(wl, idx, {"indexer_score": 0.01, "topk": 0.01, "sparse_mla": 0.01}, 1000.0, 2000.0)
    assert r["indexer_score"]["bytes"] == 69_239_808
    assert r["topk"]["bytes"] == 8 * 65536 * 4 + 8 * 2048 * 4
    assert r["sparse_mla"]["bytes"] == 8 * 2048 * LAT_FP8 + 8 * (96 * 576 * 2 + 96 * 512 * 2)
    assert r["sparse_mla"]["flops"] == 2 * 96 * (576 + 512) * 8 * 2048          # 3.42 GFLOP
    assert abs(r["sparse_mla"]["gbs"] - r["sparse_mla"]["bytes"] / 1e-5 / 1e9) < 1e-6
    assert abs(r["sparse_mla"]["frac_hbm"] - r["sparse_mla"]["gbs"] / 1000.0) < 1e-12
    assert abs(r["sparse_mla"]["tflops"] - r["sparse_mla"]["flops"] / 1e-5 / 1e12) < 1e-9
    assert abs(r["sparse_mla"]["frac_bf16"] - r["sparse_mla"]["tflops"] / 2000.0) < 1e-12
    # padding (-1) is not attended: half the selections give half the latent bytes and flops
    idx[:, 1024:] = -1
    r2 = bench.call_rooflines(wl, idx, {"indexer_score": 0.01, "topk": 0.01, "sparse_mla": 0.01}, 1000.0, 2000.0)
    assert r2["sparse_mla"]["flops"] * 2 == r["sparse_mla"]["flops"]
    assert r["sparse_mla"]["bytes"] - r2["sparse_mla"]["bytes"] == 8 * 1024 * LAT_FP8


def test_prefill_scorer_flops_and_fp8_peak():
    # every scored (query, key) pair costs 32 heads x 128 dims x 2 FLOP: for 8192
    # queries at positions 131,072 + i that is 8192 x sum_i (131,073 + i) x 8192 = 9.07 TFLOP
    wl = types.SimpleNamespace(q_pos=np.arange(131072, 131072 + 8192, dtype=np.int32))
    want = 2.0 * 32 * 128 * (8192 * 131073 + 8191 * 8192 // 2)
    assert bench.scorer_flops(wl) == want and abs(want - 9.07e12) < 0.01e12
    assert bench.fp8_peak_tflops(1914.3) == 2 * 1914.3
    assert set(bench.OTHER_CONFIGS) == {2, 3, 4}


def test_front_bytes():
    # 4096 x 1536 bf16 weights, gamma, and per token: query, head weights in and out,
    # q_idx codes, the new key in (bf16) and out (132 B)
    assert bench.front_bytes(8) == 4096 * 1536 * 2 + 1536 * 2 + 8 * (1536 * 2 + 256 + 4096 + 256 + 132)
