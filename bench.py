"""Benchmark of the DSA decode layer step on GB300.

Workload: batch-8 decode, 65,536-token context per request, FP8 index keys and
latents in a 1 GiB packed pool with a randomly permuted block table, top-2048
(the 64K decode configuration of the benchmark definition; seeded synthetic
data).  One step = one dsa_layer_step call for the whole batch: indexer scores,
exact top-2048, sparse MLA (96 heads), split-K LSE combine.

Prints one JSON line (rank 0).  `value` is layer-steps/s over all ranks
(replicas: each rank runs its own batch; weak scaling).  Inputs larger than L2:
the timed steps rotate over 4 device copies of the 1 GiB pool, so each step
reads keys and latents (80 MB) that at least 240 MB of other traffic has
evicted from the 126 MB L2 since their last use.  (A write-based L2 flush would
leave the L2 full of dirty lines whose write-back competes with the next step's
reads; that variant is reported too, as `ms_per_step_after_l2_flush`.)  The
timed steps replay a CUDA graph of four consecutive C-ABI layer-step calls (one
per pool copy), as a multi-layer forward pass would capture them; one pair of
CUDA events brackets all K steps.  `e2e` instead runs the host-buffer C-ABI call
(dsa_layer_step_host) each step, captured once into a CUDA graph as a decode loop
with fixed buffers would: the step's inputs are copied from page-locked host
memory and the output is copied back inside the timed region, and the host waits
for each step before issuing the next (`eager_value`: the same call made eagerly).

`--impl reference` times the float64 CPU oracle on the same workload (the
reference arm: the vLLM post describing the method ships no runnable code of it).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

SCORER_PROFILE = os.path.join(ROOT, "profiles", "indexer_scorer_decode_b8_64k.md")
SCORER_SOURCES = ["indexer.cu", "ptx.cuh", "common.cuh", "params.cuh"]


def scorer_code_hash():
    """sha256 of the scorer's sources with comments and blank space removed (a
    comment edit does not change the kernel the counters were taken on)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in SCORER_SOURCES:
        with open(os.path.join(ROOT, "dsa_sparse_attention_gb300", "csrc", f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("\n".join(" ".join(line.split()) for line in text.splitlines() if line.strip()).encode())
    return h.hexdigest()


def scorer_traffic():
    """DRAM bytes per scorer launch from the committed ncu summary, if the scorer
    code is unchanged since the capture (else None)."""
    try:
        text = open(SCORER_PROFILE).read()
        want = text.split("scorer_code_sha256:")[1].split()[0]
        nbytes = int(text.split("dram_bytes_per_launch:")[1].split()[0])
    except (OSError, IndexError, ValueError):
        return None
    return nbytes if scorer_code_hash() == want else None


L2_FLUSH_BYTES = 256 << 20
N_POOL_COPIES = 4
WORKLOAD = "decode b8 x 65536 ctx, FP8 keys+latents, 1 GiB packed pool, permuted block table, top-2048"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--skip-configs", action="store_true", help="measure only the headline configuration")
    ap.add_argument("--profile-config", default=None,
                    help="run configuration N's layer step (or 'prefill_small': 1024 queries on a 32,768-token "
                         "cache; or 'front': the indexer front of the headline batch, one weight copy per call) "
                         "W + K times and print nothing (for a profiler)")
    return ap.parse_args()


def dist_info():
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    return rank, world, local


def job_rate(ms_local, world, device="cpu"):
    """Replicas: the job's step time is the slowest rank's; the job's rate is the
    steps of all ranks over it.  Returns (ms, layer-steps/s)."""
    ms = ms_local
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([ms_local], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * 1000.0 / ms


def algorithmic_bytes(wl, idx):
    """Bytes the method must move for one step: every index key of each context,
    the latents of the union of selected tokens per request, the query tensors
    and the output (intermediate scores/candidates are not counted)."""
    key_b = 132 if wl.idx_fmt == 0 else 68
    lat_b = 576 if wl.lat_fmt == 0 else 352
    total = 0
    for b in range(wl.num_reqs):
        toks = np.nonzero(wl.q_req == b)[0]
        L = int(wl.ctx_lens[b])
        sel = np.unique(idx[toks][idx[toks] >= 0]) if toks.size else np.zeros(0)
        total += L * key_b + sel.size * lat_b
    total += wl.num_tokens * (4096 + 128 + 96 * 576 * 2 + 96 * 512 * 2)
    return total


def scorer_bytes(wl):
    key_b = 132 if wl.idx_fmt == 0 else 68
    q_b = 32 * 68 if getattr(wl, "q_fmt", 0) == 1 else 4096   # MXFP4 or e4m3 index query
    return int(sum(int(L) for L in wl.ctx_lens)) * key_b + wl.num_tokens * (q_b + 128)


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        # the raw samples; DSA_BENCH_CLOCKS_DIR keeps them where the caller wants them
        out_dir = os.environ.get("DSA_BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"dsa_bench_clocks_gpu{gpu_index}_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def load_bf16_peak():
    """Dense bf16 tensor peak in TFLOP/s for a kernel timed alone (burst)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def call_rooflines(wl, idx, ms, hbm_gbs, bf16_tflops):
    """Achieved rates of the three split calls from their graph-replayed times
    (`ms`: name -> milliseconds per call) against the peaks.  Bytes are the
    algorithmic bytes of each call:
      indexer_score: every index key of each context, and each query's q_idx and w;
      topk: the scores each query ranks (q_pos + 1 of them, 4 B each, written by the
            scorer just before, so mostly read from L2) and its k output indices;
      sparse_mla: each query's selected latents, its q and its output.
    The attention's tensor work is 2 x 96 heads x (576 + 512) per selected token."""
    key_b = 132 if wl.idx_fmt == 0 else 68
    lat_b = 576 if wl.lat_fmt == 0 else 352
    T = wl.num_tokens
    n_sel = int(np.count_nonzero(idx >= 0))
    b_score = scorer_bytes(wl)
    b_topk = int(np.sum(wl.q_pos.astype(np.int64) + 1)) * 4 + T * idx.shape[1] * 4
    b_mla = n_sel * lat_b + T * (96 * 576 * 2 + 96 * 512 * 2)
    flops_mla = 2.0 * 96 * (576 + 512) * n_sel

    def rate(nbytes, t_ms):
        gbs = nbytes / (t_ms * 1e-3) / 1e9
        return {"ms": t_ms, "bytes": nbytes, "gbs": gbs, "frac_hbm": gbs / hbm_gbs}

    out = {"indexer_score": rate(b_score, ms["indexer_score"]), "topk": rate(b_topk, ms["topk"]),
           "sparse_mla": rate(b_mla, ms["sparse_mla"])}
    tf = flops_mla / (ms["sparse_mla"] * 1e-3) / 1e12
    out["sparse_mla"].update({"flops": flops_mla, "tflops": tf, "frac_bf16": tf / bf16_tflops})
    return out


def cpu_baseline(wl, budget_s=12.0):
    """The float64 oracle, as it stands, on whole steps of the same workload."""
    from oracle import dsa_oracle as O
    lay = O.Layout(wl.pool, wl.row_stride, wl.idx_page_offset, wl.lat_page_offset, wl.block_size, wl.idx_fmt,
                   wl.lat_fmt)
    steps, t0 = 0, time.perf_counter()
    while True:
        O.layer_step(lay, wl.block_table, wl.ctx_lens, wl.q_req, wl.q_pos, wl.q_idx, wl.w, wl.q, topk=wl.topk,
                     sm_scale=wl.sm_scale)
        steps += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s or steps >= 50:
            break
    threads = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS") or str(os.cpu_count())
    return {"value": steps / dt, "unit": "layer-steps/s", "cores": int(threads), "kind": "oracle",
            "sample": f"{steps} whole steps ({wl.num_tokens} queries each) in {dt:.1f} s; numpy float64, "
                      f"BLAS threads = {threads} of {os.cpu_count()} host cores"}


# The other benchmark configurations, measured beside the headline one (each on its
# own synthetic workload, seed 0; one device copy of its pool).
OTHER_CONFIGS = {
    2: "MTP decode: 32 requests x 6 query tokens (causal among them), contexts log-uniform in [16384, 262144], "
       "FP8 keys and latents, permuted block table, top-2048",
    3: "decode 1 request x 1,048,576-token context, MXFP4 index keys + NVFP4 latents, permuted block table, top-2048",
    4: "chunked prefill: 8192 new queries on a 131,072-token cache (causal), FP8 keys and latents, top-2048",
}


def fp8_peak_tflops(bf16_tflops):
    """Dense FP8 tensor peak derived from the measured bf16 one by the nominal ratio
    (4.5 : 2.25 PFLOP/s dense on GB300)."""
    return 2.0 * bf16_tflops


def scorer_flops(wl):
    """Indexer MACs as FLOPs: every scored (query, key) pair costs 32 heads x 128 dims x 2."""
    return 2.0 * 32 * 128 * float(np.sum(wl.q_pos.astype(np.int64) + 1))


def oracle_query_sample(wl, tokens):
    """Seconds the float64 oracle takes for the listed query tokens of a workload."""
    from oracle import dsa_oracle as O
    lay = O.Layout(wl.pool, wl.row_stride, wl.idx_page_offset, wl.lat_page_offset, wl.block_size, wl.idx_fmt,
                   wl.lat_fmt)
    t0 = time.perf_counter()
    O.layer_step(lay, wl.block_table, wl.ctx_lens, wl.q_req, wl.q_pos, wl.q_idx, wl.w, wl.q, topk=wl.topk,
                 sm_scale=wl.sm_scale, tokens=tokens)
    return time.perf_counter() - t0


def measure_config(n, args, stream, flush, hbm_gbs, bf16_tflops, cpu=True):
    """Layer-step time of configuration n (a CUDA graph of one dsa_layer_step, the L2
    flushed by a 256 MiB write before each timed replay; median of the steps), the
    indexer scorer's roofline (HBM for decode, FP8 tensor for prefill) and an oracle
    sample on the host."""
    import torch
    import dsa_sparse_attention_gb300 as dsa
    from dsa_sparse_attention_gb300 import workloads as W
    from dsa_sparse_attention_gb300.harness import DeviceWorkload

    wl = W.config(n, seed=0)
    dw = DeviceWorkload(wl)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            dw.layer_step(stream)
    stream.synchronize()
    assert dsa.dsa_check(dw.ws, stream) == 0

    def graph_of(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    def timed_ms(g, reps):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        with torch.cuda.stream(stream):
            for a, b in ev:
                flush.zero_()
                a.record(stream)
                g.replay()
                b.record(stream)
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ev)

    reps = max(5, min(args.steps, 50))
    step_g = graph_of(lambda: dw.layer_step(torch.cuda.current_stream()))
    step_ms = timed_ms(step_g, reps)
    scores = torch.empty(wl.num_tokens, dw.ld, dtype=torch.float32, device="cuda")
    sc_g = graph_of(lambda: dsa.dsa_indexer_score(dw.layout, dw.batch, dw.q_idx, dw.w, scores, dw.ld, dw.ws,
                                                  torch.cuda.current_stream()))
    sc_ms = timed_ms(sc_g, reps)
    idx = dw.idx.cpu().numpy()
    alg = algorithmic_bytes(wl, idx)
    sb = scorer_bytes(wl)
    out = {"workload": OTHER_CONFIGS[n], "tokens": wl.num_tokens, "requests": wl.num_reqs,
           "ms_per_step": step_ms, "layer_steps_per_s": 1000.0 / step_ms, "algorithmic_bytes_per_step": alg,
           "achieved_hbm_tbs_step": alg / (step_ms * 1e-3) / 1e12,
           "timing": f"median of {reps} graph replays of one layer step, L2 flushed (256 MiB write) before each",
           "scorer_ms": sc_ms}
    if n == 4:
        fl = scorer_flops(wl)
        tf = fl / (sc_ms * 1e-3) / 1e12
        pk = fp8_peak_tflops(bf16_tflops)
        out["roofline"] = {"bound": "tensor", "kernel": "indexer scorer (FP8 tcgen05, 8 queries share a key tile)",
                           "achieved": tf, "peak": pk, "unit": "TFLOP/s", "frac": tf / pk, "flops": fl,
                           "peak_kind": "measured bf16 burst x 2 (nominal FP8 : bf16 dense ratio)"}
    else:
        gbs = sb / (sc_ms * 1e-3) / 1e9
        out["roofline"] = {"bound": "hbm", "kernel": "indexer scorer", "achieved": gbs, "peak": hbm_gbs,
                           "unit": "GB/s", "frac": gbs / hbm_gbs, "bytes": sb,
                           "peak_kind": "measured copy bandwidth (burst)"}
    if n == 3:
        # the same 1M-token context with FP8 index keys (132 B) instead of MXFP4 (68 B)
        wf = W.make_workload([1 << 20], 1, name="decode_L1M_fp8keys", seed=0, idx_fmt=W.IDX_FP8,
                             lat_fmt=W.LAT_NVFP4, permute=True)
        df = DeviceWorkload(wf)
        sf = torch.empty(1, df.ld, dtype=torch.float32, device="cuda")
        with torch.cuda.stream(stream):
            for _ in range(3):
                dsa.dsa_indexer_score(df.layout, df.batch, df.q_idx, df.w, sf, df.ld, df.ws, stream)
        fg = graph_of(lambda: dsa.dsa_indexer_score(df.layout, df.batch, df.q_idx, df.w, sf, df.ld, df.ws,
                                                    torch.cuda.current_stream()))
        f_ms = timed_ms(fg, reps)
        out["mxfp4_vs_fp8_keys"] = {"scorer_ms_mxfp4": sc_ms, "scorer_ms_fp8": f_ms, "speedup": f_ms / sc_ms,
                                    "fp8_gbs": scorer_bytes(wf) / (f_ms * 1e-3) / 1e9}
        del df, sf, fg
        # the same MXFP4 keys scored by MXFP4 queries (DSA_BATCH_QIDX_MXFP4: E2M1 x E2M1
        # block-scaled MMA, both operands' exponents from TMEM)
        wq = W.make_workload([1 << 20], 1, name="decode_L1M_mxfp4_queries", seed=0, idx_fmt=W.IDX_MXFP4,
                             lat_fmt=W.LAT_NVFP4, permute=True, q_fmt=W.Q_MXFP4)
        dq = DeviceWorkload(wq)
        sq = torch.empty(1, dq.ld, dtype=torch.float32, device="cuda")
        with torch.cuda.stream(stream):
            for _ in range(3):
                dsa.dsa_indexer_score(dq.layout, dq.batch, dq.q_idx, dq.w, sq, dq.ld, dq.ws, stream)
        qg = graph_of(lambda: dsa.dsa_indexer_score(dq.layout, dq.batch, dq.q_idx, dq.w, sq, dq.ld, dq.ws,
                                                    torch.cuda.current_stream()))
        q_ms = timed_ms(qg, reps)
        out["mxfp4_queries"] = {"scorer_ms": q_ms, "gbs": scorer_bytes(wq) / (q_ms * 1e-3) / 1e9,
                                "how": "the 1M MXFP4 keys scored by MXFP4 index queries, L2 flushed before each"}
        del dq, sq, qg
    if cpu:
        toks = [0]
        secs = oracle_query_sample(wl, toks)
        per_step = secs * wl.num_tokens / len(toks)
        out["cpu_baseline"] = {"value": 1.0 / per_step, "unit": "layer-steps/s",
                               "cores": int(os.environ.get("OPENBLAS_NUM_THREADS") or os.cpu_count()),
                               "kind": "oracle",
                               "sample": f"{len(toks)} of {wl.num_tokens} query tokens in {secs:.2f} s, scaled to the "
                                         f"whole step (extrapolated)"}
    del dw, scores, step_g, sc_g
    torch.cuda.synchronize()
    return out


FRONT_DQ = 1536


def front_bytes(T, d_q=FRONT_DQ):
    """Bytes the indexer front must move: the projection weights once, each token's
    compressed query, its head weights in and out, its q_idx and new key."""
    return 4096 * d_q * 2 + d_q * 2 + T * (d_q * 2 + 32 * 4 * 2 + 4096 + 128 * 2 + 132)


FRONT_W_COPIES = 12   # x 12.6 MB of projection weights: more than L2 holds


def measure_front(dw, stream, graph_timed_fn, hbm_gbs):
    """Mean time of one dsa_indexer_front call (replayed from a graph of 12 calls over
    the batch of `dw`, each with its own copy of the weights, so they come from HBM
    as a model's layers would), and its rate against the HBM peak."""
    import torch
    import dsa_sparse_attention_gb300 as dsa
    T = dw.wl.num_tokens
    g = torch.Generator(device="cuda").manual_seed(0)
    c_q = torch.randn(T, FRONT_DQ, generator=g, device="cuda").to(torch.bfloat16)
    gamma = (1 + 0.1 * torch.randn(FRONT_DQ, generator=g, device="cuda")).to(torch.bfloat16)
    w_qis = [(torch.randn(4096, FRONT_DQ, generator=g, device="cuda") / FRONT_DQ ** 0.5).to(torch.bfloat16)
             for _ in range(FRONT_W_COPIES)]
    head_w = torch.randn(T, 32, generator=g, device="cuda") / 32 ** 0.5
    k_new = torch.randn(T, 128, generator=g, device="cuda").to(torch.bfloat16)
    pool = dw.pool.clone()   # the front writes the new keys: a copy of the pool
    lay = dw.pool_copy_layout(pool)
    q_idx = torch.empty(T, 32, 128, dtype=torch.uint8, device="cuda")
    w_out = torch.empty(T, 32, dtype=torch.float32, device="cuda")
    turn = [0]

    def call(_lay):   # captured FRONT_W_COPIES times in a row: each capture takes the next weight copy
        w_qi = w_qis[turn[0] % FRONT_W_COPIES]
        turn[0] += 1
        dsa.dsa_indexer_front(lay, dw.batch, c_q, gamma, 1e-6, w_qi, head_w, q_idx, w_out, k_new=k_new, ws=dw.ws,
                              stream=stream)

    ms = graph_timed_fn(call, n=FRONT_W_COPIES)
    nbytes = front_bytes(T)
    gbs = nbytes / (ms * 1e-3) / 1e9
    del pool, w_qis
    return {"ms": ms, "bytes": nbytes, "gbs": gbs, "frac_hbm": gbs / hbm_gbs, "d_q": FRONT_DQ,
            "how": f"mean over {FRONT_W_COPIES} calls replayed from one CUDA graph, each with its own copy of the "
                   "weights (more than L2 holds); weights are synthetic (seeded), the compressed query width 1,536 a "
                   "reading"}


def profile_config(args):
    """Configuration N's layer step, W + K times on one stream, nothing timed or printed:
    the command a profiler wraps to capture one configuration's kernels."""
    import torch
    import dsa_sparse_attention_gb300 as dsa
    from dsa_sparse_attention_gb300 import workloads as W
    from dsa_sparse_attention_gb300.build import build
    from dsa_sparse_attention_gb300.harness import DeviceWorkload
    build()
    if args.profile_config == "front":   # the indexer front (d_q = 1,536) on the headline batch
        wl = W.config(1, seed=0)
        dw = DeviceWorkload(wl)
        T = wl.num_tokens
        g = torch.Generator(device="cuda").manual_seed(0)
        c_q = torch.randn(T, FRONT_DQ, generator=g, device="cuda").to(torch.bfloat16)
        gamma = (1 + 0.1 * torch.randn(FRONT_DQ, generator=g, device="cuda")).to(torch.bfloat16)
        n = args.warmup + args.steps
        w_qis = [(torch.randn(4096, FRONT_DQ, generator=g, device="cuda") / FRONT_DQ ** 0.5).to(torch.bfloat16)
                 for _ in range(min(n, FRONT_W_COPIES))]
        head_w = torch.randn(T, 32, generator=g, device="cuda") / 32 ** 0.5
        k_new = torch.randn(T, 128, generator=g, device="cuda").to(torch.bfloat16)
        q_idx = torch.empty(T, 32, 128, dtype=torch.uint8, device="cuda")
        w_out = torch.empty(T, 32, dtype=torch.float32, device="cuda")
        stream = torch.cuda.Stream()
        for i in range(n):
            dsa.dsa_indexer_front(dw.layout, dw.batch, c_q, gamma, 1e-6, w_qis[i % len(w_qis)], head_w, q_idx, w_out,
                                  k_new=k_new, ws=dw.ws, stream=stream)
        stream.synchronize()
        assert dsa.dsa_check(dw.ws, stream) == 0
        return
    if args.profile_config == "prefill_small":   # the prefill scorer at a size a full profile can hold
        wl = W.make_workload([32768 + 1024], 1024, name="prefill_1024_on_32768", seed=0, permute=True)
    else:
        wl = W.config(int(args.profile_config), seed=0)
    dw = DeviceWorkload(wl)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup + args.steps):
            dw.layer_step(stream)
    stream.synchronize()
    assert dsa.dsa_check(dw.ws, stream) == 0


def run_reference(args, wl):
    _, world, _ = dist_info()
    # W untimed and K timed steps of the oracle, each a whole layer step of the
    # batch (all 8 queries), timed on the host's wall clock.
    from oracle import dsa_oracle as O
    lay = O.Layout(wl.pool, wl.row_stride, wl.idx_page_offset, wl.lat_page_offset, wl.block_size, wl.idx_fmt,
                   wl.lat_fmt)

    def step():
        O.layer_step(lay, wl.block_table, wl.ctx_lens, wl.q_req, wl.q_pos, wl.q_idx, wl.w, wl.q, topk=wl.topk,
                     sm_scale=wl.sm_scale)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    ms = 1000 * (time.perf_counter() - t0) / args.steps
    value = 1000.0 / ms
    threads = os.environ.get("OPENBLAS_NUM_THREADS") or str(os.cpu_count())
    line = {"impl": "reference", "metric": "DSA decode layer-steps/s (64K context, batch 8)", "value": value,
            "unit": "layer-steps/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": value, "unit": "layer-steps/s", "cores": int(threads), "kind": "oracle",
                             "sample": f"{args.steps} whole layer steps ({wl.num_tokens} queries each) after "
                                       f"{args.warmup} untimed ones"},
            "e2e": {"value": value, "unit": "layer-steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def check_world(args, world):
    """--gpus N must match the launch: N ranks under torchrun, or 1 without it.
    Returns an error message, or None."""
    if args.gpus < 1:
        return f"--gpus {args.gpus}: at least one GPU"
    if args.gpus != world:
        how = ("launch N ranks with python -m torch.distributed.run --nproc-per-node N bench.py --gpus N"
               if world == 1 else f"this launch has WORLD_SIZE={world}")
        return f"--gpus {args.gpus} does not match {world} rank(s): {how}"
    return None


def main():
    args = parse()
    rank, world, local = dist_info()
    err = check_world(args, world)
    if err:
        print(f"bench.py: {err}", file=sys.stderr, flush=True)
        sys.exit(2)
    from dsa_sparse_attention_gb300 import workloads as W
    if args.impl == "reference":
        if rank == 0:   # the other ranks exit without work
            run_reference(args, W.config(1, seed=0))
        return
    if args.profile_config is not None:
        profile_config(args)
        return
    wl = W.config(1, seed=0)

    import torch
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    from dsa_sparse_attention_gb300.build import build
    build()
    import dsa_sparse_attention_gb300 as dsa
    from dsa_sparse_attention_gb300.harness import DeviceWorkload, HostStep

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    dw = DeviceWorkload(wl)
    stream = torch.cuda.Stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    pools = [dw.pool] + [dw.pool.clone() for _ in range(N_POOL_COPIES - 1)]
    layouts = [dw.layout] + [dw.pool_copy_layout(pl) for pl in pools[1:]]
    torch.cuda.synchronize()   # the copies (current stream) are complete before the bench stream reads them
    with torch.cuda.stream(stream):
        for lay in layouts:
            dw.layer_step(stream, lay)  # eager warm-up (sets kernel attributes)
    stream.synchronize()
    assert dsa.dsa_check(dw.ws, stream) == 0

    graphs = []
    for lay in layouts:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            dw.layer_step(torch.cuda.current_stream(), lay)
        graphs.append(g)
    # the timed steps: consecutive layer steps in one graph, one per pool copy, as a
    # multi-layer forward pass captures them (single-step graphs finish a remainder)
    chain = torch.cuda.CUDAGraph()
    with torch.cuda.graph(chain, stream=stream):
        for lay in layouts:
            dw.layer_step(torch.cuda.current_stream(), lay)
    torch.cuda.synchronize()

    # scorer, top-k (one cluster launch for rows up to 65,536 scores, else histogram,
    # candidates, resolution and emit), attention, split combine
    n_kernels_per_step = 1 + (1 if int(wl.ctx_lens.max()) <= 65536 else 4) + 1 + 1
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            chain.replay()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    t_wall = time.perf_counter()
    n_chain, n_rest = divmod(args.steps, len(layouts))
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(n_chain):
            chain.replay()
        for s in range(n_rest):
            graphs[s].replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    ms, value = job_rate(ev0.elapsed_time(ev1) / args.steps, world, device="cuda")

    # the same K-step replay repeated until about 1 s of replays: their median
    # (and spread), beside the single measurement above; the clock record covers both
    n_rep = max(3, min(2000, int(1000.0 / max(ms * args.steps, 1e-3))))
    rep = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_rep)]
    with torch.cuda.stream(stream):
        for a, b in rep:
            a.record(stream)
            for _ in range(n_chain):
                chain.replay()
            for s in range(n_rest):
                graphs[s].replay()
            b.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    rep_ms = sorted(a.elapsed_time(b) / args.steps for a, b in rep)
    replays = {"n": n_rep, "steps_each": args.steps, "ms_per_step_median": statistics.median(rep_ms),
               "ms_per_step_min": rep_ms[0], "ms_per_step_max": rep_ms[-1]}

    # the same replay after a 256 MiB write flush of the L2 (reported for comparison)
    fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(10)]
    with torch.cuda.stream(stream):
        for i in range(10):
            flush.zero_()
            fev[i][0].record(stream)
            graphs[i % len(graphs)].replay()
            fev[i][1].record(stream)
    torch.cuda.synchronize()
    ms_flushed = statistics.mean(a.elapsed_time(b) for a, b in fev)

    # each call timed alone on the bench stream, rotating over the pool copies
    def timed(fn, reps=12):
        evp = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        with torch.cuda.stream(stream):
            for i in range(reps + 4):
                lay = layouts[i % len(layouts)]
                if i >= 4:
                    evp[i - 4][0].record(stream)
                fn(lay)
                if i >= 4:
                    evp[i - 4][1].record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in evp)

    # each call replayed from a graph of 8 launches (two rounds over the pool copies),
    # so the launch overhead of the host is not counted; per-launch average
    def graph_timed(fn, n=8, reps=10):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                fn(layouts[i % len(layouts)])
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / (n * reps)

    # dominant kernel: the indexer scorer (one launch per dsa_indexer_score for a decode batch)
    scores = torch.empty(wl.num_tokens, dw.ld, dtype=torch.float32, device="cuda")
    score_call = lambda lay: dsa.dsa_indexer_score(lay, dw.batch, dw.q_idx, dw.w, scores, dw.ld, dw.ws, stream)
    sc_ms_eager = timed(score_call)
    sc_ms = graph_timed(score_call)
    peak, peak_kind = load_peaks()
    bf16_peak, bf16_kind = load_bf16_peak()
    sc_gbs = scorer_bytes(wl) / (sc_ms * 1e-3) / 1e9

    idx_b = torch.empty_like(dw.idx)
    out_b = torch.empty_like(dw.out)
    lse_b = torch.empty_like(dw.lse)
    topk_call = lambda lay: dsa.dsa_topk(lay, dw.batch, scores, dw.ld, dw.topk, idx_b, None, dw.ws, stream)
    mla_call = lambda lay: dsa.dsa_sparse_mla(lay, dw.batch, dw.q, idx_b, dw.topk, wl.sm_scale, out_b, lse_b, dw.ws,
                                              stream)
    breakdown = {
        "graph_replayed": {"indexer_score": sc_ms, "topk": graph_timed(topk_call), "sparse_mla": graph_timed(mla_call)},
        "eager_one_call": {"indexer_score": sc_ms_eager, "topk": timed(topk_call), "sparse_mla": timed(mla_call)},
    }

    # the fused indexer front of the same batch (compressed query of 1,536 dims, seeded
    # synthetic weights): a stream of the 4096 x 1536 bf16 projection weights
    front = measure_front(dw, stream, graph_timed_fn=graph_timed, hbm_gbs=load_peaks()[0])

    # whole-step algorithmic bytes
    idx_np = dw.idx.cpu().numpy()
    alg = algorithmic_bytes(wl, idx_np)
    step_tbs = alg / (ms / world * 1e-3) / 1e12 if world == 1 else alg / (ms * 1e-3) / 1e12

    # end to end through the C ABI with host buffers (dsa_layer_step_host): every step
    # copies its inputs from page-locked host memory (packed back to back, so one
    # copy), runs, and copies its output back; the host waits for each step, as a
    # decode loop whose next input depends on this output does.  The call is
    # captured once per pool copy into a CUDA graph, as a decode loop with fixed
    # buffers captures it, and each step replays one (the copies run on every
    # replay); the same call made eagerly is reported beside it.
    def e2e_host_call():
        hs = HostStep(dw, packed=True, with_lse=False, with_idx=False)
        for i in range(4):
            hs.step(stream, layouts[i % len(layouts)])
        torch.cuda.synchronize()

        def wall(step_fn):
            for i in range(4):
                step_fn(i)
                stream.synchronize()
            ms_list = []
            for i in range(args.steps):
                t0 = time.perf_counter()
                step_fn(i)
                stream.synchronize()
                ms_list.append((time.perf_counter() - t0) * 1000)
            return ms_list

        eager_ms = wall(lambda i: hs.step(stream, layouts[i % len(layouts)]))
        hgraphs = []
        for lay in layouts:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                hs.step(torch.cuda.current_stream(), lay)
            hgraphs.append(g)
        with torch.cuda.stream(stream):
            graph_ms = wall(lambda i: hgraphs[i % len(hgraphs)].replay())
        return graph_ms, eager_ms, hs.h2d_bytes, hs.d2h_bytes, (
            "dsa_layer_step_host captured into a CUDA graph (one per pool copy), one replay per step: inputs "
            "copied from one page-locked buffer, output copied back, host waits for each step")

    e2e_ms, e2e_eager_ms, h2d, d2h, e2e_how = e2e_host_call()
    _, e2e_value = job_rate(statistics.mean(e2e_ms), world, device="cuda")   # slowest rank, like `value`
    _, e2e_eager = job_rate(statistics.mean(e2e_eager_ms), world, device="cuda")
    assert dsa.dsa_check(dw.ws, stream) == 0

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl)

    # the other configurations, after the headline one's buffers are released
    others = {}
    if not args.skip_configs:
        del graphs, chain, pools, layouts
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        peak_gbs, _ = load_peaks()
        bf16_pk, _ = load_bf16_peak()
        for n in sorted(OTHER_CONFIGS):
            others[f"cfg{n}"] = measure_config(n, args, stream, flush, peak_gbs, bf16_pk,
                                               cpu=rank == 0 and not args.no_cpu_baseline)

    if rank == 0:
        line = {
            "metric": "DSA decode layer-steps/s (64K context, batch 8)", "value": value, "unit": "layer-steps/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp8/bf16/fp16 (fp32 acc)",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "batch": wl.num_reqs, "ctx_len": int(wl.ctx_lens[0]), "topk": wl.topk,
                       "l2": f"inputs larger than L2: steps rotate over {N_POOL_COPIES} device copies of the pool",
                       "graph": f"CUDA graphs of {N_POOL_COPIES} consecutive layer steps (one per pool copy)",
                       "parallelism": f"replicas x{world}"},
            "replays": replays,
            "ms_per_step_after_l2_flush": ms_flushed,
            "achieved_hbm_tbs_step": step_tbs,
            "achieved_frac_of_8tbs": step_tbs / 8.0,
            "algorithmic_bytes_per_step": alg,
            "roofline": {"bound": "hbm", "kernel": "indexer scorer (indexer_kernel, one launch per dsa_indexer_score)",
                         "achieved": sc_gbs, "peak": peak, "unit": "GB/s", "frac": sc_gbs / peak,
                         "peak_kind": f"{peak_kind} copy bandwidth (burst)",
                         "traffic": scorer_traffic(), "launch_ms": sc_ms,
                         "launch_ms_how": "mean over 8 scorer calls replayed from one CUDA graph (pool copies rotated)",
                         "launch_ms_eager": sc_ms_eager},
            "e2e": {"value": e2e_value, "unit": "layer-steps/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "how": e2e_how, "eager_value": e2e_eager,
                    "eager_how": "the same call made eagerly each step (the launches' host latency included)"},
            "gpu_launches": n_kernels_per_step * args.steps,
            "breakdown_ms": breakdown,
            "indexer_front": front,
            "call_rooflines": dict(call_rooflines(wl, idx_np, breakdown["graph_replayed"], peak, bf16_peak),
                                   peaks=f"HBM {peak:.0f} GB/s ({peak_kind}), bf16 {bf16_peak:.0f} TFLOP/s "
                                         f"({bf16_kind}, burst)"),
            "clocks": clk, "wall_s_timed": t_wall,
            "cpu_baseline": cpu,
            "other_configs": others,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
