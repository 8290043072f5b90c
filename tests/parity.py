"""Comparison of GPU results with the float64 oracle, with the tolerances of the
parity bar:

* indexer scores: |gpu - oracle| <= 1e-5 * max|oracle score| of the token (the
  e4m3 x e4m3 products are exact in fp32, so the error is that of the fp32 sum of
  128 products and of the 32-head reduction, a few 1e-7 relative);
* top-k: index sets bit-exact, except positions whose oracle score lies within
  1e-5 (relative) of the k-th oracle score; the GPU list must be ascending,
  unique, within 0..q_pos, of size min(k, q_pos + 1), then -1 padding;
* attention: relative L2 <= 2e-3 and max-abs <= 1e-2 per token against the
  oracle run on the GPU's own selection (the output is a function of the set);
  lse within 1e-3 absolute.
"""
import numpy as np

from oracle import dsa_oracle as O

SCORE_TOL = 1e-5
TIE_BAND = 1e-5
OUT_REL_L2 = 2e-3
OUT_MAX_ABS = 1e-2
LSE_ABS = 1e-3


def oracle_layout(wl):
    return O.Layout(wl.pool, wl.row_stride, wl.idx_page_offset, wl.lat_page_offset, wl.block_size,
                    wl.idx_fmt, wl.lat_fmt)


class OracleCache:
    """Oracle results of a workload, computed token by token on demand."""

    def __init__(self, wl):
        self.wl = wl
        self.lay = oracle_layout(wl)
        self._keys = {}
        self._scores = {}
        self.q_fmt = getattr(wl, "q_fmt", O.Q_FP8)
        # one entry per token in the oracle's per-token query form
        self.q_tok = (O.mxfp4_query_tokens(wl.q_idx, wl.num_tokens) if self.q_fmt == O.Q_MXFP4 else wl.q_idx)

    def keys(self, b, n):
        # one request's keys at a time (contexts of the large workloads are big)
        if b not in self._keys:
            self._keys = {b: O.gather_index_keys(self.lay, self.wl.block_table[b], int(self.wl.ctx_lens[b]))}
        return self._keys[b][:n]

    def scores(self, t):
        if t not in self._scores:
            wl = self.wl
            b, p = int(wl.q_req[t]), int(wl.q_pos[t])
            self._scores[t] = O.indexer_scores_for_token(self.keys(b, p + 1), self.q_tok[t], wl.w[t], self.q_fmt)
        return self._scores[t]

    def mla(self, t, sel):
        wl = self.wl
        lat = O.gather_latents(self.lay, wl.block_table[int(wl.q_req[t])], sel)
        return O.sparse_mla(wl.q[t], lat, wl.sm_scale)


def check_scores(oc, gpu_scores, tokens):
    worst = 0.0
    for t in tokens:
        ref = oc.scores(t)
        got = gpu_scores[t, :ref.size].astype(np.float64)
        scale = max(np.abs(ref).max(), 1e-30)
        err = np.abs(got - ref).max() / scale
        worst = max(worst, err)
        assert err <= SCORE_TOL, f"token {t}: score error {err:.3g} (relative to max |score|)"
    return worst


def check_topk(oc, gpu_idx, tokens, k):
    """Returns the number of tie-band substitutions seen."""
    subs = 0
    for t in tokens:
        sc = oc.scores(t)
        n = sc.size
        row = gpu_idx[t]
        m = min(k, n)
        assert np.all(row[m:] == -1), f"token {t}: padding"
        sel = row[:m]
        assert np.all(sel >= 0) and np.all(sel < n), f"token {t}: out of range"
        assert np.all(np.diff(sel) > 0), f"token {t}: not ascending/unique"
        ref = O.topk_select(sc, k)
        if np.array_equal(sel, ref):
            continue
        kth = O.kth_score(sc, k)
        diff = np.setxor1d(sel, ref)
        band = np.abs(sc[diff] - kth) <= TIE_BAND * abs(kth)
        assert np.all(band), f"token {t}: {np.count_nonzero(~band)} selections differ outside the tie band"
        subs += diff.size // 2
    return subs


def check_mla(oc, gpu_idx, gpu_out, gpu_lse, tokens):
    worst = (0.0, 0.0, 0.0)
    for t in tokens:
        sel = gpu_idx[t][gpu_idx[t] >= 0]
        ref_o, ref_l = oc.mla(t, sel)
        got = gpu_out[t].astype(np.float64)
        rel = np.linalg.norm(got - ref_o) / np.linalg.norm(ref_o)
        mx = np.abs(got - ref_o).max()
        le = np.abs(gpu_lse[t].astype(np.float64) - ref_l).max() if gpu_lse is not None else 0.0
        worst = tuple(max(a, b) for a, b in zip(worst, (rel, mx, le)))
        assert rel <= OUT_REL_L2, f"token {t}: rel L2 {rel:.3g}"
        assert mx <= OUT_MAX_ABS, f"token {t}: max abs {mx:.3g}"
        assert le <= LSE_ABS, f"token {t}: lse err {le:.3g}"
    return worst
