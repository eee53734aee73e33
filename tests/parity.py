"""Acceptance rules shared by the GPU parity tests.

* top-k: index sets equal except at near-ties: an index in one set but not the other must have
  an oracle score within 1e-3 relative of the oracle's k-th score; sets have equal size, no
  duplicates, all indices in range (bit-exact when both sides rank the same fp32 scores);
* sparse MLA: per (token, head) row, max_c |gpu - ref| <= 2e-2 * max(max_c |ref|, 1e-6);
  lse within 2e-2 * max(1, |ref|); the oracle runs on the GPU's own index set;
* indexer scores: |gpu - ref| <= 2^-12 * sabs + 1e-30, sabs = the score with every term
  replaced by its absolute value (a bound on fp32 accumulation-order error of the FP8 dot
  products and the head sum);
* resolve: bit-exact rows, counters, LRU state and pool bytes.
"""
import numpy as np
import torch

MLA_RTOL = 2e-2
TOPK_TIE_RTOL = 1e-3
SCORE_RTOL = 2.0 ** -12


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_mla(out_gpu, lse_gpu, out_ref, lse_ref, H=None):
    """out_gpu: bf16 tensor [T,H,512]; out_ref float64. Returns the worst normwise error."""
    g = bf16_to_f64(out_gpu)
    if H is not None:
        g = g[:, :H]
    err = np.abs(g - out_ref).max(axis=-1)
    scale = np.maximum(np.abs(out_ref).max(axis=-1), 1e-6)
    rel = err / scale
    empty = np.isneginf(lse_ref)
    assert np.all(g[empty] == 0), "rows with no valid entry must be zero"
    worst = float(rel[~empty].max()) if (~empty).any() else 0.0
    assert worst <= MLA_RTOL, "sparse MLA max normwise error %.3e > %.1e at %s" % (
        worst, MLA_RTOL, np.unravel_index(np.argmax(np.where(empty, 0, rel)), rel.shape))
    if lse_gpu is not None:
        lg = lse_gpu.detach().cpu().numpy().astype(np.float64)
        if H is not None:
            lg = lg[:, :H]
        assert np.all(np.isneginf(lg[empty]))
        d = np.abs(lg[~empty] - lse_ref[~empty]) / np.maximum(1.0, np.abs(lse_ref[~empty]))
        assert d.size == 0 or d.max() <= MLA_RTOL, "lse error %.3e" % d.max()
    return worst


def check_topk_sets(idx_gpu: np.ndarray, ref_scores: np.ndarray, kvlen: np.ndarray, k: int, ref_idx: np.ndarray):
    """Near-tie rule of the acceptance criteria. Returns the number of differing indices."""
    ndiff = 0
    for t in range(idx_gpu.shape[0]):
        n = int(kvlen[t])
        m = min(k, n)
        g = idx_gpu[t]
        r = ref_idx[t]
        gv, rv = g[g >= 0], r[r >= 0]
        assert len(gv) == m == len(rv), (t, len(gv), m)
        assert np.all(g[m:] == -1)
        assert len(np.unique(gv)) == m and np.all((gv >= 0) & (gv < n))
        assert np.all(np.diff(gv) > 0), "output must be ascending"
        if np.array_equal(gv, rv):
            continue
        s = ref_scores[t, :n]
        kth = np.sort(s)[::-1][m - 1]
        for j in np.setxor1d(gv, rv):
            ndiff += 1
            assert abs(s[j] - kth) <= TOPK_TIE_RTOL * max(abs(kth), 1e-30), (t, j, s[j], kth)
    return ndiff


def abs_codes(codes: np.ndarray) -> np.ndarray:
    """e4m3 codes of |x|: clear the sign bit."""
    return (codes & 0x7F).astype(np.uint8)
