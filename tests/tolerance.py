"""Elementwise tolerances for combine results (host-side numpy, no GPU).

Combine computes out[t] = bf16( sum over t's source rows s of c_s * y_s ) with
fp32 accumulation ("DeepEP Symmetric Memory" section 9.2, combine(x, handle,
topk_weights)).  The oracle returns the exact sum o (fp64).  Two bounds on
|g - o| per element, both checked:

loose  1e-2 * sum_s |c_s * y_s|
       The stated "1e-2 relative", made robust to cancellation by scaling
       with the sum of magnitudes instead of |o|.

tight  2^-8 * |o|  +  2 * (n + m + 1) * 2^-24 * sum_s a_s * |y_s|  +  2^-133
       What fp32 accumulation followed by one bf16 rounding can produce:
       - the coefficient c_s is an fp32 sum of at most m weights, so it is
         off by at most (m - 1) * 2^-24 * a_s with a_s = sum of |w| >= |c_s|;
       - n products are accumulated with one fp32 rounding each (fused
         multiply-add), at most n * 2^-24 of the running magnitudes;
       - the bf16 output has 8 significant bits: rounding to nearest moves a
         value by at most 2^-8 of itself;
       - 2^-133, the smallest bf16 subnormal, covers results in the subnormal
         range where the relative bound does not hold.
       The factor 2 absorbs the second-order terms.  An accumulator kept in
       bf16 instead errs by about 2^-9 of every partial sum, which is far
       outside this bound wherever the terms cancel.
"""
import numpy as np

U32 = 2.0 ** -24
U_BF16 = 2.0 ** -8
BF16_MIN_SUBNORMAL = 2.0 ** -133


def bf16_bits_to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rank_sources(idx, w, E, R, dst_row, weighted, tokens=None):
    """Source rows of the rank-row combine for the listed tokens.

    Returns (rows [n, R] int64, -1 = none; c [n, R] fp64 coefficients;
    a [n, R] fp64 sums of |w|; m = most weights summed into one coefficient).
    """
    toks = np.arange(idx.shape[0]) if tokens is None else np.asarray(tokens)
    el = E // R
    ii = idx[toks]
    rows = dst_row[toks].astype(np.int64)
    n_tok, K = ii.shape
    if not weighted:
        one = (rows >= 0).astype(np.float64)
        return rows, one, one, 0
    ww = w[toks].astype(np.float64)
    c = np.zeros((n_tok, R))
    a = np.zeros((n_tok, R))
    cnt = np.zeros((n_tok, R), np.int64)
    for k in range(K):
        e = ii[:, k]
        ok = (e >= 0) & (e < E)
        t_ok = np.flatnonzero(ok)
        r_ok = e[ok] // el
        np.add.at(c, (t_ok, r_ok), ww[ok, k])
        np.add.at(a, (t_ok, r_ok), np.abs(ww[ok, k]))
        np.add.at(cnt, (t_ok, r_ok), 1)
    return rows, c, a, int(cnt.max()) if cnt.size else 0


def expanded_sources(expanded_row, w, weighted, tokens=None):
    """Source rows of the expanded combine: one per valid top-k slot, the
    coefficient being that slot's weight (no sum: m = 1)."""
    toks = np.arange(expanded_row.shape[0]) if tokens is None else np.asarray(tokens)
    rows = expanded_row[toks].astype(np.int64)
    if weighted:
        c = np.where(rows >= 0, w[toks].astype(np.float64), 0.0)
    else:
        c = (rows >= 0).astype(np.float64)
    return rows, c, np.abs(c), 1


def combine_bounds(y_bits, rows, c, a, ref, m, num_y_rows=None):
    """(loose, tight) elementwise bounds for the listed tokens (see the module
    docstring).  Rows at or beyond num_y_rows are skipped, as by combine."""
    ref = np.asarray(ref, np.float64)
    n_tok = rows.shape[0]
    H = y_bits.shape[1]
    lim = y_bits.shape[0] if num_y_rows is None else num_y_rows
    s_c = np.zeros((n_tok, H))
    s_a = np.zeros((n_tok, H))
    n = np.zeros(n_tok)
    for j in range(rows.shape[1]):
        rj = rows[:, j]
        ok = (rj >= 0) & (rj < lim)
        if not ok.any():
            continue
        yabs = np.abs(bf16_bits_to_f64(y_bits[rj[ok]]))
        s_c[ok] += np.abs(c[ok, j])[:, None] * yabs
        s_a[ok] += a[ok, j][:, None] * yabs
        n += ok
    loose = 1e-2 * s_c
    tight = U_BF16 * np.abs(ref) + 2.0 * (n[:, None] + m + 1) * U32 * s_a + BF16_MIN_SUBNORMAL
    return loose, tight


def sum_bound(ref, mag, n_parts):
    """Tight bound for bf16( fp32 sum of some parts ) against their exact sum
    ref, given the sum of the parts' magnitudes mag [n, H] and the number of
    parts per row n_parts [n] (coefficients 1: no weight sums)."""
    return U_BF16 * np.abs(ref) + 2.0 * (np.asarray(n_parts)[:, None] + 1) * U32 * mag + BF16_MIN_SUBNORMAL


def check_close(gpu_bits, ref, loose, tight):
    """Assert |g - ref| within both bounds; g given as bf16 bit patterns."""
    g = bf16_bits_to_f64(gpu_bits)
    err = np.abs(g - ref)
    bad = err > loose
    assert not bad.any(), ("1e-2 bound", np.argwhere(bad)[:5], err[bad][:5], loose[bad][:5])
    bad = err > tight
    assert not bad.any(), ("fp32-accumulation bound", np.argwhere(bad)[:5], err[bad][:5], tight[bad][:5])


def rank_combine_bounds(y_bits, idx, w, E, R, dst_row, weighted, ref, tokens=None, num_y_rows=None):
    """(loose, tight) for the rank-row combine of the listed tokens."""
    rows, c, a, m = rank_sources(idx, w, E, R, dst_row, weighted, tokens)
    return combine_bounds(y_bits, rows, c, a, ref, m, num_y_rows)
