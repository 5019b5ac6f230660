"""Where floating point decides an E4M3 code: a code (or a block scale) that differs from the
oracle's must be explained by the oracle's value lying within the kernel's stated arithmetic
error of the rounding boundary between the two results.  Everything else must match exactly.

The fused SwiGLU kernels quantize an fp32 value that they form with the special-function
unit (2^x and 1/x approximations) and fp32 products, while the oracle forms the same value
in double precision and rounds it once to fp32.  The two fp32 values differ by a bounded
amount, so a value closer than that bound to an E4M3 rounding midpoint (or a block maximum
closer than that to a power of two, which decides the scale byte) may legitimately come out
on the other side.  The bound of each element is supplied by the caller (from the inputs);
this module only checks that every difference is explained by it.

Test infrastructure: it uses the oracle's E4M3 decoder and encoder; no kernel output feeds an
expected value."""
import numpy as np

import oracle

_CODES = np.arange(256, dtype=np.uint8)
_VALS = oracle.e4m3_decode(_CODES)                          # NaN for the two NaN codes
_FINITE = np.sort(np.unique(np.abs(_VALS[np.isfinite(_VALS)])))   # 0, 2^-9, ..., 448


def _between_has_code(a, b):
    """True where some finite |E4M3| value lies strictly between |a| and |b| (same sign)."""
    lo, hi = np.minimum(np.abs(a), np.abs(b)), np.maximum(np.abs(a), np.abs(b))
    i_lo = np.searchsorted(_FINITE, lo, side="right")
    i_hi = np.searchsorted(_FINITE, hi, side="left")
    return i_hi > i_lo


def check_blocks(v, bound, q_gpu, sf_gpu):
    """v: the oracle's values (float64 [rows, n], n % 32 == 0, blocks of 32 along axis 1);
    bound: largest |kernel value - exact value| per element (same shape);
    q_gpu: the kernel's codes [rows, n]; sf_gpu: its scale bytes [rows, n / 32].
    Returns (number of differing codes, number of differing scales); raises AssertionError with
    the first unexplained differences."""
    v = np.asarray(v, np.float64)
    bound = np.broadcast_to(np.asarray(bound, np.float64), v.shape)
    rows, n = v.shape
    nb = n // 32
    q_ref, sf_ref = oracle.quantize_rowwise_ex(v.astype(np.float32))   # v is already an fp32 value
    q_gpu = np.asarray(q_gpu, np.uint8).reshape(rows, n)
    sf_gpu = np.asarray(sf_gpu, np.uint8).reshape(rows, nb)

    # 1. scale bytes: a difference of one, with the block maximum within its bound of the power
    #    of two that separates the two scales
    vb = np.abs(v).reshape(rows, nb, 32)
    bb = bound.reshape(rows, nb, 32)
    amax = vb.max(axis=2)
    arg = vb.argmax(axis=2)
    amax_bound = np.take_along_axis(bb, arg[..., None], axis=2)[..., 0]
    dsf = sf_gpu.astype(np.int64) - sf_ref.astype(np.int64)
    bad_sf = np.nonzero(dsf != 0)
    for r, b in zip(*bad_sf):
        d = int(dsf[r, b])
        assert abs(d) == 1 and sf_ref[r, b] not in (0, 255), \
            "scale byte %d vs oracle %d at block (%d, %d)" % (sf_gpu[r, b], sf_ref[r, b], r, b)
        e_ref = int(sf_ref[r, b]) - 127 + 8                 # floor(log2 amax) of the oracle's block
        edge = 2.0 ** (e_ref + 1) if d == 1 else 2.0 ** e_ref
        assert abs(amax[r, b] - edge) <= amax_bound[r, b], \
            "scale byte %d vs oracle %d at block (%d, %d): amax %.9g is %.3g from the power of two %.9g, " \
            "bound %.3g" % (sf_gpu[r, b], sf_ref[r, b], r, b, amax[r, b], abs(amax[r, b] - edge), edge,
                            amax_bound[r, b])

    # 2. codes, each taken against the oracle's rounding of v under the kernel's block scale
    scale = np.repeat(np.exp2(sf_gpu.astype(np.float64) - 127.0), 32, axis=1)
    q_exp = q_ref.copy()
    if len(bad_sf[0]):
        blk = np.zeros((rows, nb), bool)
        blk[bad_sf] = True
        m = np.repeat(blk, 32, axis=1)
        q_exp[m] = oracle.e4m3_encode(v[m] / scale[m])
    diff = np.nonzero(q_gpu != q_exp)
    if len(diff[0]):
        y = v[diff] / scale[diff]
        yb = bound[diff] / scale[diff]
        a, g = _VALS[q_exp[diff]], _VALS[q_gpu[diff]]
        mid = 0.5 * (a + g)
        both_zero = (a == 0) & (g == 0)
        ok = np.isfinite(a) & np.isfinite(g) & ((np.sign(a) == np.sign(g)) | (a == 0) | (g == 0))
        ok &= ~_between_has_code(a, g)
        ok &= (np.abs(y - mid) <= yb) | (both_zero & (np.abs(y) <= yb))
        if not ok.all():
            i = np.nonzero(~ok)[0][:8]
            raise AssertionError("%d of %d differing codes unexplained; first: %s" % (
                int((~ok).sum()), len(ok), ", ".join(
                    "(%d,%d) v/scale=%.9g code %#x vs oracle %#x (%.6g vs %.6g), bound %.3g" % (
                        diff[0][j], diff[1][j], y[j], q_gpu[diff][j], q_exp[diff][j], g[j], a[j], yb[j])
                    for j in i)))
    return len(diff[0]), len(bad_sf[0])


def swiglu_bounds(g, u, d=None):
    """Largest |kernel - exact| of the fused SwiGLU values, per element, from the inputs (float64).

    The kernel: e = 2^(-|g| log2 e) on the special-function unit (argument rounded to fp32:
    relative error <= |g| log2(e) 2^-24 ln 2 in e; the approximation itself <= 2^-21), r = 1/(1+e)
    (1 + e rounded, reciprocal approximation <= 2^-23), sigmoid = r or e r, then fp32 products.
    So rel(sigmoid) <= (1.1 |g| + 20) 2^-24, and
      forward  h = g s u                      : rel(s) + 2^-22
      backward du = d g s                     : rel(s) + 2^-22
      backward dg = d u s (1 + g (1 - s))     : |d u s| (|t| (rel(s) + 2^-22) + |g| s rel(s) + 2^-23 (1 + |g (1-s)|))
                                                with t = 1 + g (1 - s) (cancels for g near -1.28)
    The oracle's own fp32 rounding (2^-24 relative) is added to each."""
    g = np.asarray(g, np.float64)
    u = np.asarray(u, np.float64)
    s = 1.0 / (1.0 + np.exp(-g))
    rs = (1.1 * np.abs(g) + 20.0) * 2.0 ** -24
    if d is None:
        h = g * s * u
        return np.abs(h) * (rs + 2.0 ** -22 + 2.0 ** -24)
    d = np.asarray(d, np.float64)
    du = d * g * s
    t = 1.0 + g * (1.0 - s)
    dg = d * u * s * t
    b_du = np.abs(du) * (rs + 2.0 ** -22 + 2.0 ** -24)
    b_dg = np.abs(d * u * s) * (np.abs(t) * (rs + 2.0 ** -22) + np.abs(g) * s * rs +
                                2.0 ** -23 * (1.0 + np.abs(g * (1.0 - s)))) + np.abs(dg) * 2.0 ** -24
    return b_dg, b_du
