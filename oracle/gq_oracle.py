"""Plain, slow, float64 oracle of the group-quantized weight-only GEMM.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never imports it.

Sources (the pages this follows):
  * P1 = "GPU Kernel 工程（09）：量化与融合 kernel" (arganzheng.life,
    quantization-and-fused-kernels).
  * P2 = "04 · 分组量化 GEMM 内核" (developer.aliyun.com article 1770277).

What it computes (P2 section 2, the block-wise dot then scale; P1 section 2.1, x ≈ s·(q − z);
P1 section 8 rule 2, compare against the dequantized weights, not the unquantized ones):

    out[m][n] = Σ_g s[g][n] · Σ_{k ∈ group g} A[m][k] · (q[k][n] − z[g][n])

with activation scale 1 (float activations).  The per-group integer-weighted dot is
finished before the scale is applied, exactly as the formula states.  The variants the
library also computes have their own functions here: float zero points subtracted after
scaling (``group_gemm_zf``, P1 section 3.4), the fused SiLU-and-mul epilogue
(``silu_mul_reference``, P1 section 5.2), int8 activations with per-group scales
(``quantize_act_i8``, ``group_gemm_a8``; P2 section 2, P1 section 4.5) and the FP8
block-scaled GEMM with its activation quantizer (``quantize_act_fp8``, ``fp8_block_gemm``;
P1 section 4.3).  All arithmetic is
float64; products of a bf16/fp32 activation and a small integer are exact in float64 and
sums of at most a few thousand such terms lose at most a few ulps of float64, far below
every tolerance used against the GPU.
"""
from __future__ import annotations

import math
import numpy as np

__all__ = [
    "fp16_bits_to_f64", "bf16_bits_to_f64", "f32_to_f64", "f64_to_bf16_bits",
    "f64_to_f32", "unpack_int4_k", "unpack_int4_n", "dequantize", "group_gemm",
    "group_gemm_magnitude", "reference", "tolerance", "check", "quantize_w4_g",
    "bits_per_weight", "dequantize_brute", "silu", "silu_mul_reference",
    "quantize_act_i8", "group_gemm_a8", "reference_a8", "e4m3_bits_to_f64",
    "fp8_block_gemm", "f64_to_e4m3_bits", "quantize_act_fp8", "group_gemm_zf",
]


# ---------------------------------------------------------------------------------------
# IEEE-754 binary16 / bfloat16 / binary32 codecs, written from the format definitions.
# (P1 section 2.1 lists the layouts: FP16 = 1 sign, 5 exponent, 10 mantissa bits;
#  BF16 = the high 16 bits of an FP32: 1 sign, 8 exponent, 7 mantissa bits.)
# ---------------------------------------------------------------------------------------

def _decode_ieee(bits: np.ndarray, exp_bits: int, man_bits: int) -> np.ndarray:
    b = np.asarray(bits).astype(np.int64) & ((1 << (1 + exp_bits + man_bits)) - 1)
    sign = np.where((b >> (exp_bits + man_bits)) & 1, -1.0, 1.0)
    e = (b >> man_bits) & ((1 << exp_bits) - 1)
    f = (b & ((1 << man_bits) - 1)).astype(np.float64)
    bias = (1 << (exp_bits - 1)) - 1
    emax = (1 << exp_bits) - 1
    frac = f / float(1 << man_bits)
    normal = np.ldexp(1.0 + frac, (e - bias).astype(np.int64))
    subnormal = np.ldexp(frac, 1 - bias)
    val = np.where(e == 0, subnormal, normal)
    val = np.where(e == emax, np.where(f == 0, np.inf, np.nan), val)
    return sign * val


def fp16_bits_to_f64(bits) -> np.ndarray:
    """binary16 bit patterns -> float64 (exact), including subnormals, inf and NaN."""
    return _decode_ieee(bits, 5, 10)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bfloat16 bit patterns -> float64 (exact)."""
    return _decode_ieee(bits, 8, 7)


def f32_to_f64(x) -> np.ndarray:
    """binary32 values -> float64 (exact widening)."""
    return np.asarray(x, dtype=np.float32).astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """float64 -> bfloat16 bits, round to nearest even (P1 section 2.3: FP32 -> BF16 is
    RNE), computed directly from float64 (no intermediate fp32 rounding).  Finite inputs
    beyond the bf16 range round to inf like the hardware conversion."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.uint16)
    sign = (np.signbit(x)).astype(np.uint16) << 15
    ax = np.abs(x)
    nan = np.isnan(x)
    with np.errstate(all="ignore"):
        m, e = np.frexp(ax)          # ax = m * 2^e, m in [0.5, 1)
        # a normal bf16 has 8 significant bits: value = integer(2^7..2^8-1) * 2^(E-7)
        # exponent of the leading bit: E = e - 1; subnormals fix E at -126
        E = np.maximum(e - 1, -126)
        scaled = np.ldexp(ax, (7 - E).astype(np.int64))   # integer part holds the significand
        r = np.rint(scaled)                                # round half to even
        # renormalize when rounding carried into a new binade
        carry = r >= 256
        r = np.where(carry, r / 2, r)
        E = np.where(carry, E + 1, E)
        is_sub = r < 128
        expfield = np.where(is_sub, 0, E + 127).astype(np.int64)
        manfield = np.where(is_sub, r, r - 128).astype(np.int64)
        bits = (expfield << 7) | manfield
        bits = np.where(ax == 0, 0, bits)
        bits = np.where((expfield >= 255) | np.isinf(ax), 0x7F80, bits)
    out = (bits.astype(np.uint16) | sign)
    out = np.where(nan, np.uint16(0x7FC0), out).astype(np.uint16)
    return out


def f64_to_f32(x) -> np.ndarray:
    """float64 -> float32 with round to nearest even (numpy's conversion)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)


# ---------------------------------------------------------------------------------------
# Canonical INT4 layouts (P1 section 2.4: eight INT4 values per uint32, element j at
# bits 4j..4j+3; P1 section 3.1: scales [K/g, N], zero points INT4-packed [K/g, N/8];
# P1 section 9.4 packs eight consecutive k into one word).
# ---------------------------------------------------------------------------------------

def unpack_int4_k(words: np.ndarray) -> np.ndarray:
    """uint32 [K/8][N] -> codes int64 [K][N]; k = 8r + j is read from bits 4j..4j+3."""
    w = np.asarray(words, dtype=np.uint32)
    R, N = w.shape
    q = np.empty((R, 8, N), dtype=np.int64)
    for j in range(8):
        q[:, j, :] = (w >> np.uint32(4 * j)) & np.uint32(0xF)
    return q.reshape(R * 8, N)


def unpack_int4_n(words: np.ndarray) -> np.ndarray:
    """uint32 [R][N/8] -> codes int64 [R][N]; n = 8c + j is read from bits 4j..4j+3."""
    w = np.asarray(words, dtype=np.uint32)
    R, C = w.shape
    z = np.empty((R, C, 8), dtype=np.int64)
    for j in range(8):
        z[:, :, j] = (w >> np.uint32(4 * j)) & np.uint32(0xF)
    return z.reshape(R, C * 8)


# ---------------------------------------------------------------------------------------
# The method.
# ---------------------------------------------------------------------------------------

def dequantize(q: np.ndarray, z: np.ndarray, s: np.ndarray, G: int) -> np.ndarray:
    """W_hat[k][n] = s[g][n] * (q[k][n] - z[g][n]), g = k // G   (P1 section 2.1, the
    affine relation x ≈ s·(q − z); P1 section 9.4 builds W_hat = s·(q − 8) as the
    reference weights)."""
    K, N = q.shape
    qz = q.astype(np.float64).reshape(K // G, G, N) - np.asarray(z, np.float64)[:, None, :]
    return (qz * np.asarray(s, np.float64)[:, None, :]).reshape(K, N)


def group_gemm(A: np.ndarray, q: np.ndarray, z: np.ndarray, s: np.ndarray, G: int) -> np.ndarray:
    """out[m][n] = Σ_g s[g][n] · Σ_{k∈g} A[m][k]·(q[k][n] − z[g][n])   (P2 section 2: the
    integer-weighted dot of a whole group finishes before its scale multiplies it).

    A [M][K] float64, q [K][N] integer codes, z [K/G][N] integer zero points,
    s [K/G][N] float64 scales.  The inner dot is a library matmul over one group.
    """
    A = np.asarray(A, np.float64)
    M, K = A.shape
    N = q.shape[1]
    assert K % G == 0 and q.shape[0] == K
    out = np.zeros((M, N), dtype=np.float64)
    for g in range(K // G):
        ks = slice(g * G, (g + 1) * G)
        d = q[ks, :].astype(np.float64) - np.asarray(z[g], np.float64)[None, :]
        partial = A[:, ks] @ d
        out += np.asarray(s[g], np.float64)[None, :] * partial
    return out


def group_gemm_magnitude(A, q, z, s, G) -> np.ndarray:
    """mag[m][n] = Σ_k |A[m][k] · w[k][n]| with w = s·(q − z): the conditioning term of
    the tolerance (the size of the terms the sum cancels)."""
    A = np.abs(np.asarray(A, np.float64))
    M, K = A.shape
    N = q.shape[1]
    out = np.zeros((M, N), dtype=np.float64)
    for g in range(K // G):
        ks = slice(g * G, (g + 1) * G)
        d = np.abs(q[ks, :].astype(np.float64) - np.asarray(z[g], np.float64)[None, :])
        out += np.abs(np.asarray(s[g], np.float64))[None, :] * (A[:, ks] @ d)
    return out


def group_gemm_zf(A: np.ndarray, q: np.ndarray, zf: np.ndarray, s: np.ndarray, G: int):
    """Float zero points: out = A @ W_hat with W_hat[k][n] = q[k][n] · s[g][n] − zf[g][n],
    g = k // G (P1 section 3.4: Machete's out = (w_q · w_s − w_z) @ a, the zero point a float
    in the scale type, subtracted after scaling rather than from the code).  Returns
    (out, mag) with mag[m][n] = Σ_k |A[m][k] · W_hat[k][n]|.

    A [M][K] float64, q [K][N] integer codes, zf and s [K/G][N] float64.  The dequantized
    weights are formed first, as the formula is written, then one library matmul.
    """
    A = np.asarray(A, np.float64)
    K, N = q.shape
    assert K % G == 0 and A.shape[1] == K
    W = (q.astype(np.float64).reshape(K // G, G, N) * np.asarray(s, np.float64)[:, None, :]
         - np.asarray(zf, np.float64)[:, None, :]).reshape(K, N)
    return A @ W, np.abs(A) @ np.abs(W)


def reference(A_raw, codes, scales, zeros, *, K: int, N: int, G: int, w4: bool,
              act: str, sc: str, rows=None, cols=None, zp_float: bool = False):
    """Decode canonical inputs with this module's own codecs and return (ref, mag), both
    float64 [len(rows)][len(cols)].

    A_raw:  [M][K] bf16 bits (uint16) if act == "bf16", else float32.
    codes:  W4: uint32 [K/8][N]; W8: int8 [K][N] (zero point 0).
    scales: [K/G][N] fp16 / bf16 bits (uint16) or float32, per ``sc``.
    zeros:  W4 only: uint32 [K/G][N/8] or None (then z = 8, the symmetric point of the
            INT4 teaching kernel, P1 section 9.4); with ``zp_float``, float zero points
            [K/G][N] in the scales' format, subtracted after scaling (``group_gemm_zf``).
    """
    A_raw = np.asarray(A_raw)
    if rows is not None:
        A_raw = A_raw[np.asarray(rows)]
    A = bf16_bits_to_f64(A_raw) if act == "bf16" else f32_to_f64(A_raw)
    ng = K // G
    cols_ = np.arange(N) if cols is None else np.asarray(cols)
    if w4:
        q = unpack_int4_k(np.asarray(codes)[:, cols_])
        if zeros is None or zp_float:
            z = np.full((ng, len(cols_)), 8, dtype=np.int64)
        else:
            z = unpack_int4_n(np.asarray(zeros))[:, cols_]
    else:
        q = np.asarray(codes)[:, cols_].astype(np.int64)
        z = np.zeros((ng, len(cols_)), dtype=np.int64)
    def dec(raw):
        raw = np.asarray(raw)[:, cols_]
        if sc == "fp16":
            return fp16_bits_to_f64(raw)
        if sc == "bf16":
            return bf16_bits_to_f64(raw)
        return f32_to_f64(raw)
    s = dec(scales)
    if zp_float:
        assert w4
        return group_gemm_zf(A, unpack_int4_k(np.asarray(codes)[:, cols_]), dec(zeros), s, G)
    return group_gemm(A, q, z, s, G), group_gemm_magnitude(A, q, z, s, G)


# ---------------------------------------------------------------------------------------
# Fused gate+up epilogue (P1 section 五.2, SiLU-and-mul): the gate_up GEMM's N = 2F columns
# are F gate columns then F up columns, and the epilogue returns silu(gate) · up, [M][F].
# ---------------------------------------------------------------------------------------

def silu(x) -> np.ndarray:
    """silu(x) = x · σ(x) = x / (1 + e^(−x)), in float64."""
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def silu_mul_reference(A_raw, codes, scales, zeros, *, K: int, N: int, G: int, act: str,
                       sc: str, rows=None, cols=None, w4: bool = True):
    """out[m][j] = silu(gate[m][j]) · up[m][j] with gate = column j < F = N/2 and up = column
    F + j of the group GEMM (W4 or W8 codes).  Returns (ref, mag) over output columns ``cols``
    (default all F).  mag carries the GEMM's own error bound through the product to first
    order: max|silu'| · mag_gate · |up| + |silu(gate)| · mag_up, where |silu'(x)| =
    |σ(x)·(1 + x·(1 − σ(x)))| < 1.1 for every x, so ``tolerance``/``check`` apply unchanged."""
    F = N // 2
    jc = np.arange(F) if cols is None else np.asarray(cols)
    g, mg = reference(A_raw, codes, scales, zeros, K=K, N=N, G=G, w4=w4, act=act, sc=sc,
                      rows=rows, cols=jc)
    u, mu = reference(A_raw, codes, scales, zeros, K=K, N=N, G=G, w4=w4, act=act, sc=sc,
                      rows=rows, cols=F + jc)
    sg = silu(g)
    return sg * u, 1.1 * mg * np.abs(u) + np.abs(sg) * mu


# ---------------------------------------------------------------------------------------
# INT8-activation variant.  P2 section 2: out[m][n] = Σ_g a_scale[m][g] · b_scale[g][n] ·
# (Σ_{k ∈ g} Aq[m][k] · Wq[k][n]), the integer dot of a whole group before either scale.
# The activation codes come from the per-group absmax quantization of P1 section 四.5
# (s = max|x| / 127, divide, round, saturate, cast).
# ---------------------------------------------------------------------------------------

def quantize_act_i8(A_raw, G: int, act: str):
    """Per (row, group of G): s = max|x| / 127 and q = rint(x / s) clamped to [-127, 127];
    s = 0 and q = 0 for a group of zeros.  Both divisions are IEEE binary32 and the rounding
    is to nearest, ties to even: the integer each code is decided in the same precision as
    the GPU kernel.  Returns (Aq int8 [M][K], a_scales float32 [M][K/G])."""
    A = bf16_bits_to_f64(A_raw) if act == "bf16" else f32_to_f64(A_raw)
    A32 = A.astype(np.float32)                      # exact: bf16 and fp32 inputs
    M, K = A32.shape
    Ag = A32.reshape(M, K // G, G)
    amax = np.abs(Ag).max(axis=2)                   # exact
    s = (amax / np.float32(127)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (Ag / s[:, :, None]).astype(np.float32)
    q = np.where(s[:, :, None] > 0, np.clip(np.rint(r), -127, 127), 0)
    return q.reshape(M, K).astype(np.int8), s


def group_gemm_a8(Aq, a_s, q, s, G: int):
    """Σ_g a_s[m][g] · s[g][n] · Σ_{k ∈ g} Aq[m][k] · q[k][n], the group dots in exact int64,
    the scales in float64.  Returns (out, mag) with mag = Σ_g |a_s · s| · Σ_k |Aq · q|."""
    Aq = np.asarray(Aq, dtype=np.int64)
    q = np.asarray(q, dtype=np.int64)
    a_s = np.asarray(a_s, dtype=np.float64)
    s = np.asarray(s, dtype=np.float64)
    M, K = Aq.shape
    N = q.shape[1]
    out = np.zeros((M, N))
    mag = np.zeros((M, N))
    for g in range(K // G):
        ks = slice(g * G, (g + 1) * G)
        dot = Aq[:, ks] @ q[ks, :]                  # exact integers
        adot = np.abs(Aq[:, ks]) @ np.abs(q[ks, :])
        w = a_s[:, g][:, None] * s[g][None, :]
        out += w * dot.astype(np.float64)
        mag += np.abs(w) * adot.astype(np.float64)
    return out, mag


def reference_a8(Aq, a_scales, codes, scales, *, K: int, N: int, G: int, rows=None, cols=None):
    """(ref, mag) of the W8A8 group GEMM from int8 activation codes [M][K], fp32 activation
    scales [M][K/G], int8 weight codes [K][N] and fp32 weight scales [K/G][N]."""
    Aq = np.asarray(Aq)
    a_s = f32_to_f64(a_scales)
    if rows is not None:
        Aq, a_s = Aq[np.asarray(rows)], a_s[np.asarray(rows)]
    cols_ = np.arange(N) if cols is None else np.asarray(cols)
    q = np.asarray(codes)[:, cols_]
    s = f32_to_f64(np.asarray(scales)[:, cols_])
    return group_gemm_a8(Aq, a_s, q, s, G)


# ---------------------------------------------------------------------------------------
# FP8 W8A8 GEMM with block scales (P1 section 四.3).  E4M3 ("FN": no infinities): 1 sign bit,
# 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 is subnormal (m/8 · 2^-6); the
# pattern S.1111.111 is NaN, so the largest finite magnitude is 1.75 · 2^8 = 448.
# ---------------------------------------------------------------------------------------

def e4m3_bits_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits).astype(np.int64) & 0xFF
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def f64_to_e4m3_bits(x) -> np.ndarray:
    """Nearest E4M3 value, ties to the even code, finite values beyond ±448 saturated to ±448
    (the "satfinite" conversion); the sign of a zero is kept.  Written from the format: the
    finite magnitudes are the 127 codes 0x00 .. 0x7E in increasing order."""
    x = np.asarray(x, dtype=np.float64)
    grid = e4m3_bits_to_f64(np.arange(0x7F))       # increasing, 0 .. 448
    a = np.minimum(np.abs(x), 448.0)
    hi = np.clip(np.searchsorted(grid, a, side="left"), 0, 0x7E)
    lo = np.clip(hi - 1, 0, 0x7E)
    d_lo, d_hi = a - grid[lo], grid[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(take_hi, hi, lo)
    code = np.where(a == grid[hi], hi, code)       # exact grid values
    return (code | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


def quantize_act_fp8(A_raw, act: str, block: int = 128):
    """Per (row, block of 128 k): s = max|x| / 448 and code = E4M3(x / s), both divisions in
    binary32 as on the GPU (the code is decided in the kernel's precision); s = 0 and codes 0
    for a block of zeros.  Returns (Aq uint8 [M][K], a_scales float32 [K/block][M])."""
    A = bf16_bits_to_f64(A_raw) if act == "bf16" else f32_to_f64(A_raw)
    A32 = A.astype(np.float32)
    M, K = A32.shape
    Ag = A32.reshape(M, K // block, block)
    s = (np.abs(Ag).max(axis=2) / np.float32(448)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (Ag / s[:, :, None]).astype(np.float32)
    codes = np.where(s[:, :, None] > 0, f64_to_e4m3_bits(r.astype(np.float64)), 0)
    return codes.reshape(M, K).astype(np.uint8), np.ascontiguousarray(s.T)


def fp8_block_gemm(A_bits, a_scales, W_bits, w_scales, block: int = 128):
    """out[m][n] = Σ_b a_scales[b][m] · w_scales[n // block][b] · Σ_{k ∈ b} A[m][k] · W[n][k]
    in float64 (each product of two E4M3 values is exact), with mag = the same sum of
    absolute values for the tolerance.  A_bits [M][K], W_bits [N][K] (E4M3 bytes), a_scales
    float32 [K/block][M], w_scales float32 [ceil(N/block)][K/block]."""
    A = e4m3_bits_to_f64(A_bits)
    W = e4m3_bits_to_f64(W_bits)
    a_s = f32_to_f64(a_scales)
    w_s = f32_to_f64(w_scales)
    M, K = A.shape
    N = W.shape[0]
    nrow_blk = np.arange(N) // block
    out = np.zeros((M, N))
    mag = np.zeros((M, N))
    for b in range(K // block):
        ks = slice(b * block, (b + 1) * block)
        part = A[:, ks] @ W[:, ks].T
        apart = np.abs(A[:, ks]) @ np.abs(W[:, ks]).T
        sc = a_s[b][:, None] * w_s[nrow_blk, b][None, :]
        out += sc * part
        mag += np.abs(sc) * apart
    return out, mag


# ---------------------------------------------------------------------------------------
# Tolerance.  P1 section 8: error of a K-term FP32 accumulation grows like ε·sqrt(K) times
# the typical product and relative error blows up where the output cancels; so the bound
# has a relative term (the final rounding of the output) and a conditioning term.
# ---------------------------------------------------------------------------------------

def tolerance(ref: np.ndarray, mag: np.ndarray, out_dtype: str) -> np.ndarray:
    """bf16 out: 2^-8·|ref| + 1e-4·mag.  fp32 out: 1e-5·|ref| + 1e-6·mag."""
    if out_dtype == "bf16":
        return 2.0 ** -8 * np.abs(ref) + 1e-4 * mag
    return 1e-5 * np.abs(ref) + 1e-6 * mag


def check(out_f64: np.ndarray, ref: np.ndarray, mag: np.ndarray, out_dtype: str):
    """Return (n_bad, worst err/tol) of a decoded GPU output against the oracle."""
    tol = tolerance(ref, mag, out_dtype)
    err = np.abs(np.asarray(out_f64, np.float64) - ref)
    bad = ~(err <= tol)
    ratio = float(np.max(err / np.maximum(tol, 1e-300))) if err.size else 0.0
    return int(bad.sum()), ratio


# ---------------------------------------------------------------------------------------
# The reference quantizer of P1 section 9.4 (symmetric, per-group amax / 7, zero point 8),
# kept to generate quantized weights from real ones in the checks.
# ---------------------------------------------------------------------------------------

def quantize_w4_g(W: np.ndarray, G: int = 128):
    """W [N][K] real -> (q uint8 [N][K] in [0,15], s float64 [N][K/G], W_hat float64 [N][K]).

    s = max(amax(|W_group|) / 7, 1e-8); q = clamp(round(W / s) + 8, 0, 15);
    W_hat = (q − 8)·s.  round() is round-half-to-even (numpy rint).
    """
    N, K = W.shape
    assert K % G == 0
    Wg = np.asarray(W, np.float64).reshape(N, K // G, G)
    s = np.maximum(np.abs(Wg).max(axis=-1, keepdims=True) / 7.0, 1e-8)
    q = np.clip(np.rint(Wg / s) + 8, 0, 15)
    W_hat = ((q - 8.0) * s).reshape(N, K)
    return q.astype(np.uint8).reshape(N, K), s.reshape(N, K // G), W_hat


def bits_per_weight(code_bits: int, G: int, scale_bits: int, zero_point_bits: int = 0) -> float:
    """Storage cost per weight: the code, plus one scale and (optionally) one packed zero
    point shared by each group of G weights (P1 section 3.1: a g128 fp16 scale adds 0.125
    bit, an INT4 zero point about 0.03 bit)."""
    return code_bits + (scale_bits + zero_point_bits) / G


def dequantize_brute(q_raw, z_raw, s_vals, G: int, K: int, N: int):
    """Element-by-element dequantization with Python loops (tiny shapes only): the
    brute-force side of the oracle's self-check.  q_raw [K][N] ints, z_raw [K/G][N] ints
    (or a scalar), s_vals [K/G][N] floats."""
    W = [[0.0] * N for _ in range(K)]
    for k in range(K):
        g = k // G
        for n in range(N):
            zz = z_raw if np.isscalar(z_raw) else int(z_raw[g][n])
            W[k][n] = float(s_vals[g][n]) * (int(q_raw[k][n]) - zz)
    return W
