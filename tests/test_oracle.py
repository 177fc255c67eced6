"""Pins of the float64 oracle against things other than itself (CPU only).

Each test names what fixes the expected value: a value the pages print (tests/golden),
a closed form, a library routine in a special case, or brute force on tiny inputs.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import gq_synth
import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ------------------------------------------------------------------ IEEE codecs

def test_fp16_decoder_matches_library_on_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = orc.fp16_bits_to_f64(bits)
    lib = bits.view(np.float16).astype(np.float64)
    same = (ours == lib) | (np.isnan(ours) & np.isnan(lib))
    assert same.all()


def test_bf16_decoder_matches_library_on_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    lib = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    ours = orc.bf16_bits_to_f64(bits)
    same = (ours == lib) | (np.isnan(ours) & np.isnan(lib))
    assert same.all()


def test_bf16_encoder_matches_library_rne():
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-40, 38, 20000),
        # exact ties between neighbouring bf16 values: round half to even
        orc.bf16_bits_to_f64(np.arange(0x3F80, 0x3FA0)) + 2.0 ** -8,
        orc.bf16_bits_to_f64(np.arange(0x0001, 0x0040)) * 1.5,   # subnormal ties
        np.array([0.0, -0.0, 3.3895313892515355e38, 3.4e38, -1e-45, 1e-39]),
    ]).astype(np.float32).astype(np.float64)   # exactly representable in fp32
    lib = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16)
    lib = lib.numpy().view(np.uint16)
    assert np.array_equal(orc.f64_to_bf16_bits(x), lib)


def test_bf16_encoder_roundtrip_all_finite_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = orc.bf16_bits_to_f64(bits)
    fin = np.isfinite(vals)
    back = orc.f64_to_bf16_bits(vals[fin])
    # -0.0 and +0.0 both survive with their sign
    assert np.array_equal(back, bits[fin])


# ------------------------------------------------------------------ magic numbers

def test_magic_constants_printed_on_the_page():
    for fmt, bits, value in _golden("magic_constants.txt"):
        b = np.array([int(bits, 16)], dtype=np.uint16)
        dec = orc.fp16_bits_to_f64(b) if fmt == "fp16" else orc.bf16_bits_to_f64(b)
        assert dec[0] == float(value), (fmt, bits)


def test_magic_identities_exhaustive():
    """All 16 INT4 codes: the decode forms the CUDA path relies on reach q - 8 exactly."""
    f16 = lambda b: float(orc.fp16_bits_to_f64(np.array([b], dtype=np.uint16))[0])
    b16 = lambda b: float(orc.bf16_bits_to_f64(np.array([b], dtype=np.uint16))[0])
    f32 = lambda b: float(np.array([b], dtype=np.uint32).view(np.float32)[0])
    for q in range(16):
        assert f16(0x6400 | q) - f16(0x6408) == q - 8                      # lo nibble, FP16
        assert f16(0x6400 | (q << 4)) * f16(0x2C00) + f16(0xD480) == q - 8  # hi nibble, FP16
        assert b16(0x4300 | q) - 136.0 == q - 8                            # lo nibble, BF16
        assert f32(0x4B000000 | q) - (2.0 ** 23 + 8) == q - 8              # FP32 2^23 form
        for zp in range(16):                                               # asymmetric point
            assert b16(0x4300 | q) - b16(0x4300 | zp) == q - zp
    # the hi-nibble form does not carry over to BF16: bit 7 of the half-word is the
    # exponent's lowest bit there, so codes >= 8 change the binade (q = 8 lands on 256,
    # which happens to give 0 = q - 8; every code above it is wrong)
    wrong = [q for q in range(16) if b16(0x4300 | (q << 4)) / 16.0 - 16.0 != q - 8]
    assert wrong == list(range(9, 16))


def test_int8_magic_identity_all_codes():
    """Signed INT8 code c -> (c xor 0x80) in the low byte of 2^23 gives 2^23 + c + 128."""
    for c in range(-128, 128):
        u = (c & 0xFF) ^ 0x80
        v = float(np.array([0x4B000000 | u], dtype=np.uint32).view(np.float32)[0])
        assert v - (2.0 ** 23 + 128) == c


# ------------------------------------------------------------------ layouts

def test_int4_word_convention():
    w = np.array([[0x76543210, 0xFEDCBA98]], dtype=np.uint32)
    assert orc.unpack_int4_k(w)[:, 0].tolist() == list(range(8))
    assert orc.unpack_int4_k(w)[:, 1].tolist() == list(range(8, 16))
    assert orc.unpack_int4_n(w)[0].tolist() == list(range(16))


@pytest.mark.parametrize("name", ["tiny_gemv", "asym_m16"])
def test_unpack_matches_generator_codes(name):
    cfg = gq_synth.CONFIGS[name]
    if cfg.K * cfg.N > 1 << 22:
        cfg = cfg.replace(K=1024, N=512)
    w = gq_synth.make_weights(cfg, seed=3)
    assert np.array_equal(orc.unpack_int4_k(w["codes"]), w["q"].astype(np.int64))
    if w["zeros"] is not None:
        assert np.array_equal(orc.unpack_int4_n(w["zeros"]), w["z"].astype(np.int64))


# ------------------------------------------------------------------ the GEMM itself

def _brute(cfg, inp):
    """Dequantize element by element, then a triple loop with exact fsum.  Reads the
    generator's raw integer codes and decodes scales/activations with library routines,
    so it shares no decoding step with the oracle."""
    K, N, G = cfg.K, cfg.N, cfg.G
    if cfg.sc == "fp16":
        s = inp["scales"].view(np.float16).astype(np.float64)
    elif cfg.sc == "bf16":
        s = torch.from_numpy(inp["scales"].view(np.int16)).view(torch.bfloat16).double().numpy()
    else:
        s = inp["scales"].astype(np.float64)
    if cfg.act == "bf16":
        A = torch.from_numpy(inp["A"].view(np.int16)).view(torch.bfloat16).double().numpy()
    else:
        A = inp["A"].astype(np.float64)
    z = inp["z"] if inp["z"] is not None else (8 if cfg.w4 else 0)
    W = orc.dequantize_brute(inp["q"], z, s, G, K, N)
    M = A.shape[0]
    out = [[math.fsum(A[m][k] * W[k][n] for k in range(K)) for n in range(N)] for m in range(M)]
    return np.array(out)


SMALL = [
    gq_synth.Config("w4_sym", M=3, K=256, N=24, G=128),
    gq_synth.Config("w4_asym", M=2, K=256, N=16, G=32, zp=True, sc="bf16"),
    gq_synth.Config("w8", M=2, K=96, N=8, G=32, w4=False, act="f32", sc="f32", out="f32",
                    s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("w4_g128_single_group", M=4, K=128, N=40, G=128, outlier_frac=0.02),
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_oracle_matches_brute_force(cfg):
    inp = gq_synth.make_inputs(cfg, seed=11)
    ref, mag = orc.reference(inp["A"], inp["codes"], inp["scales"], inp["zeros"], K=cfg.K,
                             N=cfg.N, G=cfg.G, w4=cfg.w4, act=cfg.act, sc=cfg.sc)
    brute = _brute(cfg, inp)
    assert np.allclose(ref, brute, rtol=1e-12, atol=1e-12 * float(np.max(mag)))
    assert (mag >= np.abs(ref) * (1 - 1e-12)).all()


def test_oracle_subset_rows_cols_match_full():
    cfg = gq_synth.Config("sub", M=5, K=256, N=64, G=128, zp=True, sc="bf16")
    inp = gq_synth.make_inputs(cfg, seed=2)
    kw = dict(K=cfg.K, N=cfg.N, G=cfg.G, w4=True, act="bf16", sc="bf16")
    full, _ = orc.reference(inp["A"], inp["codes"], inp["scales"], inp["zeros"], **kw)
    rows, cols = [4, 0, 2], [63, 1, 8, 9, 40]
    part, _ = orc.reference(inp["A"], inp["codes"], inp["scales"], inp["zeros"], rows=rows,
                            cols=cols, **kw)
    assert np.array_equal(part, full[np.ix_(rows, cols)])


def test_identity_weights_return_activations():
    """K = N, s = 1, z = 8, q = 9 on the diagonal and 8 elsewhere: W_hat = I, out = A."""
    K = N = 256
    q = np.full((K, N), 8, dtype=np.uint8)
    np.fill_diagonal(q, 9)
    codes = gq_synth.pack_int4_along_k(q)
    scales = np.full((K // 128, N), 0x3C00, dtype=np.uint16)       # fp16 1.0
    A = gq_synth.make_activations(gq_synth.Config("id", M=3, K=K, N=N, G=128), seed=1)
    ref, _ = orc.reference(A, codes, scales, None, K=K, N=N, G=128, w4=True, act="bf16",
                           sc="fp16")
    assert np.array_equal(ref, orc.bf16_bits_to_f64(A))


def test_one_hot_weight_selects_one_activation_column():
    K, N, G = 256, 16, 128
    q = np.full((K, N), 8, dtype=np.uint8)
    k0, n0, code = 200, 5, 3
    q[k0, n0] = code
    s = np.full((K // G, N), 0.5, dtype=np.float32)
    codes = gq_synth.pack_int4_along_k(q)
    scales = gq_synth.f32_to_fp16_bits(s)
    A = gq_synth.make_activations(gq_synth.Config("oh", M=4, K=K, N=N, G=G), seed=9)
    ref, _ = orc.reference(A, codes, scales, None, K=K, N=N, G=G, w4=True, act="bf16",
                           sc="fp16")
    expect = np.zeros((4, N))
    expect[:, n0] = 0.5 * (code - 8) * orc.bf16_bits_to_f64(A[:, k0])
    assert np.array_equal(ref, expect)


def test_doubling_scales_doubles_output_exactly():
    cfg = gq_synth.Config("lin", M=2, K=512, N=32, G=128, zp=True, sc="fp16")
    inp = gq_synth.make_inputs(cfg, seed=4)
    kw = dict(K=cfg.K, N=cfg.N, G=cfg.G, w4=True, act="bf16", sc="fp16")
    r1, _ = orc.reference(inp["A"], inp["codes"], inp["scales"], inp["zeros"], **kw)
    s2 = gq_synth.f32_to_fp16_bits(orc.fp16_bits_to_f64(inp["scales"]) * 2)
    r2, _ = orc.reference(inp["A"], inp["codes"], s2, inp["zeros"], **kw)
    assert np.array_equal(r2, 2 * r1)


def test_integer_case_is_exact():
    """Integer activations and power-of-two scales: every partial sum is an exact
    rational; the oracle must equal the exact Fraction sum."""
    cfg = gq_synth.Config("exact", M=2, K=256, N=8, G=128, zp=True, sc="fp16", a_kind="int",
                          pow2_scales=True)
    inp = gq_synth.make_inputs(cfg, seed=6)
    ref, _ = orc.reference(inp["A"], inp["codes"], inp["scales"], inp["zeros"], K=cfg.K,
                           N=cfg.N, G=cfg.G, w4=True, act="bf16", sc="fp16")
    A = torch.from_numpy(inp["A"].view(np.int16)).view(torch.bfloat16).double().numpy()
    s = inp["scales"].view(np.float16).astype(np.float64)
    for m in range(cfg.M):
        for n in range(cfg.N):
            tot = Fraction(0)
            for k in range(cfg.K):
                g = k // cfg.G
                tot += Fraction(A[m, k]) * Fraction(s[g, n]) * (int(inp["q"][k, n]) - int(inp["z"][g, n]))
            assert Fraction(ref[m, n]) == tot


# ------------------------------------------------------------------ planted mistakes

def _mutant_gemm_no_zero_point(A, q, z, s, G):
    return orc.group_gemm(A, q, np.zeros_like(z), s, G)


def _mutant_gemm_wrong_group_index(A, q, z, s, G):
    K = q.shape[0]
    ng = K // G
    out = np.zeros((A.shape[0], q.shape[1]))
    for k in range(K):
        g = k % ng                       # wrong: interleaved instead of contiguous groups
        out += np.outer(A[:, k], s[g] * (q[k] - z[g]))
    return out


def _mutant_gemm_scale_after_sum(A, q, z, s, G):
    return (A @ (q.astype(np.float64) - np.repeat(z, G, axis=0))) * s.mean(axis=0)


@pytest.mark.parametrize("mutant", [_mutant_gemm_no_zero_point, _mutant_gemm_wrong_group_index,
                                    _mutant_gemm_scale_after_sum])
def test_brute_force_pin_catches_planted_mistakes(mutant, monkeypatch):
    cfg = SMALL[1]   # asymmetric, several groups, non-square
    inp = gq_synth.make_inputs(cfg, seed=11)
    brute = _brute(cfg, inp)
    monkeypatch.setattr(orc.gq_oracle, "group_gemm", mutant)
    ref, _ = orc.gq_oracle.reference(inp["A"], inp["codes"], inp["scales"], inp["zeros"],
                                     K=cfg.K, N=cfg.N, G=cfg.G, w4=True, act=cfg.act, sc=cfg.sc)
    assert not np.allclose(ref, brute, rtol=1e-6, atol=1e-9)


def test_identity_pin_catches_reversed_nibble_order(monkeypatch):
    real = orc.gq_oracle.unpack_int4_k

    def reversed_nibbles(words):
        q = real(words)
        R = q.shape[0] // 8
        return q.reshape(R, 8, -1)[:, ::-1, :].reshape(R * 8, -1)

    monkeypatch.setattr(orc.gq_oracle, "unpack_int4_k", reversed_nibbles)
    K = N = 128
    q = np.full((K, N), 8, dtype=np.uint8)
    np.fill_diagonal(q, 9)
    A = gq_synth.make_activations(gq_synth.Config("id", M=2, K=K, N=N, G=128), seed=1)
    ref, _ = orc.gq_oracle.reference(A, gq_synth.pack_int4_along_k(q),
                                     np.full((1, N), 0x3C00, dtype=np.uint16), None, K=K, N=N,
                                     G=128, w4=True, act="bf16", sc="fp16")
    assert not np.array_equal(ref, orc.bf16_bits_to_f64(A))


# ------------------------------------------------------------------ quantizer and costs

def test_reference_quantizer_error_bound():
    """P1 section 9.4's quantizer: |W - W_hat| <= s/2 everywhere (W/s stays in [-7, 7], so
    the clamp never fires), and the largest element of each group is reproduced exactly
    up to its sign (q - 8 = ±7)."""
    W = gq_synth.real_weights(16, 512, seed=1)
    q, s, W_hat = orc.quantize_w4_g(W, G=128)
    err = np.abs(W.astype(np.float64) - W_hat)
    s_full = np.repeat(s, 128, axis=1)
    assert (err <= s_full / 2 * (1 + 1e-12)).all()
    assert q.min() >= 1 and q.max() <= 15
    Wg = W.astype(np.float64).reshape(16, 4, 128)
    idx = np.abs(Wg).argmax(-1)
    qg = q.reshape(16, 4, 128).astype(int)
    picked = np.take_along_axis(qg, idx[..., None], -1)[..., 0]
    assert set(np.unique(picked)) <= {1, 15}


def test_format_costs_printed_on_the_page():
    g = {r[0]: (float(r[1]), float(r[2])) for r in _golden("format_costs.txt")}
    bpw = orc.bits_per_weight(4, 128, 16, 4)
    checks = {
        "scale_bits_g128": orc.bits_per_weight(0, 128, 16),
        "zero_point_bits_g128": orc.bits_per_weight(0, 128, 0, 4),
        "w4_g128_bits_per_weight": bpw,
        "w4_g128_fraction_of_bf16": bpw / 16,
        "decode_speedup_bound": 16 / bpw,
        "int8_dot_bound_k4096": 127 * 127 * 4096,
    }
    for k, v in checks.items():
        val, tol = g[k]
        assert abs(v - val) <= tol, (k, v, val)
    assert 127 * 127 * 4096 < 2 ** 31
    assert orc.bits_per_weight(4, 128, 16) == 4.125
    assert orc.bits_per_weight(8, 32, 32) == 9.0


def test_layer_byte_counts_printed_on_the_page():
    g = {r[0]: (float(r[1]), float(r[2])) for r in _golden("byte_counts.txt")}
    d, dff, kv = 4096, 14336, 8 * 128
    shapes = [(d, d + 2 * kv), (d, d), (d, 2 * dff), (dff, d)]      # (K, N) of qkv, o, gate_up, down
    params = sum(K * N for K, N in shapes)
    w4 = orc.bits_per_weight(4, 128, 16, 4)
    vals = {
        "gemv4096_int4_weight_bytes": 4096 * 4096 * 4 / 8,
        "gemv4096_int4_scale_bytes": 4096 * 4096 * orc.bits_per_weight(0, 128, 16) / 8,
        "gemv4096_bf16_weight_bytes": 4096 * 4096 * 2,
        "layer_bf16_bytes": params * 2,
        "layer_int4_g128_bytes": params * w4 / 8,
        "prefill4096_int4_saving_bytes": 4096 * 4096 * (2 - 0.5),
    }
    for k, v in vals.items():
        val, tol = g[k]
        assert abs(v - val) <= tol, (k, v, val)


def test_tolerance_formula():
    ref = np.array([1.0, -2.0, 0.0])
    mag = np.array([10.0, 10.0, 10.0])
    assert np.allclose(orc.tolerance(ref, mag, "bf16"), [2 ** -8 + 1e-3, 2 ** -7 + 1e-3, 1e-3])
    assert np.allclose(orc.tolerance(ref, mag, "f32"), [1e-5 + 1e-5, 2e-5 + 1e-5, 1e-5])
    bad, ratio = orc.check(ref + np.array([0.0, 0.0, 2e-3]), ref, mag, "bf16")
    assert bad == 1 and ratio == pytest.approx(2.0)


# ------------------------------------------------------------------ fused gate+up epilogue

def test_silu_closed_forms_and_odd_part():
    """silu(x) = x·σ(x): silu(0) = 0; σ(ln 3) = 3/4 and σ(−ln 3) = 1/4, so silu(±ln 3) =
    ±ln 3 · {3/4, 1/4}; σ(x) + σ(−x) = 1 gives silu(x) − silu(−x) = x for every x; and
    silu(x) → x, silu(−x) → 0 for large x."""
    ln3 = math.log(3.0)
    assert orc.silu(0.0) == 0.0
    assert abs(orc.silu(ln3) - 0.75 * ln3) <= 1e-15
    assert abs(orc.silu(-ln3) + 0.25 * ln3) <= 1e-15
    x = np.random.default_rng(3).normal(0, 4, 1000)
    assert np.allclose(orc.silu(x) - orc.silu(-x), x, rtol=1e-14, atol=1e-14)
    assert orc.silu(40.0) == 40.0 and abs(orc.silu(-40.0)) < 1e-15


def test_silu_mul_takes_gate_from_the_first_half_and_up_from_the_second():
    """One-hot weights: gate column j0 = 40·(selected activation 1.0) so silu(gate) = 40 to
    double precision, up column F + j0 = 0.5·(code − 8)·A[:, k2]; out[:, j0] = 40·up and
    every other output is silu(0)·0 = 0.  Swapping the halves would give silu(up)·40."""
    K, N, G = 256, 32, 128
    F = N // 2
    q = np.full((K, N), 8, dtype=np.uint8)
    j0, k1, k2 = 5, 17, 200
    q[k1, j0] = 9                                  # gate: s·1 at k1
    q[k2, F + j0] = 3                              # up: s·(3 − 8) at k2
    s = np.ones((K // G, N), dtype=np.float32)
    s[:, F + j0] = 0.5
    s[:, j0] = 40.0
    codes = gq_synth.pack_int4_along_k(q)
    scales = gq_synth.f32_to_fp16_bits(s)
    A = gq_synth.make_activations(gq_synth.Config("gu", M=3, K=K, N=N, G=G), seed=2)
    A[:, k1] = 0x3F80                              # bf16 1.0
    ref, mag = orc.silu_mul_reference(A, codes, scales, None, K=K, N=N, G=G, act="bf16",
                                      sc="fp16")
    up = 0.5 * (3 - 8) * orc.bf16_bits_to_f64(A[:, k2])
    expect = np.zeros((3, F))
    expect[:, j0] = 40.0 * up
    assert ref.shape == (3, F)
    assert np.array_equal(ref, expect)
    assert (mag >= 0).all() and (mag[:, j0] > 0).all()


# ------------------------------------------------------------------ INT8-activation variant

def test_activation_quantizer_special_cases():
    """A group whose largest magnitude is 127 has scale exactly 1, so codes are the values
    rounded to nearest with ties to even (2.5 -> 2, 3.5 -> 4, -2.5 -> -2), ±127 map to ±127,
    and an all-zero group has scale 0 and codes 0."""
    G = 32
    row = np.zeros(2 * G, dtype=np.float32)
    row[:8] = [127.0, -127.0, 2.5, 3.5, -2.5, 0.25, 126.5, 0.0]
    Aq, s = orc.quantize_act_i8(row[None, :], G, "f32")
    assert s[0, 0] == 1.0 and s[0, 1] == 0.0
    assert Aq[0, :8].tolist() == [127, -127, 2, 4, -2, 0, 126, 0]
    assert (Aq[0, G:] == 0).all()


def test_activation_quantizer_error_bound_and_range():
    """|x − s·q| ≤ s/2 (to float32 rounding of x/s) and |q| ≤ 127, with the group's largest
    magnitude at ±127, on bf16 N(0,1) activations with outliers."""
    cfg = gq_synth.Config("aq", M=4, K=1024, N=16, G=64, outlier_frac=0.01)
    A = gq_synth.make_activations(cfg, seed=5)
    Aq, s = orc.quantize_act_i8(A, 64, "bf16")
    x = orc.bf16_bits_to_f64(A).reshape(4, 16, 64)
    qq = Aq.astype(np.int64).reshape(4, 16, 64)
    ss = s.astype(np.float64)[:, :, None]
    assert (np.abs(qq) <= 127).all()
    assert (np.abs(qq).max(axis=2) == 127).all()
    assert (np.abs(x - ss * qq) <= ss * (0.5 + 1e-6)).all()


def test_a8_group_gemm_matches_brute_force_and_integer_product():
    rng = np.random.default_rng(8)
    M, K, N, G = 3, 96, 5, 32
    Aq = rng.integers(-127, 128, (M, K)).astype(np.int8)
    q = rng.integers(-127, 128, (K, N)).astype(np.int8)
    a_s = rng.uniform(0.01, 0.1, (M, K // G)).astype(np.float32)
    s = rng.uniform(1e-3, 1e-2, (K // G, N)).astype(np.float32)
    out, mag = orc.reference_a8(Aq, a_s, q, s, K=K, N=N, G=G)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(float(a_s[m, k // G])) * Fraction(float(s[k // G, n])) *
                        int(Aq[m, k]) * int(q[k, n]) for k in range(K))
            assert abs(out[m, n] - float(exact)) <= 1e-12 * mag[m, n]
    # unit scales reduce it to the integer matrix product
    one_a, one_s = np.ones_like(a_s), np.ones_like(s)
    out1, _ = orc.reference_a8(Aq, one_a, q, one_s, K=K, N=N, G=G)
    assert np.array_equal(out1, (Aq.astype(np.int64) @ q.astype(np.int64)).astype(np.float64))


# ------------------------------------------------------------------ float zero points

def _lib_decode(bits, fmt):
    """Scale-format bits -> float64 with library routines (numpy fp16, torch bf16)."""
    if fmt == "fp16":
        return np.asarray(bits).view(np.float16).astype(np.float64)
    if fmt == "bf16":
        return torch.from_numpy(np.asarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()
    return np.asarray(bits).astype(np.float64)


ZF_SMALL = [
    gq_synth.Config("zf_bf16", M=2, K=64, N=5, G=32, zf=True, sc="bf16"),
    gq_synth.Config("zf_fp16_g128", M=3, K=256, N=8, G=128, zf=True),
    gq_synth.Config("zf_f32", M=1, K=96, N=16, G=32, zf=True, sc="f32", out="f32"),
]


@pytest.mark.parametrize("cfg", ZF_SMALL, ids=lambda c: c.name)
def test_float_zero_oracle_matches_exact_rational_sum(cfg):
    """Σ_k A·(q·s − zf) in exact rationals from the generator's raw codes and library-decoded
    scales, zero points and activations (nothing shared with the oracle's decoders)."""
    inp = gq_synth.make_inputs(cfg, seed=5)
    ref, mag = orc.reference(inp["A"], inp["codes"], inp["scales"], inp["zeros"], K=cfg.K,
                             N=cfg.N, G=cfg.G, w4=True, act=cfg.act, sc=cfg.sc, zp_float=True)
    s, zf = _lib_decode(inp["scales"], cfg.sc), _lib_decode(inp["zeros"], cfg.sc)
    A = torch.from_numpy(inp["A"].view(np.int16)).view(torch.bfloat16).double().numpy()
    q = inp["q"]
    for m in range(A.shape[0]):
        for n in range(cfg.N):
            exact = sum(Fraction(float(A[m, k])) * (int(q[k, n]) * Fraction(float(s[k // cfg.G, n]))
                                                     - Fraction(float(zf[k // cfg.G, n])))
                        for k in range(cfg.K))
            assert abs(ref[m, n] - float(exact)) <= 1e-13 * mag[m, n] + 1e-300
    assert (mag >= np.abs(ref) * (1 - 1e-12)).all()


def test_float_zero_equal_to_scaled_integer_zero_gives_the_integer_form():
    """With power-of-two scales and zf = s·z for integer z (exact), W_hat = q·s − zf equals
    s·(q − z): the float form must agree with the integer-zero group GEMM."""
    cfg = gq_synth.Config("zf_int", M=3, K=256, N=24, G=64, zf=True, sc="bf16", pow2_scales=True)
    inp = gq_synth.make_inputs(cfg, seed=2)
    s, zf = _lib_decode(inp["scales"], "bf16"), _lib_decode(inp["zeros"], "bf16")
    z = zf / s
    assert np.array_equal(z, np.round(z)) and z.min() >= cfg.z_lo and z.max() <= cfg.z_hi
    assert len(np.unique(z)) > 3                     # zero points vary over groups and columns
    A = torch.from_numpy(inp["A"].view(np.int16)).view(torch.bfloat16).double().numpy()
    out_f, _ = orc.group_gemm_zf(A, inp["q"].astype(np.int64), zf, s, cfg.G)
    out_i = orc.group_gemm(A, inp["q"].astype(np.int64), z.astype(np.int64), s, cfg.G)
    mag = orc.group_gemm_magnitude(A, inp["q"].astype(np.int64), z.astype(np.int64), s, cfg.G)
    assert np.allclose(out_f, out_i, rtol=0, atol=1e-12 * float(mag.max()))


def test_float_zero_enters_through_the_group_sums_of_the_activations():
    """out(zf) − out(0) = −Σ_g (Σ_{k∈g} A[m][k]) · zf[g][n]: the sign, the group of each k and
    the column of each zero point (group sums by a numpy reshape)."""
    rng = np.random.default_rng(4)
    M, K, N, G = 3, 128, 6, 32
    A = rng.standard_normal((M, K))
    q = rng.integers(0, 16, (K, N))
    s = rng.uniform(0.005, 0.02, (K // G, N))
    zf = rng.uniform(-0.2, 0.2, (K // G, N))
    out, _ = orc.group_gemm_zf(A, q, zf, s, G)
    out0, _ = orc.group_gemm_zf(A, q, np.zeros_like(zf), s, G)
    gsum = A.reshape(M, K // G, G).sum(axis=2)
    assert np.allclose(out - out0, -(gsum @ zf), rtol=1e-12, atol=1e-12)


def test_float_zero_pins_catch_a_planted_sign_error(monkeypatch):
    real = orc.group_gemm_zf
    monkeypatch.setattr(orc, "group_gemm_zf", lambda A, q, zf, s, G: real(A, q, -np.asarray(zf), s, G))
    with pytest.raises(AssertionError):
        test_float_zero_enters_through_the_group_sums_of_the_activations()


# ------------------------------------------------------------------ FP8 block-scaled GEMM

def test_e4m3_decoder_matches_library_on_all_patterns():
    bits = np.arange(256, dtype=np.uint8)
    lib = torch.from_numpy(bits).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = orc.e4m3_bits_to_f64(bits)
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    ok = ~np.isnan(lib)
    assert np.array_equal(ours[ok], lib[ok])
    assert np.nanmax(ours) == 448.0 and orc.e4m3_bits_to_f64(0x01) == 2.0 ** -9


def test_fp8_block_gemm_matches_brute_force_and_block_scaling():
    rng = np.random.default_rng(2)
    M, K, N = 3, 256, 136                          # two k blocks, two weight row blocks
    A = rng.integers(0, 256, (M, K)).astype(np.uint8)
    W = rng.integers(0, 256, (N, K)).astype(np.uint8)
    A[(A & 0x7F) == 0x7F] = 0x38                   # no NaN patterns (0x38 = 1.0)
    W[(W & 0x7F) == 0x7F] = 0x38
    a_s = rng.uniform(0.01, 0.1, (K // 128, M)).astype(np.float32)
    w_s = rng.uniform(0.01, 0.1, (2, K // 128)).astype(np.float32)
    out, mag = orc.fp8_block_gemm(A, a_s, W, w_s)
    Af, Wf = orc.e4m3_bits_to_f64(A), orc.e4m3_bits_to_f64(W)
    for m in range(M):
        for n in (0, 7, 127, 128, 135):
            exact = sum(Fraction(float(a_s[k // 128, m])) * Fraction(float(w_s[n // 128, k // 128])) *
                        Fraction(Af[m, k]) * Fraction(Wf[n, k]) for k in range(K))
            assert abs(out[m, n] - float(exact)) <= 1e-12 * mag[m, n]
    # doubling one block's activation scales doubles exactly that block's share
    a2 = a_s.copy()
    a2[1] *= 2
    out2, _ = orc.fp8_block_gemm(A, a2, W, w_s)
    one_block, _ = orc.fp8_block_gemm(A[:, 128:], a_s[1:], W[:, 128:], w_s[:, 1:])
    assert np.allclose(out2 - out, one_block, rtol=1e-12, atol=1e-12)


def test_e4m3_encoder_matches_library_rounding_and_saturates():
    """Inside ±448 the encoder is torch's round-to-nearest-even cast; beyond, it saturates;
    every code decodes back to itself."""
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.normal(0, 30, 20000), rng.uniform(-448, 448, 20000),
                        orc.e4m3_bits_to_f64(np.arange(0x7F))])
    # midpoints between neighbouring codes: ties go to the even code
    grid = orc.e4m3_bits_to_f64(np.arange(0x7F))
    x = np.concatenate([x, (grid[1:] + grid[:-1]) / 2, -(grid[1:] + grid[:-1]) / 2])
    ours = orc.f64_to_e4m3_bits(x)
    lib = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, lib)
    assert orc.f64_to_e4m3_bits(np.array([1000.0, -1e6]))[0] == 0x7E
    assert orc.f64_to_e4m3_bits(np.array([-1e6]))[0] == 0xFE
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(orc.f64_to_e4m3_bits(orc.e4m3_bits_to_f64(codes)), codes)


def test_fp8_activation_quantizer_block_maximum_and_error_bound():
    cfg = gq_synth.Config("q8f", M=3, K=512, N=16, G=128, outlier_frac=0.01)
    A = gq_synth.make_activations(cfg, seed=6)
    Aq, s = orc.quantize_act_fp8(A, "bf16")
    x = orc.bf16_bits_to_f64(A).reshape(3, 4, 128)
    q = orc.e4m3_bits_to_f64(Aq).reshape(3, 4, 128)
    ss = s.T.astype(np.float64)[:, :, None]
    assert (np.abs(q).max(axis=2) == 448.0).all()        # each block's largest element
    # E4M3 has 3 mantissa bits: the relative error of a normal code is at most 2^-4
    assert (np.abs(x - ss * q) <= np.abs(x) * 2.0 ** -4 + ss * 2.0 ** -10).all()


# ------------------------------------------------------------------ the tolerance's magnitude term
#
# Every GPU parity bound is 2^-8·|ref| + 1e-4·mag (bf16) or 1e-5·|ref| + 1e-6·mag (fp32), so an
# inflated mag would silently loosen every parity test.  These pins compute mag term by term
# (exact rational sums of |A[m][k]·W_hat[k][n]| from the generator's raw codes and library
# decoders) and require equality to float64 rounding: a mag that is too large fails as surely
# as one that is too small.  P1 section 8: the error of the K-term sum scales with the size of
# the terms it adds, not with the size of the result.

def _lib_act(inp, act):
    if act == "bf16":
        return torch.from_numpy(inp["A"].view(np.int16)).view(torch.bfloat16).double().numpy()
    return inp["A"].astype(np.float64)


def _exact_abs_sum(terms):
    return float(sum((abs(Fraction(float(t))) for t in terms), Fraction(0)))


def _brute_mag(cfg, inp):
    s = _lib_decode(inp["scales"], cfg.sc)
    A = _lib_act(inp, cfg.act)
    q = inp["q"].astype(np.int64)
    z = inp["z"] if inp["z"] is not None else None
    z0 = 8 if cfg.w4 else 0
    M = A.shape[0]
    mag = np.zeros((M, cfg.N))
    for m in range(M):
        for n in range(cfg.N):
            terms = []
            for k in range(cfg.K):
                g = k // cfg.G
                zz = int(z[g, n]) if z is not None else z0
                # A·s and the integer (q − z) are exact in float64; |·| of their product is
                # formed as an exact rational
                terms.append(Fraction(float(A[m, k])) * Fraction(float(s[g, n])) * (int(q[k, n]) - zz))
            mag[m, n] = float(sum((abs(t) for t in terms), Fraction(0)))
    return mag


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_magnitude_equals_the_exact_sum_of_absolute_terms(cfg):
    inp = gq_synth.make_inputs(cfg, seed=11)
    _, mag = orc.reference(inp["A"], inp["codes"], inp["scales"], inp["zeros"], K=cfg.K,
                           N=cfg.N, G=cfg.G, w4=cfg.w4, act=cfg.act, sc=cfg.sc)
    exact = _brute_mag(cfg, inp)
    assert np.allclose(mag, exact, rtol=1e-13, atol=0)


def _mutant_mag_doubled(A, q, z, s, G):
    return 2.0 * _REAL_MAG(A, q, z, s, G)


def _mutant_mag_abs_code(A, q, z, s, G):
    # |q| in place of |q − z|
    return _REAL_MAG(A, q, np.zeros_like(z), s, G)


def _mutant_mag_abs_after_sum(A, q, z, s, G):
    # |Σ| in place of Σ|·|: the magnitude collapses to |ref| where the terms cancel
    return np.abs(orc.group_gemm(A, q, z, s, G))


_REAL_MAG = orc.gq_oracle.group_gemm_magnitude


@pytest.mark.parametrize("mutant", [_mutant_mag_doubled, _mutant_mag_abs_code,
                                    _mutant_mag_abs_after_sum])
def test_magnitude_pin_catches_planted_mistakes(mutant, monkeypatch):
    cfg = SMALL[1]                                  # asymmetric zero points, several groups
    inp = gq_synth.make_inputs(cfg, seed=11)
    exact = _brute_mag(cfg, inp)
    monkeypatch.setattr(orc.gq_oracle, "group_gemm_magnitude", mutant)
    _, mag = orc.gq_oracle.reference(inp["A"], inp["codes"], inp["scales"], inp["zeros"],
                                     K=cfg.K, N=cfg.N, G=cfg.G, w4=True, act=cfg.act, sc=cfg.sc)
    assert not np.allclose(mag, exact, rtol=1e-6, atol=0)


def test_a8_magnitude_equals_the_exact_sum_of_absolute_terms():
    rng = np.random.default_rng(12)
    M, K, N, G = 3, 96, 7, 32
    Aq = rng.integers(-127, 128, (M, K)).astype(np.int8)
    q = rng.integers(-127, 128, (K, N)).astype(np.int8)
    a_s = rng.uniform(0.01, 0.1, (M, K // G)).astype(np.float32)
    s = rng.uniform(1e-3, 1e-2, (K // G, N)).astype(np.float32)
    _, mag = orc.reference_a8(Aq, a_s, q, s, K=K, N=N, G=G)
    for m in range(M):
        for n in range(N):
            exact = _exact_abs_sum(
                float(Fraction(float(a_s[m, k // G])) * Fraction(float(s[k // G, n])) *
                      int(Aq[m, k]) * int(q[k, n])) for k in range(K))
            assert mag[m, n] == pytest.approx(exact, rel=1e-13)
    # planted: the magnitude of the group sums (|Σ|) is not the sum of magnitudes
    out, _ = orc.reference_a8(Aq, a_s, q, s, K=K, N=N, G=G)
    assert (mag > np.abs(out) * (1 + 1e-3)).any()


@pytest.mark.parametrize("cfg", ZF_SMALL, ids=lambda c: c.name)
def test_float_zero_magnitude_equals_the_exact_sum_of_absolute_terms(cfg):
    inp = gq_synth.make_inputs(cfg, seed=5)
    _, mag = orc.reference(inp["A"], inp["codes"], inp["scales"], inp["zeros"], K=cfg.K,
                           N=cfg.N, G=cfg.G, w4=True, act=cfg.act, sc=cfg.sc, zp_float=True)
    s, zf = _lib_decode(inp["scales"], cfg.sc), _lib_decode(inp["zeros"], cfg.sc)
    A = _lib_act(inp, cfg.act)
    q = inp["q"]
    for m in range(A.shape[0]):
        for n in range(cfg.N):
            exact = sum((abs(Fraction(float(A[m, k])) *
                             (int(q[k, n]) * Fraction(float(s[k // cfg.G, n])) -
                              Fraction(float(zf[k // cfg.G, n]))))
                         for k in range(cfg.K)), Fraction(0))
            # W_hat = q·s − zf is formed in float64 first (one rounding per weight)
            assert mag[m, n] == pytest.approx(float(exact), rel=1e-13)


def test_fp8_magnitude_equals_the_exact_sum_of_absolute_terms():
    rng = np.random.default_rng(21)
    M, K, N = 2, 256, 136
    A = rng.integers(0, 256, (M, K)).astype(np.uint8)
    W = rng.integers(0, 256, (N, K)).astype(np.uint8)
    A[(A & 0x7F) == 0x7F] = 0x38
    W[(W & 0x7F) == 0x7F] = 0x38
    a_s = rng.uniform(0.01, 0.1, (K // 128, M)).astype(np.float32)
    w_s = rng.uniform(0.01, 0.1, (2, K // 128)).astype(np.float32)
    _, mag = orc.fp8_block_gemm(A, a_s, W, w_s)
    Af = torch.from_numpy(A).view(torch.float8_e4m3fn).double().numpy()
    Wf = torch.from_numpy(W).view(torch.float8_e4m3fn).double().numpy()
    for m in range(M):
        for n in (0, 1, 127, 128, 135):
            exact = sum((abs(Fraction(float(a_s[k // 128, m])) * Fraction(float(w_s[n // 128, k // 128])) *
                             Fraction(float(Af[m, k])) * Fraction(float(Wf[n, k])))
                         for k in range(K)), Fraction(0))
            assert mag[m, n] == pytest.approx(float(exact), rel=1e-13)


def test_silu_derivative_bound_is_tight():
    """|silu'(x)| = |σ(x)·(1 + x·(1 − σ(x)))| peaks just below 1.1 (about 1.0998 near x ≈ 2.4),
    so the factor 1.1 of the SiLU-and-mul magnitude is an upper bound, and 1.0 would not be.
    The derivative is taken by central differences of silu itself."""
    x = np.linspace(-30, 30, 600001)
    h = 1e-6
    d = (orc.silu(x + h) - orc.silu(x - h)) / (2 * h)
    assert np.max(np.abs(d)) < 1.1
    assert np.max(np.abs(d)) > 1.099


def test_silu_mul_magnitude_bounds_the_propagated_gemm_error(monkeypatch):
    """First-order propagation: if gate and up each carry an error up to ε·(their own mag),
    silu(gate)·up moves by at most ε·mag_out (+ O(ε²)).  The gate and up values are planted
    through a stand-in for the GEMM: worst-case signs, gate at the steepest point of silu."""
    gvals = np.array([[2.3994, -1.0, 0.5, 8.0]])
    uvals = np.array([[3.0, -2.0, 7.0, 0.25]])
    mg = np.array([[40.0, 5.0, 2.0, 1.0]])
    mu = np.array([[10.0, 3.0, 30.0, 2.0]])

    def fake_reference(A_raw, codes, scales, zeros, *, K, N, G, w4, act, sc, rows=None, cols=None,
                       zp_float=False):
        cols = np.asarray(cols)
        if cols[0] < N // 2:
            return gvals[:, cols], mg[:, cols]
        return uvals[:, cols - N // 2], mu[:, cols - N // 2]

    monkeypatch.setattr(orc.gq_oracle, "reference", fake_reference)
    ref, mag = orc.gq_oracle.silu_mul_reference(None, None, None, None, K=128, N=8, G=128,
                                                act="bf16", sc="fp16")
    eps = 1e-7
    worst = np.zeros_like(ref)
    for sg in (-1, 1):
        for su in (-1, 1):
            g2 = gvals + sg * eps * mg
            u2 = uvals + su * eps * mu
            worst = np.maximum(worst, np.abs(orc.silu(g2) * u2 - ref))
    assert (worst <= eps * mag * (1 + 1e-4)).all()
    # planted: without the 1.1 the bound fails at the steepest point of silu
    mag_no_factor = mg * np.abs(uvals) + np.abs(orc.silu(gvals)) * mu
    assert (worst > eps * mag_no_factor * (1 + 1e-4)).any()


def test_dequantize_matches_the_element_by_element_loop():
    cfg = gq_synth.Config("dq", M=1, K=128, N=16, G=32, zp=True, sc="bf16")
    inp = gq_synth.make_weights(cfg, seed=3)
    s = _lib_decode(inp["scales"], "bf16")
    W = orc.dequantize(inp["q"].astype(np.int64), inp["z"].astype(np.int64), s, cfg.G)
    brute = np.array(orc.dequantize_brute(inp["q"], inp["z"], s, cfg.G, cfg.K, cfg.N))
    assert np.array_equal(W, brute)
    # and the group GEMM is A @ W_hat (one product per weight, no reassociation in W_hat)
    A = np.random.default_rng(1).standard_normal((3, cfg.K))
    out = orc.group_gemm(A, inp["q"].astype(np.int64), inp["z"].astype(np.int64), s, cfg.G)
    assert np.allclose(out, A @ W, rtol=1e-12, atol=1e-12)
