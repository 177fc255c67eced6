"""Parity of the CUDA path with the float64 oracle (GPU).

Every test calls the library through its C ABI (ctypes) on seeded synthetic inputs and
compares element by element with the oracle: per element
  bf16 out: |gpu - ref| <= 2^-8 |ref| + 1e-4 mag,   fp32 out: |gpu - ref| <= 1e-5 |ref| + 1e-6 mag
with mag = Σ_k |A[m][k] w[k][n]|.  Integer-valued activations with power-of-two scales make
every partial sum exact, and there the output must equal the oracle bit for bit.
"""
import numpy as np
import pytest

import gq_synth
import oracle
from helpers import alloc_out, load, np_to_dev, out_to_f64, prec_of, run_gemm

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return load()


def _oracle(cfg, inp, rows=None, cols=None):
    return oracle.reference(inp["A"], inp["codes"], inp["scales"], inp["zeros"], K=cfg.K,
                            N=cfg.N, G=cfg.G, w4=cfg.w4, act=cfg.act, sc=cfg.sc, rows=rows,
                            cols=cols, zp_float=cfg.zf)


def _assert_parity(cfg, got, ref, mag):
    assert np.isfinite(got).all()
    bad, ratio = oracle.check(got, ref, mag, cfg.out)
    assert bad == 0, f"{cfg.name}: {bad} elements out of tolerance (worst err/tol {ratio:.3g})"
    return ratio


def _full_case(gq, cfg, seed=0):
    inp = gq_synth.make_inputs(cfg, seed=seed)
    out, _ = run_gemm(gq, cfg, inp)
    ref, mag = _oracle(cfg, inp)
    return _assert_parity(cfg, out_to_f64(out, cfg.out), ref, mag)


# ------------------------------------------------------------------ small, full compare

W4_SHAPES = [
    gq_synth.Config("w4_tiny", M=1, K=512, N=512, G=128),
    gq_synth.Config("w4_single_group", M=2, K=128, N=64, G=128),
    gq_synth.Config("w4_ragged_n", M=3, K=1024, N=264, G=128),
    gq_synth.Config("w4_g32", M=5, K=512, N=136, G=32, zp=True, sc="bf16"),
    gq_synth.Config("w4_g64_f32scale", M=4, K=768, N=128, G=64, sc="f32"),
    gq_synth.Config("w4_g256", M=1, K=2048, N=96, G=256, zp=True),
    gq_synth.Config("w4_out_f32", M=7, K=1024, N=80, G=128, out="f32"),
    gq_synth.Config("w4_outliers", M=1, K=4096, N=2048, G=128, outlier_frac=0.001),
    gq_synth.Config("w4_asym_m16", M=16, K=8192, N=512, G=128, zp=True, sc="bf16"),
    # small-batch kernel with split K: two row blocks and a ragged last tile; eight slices
    gq_synth.Config("w4_m40_g32_split", M=40, K=4096, N=264, G=32, zp=True),
    gq_synth.Config("w4_m24_split_ragged", M=24, K=8192, N=136, G=64, sc="f32", out="f32"),
]


@pytest.mark.parametrize("cfg", W4_SHAPES, ids=lambda c: c.name)
def test_w4_small_shapes(gq, cfg):
    _full_case(gq, cfg)


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 9, 15, 16, 17, 31, 32, 33, 64, 65, 127, 128, 129])
def test_w4_m_sweep(gq, M):
    cfg = gq_synth.Config(f"w4_m{M}", M=M, K=512, N=264, G=128, zp=(M % 2 == 0))
    _full_case(gq, cfg, seed=M)


Q8_SHAPES = [
    gq_synth.Config("q8_m1", M=1, K=2048, N=1024, G=32, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("q8_m3_g64", M=3, K=512, N=136, G=64, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("q8_m33_g128", M=33, K=1024, N=72, G=128, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("q8_bf16_out", M=2, K=256, N=64, G=32, w4=False, act="f32", sc="f32",
                    out="bf16", s_lo=1e-3, s_hi=1e-2),
    # rows padded to the warps' row blocks, several K slices, a ragged last column block
    gq_synth.Config("q8_m12_split", M=12, K=1024, N=200, G=32, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("q8_m24_g256", M=24, K=2048, N=136, G=256, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("q8_m32_g64_bf16", M=32, K=512, N=328, G=64, w4=False, act="f32",
                    sc="f32", out="bf16", s_lo=1e-3, s_hi=1e-2),
    # several column blocks per CTA (the last narrow), K slices of one group for one K part
    gq_synth.Config("q8_m7_g128", M=7, K=1024, N=1000, G=128, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("q8_m20_blocks", M=20, K=2048, N=4040, G=32, w4=False, act="f32",
                    sc="f32", out="f32", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("q8_m24_2blocks", M=24, K=512, N=12248, G=32, w4=False, act="f32",
                    sc="f32", out="f32", s_lo=1e-3, s_hi=1e-2),     # 2 blocks per CTA
    gq_synth.Config("q8_m16_5blocks", M=16, K=1024, N=20008, G=64, w4=False, act="f32",
                    sc="f32", out="bf16", s_lo=1e-3, s_hi=1e-2),    # 5 blocks per CTA
    # the warp-specialized INT8 decode kernel (M <= 4, N a multiple of 64): G = 64 and 128, a
    # padded fourth row, blocks split between warps and CTAs, whole blocks per CTA (304 blocks
    # on 152 SMs, no scratch), a CTA whose later warps hold no unit
    gq_synth.Config("q8g_m2_g64", M=2, K=1024, N=640, G=64, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("q8g_m3_g64", M=3, K=1024, N=640, G=64, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("q8g_m4_g128_bf16", M=4, K=2048, N=448, G=128, w4=False, act="f32",
                    sc="f32", out="bf16", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("q8g_m2_whole_blocks", M=2, K=512, N=19456, G=32, w4=False, act="f32",
                    sc="f32", out="f32", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("q8g_m1_three_units", M=1, K=96, N=64, G=32, w4=False, act="f32",
                    sc="f32", out="f32", s_lo=1e-3, s_hi=1e-2),
]


@pytest.mark.parametrize("cfg", Q8_SHAPES, ids=lambda c: c.name)
def test_q8_small_shapes(gq, cfg):
    _full_case(gq, cfg)


# ------------------------------------------------------------------ exact arithmetic

@pytest.mark.parametrize("M,spread", [(1, 100), (2, 50), (3, 25), (4, 25), (7, 25)])
def test_wide_dynamic_range_activations(gq, M, spread):
    """Activations spread over 2^(2 * spread) within a row: the decode path carries bf16
    activations into fp16 MMA operands by exponent bands, which must stay exact."""
    cfg = gq_synth.Config(f"wide_m{M}", M=M, K=2048, N=264, G=128, zp=(M % 2 == 1),
                          a_kind="wide", a_spread=spread)
    _full_case(gq, cfg, seed=M)


@pytest.mark.parametrize("cfg", [
    gq_synth.Config("exact_w4", M=3, K=4096, N=264, G=128, zp=True, a_kind="int", pow2_scales=True),
    gq_synth.Config("exact_w4_f32out", M=16, K=1024, N=128, G=32, a_kind="int", pow2_scales=True,
                    out="f32", sc="f32"),
    gq_synth.Config("exact_q8", M=2, K=2048, N=256, G=32, w4=False, act="f32", sc="f32", out="f32",
                    a_kind="int", pow2_scales=True),
], ids=lambda c: c.name)
def test_integer_inputs_are_bit_exact(gq, cfg):
    inp = gq_synth.make_inputs(cfg, seed=1)
    out, _ = run_gemm(gq, cfg, inp)
    ref, _ = _oracle(cfg, inp)
    if cfg.out == "bf16":
        h = out.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(h, oracle.f64_to_bf16_bits(ref))
    else:
        assert np.array_equal(out.cpu().numpy().astype(np.float64), ref)


# ------------------------------------------------------------------ large M (tcgen05 path)

PREFILL_SHAPES = [
    gq_synth.Config("pf_base", M=256, K=512, N=256, G=128),
    gq_synth.Config("pf_ragged", M=300, K=1024, N=392, G=128, zp=True, sc="bf16"),
    gq_synth.Config("pf_g64_f32", M=128, K=256, N=136, G=64, sc="f32", out="f32"),
    gq_synth.Config("pf_g256", M=520, K=2048, N=264, G=256, zp=True),
    gq_synth.Config("pf_tall", M=1100, K=512, N=128, G=128, outlier_frac=0.01),
    # the smallest row counts the prefill kernel takes: one 256-row tile, mostly past M
    gq_synth.Config("pf_m33", M=33, K=512, N=136, G=128),
    gq_synth.Config("pf_m64_zp", M=64, K=1024, N=256, G=64, zp=True, sc="bf16", out="f32"),
    # the mid-M tiles: 64- and 128-row activation tiles over the full K = 4096 (64 stages
    # through the ring) with a ragged last 128-column tile, rows past M in the last tile
    gq_synth.Config("pf_m33_k4096", M=33, K=4096, N=1032, G=128, zp=True),
    gq_synth.Config("pf_m64_k4096", M=64, K=4096, N=2056, G=128, outlier_frac=0.001),
    gq_synth.Config("pf_m100_bm128", M=100, K=2048, N=520, G=64, sc="bf16"),
    gq_synth.Config("pf_m128_f32", M=128, K=1024, N=392, G=128, sc="f32", out="f32"),
    gq_synth.Config("pf_m300_ragged", M=300, K=1024, N=392, G=256, zp=True),
]


@pytest.mark.parametrize("cfg", PREFILL_SHAPES, ids=lambda c: c.name)
def test_prefill_shapes(gq, cfg):
    from group_quantized_weight_gb300.constants import prec_flags
    plan = gq.gq_plan(cfg.M, cfg.K, cfg.N, cfg.G, prec_flags(cfg.w4, cfg.zp, cfg.act, cfg.sc, cfg.out))
    assert plan["path"] == 2
    _full_case(gq, cfg)
    assert gq.gq_device_error() == 0


@pytest.mark.parametrize("M,K,N", [(384, 1024, 256), (64, 4096, 1032), (128, 2048, 264)])
def test_prefill_integer_inputs_are_bit_exact(gq, M, K, N):
    """Integer activations and power-of-two scales: every partial sum is exact in FP32, so the
    output equals the oracle bit for bit, unsplit and with K split in four slices."""
    cfg = gq_synth.Config("pf_exact", M=M, K=K, N=N, G=128, zp=True, a_kind="int",
                          pow2_scales=True)
    inp = gq_synth.make_inputs(cfg, seed=2)
    ref, _ = _oracle(cfg, inp)
    try:
        for n in (0, 4):
            gq.gq_set_split_override(n)
            out, _ = run_gemm(gq, cfg, inp)
            h = out.view(torch.int16).cpu().numpy().view(np.uint16)
            assert np.array_equal(h, oracle.f64_to_bf16_bits(ref)), n
    finally:
        gq.gq_set_split_override(0)


def test_prefill_forced_split_counts_match_the_oracle(gq):
    """The tcgen05 kernel's K split at one, two and the largest slice count (16 here), on a
    64-row problem with a ragged last tile."""
    cfg = gq_synth.Config("pf_split", M=64, K=4096, N=392, G=128, zp=True, sc="bf16")
    inp = gq_synth.make_inputs(cfg, seed=9)
    ref, mag = _oracle(cfg, inp)
    prec = prec_of(cfg)
    counts = []
    try:
        for n in (1, 2, -1):
            gq.gq_set_split_override(n)
            plan = gq.gq_plan(cfg.M, cfg.K, cfg.N, cfg.G, prec)
            assert plan["path"] == 2
            counts.append(plan["nsplit"])
            out, _ = run_gemm(gq, cfg, inp)
            _assert_parity(cfg, out_to_f64(out, cfg.out), ref, mag)
    finally:
        gq.gq_set_split_override(0)
    assert counts == [1, 2, 16]
    assert gq.gq_device_error() == 0


# ------------------------------------------------------------------ float zero points

ZF_SHAPES = [
    gq_synth.Config("zf_m1", M=1, K=512, N=264, G=128, zf=True, sc="bf16"),
    gq_synth.Config("zf_m5_g32", M=5, K=1024, N=136, G=32, zf=True),
    gq_synth.Config("zf_m16_split", M=16, K=8192, N=512, G=128, zf=True, sc="bf16"),
    gq_synth.Config("zf_m24_f32", M=24, K=2048, N=200, G=64, zf=True, sc="f32", out="f32"),
    gq_synth.Config("zf_m32_g256", M=32, K=4096, N=152, G=256, zf=True),
    gq_synth.Config("zf_m40_rows", M=40, K=2048, N=264, G=128, zf=True, sc="bf16"),
    gq_synth.Config("zf_m64_g32", M=64, K=1024, N=128, G=32, zf=True, sc="f32", out="f32"),
    gq_synth.Config("zf_outliers", M=8, K=4096, N=512, G=128, zf=True, outlier_frac=0.001),
]


@pytest.mark.parametrize("cfg", ZF_SHAPES, ids=lambda c: c.name)
def test_float_zero_points(gq, cfg):
    _full_case(gq, cfg)


def test_float_zero_points_integer_inputs_are_bit_exact(gq):
    """Integer activations, power-of-two scales and zf = s·z: every group dot, product and
    sum is exact in FP32, so the output equals the oracle bit for bit."""
    cfg = gq_synth.Config("zf_exact", M=16, K=1024, N=128, G=64, zf=True, sc="bf16",
                          a_kind="int", pow2_scales=True, out="f32")
    inp = gq_synth.make_inputs(cfg, seed=3)
    out, _ = run_gemm(gq, cfg, inp)
    ref, _ = _oracle(cfg, inp)
    assert np.array_equal(out.cpu().numpy(), ref.astype(np.float32))


def test_float_zero_points_full_size_sampled_and_repeatable(gq):
    cfg = gq_synth.CONFIGS["asym_m16"].replace(name="asym_m16_zf", zp=False, zf=True)
    inp = gq_synth.make_inputs(cfg, seed=0)
    out, packed = run_gemm(gq, cfg, inp)
    rng = np.random.default_rng(9)
    rows = np.arange(cfg.M)
    cols = np.unique(np.concatenate([[0, 1, 15, 16, cfg.N - 1], rng.choice(cfg.N, 512, replace=False)]))
    ref, mag = _oracle(cfg, inp, rows=rows, cols=cols)
    _assert_parity(cfg, out_to_f64(out, cfg.out)[np.ix_(rows, cols)], ref, mag)
    out2 = alloc_out(cfg.M, cfg.N, cfg.out)
    gq.gemm_t(np_to_dev(inp["A"]), packed, np_to_dev(inp["scales"]), np_to_dev(inp["zeros"]),
              out2, cfg.M, cfg.K, cfg.N, cfg.G, prec_of(cfg))
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


# ------------------------------------------------------------------ the workloads

@pytest.mark.parametrize("name", ["tiny_gemv", "decode_gateup", "q8_m1", "q8_m32"])
def test_workload_full_compare(gq, name):
    _full_case(gq, gq_synth.CONFIGS[name])


@pytest.mark.parametrize("name", ["asym_m16", "prefill"])
def test_workload_sampled(gq, name):
    """Full-size run; the oracle recomputes a sample of rows and columns (ragged edges
    included) one by one."""
    cfg = gq_synth.CONFIGS[name]
    inp = gq_synth.make_inputs(cfg, seed=0)
    out, _ = run_gemm(gq, cfg, inp)
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([[0, cfg.M - 1], rng.choice(cfg.M, min(cfg.M, 24), replace=False)]))
    cols = np.unique(np.concatenate([[0, 1, 127, 128, cfg.N - 1],
                                     rng.choice(cfg.N, 1024, replace=False)]))
    ref, mag = _oracle(cfg, inp, rows=rows, cols=cols)
    got = out_to_f64(out, cfg.out)[np.ix_(rows, cols)]
    _assert_parity(cfg, got, ref, mag)


@pytest.mark.parametrize("name", ["tiny_gemv", "decode_gateup", "asym_m16", "q8_m1", "q8_m32",
                                  "prefill"])
def test_bitwise_deterministic(gq, name):
    cfg = gq_synth.CONFIGS[name]
    inp = gq_synth.make_inputs(cfg, seed=0)
    prec = prec_of(cfg)
    packed = gq.pack_weights_t(np_to_dev(inp["codes"]), cfg.K, cfg.N, cfg.G, prec)
    A, S = np_to_dev(inp["A"]), np_to_dev(inp["scales"])
    Z = np_to_dev(inp["zeros"]) if inp["zeros"] is not None else None
    outs = []
    for _ in range(3):
        o = alloc_out(cfg.M, cfg.N, cfg.out)
        gq.gemm_t(A, packed, S, Z, o, cfg.M, cfg.K, cfg.N, cfg.G, prec)
        outs.append(o)
    torch.cuda.synchronize()
    b = [o.view(torch.int16 if cfg.out == "bf16" else torch.int32) for o in outs]
    assert torch.equal(b[0], b[1]) and torch.equal(b[0], b[2])


# ------------------------------------------------------------------ forced split counts
#
# The z-split of "分组量化 GEMM 内核" section 3.3 partitions K into slices of whole groups and
# adds the slices' partial sums in slice order.  The same problem at one slice, two slices and
# the largest count each path supports must stay within the tolerance of the oracle.

SPLIT_SHAPES = [
    gq_synth.Config("split_w4_batch", M=16, K=2048, N=1032, G=128, zp=True, sc="bf16"),
    gq_synth.Config("split_w4_mma_decode", M=3, K=1088, N=264, G=64),        # K % 256 != 0
    gq_synth.Config("split_w8_block", M=2, K=2048, N=1000, G=32, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("split_w8_mma", M=12, K=512, N=520, G=32, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("split_w8_decode", M=40, K=512, N=264, G=32, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),
]


@pytest.mark.parametrize("cfg", SPLIT_SHAPES, ids=lambda c: c.name)
def test_forced_split_counts_one_two_and_max_match_the_oracle(gq, cfg):
    inp = gq_synth.make_inputs(cfg, seed=7)
    ref, mag = _oracle(cfg, inp)
    prec = prec_of(cfg)
    path = gq.gq_plan(cfg.M, cfg.K, cfg.N, cfg.G, prec)["path"]
    counts = []
    try:
        for n in (1, 2, -1):
            gq.gq_set_split_override(n)
            plan = gq.gq_plan(cfg.M, cfg.K, cfg.N, cfg.G, prec)
            assert plan["path"] == path
            if n > 0:
                assert plan["nsplit"] == n
            counts.append(plan["nsplit"])
            out, _ = run_gemm(gq, cfg, inp)
            _assert_parity(cfg.replace(name=f"{cfg.name}_nsplit{plan['nsplit']}"),
                           out_to_f64(out, cfg.out), ref, mag)
            again, _ = run_gemm(gq, cfg, inp)
            view = torch.int16 if cfg.out == "bf16" else torch.int32
            assert torch.equal(out.view(view), again.view(view))
    finally:
        gq.gq_set_split_override(0)
    assert counts[0] == 1 and counts[1] == 2 and counts[2] > 2


# ------------------------------------------------------------------ layout, API edges

def _unpack_w4_device_layout(packed: np.ndarray, K: int, N: int) -> np.ndarray:
    """Host reading of the documented packed layout (include/gq.h and gq_pack.cu):
    [tile][chunk][lane][word j], pair i of word j = rows L/4 + 8(i&1), k = 16j + 2(L%4)
    + 8(i>>1) + {0, 1} at bits 4i and 4i+16."""
    words = packed.view(np.uint32)
    tiles = (N + 15) // 16
    nch = K // 64
    w = words.reshape(tiles, nch, 32, 4)
    q = np.zeros((K, tiles * 16), dtype=np.int64)
    for lane in range(32):
        for j in range(4):
            for i in range(4):
                r = lane // 4 + 8 * (i & 1)
                kk = 16 * j + 2 * (lane % 4) + 8 * (i >> 1)
                ww = w[:, :, lane, j]                         # [tiles][chunks]
                for e, sh in ((0, 4 * i), (1, 4 * i + 16)):
                    vals = (ww >> sh) & 0xF
                    for t in range(tiles):
                        q[np.arange(nch) * 64 + kk + e, t * 16 + r] = vals[t]
    return q[:, :N]


def test_pack_roundtrip_w4(gq):
    cfg = gq_synth.Config("pack", M=1, K=256, N=40, G=128)
    inp = gq_synth.make_weights(cfg, seed=5)
    from group_quantized_weight_gb300.constants import GQ_W4
    packed = gq.pack_weights_t(np_to_dev(inp["codes"]), cfg.K, cfg.N, cfg.G, GQ_W4)
    q = _unpack_w4_device_layout(packed.cpu().numpy(), cfg.K, cfg.N)
    assert np.array_equal(q, inp["q"].astype(np.int64))


def _unpack_w8_device_layout(packed: np.ndarray, K: int, N: int) -> np.ndarray:
    """Inverse of the W8 device layout: 64-column blocks one after another, each holding its
    K/16 rows of 16-byte chunks (16 consecutive k of one column) contiguously; the last
    block is N mod 64 columns wide when N is not a multiple of 64."""
    flat = packed.view(np.int8).reshape(-1)
    q = np.empty((K, N), dtype=np.int8)
    off = 0
    for n0 in range(0, N, 64):
        wb = min(64, N - n0)
        blk = flat[off:off + (K // 16) * wb * 16].reshape(K // 16, wb, 16)
        q[:, n0:n0 + wb] = blk.transpose(0, 2, 1).reshape(K, wb)
        off += (K // 16) * wb * 16
    assert off == K * N
    return q


def test_pack_roundtrip_w8(gq):
    cfg = gq_synth.Config("pack8", M=1, K=64, N=152, G=32, w4=False, act="f32", sc="f32",
                          out="f32")   # two full column blocks and one of 24 columns
    inp = gq_synth.make_weights(cfg, seed=5)
    from group_quantized_weight_gb300.constants import GQ_ACT_F32, GQ_SC_F32
    packed = gq.pack_weights_t(np_to_dev(inp["codes"]), cfg.K, cfg.N, cfg.G, GQ_ACT_F32 | GQ_SC_F32)
    q = _unpack_w8_device_layout(packed.cpu().numpy(), cfg.K, cfg.N)
    assert np.array_equal(q, inp["q"])


def test_empty_problem_leaves_output_untouched(gq):
    from group_quantized_weight_gb300.constants import GQ_W4
    o = torch.full((4, 16), 3.0, dtype=torch.bfloat16, device="cuda")
    d = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    assert gq.gq_gemm(0, 512, 16, 128, GQ_W4, d.data_ptr(), d.data_ptr(), d.data_ptr(), None,
                      o.data_ptr(), None) == 0
    torch.cuda.synchronize()
    assert (o == 3.0).all()


def test_misaligned_pointer_is_rejected_on_device(gq):
    from group_quantized_weight_gb300.constants import GQ_W4
    d = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    base = d.data_ptr()
    assert gq.gq_gemm(1, 512, 16, 128, GQ_W4, base + 2, base, base, None, base, None) == 3


def test_user_workspace_matches_library_workspace(gq):
    cfg = gq_synth.CONFIGS["decode_gateup"].replace(N=4096)
    inp = gq_synth.make_inputs(cfg, seed=2)
    ref_out, packed = run_gemm(gq, cfg, inp)
    prec = prec_of(cfg)
    need = gq.gq_workspace_size(cfg.M, cfg.K, cfg.N, cfg.G, prec)
    assert need > 0
    A, S = np_to_dev(inp["A"]), np_to_dev(inp["scales"])
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    try:
        assert gq.gq_set_workspace(small.data_ptr(), 256) == 0
        o = alloc_out(cfg.M, cfg.N, cfg.out)
        st = gq.gq_gemm(cfg.M, cfg.K, cfg.N, cfg.G, prec, A.data_ptr(), packed.data_ptr(),
                        S.data_ptr(), None, o.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert st == 4                                             # GQ_ERR_WORKSPACE
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        assert gq.gq_set_workspace(ws.data_ptr(), need) == 0
        for _ in range(2):
            o = alloc_out(cfg.M, cfg.N, cfg.out)
            gq.gemm_t(A, packed, S, None, o, cfg.M, cfg.K, cfg.N, cfg.G, prec)
            torch.cuda.synchronize()
            assert torch.equal(o.view(torch.int16), ref_out.view(torch.int16))
    finally:
        assert gq.gq_set_workspace(None, 0) == 0


def test_graph_capture_of_gemm(gq):
    """gq_gemm enqueues only kernels (after its scratch exists), so it can be captured."""
    cfg = gq_synth.CONFIGS["tiny_gemv"]
    inp = gq_synth.make_inputs(cfg, seed=0)
    ref_out, packed = run_gemm(gq, cfg, inp)
    prec = prec_of(cfg)
    A, S = np_to_dev(inp["A"]), np_to_dev(inp["scales"])
    o = alloc_out(cfg.M, cfg.N, cfg.out)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        gq.gemm_t(A, packed, S, None, o, cfg.M, cfg.K, cfg.N, cfg.G, prec)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), ref_out.view(torch.int16))


# ------------------------------------------------------------------ static-weight launches

@pytest.mark.parametrize("cfg", [
    gq_synth.Config("static_stripe_m1", M=1, K=4096, N=4096, G=128),
    gq_synth.Config("static_batch_m16", M=16, K=8192, N=512, G=128, zp=True, sc="bf16"),
    gq_synth.Config("static_q8_m12", M=12, K=1024, N=200, G=32, w4=False, act="f32",
                    sc="f32", out="f32", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("static_q8g_m1", M=1, K=2048, N=1024, G=32, w4=False, act="f32",
                    sc="f32", out="f32", s_lo=1e-3, s_hi=1e-2),
], ids=lambda c: c.name)
def test_static_weight_flag_gives_the_same_bits(gq, cfg):
    """GQ_STATIC_W lets a kernel stream its weights before the preceding kernel on the stream
    has ended; the activations still wait for it.  Back-to-back calls, the second one's
    activations written by a kernel just before it, give the bits of the plain calls."""
    from group_quantized_weight_gb300.constants import GQ_STATIC_W
    inp = gq_synth.make_inputs(cfg, seed=6)
    prec = prec_of(cfg)
    packed = gq.pack_weights_t(np_to_dev(inp["codes"]), cfg.K, cfg.N, cfg.G, prec)
    A = np_to_dev(inp["A"])
    S = np_to_dev(inp["scales"])
    Z = np_to_dev(inp["zeros"]) if inp["zeros"] is not None else None
    ref = alloc_out(cfg.M, cfg.N, cfg.out)
    gq.gemm_t(A, packed, S, Z, ref, cfg.M, cfg.K, cfg.N, cfg.G, prec)
    got = [alloc_out(cfg.M, cfg.N, cfg.out) for _ in range(3)]
    A2 = torch.zeros_like(A)
    for o in got:
        A2.zero_()
        A2.copy_(A)                      # written on the stream right before the call
        gq.gemm_t(A2, packed, S, Z, o, cfg.M, cfg.K, cfg.N, cfg.G, prec | GQ_STATIC_W)
    torch.cuda.synchronize()
    view = torch.int16 if cfg.out == "bf16" else torch.int32
    for o in got:
        assert torch.equal(o.view(view), ref.view(view))


# ------------------------------------------------------------------ fused gate+up epilogue

GATE_UP_SHAPES = [
    gq_synth.Config("gu_m1", M=1, K=1024, N=512, G=128),
    gq_synth.Config("gu_m3_zp", M=3, K=2048, N=1024, G=128, zp=True, sc="bf16"),
    gq_synth.Config("gu_m8_f32", M=8, K=512, N=272, G=64, sc="f32", out="f32"),
    # 128 tiles on 152 SMs: CTAs split tiles, so the cross-CTA reduction stores the epilogue
    gq_synth.Config("gu_m1_split", M=1, K=4096, N=2048, G=128, outlier_frac=0.001),
    gq_synth.Config("gu_m5_g32", M=5, K=1024, N=320, G=32, zp=True),
    # the small-batch kernel: one slice, K split into slices, two row blocks, fp32 scales
    gq_synth.Config("gu_m16_zp", M=16, K=2048, N=1056, G=128, zp=True, sc="bf16"),
    gq_synth.Config("gu_m12_split_f32", M=12, K=8192, N=288, G=64, sc="f32", out="f32"),
    gq_synth.Config("gu_m40_g32_split", M=40, K=4096, N=544, G=32, zp=True),
    gq_synth.Config("gu_m33_g64", M=33, K=1024, N=160, G=64),
    # INT8 codes (Q8_0 form): the warp-specialized kernel (M <= 4), the CUDA-core block kernel
    # (G = 256) and the tensor-core one, with and without a K split, fp32 and bf16 output
    gq_synth.Config("gu_q8_m1", M=1, K=2048, N=1024, G=32, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("gu_q8_m2_g256", M=2, K=2048, N=128, G=256, w4=False, act="f32",
                    sc="f32", out="f32", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("gu_q8_m3_split", M=3, K=2048, N=128, G=32, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("gu_q8_m12", M=12, K=1024, N=640, G=32, w4=False, act="f32", sc="f32",
                    out="bf16", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("gu_q8_m32_g64", M=32, K=2048, N=256, G=64, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),
]


def _gate_up_case(gq, cfg, seed, cols=None):
    from group_quantized_weight_gb300.constants import GQ_GATE_UP
    inp = gq_synth.make_inputs(cfg, seed=seed)
    prec = prec_of(cfg) | GQ_GATE_UP
    packed = gq.pack_weights_t(np_to_dev(inp["codes"]), cfg.K, cfg.N, cfg.G, prec)
    A, S = np_to_dev(inp["A"]), np_to_dev(inp["scales"])
    Z = np_to_dev(inp["zeros"]) if inp["zeros"] is not None else None
    out = alloc_out(cfg.M, cfg.N // 2, cfg.out)
    gq.gemm_t(A, packed, S, Z, out, cfg.M, cfg.K, cfg.N, cfg.G, prec)
    torch.cuda.synchronize()
    got = out_to_f64(out, cfg.out)
    ref, mag = oracle.silu_mul_reference(inp["A"], inp["codes"], inp["scales"], inp["zeros"],
                                         K=cfg.K, N=cfg.N, G=cfg.G, act=cfg.act, sc=cfg.sc,
                                         cols=cols, w4=cfg.w4)
    if cols is not None:
        got = got[:, cols]
    return _assert_parity(cfg, got, ref, mag), (A, packed, S, Z, prec)


@pytest.mark.parametrize("cfg", GATE_UP_SHAPES, ids=lambda c: c.name)
def test_gate_up_silu_mul(gq, cfg):
    _gate_up_case(gq, cfg, seed=7)


def test_gate_up_full_size_sampled_and_repeatable(gq):
    """The fused gate+up GEMV at the decode size (N = 2·14336), 512 sampled output columns
    against the oracle; a second call gives the same bits."""
    cfg = gq_synth.CONFIGS["decode_gateup"]
    cols = np.random.default_rng(11).choice(cfg.N // 2, 512, replace=False)
    _, (A, packed, S, Z, prec) = _gate_up_case(gq, cfg, seed=0, cols=cols)
    o1 = alloc_out(cfg.M, cfg.N // 2, cfg.out)
    o2 = alloc_out(cfg.M, cfg.N // 2, cfg.out)
    gq.gemm_t(A, packed, S, Z, o1, cfg.M, cfg.K, cfg.N, cfg.G, prec)
    gq.gemm_t(A, packed, S, Z, o2, cfg.M, cfg.K, cfg.N, cfg.G, prec)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_gate_up_small_batch_full_size_sampled_and_repeatable(gq):
    """The fused gate+up GEMM at the asymmetric small-batch size (M = 16, K = 8192,
    N = 2·14336, INT4 zero points), 384 sampled output columns of every row against the
    oracle; a second call gives the same bits."""
    cfg = gq_synth.CONFIGS["asym_m16"]
    cols = np.random.default_rng(12).choice(cfg.N // 2, 384, replace=False)
    _, (A, packed, S, Z, prec) = _gate_up_case(gq, cfg, seed=0, cols=cols)
    assert gq.gq_plan(cfg.M, cfg.K, cfg.N, cfg.G, prec)["path"] == 4
    o1 = alloc_out(cfg.M, cfg.N // 2, cfg.out)
    o2 = alloc_out(cfg.M, cfg.N // 2, cfg.out)
    gq.gemm_t(A, packed, S, Z, o1, cfg.M, cfg.K, cfg.N, cfg.G, prec)
    gq.gemm_t(A, packed, S, Z, o2, cfg.M, cfg.K, cfg.N, cfg.G, prec)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_gate_up_q8_full_size_sampled_and_repeatable(gq):
    """The fused gate+up Q8_0 GEMM at its full size (K = 2048, N = 2·6144, G = 32) for one and
    32 rows, 512 sampled output columns against the oracle; a second call gives the same bits."""
    for name in ("q8_m1", "q8_m32"):
        cfg = gq_synth.CONFIGS[name]
        cols = np.random.default_rng(13).choice(cfg.N // 2, 512, replace=False)
        _, (A, packed, S, Z, prec) = _gate_up_case(gq, cfg, seed=0, cols=cols)
        o1 = alloc_out(cfg.M, cfg.N // 2, cfg.out)
        o2 = alloc_out(cfg.M, cfg.N // 2, cfg.out)
        gq.gemm_t(A, packed, S, Z, o1, cfg.M, cfg.K, cfg.N, cfg.G, prec)
        gq.gemm_t(A, packed, S, Z, o2, cfg.M, cfg.K, cfg.N, cfg.G, prec)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2)


def test_pack_gate_up_interleaves_gate_and_up_columns(gq):
    """Tile t of the gate+up packing holds gate columns 8t .. 8t+7 and up columns
    N/2 + 8t .. N/2 + 8t + 7, each in the plain packed tile format."""
    from group_quantized_weight_gb300.constants import GQ_GATE_UP, GQ_W4
    cfg = gq_synth.Config("pgu", M=1, K=128, N=64, G=128)
    inp = gq_synth.make_weights(cfg, seed=8)
    packed = gq.pack_weights_t(np_to_dev(inp["codes"]), cfg.K, cfg.N, cfg.G, GQ_W4 | GQ_GATE_UP)
    qp = _unpack_w4_device_layout(packed.cpu().numpy(), cfg.K, cfg.N)   # packed column order
    F = cfg.N // 2
    order = np.concatenate([np.r_[8 * t:8 * t + 8, F + 8 * t:F + 8 * t + 8]
                            for t in range(cfg.N // 16)])
    assert np.array_equal(qp, inp["q"].astype(np.int64)[:, order])


# ------------------------------------------------------------------ INT8-activation variant

def _a8_inputs(cfg, seed):
    """W8 weights of cfg plus its fp32 activations, quantized by the oracle."""
    inp = gq_synth.make_inputs(cfg, seed=seed)
    Aq, As = oracle.quantize_act_i8(inp["A"], cfg.G, cfg.act)
    return inp, Aq, As


@pytest.mark.parametrize("act", ["f32", "bf16"])
def test_activation_quantizer_is_bit_exact(gq, act):
    from group_quantized_weight_gb300.constants import GQ_ACT_F32
    cfg = gq_synth.Config("aq", M=5, K=1024, N=16, G=32, w4=False, act=act, sc="f32",
                          outlier_frac=0.01)
    A = gq_synth.make_activations(cfg, seed=3)
    A[1, 32:64] = 0                                # a group of zeros
    if act == "f32":                               # ties: largest magnitude 127, halves
        A[2, :32] = np.arange(32, dtype=np.float32) + 0.5
        A[2, 0] = 127.0
    Aq_ref, As_ref = oracle.quantize_act_i8(A, cfg.G, act)
    Aq, As = gq.quantize_act_t(np_to_dev(A), cfg.K, cfg.G, GQ_ACT_F32 if act == "f32" else 0)
    torch.cuda.synchronize()
    assert np.array_equal(Aq.cpu().numpy(), Aq_ref)
    assert np.array_equal(As.cpu().numpy().view(np.uint32), As_ref.view(np.uint32))


A8_SHAPES = [
    gq_synth.Config("a8_m1", M=1, K=2048, N=1024, G=32, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("a8_m3_g64", M=3, K=512, N=136, G=64, w4=False, act="f32", sc="f32",
                    out="bf16", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("a8_m16_split", M=16, K=2048, N=1000, G=32, w4=False, act="f32",
                    sc="f32", out="f32", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("a8_m40_rows", M=40, K=1024, N=328, G=128, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("a8_m32_g256", M=32, K=2048, N=200, G=256, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),
    # the warp-specialized decode kernel (N a multiple of 64, M <= 4): G = 64 with bf16
    # output, a padded fourth row at G = 128, whole blocks per CTA (304 blocks, no scratch)
    gq_synth.Config("a8g_m2_g64_bf16", M=2, K=1024, N=640, G=64, w4=False, act="f32",
                    sc="f32", out="bf16", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("a8g_m3_g128", M=3, K=2048, N=448, G=128, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("a8g_m4_whole_blocks", M=4, K=512, N=19456, G=32, w4=False, act="f32",
                    sc="f32", out="f32", s_lo=1e-3, s_hi=1e-2),
    gq_synth.Config("a8g_m1_g128", M=1, K=2048, N=448, G=128, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),
]


@pytest.mark.parametrize("cfg", A8_SHAPES, ids=lambda c: c.name)
def test_a8_group_gemm(gq, cfg):
    from group_quantized_weight_gb300.constants import GQ_ACT_I8, GQ_OUT_F32, GQ_SC_F32
    inp, Aq, As = _a8_inputs(cfg, seed=9)
    prec = GQ_ACT_I8 | GQ_SC_F32 | (GQ_OUT_F32 if cfg.out == "f32" else 0)
    packed = gq.pack_weights_t(np_to_dev(inp["codes"]), cfg.K, cfg.N, cfg.G, prec)
    out = alloc_out(cfg.M, cfg.N, cfg.out)
    gq.gemm_a8_t(np_to_dev(Aq), np_to_dev(As), packed, np_to_dev(inp["scales"]), out,
                 cfg.M, cfg.K, cfg.N, cfg.G, prec)
    torch.cuda.synchronize()
    ref, mag = oracle.reference_a8(Aq, As, inp["codes"], inp["scales"], K=cfg.K, N=cfg.N,
                                   G=cfg.G)
    _assert_parity(cfg, out_to_f64(out, cfg.out), ref, mag)


def test_a8_quantize_then_gemm_and_integer_exactness(gq):
    """gq_quantize_act feeding gq_gemm_a8 on the device equals the oracle's chain; with
    power-of-two scales and integer activations the result is exact and equal bit for bit."""
    from group_quantized_weight_gb300.constants import GQ_ACT_F32, GQ_ACT_I8, GQ_OUT_F32, GQ_SC_F32
    cfg = gq_synth.Config("a8_chain", M=4, K=1024, N=264, G=32, w4=False, act="f32", sc="f32",
                          out="f32", s_lo=1e-3, s_hi=1e-2)
    inp = gq_synth.make_inputs(cfg, seed=12)
    prec = GQ_ACT_I8 | GQ_SC_F32 | GQ_OUT_F32
    packed = gq.pack_weights_t(np_to_dev(inp["codes"]), cfg.K, cfg.N, cfg.G, prec)
    Aq, As = gq.quantize_act_t(np_to_dev(inp["A"]), cfg.K, cfg.G, GQ_ACT_F32)
    out = alloc_out(cfg.M, cfg.N, "f32")
    gq.gemm_a8_t(Aq, As, packed, np_to_dev(inp["scales"]), out, cfg.M, cfg.K, cfg.N, cfg.G, prec)
    torch.cuda.synchronize()
    Aq_r, As_r = oracle.quantize_act_i8(inp["A"], cfg.G, "f32")
    ref, mag = oracle.reference_a8(Aq_r, As_r, inp["codes"], inp["scales"], K=cfg.K, N=cfg.N,
                                   G=cfg.G)
    _assert_parity(cfg, out_to_f64(out, "f32"), ref, mag)
    # exact case: activation codes in [-8, 8], scales 2^-4 or 2^-3 and 2^-6 or 2^-5: every
    # product and partial sum is a multiple of 2^-10 below 2^11 (21 bits), exact in FP32
    rng = np.random.default_rng(4)
    Aq_i = rng.integers(-8, 9, (cfg.M, cfg.K)).astype(np.int8)
    As_i = np.ldexp(1.0, rng.integers(-4, -2, (cfg.M, cfg.K // cfg.G))).astype(np.float32)
    S_i = np.ldexp(1.0, rng.integers(-6, -4, (cfg.K // cfg.G, cfg.N))).astype(np.float32)
    out_i = alloc_out(cfg.M, cfg.N, "f32")
    gq.gemm_a8_t(np_to_dev(Aq_i), np_to_dev(As_i), packed, np_to_dev(S_i), out_i, cfg.M, cfg.K,
                 cfg.N, cfg.G, prec)
    torch.cuda.synchronize()
    ref_i, _ = oracle.reference_a8(Aq_i, As_i, inp["codes"], S_i, K=cfg.K, N=cfg.N, G=cfg.G)
    assert np.array_equal(out_to_f64(out_i, "f32"), ref_i)


def test_a8_decode_kernel_integer_inputs_exact_and_repeatable(gq):
    """The warp-specialized decode kernel's W8A8 form (N a multiple of 64): integer inputs
    with power-of-two scales give the oracle's exact result bit for bit, and the Q8_0 M=1
    workload gives the same bits call after call."""
    from group_quantized_weight_gb300.constants import GQ_ACT_I8, GQ_OUT_F32, GQ_SC_F32
    prec = GQ_ACT_I8 | GQ_SC_F32 | GQ_OUT_F32
    cfg = gq_synth.Config("a8g_exact", M=3, K=1024, N=256, G=32, w4=False, act="f32",
                          sc="f32", out="f32", s_lo=1e-3, s_hi=1e-2)
    assert gq.gq_plan(cfg.M, cfg.K, cfg.N, cfg.G, prec)["path"] == 9
    inp = gq_synth.make_inputs(cfg, seed=13)
    packed = gq.pack_weights_t(np_to_dev(inp["codes"]), cfg.K, cfg.N, cfg.G, prec)
    rng = np.random.default_rng(5)
    Aq_i = rng.integers(-8, 9, (cfg.M, cfg.K)).astype(np.int8)
    As_i = np.ldexp(1.0, rng.integers(-4, -2, (cfg.M, cfg.K // cfg.G))).astype(np.float32)
    S_i = np.ldexp(1.0, rng.integers(-6, -4, (cfg.K // cfg.G, cfg.N))).astype(np.float32)
    out_i = alloc_out(cfg.M, cfg.N, "f32")
    gq.gemm_a8_t(np_to_dev(Aq_i), np_to_dev(As_i), packed, np_to_dev(S_i), out_i, cfg.M, cfg.K,
                 cfg.N, cfg.G, prec)
    torch.cuda.synchronize()
    ref_i, _ = oracle.reference_a8(Aq_i, As_i, inp["codes"], S_i, K=cfg.K, N=cfg.N, G=cfg.G)
    assert np.array_equal(out_to_f64(out_i, "f32"), ref_i)
    full = gq_synth.CONFIGS["q8_m1"]
    assert gq.gq_plan(full.M, full.K, full.N, full.G, prec)["path"] == 9
    inp, Aq, As = _a8_inputs(full, seed=2)
    packed = gq.pack_weights_t(np_to_dev(inp["codes"]), full.K, full.N, full.G, prec)
    Aq_d, As_d, S = np_to_dev(Aq), np_to_dev(As), np_to_dev(inp["scales"])
    outs = []
    for _ in range(3):
        o = alloc_out(full.M, full.N, "f32")
        gq.gemm_a8_t(Aq_d, As_d, packed, S, o, full.M, full.K, full.N, full.G, prec)
        outs.append(o.view(torch.int32))
    torch.cuda.synchronize()
    assert gq.gq_device_error(clear=True) == 0
    assert all(torch.equal(outs[0], x) for x in outs[1:])
    ref, mag = oracle.reference_a8(Aq, As, inp["codes"], inp["scales"], K=full.K, N=full.N,
                                   G=full.G)
    _assert_parity(full.replace(name="a8g_q8_m1"), out_to_f64(outs[0].view(torch.float32), "f32"),
                   ref, mag)


# ------------------------------------------------------------------ FP8 block-scaled GEMM

def _fp8_inputs(M, K, N, seed):
    """E4M3 activations ~N(0, 1) and weights ~N(0, 0.25) as bytes (torch's round to nearest
    E4M3), activation scales U[0.01, 0.1] per (128-k block, row), weight scales U[0.01, 0.1]
    per 128 x 128 block."""
    g = torch.Generator().manual_seed(seed)
    A = torch.randn(M, K, generator=g).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    W = (0.5 * torch.randn(N, K, generator=g)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    rng = np.random.default_rng(seed)
    a_s = rng.uniform(0.01, 0.1, (K // 128, M)).astype(np.float32)
    w_s = rng.uniform(0.01, 0.1, (-(-N // 128), K // 128)).astype(np.float32)
    return A, a_s, W, w_s


@pytest.mark.parametrize("M,K,N,out", [
    (256, 128, 128, "bf16"),        # one tile, one block
    (300, 512, 400, "bf16"),        # ragged rows and columns
    (1, 256, 256, "bf16"),          # a single activation row
    (1024, 1024, 640, "f32"),       # several tiles per CTA
    (700, 384, 128, "f32"),
])
def test_fp8_block_gemm(gq, M, K, N, out):
    from group_quantized_weight_gb300.constants import GQ_OUT_F32
    A, a_s, W, w_s = _fp8_inputs(M, K, N, seed=M + K + N)
    o = alloc_out(M, N, out)
    gq.gemm_fp8_t(np_to_dev(A), np_to_dev(a_s), np_to_dev(W), np_to_dev(w_s), o, M, K, N,
                  GQ_OUT_F32 if out == "f32" else 0)
    torch.cuda.synchronize()
    assert gq.gq_device_error(clear=True) == 0
    ref, mag = oracle.fp8_block_gemm(A, a_s, W, w_s)
    cfg = gq_synth.Config(f"fp8_{M}x{K}x{N}", M=M, K=K, N=N, G=128, out=out)
    _assert_parity(cfg, out_to_f64(o, out), ref, mag)


def test_a8_and_fp8_paths_are_bitwise_repeatable(gq):
    """The W8A8 group GEMM at the Q8_0 M=32 workload (split K, fixed-order reduction) and the
    FP8 block-scaled GEMM on a multi-tile shape give the same bits call after call."""
    from group_quantized_weight_gb300.constants import GQ_ACT_I8, GQ_OUT_F32, GQ_SC_F32
    cfg = gq_synth.CONFIGS["q8_m32"]
    inp, Aq, As = _a8_inputs(cfg, seed=0)
    prec = GQ_ACT_I8 | GQ_SC_F32 | GQ_OUT_F32
    packed = gq.pack_weights_t(np_to_dev(inp["codes"]), cfg.K, cfg.N, cfg.G, prec)
    Aq_d, As_d, S = np_to_dev(Aq), np_to_dev(As), np_to_dev(inp["scales"])
    outs = []
    for _ in range(3):
        o = alloc_out(cfg.M, cfg.N, "f32")
        gq.gemm_a8_t(Aq_d, As_d, packed, S, o, cfg.M, cfg.K, cfg.N, cfg.G, prec)
        outs.append(o.view(torch.int32))
    M, K, N = 1024, 4096, 4096
    A, a_s, W, w_s = _fp8_inputs(M, K, N, seed=21)
    A_d, as_d, W_d, ws_d = np_to_dev(A), np_to_dev(a_s), np_to_dev(W), np_to_dev(w_s)
    f8 = []
    for _ in range(3):
        o = alloc_out(M, N, "bf16")
        gq.gemm_fp8_t(A_d, as_d, W_d, ws_d, o, M, K, N, 0)
        f8.append(o.view(torch.int16))
    torch.cuda.synchronize()
    assert gq.gq_device_error(clear=True) == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    assert torch.equal(f8[0], f8[1]) and torch.equal(f8[0], f8[2])


@pytest.mark.parametrize("act", ["bf16", "f32"])
def test_fp8_activation_quantizer_is_bit_exact(gq, act):
    from group_quantized_weight_gb300.constants import GQ_ACT_F32
    cfg = gq_synth.Config("q8f", M=7, K=1024, N=16, G=128, w4=False, act=act, sc="f32",
                          outlier_frac=0.01)
    A = gq_synth.make_activations(cfg, seed=8)
    A[2, 128:256] = 0                              # a block of zeros
    if act == "f32":
        A[3, 0] = -0.0
    Aq_ref, s_ref = oracle.quantize_act_fp8(A, act)
    Aq, s = gq.quantize_act_fp8_t(np_to_dev(A), cfg.K, GQ_ACT_F32 if act == "f32" else 0)
    torch.cuda.synchronize()
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(Aq.cpu().numpy(), Aq_ref)


def test_fp8_quantize_then_gemm(gq):
    """bf16 activations quantized on the device, then the block-scaled FP8 GEMM, against the
    oracle's quantizer and GEMM."""
    M, K, N = 200, 512, 384
    cfg = gq_synth.Config("fp8chain", M=M, K=K, N=N, G=128)
    A = gq_synth.make_activations(cfg, seed=10)
    _, _, W, w_s = _fp8_inputs(M, K, N, seed=10)
    Aq, a_s = gq.quantize_act_fp8_t(np_to_dev(A), K, 0)
    o = alloc_out(M, N, "bf16")
    gq.gemm_fp8_t(Aq, a_s, np_to_dev(W), np_to_dev(w_s), o, M, K, N, 0)
    torch.cuda.synchronize()
    Aq_r, a_s_r = oracle.quantize_act_fp8(A, "bf16")
    ref, mag = oracle.fp8_block_gemm(Aq_r, a_s_r, W, w_s)
    _assert_parity(cfg, out_to_f64(o, "bf16"), ref, mag)


@pytest.mark.parametrize("cfg", [
    gq_synth.Config("host_gemv", M=1, K=4096, N=2048, G=128),
    gq_synth.Config("host_asym_f32", M=3, K=1024, N=264, G=128, zp=True, sc="bf16", out="f32"),
    gq_synth.Config("host_prefill", M=200, K=1024, N=392, G=64),
    gq_synth.Config("host_q8_f32", M=2, K=1024, N=384, G=32, w4=False, act="f32", sc="f32",
                    out="f32"),
], ids=lambda c: c.name)
def test_host_buffer_call_matches_the_device_call(gq, cfg):
    """gq_gemm_host on page-locked host activations and output: the same bits as gq_gemm on
    device buffers, and the oracle's values."""
    inp = gq_synth.make_inputs(cfg, seed=4)
    out_dev_ref, packed = run_gemm(gq, cfg, inp)
    ref, mag = _oracle(cfg, inp)
    prec = prec_of(cfg)
    a = np.ascontiguousarray(inp["A"])
    a = a.view(np.int16) if a.dtype == np.uint16 else a
    A_h = torch.from_numpy(a).pin_memory()
    A_d = torch.empty(A_h.shape, dtype=A_h.dtype, device="cuda")
    S = np_to_dev(inp["scales"])
    Z = np_to_dev(inp["zeros"]) if inp["zeros"] is not None else None
    out_d = alloc_out(cfg.M, cfg.N, cfg.out)
    out_h = torch.empty(tuple(out_d.shape), dtype=out_d.dtype).pin_memory()
    st = gq.gq_gemm_host(cfg.M, cfg.K, cfg.N, cfg.G, prec, A_h.data_ptr(), A_d.data_ptr(),
                         packed.data_ptr(), S.data_ptr(), Z.data_ptr() if Z is not None else None,
                         out_d.data_ptr(), out_h.data_ptr(),
                         torch.cuda.current_stream().cuda_stream)
    assert st == 0, gq.gq_status_string(st)
    torch.cuda.synchronize()
    assert torch.equal(out_h.view(torch.int16 if cfg.out != "f32" else torch.int32),
                       out_dev_ref.cpu().view(torch.int16 if cfg.out != "f32" else torch.int32))
    _assert_parity(cfg, out_to_f64(out_h, cfg.out), ref, mag)
    assert gq.gq_device_error() == 0
