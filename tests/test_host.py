"""Host-side checks of libgq (CPU only): the library loads and exports every symbol of
include/gq.h, argument validation, the launch plan, the z-split and the work model."""
import os
import re

import pytest

import gq_synth
from helpers import ROOT, load

gq = load()
from group_quantized_weight_gb300 import constants as C  # noqa: E402


def _header_functions():
    src = open(os.path.join(ROOT, "include", "gq.h"), encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(gq_\w+)\s*\(", src, flags=re.M)))


def test_library_exports_every_declared_function():
    import ctypes
    names = _header_functions()
    assert len(names) >= 10
    lib = ctypes.CDLL(gq.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(gq.EXPORTED)


def test_binding_flags_and_statuses_match_the_header():
    """Every GQ_* constant the binding defines has the header's value, and the reverse."""
    src = open(os.path.join(ROOT, "include", "gq.h"), encoding="utf-8").read()
    flags = {m.group(1): int(m.group(2), 16)
             for m in re.finditer(r"#define\s+(GQ_\w+)\s+0x([0-9a-fA-F]+)", src)}
    statuses = {m.group(1): int(m.group(2))
                for m in re.finditer(r"\b(GQ_(?:OK|ERR_\w+))\s*=\s*(\d+)", src)}
    assert len(flags) >= 10 and "GQ_ZP_FLOAT" in flags
    for name, val in flags.items():
        assert getattr(C, name) == val, name
    for name, val in statuses.items():
        assert C.STATUS_NAMES[val] == name
    binding = {n for n in dir(C) if n.startswith("GQ_") and isinstance(getattr(C, n), int)
               and n not in ("GQ_OK",)}
    assert binding <= set(flags), binding - set(flags)


def test_status_strings():
    assert gq.gq_status_string(0) == "ok"
    for s in range(1, 8):
        assert gq.gq_status_string(s) not in ("ok", "unknown status")


def test_zsplit_is_the_pages_partition():
    """The z-split of the group-wise GEMM blog (section 3.3): contiguous, disjoint,
    covering, sizes differing by at most one, larger slices first."""
    for units in (1, 2, 5, 32, 64, 97):
        for nsplit in range(1, min(units, 70) + 1):
            spans = [gq.gq_zsplit(units, nsplit, z) for z in range(nsplit)]
            assert spans[0][0] == 0 and spans[-1][1] == units
            for (b0, e0), (b1, e1) in zip(spans, spans[1:]):
                assert e0 == b1
            sizes = [e - b for b, e in spans]
            assert max(sizes) - min(sizes) <= 1 and sizes == sorted(sizes, reverse=True)
            base, rem = divmod(units, nsplit)
            assert sizes.count(base + 1) == rem
    with pytest.raises(C.GqError):
        gq.gq_zsplit(4, 0, 0)


def test_packed_bytes():
    assert gq.gq_packed_bytes(4096, 28672, 128, C.GQ_W4) == 4096 * 28672 // 2
    assert gq.gq_packed_bytes(512, 24, 128, C.GQ_W4) == 512 * 32 // 2        # padded to 2 tiles
    assert gq.gq_packed_bytes(2048, 12288, 32, C.GQ_ACT_F32 | C.GQ_SC_F32) == 2048 * 12288


@pytest.mark.parametrize("args,status", [
    ((1, 4096, 28672, 100, C.GQ_W4), 2),          # G outside {32, 64, 128, 256}
    ((1, 4000, 512, 32, C.GQ_W4), 2),             # W4 needs K % 64 == 0
    ((1, 192, 512, 128, C.GQ_W4), 1),             # K % G != 0
    ((1, 512, 12, 128, C.GQ_W4), 1),              # N % 8 != 0
    ((1, 512, 16, 128, C.GQ_W4 | C.GQ_SC_BF16 | C.GQ_SC_F32), 1),
    ((1, 512, 16, 128, C.GQ_W4 | C.GQ_ACT_F32), 2),
    ((1, 512, 16, 32, C.GQ_ZP | C.GQ_ACT_F32 | C.GQ_SC_F32), 1),   # INT8 has no zero point
    ((1, 512, 16, 32, C.GQ_ACT_F32), 2),          # INT8 needs fp32 scales
    ((-1, 512, 16, 128, C.GQ_W4), 1),
    ((1, 512, 16, 128, 0x400), 1),                # unknown flag
])
def test_invalid_calls_are_rejected_before_any_launch(args, status):
    """No device exists here: an invalid call must return its status before touching one."""
    M, K, N, G, prec = args
    st = gq.gq_gemm(M, K, N, G, prec, 16, 16, 16, None, 16, None)
    assert st == status
    with pytest.raises(C.GqError) as e:
        gq.gq_plan(M, K, N, G, prec, sm_count=152)
    assert e.value.status == status


def test_null_and_misaligned_pointers():
    assert gq.gq_gemm(1, 512, 16, 128, C.GQ_W4, None, 16, 16, None, 16, None) == 1
    assert gq.gq_gemm(1, 512, 16, 128, C.GQ_W4, 8, 16, 16, None, 16, None) == 3
    # zero points passed without GQ_ZP (and the reverse)
    assert gq.gq_gemm(1, 512, 16, 128, C.GQ_W4, 16, 16, 16, 16, 16, None) == 1
    assert gq.gq_gemm(1, 512, 16, 128, C.GQ_W4 | C.GQ_ZP, 16, 16, 16, None, 16, None) == 1
    assert gq.gq_pack_weights(512, 16, 128, C.GQ_W4, 8, 16, None) == 3
    # empty problems are valid and launch nothing
    assert gq.gq_gemm(0, 512, 16, 128, C.GQ_W4, 16, 16, 16, None, 16, None) == 0
    assert gq.gq_gemm(4, 512, 0, 128, C.GQ_W4, 16, 16, 16, None, 16, None) == 0


def test_host_buffer_call_checks_its_arguments_before_any_copy():
    """gq_gemm_host: a NULL host buffer, a NULL or misaligned device buffer and a bad shape
    come back as statuses before anything is issued (no device is touched for them here);
    an empty problem is a no-op."""
    W4 = C.GQ_W4
    h = gq.gq_gemm_host
    assert h(1, 512, 16, 128, W4, None, 16, 16, 16, None, 16, 16, None) == 1     # A_host
    assert h(1, 512, 16, 128, W4, 16, 16, 16, 16, None, 16, None, None) == 1     # out_host
    assert h(1, 500, 16, 128, W4, 16, 16, 16, 16, None, 16, 16, None) != 0       # K % G
    assert h(1, 512, 16, 128, W4 | C.GQ_ACT_I8, 16, 16, 16, 16, None, 16, 16, None) != 0
    assert h(1, 512, 16, 128, W4, 16, None, 16, 16, None, 16, 16, None) == 1     # A_dev
    assert h(1, 512, 16, 128, W4, 16, 8, 16, 16, None, 16, 16, None) == 3        # alignment
    assert h(0, 512, 16, 128, W4, None, None, None, None, None, None, None, None) == 0



def _q8_row_blocks(M):
    """Row blocks of 8 rows a CTA of the INT8 CUDA-core kernel splits M rows into."""
    rb = 1
    while rb * 8 < M:
        rb *= 2
    return rb


@pytest.mark.parametrize("name", list(gq_synth.CONFIGS))
def test_plan_is_a_pure_function_of_shape(name):
    cfg = gq_synth.CONFIGS[name]
    from helpers import prec_of
    p1 = gq.gq_plan(cfg.M, cfg.K, cfg.N, cfg.G, prec_of(cfg), sm_count=152)
    p2 = gq.gq_plan(cfg.M, cfg.K, cfg.N, cfg.G, prec_of(cfg), sm_count=152)
    assert p1 == p2
    units = cfg.K // max(cfg.G, 64 if cfg.w4 else cfg.G)
    if p1["path"] == 2:
        # tcgen05 prefill: persistent, at most one CTA per SM; one CTA holds the shared-memory
        # ring (at most 227 KiB per CTA on sm_103a); activation tiles of 64, 128 or 256 rows;
        # scratch only with a K split
        assert cfg.M >= (33 if cfg.zp else 25) and cfg.w4
        assert 1 <= p1["grid_x"] <= 152
        assert p1["m_tile"] == (64 if cfg.M <= 64 else 128 if cfg.M <= 128 else 256)
        assert (p1["workspace_bytes"] > 0) == (p1["nsplit"] > 1)
        assert p1["smem_bytes"] <= 227 * 1024
        return
    if p1["path"] == 3:
        # striped decode: one CTA per SM at most, each over a contiguous range of (tile,
        # 256-k slot) pairs; whole tiles per CTA need no scratch, equal slot ranges need
        # per-CTA partial sums and per-tile counters
        tiles = (cfg.N + 15) // 16
        assert cfg.M <= 8 and cfg.K % 256 == 0
        assert 1 <= p1["grid_x"] <= min(152, tiles * cfg.K // 256)
        assert p1["nsplit"] == p1["grid_x"]
        assert p1["smem_bytes"] <= 227 * 1024
        if p1["workspace_bytes"]:
            assert p1["workspace_bytes"] >= p1["grid_x"] * 8 * 16 * 4 + 4 * tiles
        else:
            assert tiles >= 152
        return
    if p1["path"] == 8:
        # warp-specialized decode (M <= 4): a producer warp and eight consumer warps per CTA,
        # at most one CTA per SM in the grid; two fit on an SM where the shape allows, so the
        # next call's CTAs can start while this call's finish
        tiles = (cfg.N + 15) // 16
        assert cfg.M <= 4 and cfg.K % 256 == 0
        assert p1["block_threads"] == 17 * 32
        assert 1 <= p1["grid_x"] <= min(152, tiles * cfg.K // 256)
        assert p1["nsplit"] == p1["grid_x"]
        assert p1["smem_bytes"] <= 227 * 1024
        if p1["workspace_bytes"]:
            assert p1["workspace_bytes"] >= p1["grid_x"] * 2 * 4 * 16 * 4 + 4 * tiles
        else:
            assert tiles >= 152
        return
    if p1["path"] == 9:
        # warp-specialized INT8 decode (M <= 4, N a multiple of 64): a producer warp and
        # sixteen consumer warps per CTA over (64-column block, group) units, at most one CTA
        # per SM; whole blocks per CTA need no scratch, equal unit ranges per-CTA partial sums
        # and per-block counters
        blocks = cfg.N // 64
        units = blocks * (cfg.K // cfg.G)
        assert not cfg.w4 and cfg.M <= 4 and cfg.N % 64 == 0
        assert p1["block_threads"] == 17 * 32
        assert 1 <= p1["grid_x"] <= min(152, units)
        assert p1["nsplit"] == p1["grid_x"] and p1["n_tile"] == 64
        assert p1["smem_bytes"] <= 227 * 1024 - 1024 - 256
        if p1["workspace_bytes"]:
            assert p1["workspace_bytes"] >= p1["grid_x"] * 2 * 4 * 64 * 4 + 4 * blocks
        else:
            assert blocks >= 152
        return
    if p1["path"] == 4:
        # small-batch kernel: (K slice, tile range) CTAs x 32-row blocks, at most one wave
        assert 1 <= cfg.M <= 64 and cfg.K % 256 == 0
        ks = p1["nsplit"]
        assert cfg.K % ks == 0 and (cfg.K // ks) % 256 == 0
        assert min(cfg.M, 32) * (cfg.K // ks) * 2 <= 64 * 1024
        assert p1["grid_z"] == -(-cfg.M // 32)
        assert p1["grid_x"] * p1["grid_z"] <= 152
        assert p1["smem_bytes"] <= 227 * 1024
        if ks > 1:
            assert p1["workspace_bytes"] >= ks * cfg.M * cfg.N * 4
        return
    if p1["path"] == 5:
        # INT8 CUDA-core kernel (M <= 4): 64 columns x one K slice of whole groups per CTA, two CTAs
        # per SM (at most 113 KiB of shared memory each), every warp of a split CTA with a
        # group; up to 8 rows the fewest slices that fit
        assert not cfg.w4 and 1 <= cfg.M <= 4
        ks = p1["nsplit"]
        groups = cfg.K // cfg.G
        assert 1 <= ks <= groups
        assert ks == 1 or groups // ks >= 8 // _q8_row_blocks(cfg.M)
        assert p1["n_tile"] == 64 and p1["grid_x"] == -(-cfg.N // 64) * ks
        assert p1["block_threads"] == 256 and p1["grid_y"] == p1["grid_z"] == 1
        assert p1["smem_bytes"] <= 113 * 1024
        if cfg.M <= 8 and cfg.M * cfg.K * 4 + 8 * 8 * 1024 <= 113 * 1024:
            assert ks == 1
        if ks > 1:
            assert p1["workspace_bytes"] >= ks * cfg.M * cfg.N * 4
        else:
            assert p1["workspace_bytes"] == 0
        return
    if p1["path"] == 6:
        # INT8 on tensor cores: one K slice x some 64-column blocks per CTA (about one wave of
        # two CTAs per SM), 8 warps = 4 MMA tiles of 16 columns x 2 K parts, three BF16
        # activation planes of 8-row blocks in shared memory
        assert not cfg.w4 and 5 <= cfg.M <= 32
        ks = p1["nsplit"]
        groups = cfg.K // cfg.G
        assert 1 <= ks <= groups and (ks == 1 or groups // ks >= 2)
        assert p1["n_tile"] % 64 == 0 and p1["grid_x"] == -(-cfg.N // p1["n_tile"]) * ks
        assert p1["m_tile"] == -(-cfg.M // 8) * 8
        assert p1["smem_bytes"] <= 113 * 1024
        assert p1["smem_bytes"] >= 3 * p1["m_tile"] * (-(-groups // ks) * cfg.G) * 2
        if ks > 1:
            assert p1["workspace_bytes"] >= ks * cfg.M * cfg.N * 4
        return
    assert p1["smem_bytes"] <= 200 * 1024
    assert 1 <= p1["nsplit"] <= units
    assert p1["grid_y"] == p1["nsplit"]
    assert p1["grid_x"] * p1["n_tile"] >= cfg.N
    assert p1["grid_z"] * p1["m_tile"] >= cfg.M
    if p1["nsplit"] == 1:
        assert p1["workspace_bytes"] == 0
    else:
        assert p1["workspace_bytes"] >= p1["nsplit"] * cfg.M * cfg.N * 4


def test_decode_plan_fills_the_machine():
    cfg = gq_synth.CONFIGS["decode_gateup"]
    p = gq.gq_plan(cfg.M, cfg.K, cfg.N, cfg.G, C.GQ_W4, sm_count=152)
    assert p["path"] == 8 and p["block_threads"] == 17 * 32
    assert p["grid_x"] == 152
    # 1792 tiles over 152 SMs: whole tiles per CTA (11 or 12), no scratch
    assert p["workspace_bytes"] == 0
    # five to eight rows take the striped kernel
    assert gq.gq_plan(5, cfg.K, cfg.N, cfg.G, C.GQ_W4, sm_count=152)["path"] == 3
    # activations too large for the decode kernels' shared memory: the small-batch kernel
    assert gq.gq_plan(4, 32768, 28672, 128, C.GQ_W4, sm_count=152)["path"] == 4


def test_small_batch_plan_warps_follow_the_rows_and_fill_one_wave():
    """The small-batch kernel runs as many warps as its registers allow without spills (32 up
    to 8 rows, 24 up to 16, 16 above), one CTA per SM, K slices x tile ranges = #SM."""
    zp = C.GQ_W4 | C.GQ_ZP | C.GQ_SC_BF16
    for M, warps in ((9, 24), (16, 24), (17, 16), (32, 16)):
        p = gq.gq_plan(M, 8192, 28672, 128, zp, sm_count=152)
        assert p["path"] == 4 and p["block_threads"] == 32 * warps, (M, p)
        assert p["grid_x"] * p["grid_z"] <= 152 and p["grid_x"] >= 150
        assert p["smem_bytes"] <= 226 * 1024
    # float zero points take the same kernel from one row: 32 warps up to 8 rows
    p = gq.gq_plan(1, 4096, 28672, 128, zp & ~C.GQ_ZP | C.GQ_ZP_FLOAT, sm_count=152)
    assert p["path"] == 4 and p["block_threads"] == 32 * 32
    # the asymmetric M=16 workload: 4 K slices of 2048 x 38 tile ranges, split-K scratch
    p = gq.gq_plan(16, 8192, 28672, 128, zp, sm_count=152)
    assert (p["nsplit"], p["grid_x"]) == (4, 152)
    assert p["workspace_bytes"] >= 4 * 16 * 28672 * 4


def test_q8_decode_plan_partitions_block_group_units():
    """INT8 rows M <= 4 with N a multiple of 64: the warp-specialized kernel, one CTA per SM at
    most over contiguous (64-column block, group) ranges; the split override (a K-slice
    count) does not apply to it."""
    W8 = C.GQ_ACT_F32 | C.GQ_SC_F32 | C.GQ_OUT_F32
    # the Q8_0 projection: 192 blocks x 64 groups on 152 SMs, equal unit ranges
    p = gq.gq_plan(1, 2048, 12288, 32, W8, sm_count=152)
    assert p["path"] == 9 and p["grid_x"] == 152 and p["workspace_bytes"] > 0
    # 304 blocks: two whole blocks per CTA, no scratch
    p = gq.gq_plan(2, 1024, 304 * 64, 64, W8, sm_count=152)
    assert p["path"] == 9 and p["grid_x"] == 152 and p["workspace_bytes"] == 0
    # a small shape (4 blocks x 16 groups): at least two units per consumer warp
    p = gq.gq_plan(2, 512, 256, 32, W8, sm_count=152)
    assert p["path"] == 9 and p["grid_x"] == 2
    # not taken: N not a multiple of 64, G of 256, five rows, activations too wide
    assert gq.gq_plan(1, 2048, 1000, 32, W8, sm_count=152)["path"] == 5
    assert gq.gq_plan(1, 2048, 1024, 256, W8, sm_count=152)["path"] == 5
    assert gq.gq_plan(3, 2048, 1024, 32, W8, sm_count=152)["path"] == 9
    assert gq.gq_plan(5, 2048, 1024, 32, W8, sm_count=152)["path"] == 6
    assert gq.gq_plan(2, 32768, 1024, 32, W8, sm_count=152)["path"] == 5
    # the GPU parity shapes named q8g_* and the gate+up ones meant for it take this kernel
    for M, K, N, G in ((3, 1024, 640, 64), (4, 2048, 448, 128), (2, 512, 19456, 32),
                       (1, 96, 64, 32)):
        assert gq.gq_plan(M, K, N, G, W8, sm_count=152)["path"] == 9, (M, K, N, G)
    assert gq.gq_plan(2, 512, 19456, 32, W8, sm_count=152)["workspace_bytes"] == 0
    gu = W8 | C.GQ_GATE_UP
    assert gq.gq_plan(1, 2048, 1024, 32, gu, sm_count=152)["path"] == 9
    assert gq.gq_plan(3, 2048, 128, 32, gu, sm_count=152)["path"] == 9
    assert gq.gq_plan(2, 2048, 128, 256, gu, sm_count=152)["path"] == 5
    prev = gq.gq_set_split_override(2)
    try:
        q = gq.gq_plan(1, 2048, 12288, 32, W8, sm_count=152)
        assert q["path"] == 9 and q["grid_x"] == 152
    finally:
        gq.gq_set_split_override(prev)


def test_small_decode_plan_splits_slots_between_ctas():
    p = gq.gq_plan(1, 4096, 1024, 128, C.GQ_W4, sm_count=152)
    assert p["path"] == 8
    assert p["grid_x"] == -(-64 * 16 // 32)      # 64 tiles x 16 slots, two slots per consumer
    assert p["workspace_bytes"] > 0
    p = gq.gq_plan(6, 4096, 1024, 128, C.GQ_W4, sm_count=152)
    assert p["path"] == 3
    warps = p["block_threads"] // 32
    assert p["grid_x"] == -(-64 * 16 // warps)   # one slot per warp or more
    assert p["workspace_bytes"] > 0


def test_algorithmic_bytes_match_the_worked_figures():
    # configurations' byte counts, and the page's M=1 N=K=4096 INT4 GEMV (8 MiB of
    # weights + 256 KiB of fp16 scales, plus 8 KiB of activations and 8 KiB of output)
    assert C.algorithmic_bytes(1, 4096, 28672, 128, True, False, "bf16", "fp16", "bf16") == 60620800
    assert C.algorithmic_bytes(1, 512, 512, 128, True, False, "bf16", "fp16", "bf16") == 137216
    assert C.algorithmic_bytes(1, 2048, 12288, 32, False, False, "f32", "f32", "f32") == 28368896
    assert C.algorithmic_bytes(16, 8192, 28672, 128, True, True, "bf16", "bf16", "bf16") == 123207680
    assert C.algorithmic_bytes(4096, 4096, 14336, 128, True, False, "bf16", "fp16", "bf16") == 181272576
    assert C.algorithmic_bytes(1, 4096, 4096, 128, True, False, "bf16", "fp16", "bf16") == \
        (8 << 20) + (256 << 10) + 8192 + 8192
    assert C.gemm_flops(4096, 4096, 14336) == 481036337152


def test_gate_up_flag_is_validated_and_planned_on_the_decode_kernels():
    gu = C.GQ_W4 | C.GQ_GATE_UP
    # N must hold whole 16-column tiles of 8 gate and 8 up columns (W4) or whole 64-column
    # blocks of 32 and 32 (W8)
    W8GU = C.GQ_ACT_F32 | C.GQ_SC_F32 | C.GQ_GATE_UP
    assert gq.gq_gemm(1, 512, 24, 128, gu, 16, 16, 16, None, 16, None) == 1
    assert gq.gq_gemm(1, 512, 32, 32, W8GU, 16, 16, 16, None, 16, None) == 1
    # INT8: the warp-specialized kernel up to four rows (the CUDA-core block kernel where it
    # does not take the shape), the tensor-core one to 32; not above
    for M in (1, 2, 3, 4):
        assert gq.gq_plan(M, 2048, 12288, 32, W8GU, sm_count=152)["path"] == 9
    assert gq.gq_plan(2, 2048, 12288, 256, W8GU, sm_count=152)["path"] == 5
    assert gq.gq_plan(1, 2048, 12224, 32, W8GU, sm_count=152)["path"] == 9
    assert gq.gq_plan(32, 2048, 12288, 32, W8GU, sm_count=152)["path"] == 6
    with pytest.raises(C.GqError) as e:
        gq.gq_plan(33, 2048, 12288, 32, W8GU, sm_count=152)
    assert e.value.status == 2
    # the decode and small-batch kernels (K % 256 == 0) carry the epilogue: the
    # warp-specialized one up to four rows, the striped one to eight, the small-batch one to
    # 64 rows; not the prefill kernel, which would take 25 rows and more without it
    assert gq.gq_plan(1, 4096, 28672, 128, gu, sm_count=152)["path"] == 8
    assert gq.gq_plan(1, 4096, 2048, 128, gu, sm_count=152)["path"] == 8
    assert gq.gq_plan(8, 1024, 512, 64, gu | C.GQ_ZP, sm_count=152)["path"] == 3
    assert gq.gq_plan(16, 8192, 28672, 128, gu | C.GQ_ZP, sm_count=152)["path"] == 4
    assert gq.gq_plan(9, 4096, 1024, 64, gu, sm_count=152)["path"] == 4
    assert gq.gq_plan(64, 4096, 1024, 32, gu, sm_count=152)["path"] == 4
    assert gq.gq_plan(33, 4096, 1024, 64, gu, sm_count=152)["path"] == 4
    assert gq.gq_plan(33, 4096, 1024, 64, C.GQ_W4, sm_count=152)["path"] == 2
    assert gq.gq_plan(25, 4096, 1024, 64, gu, sm_count=152)["path"] == 4
    assert gq.gq_plan(25, 4096, 1024, 64, C.GQ_W4, sm_count=152)["path"] == 2
    assert gq.gq_plan(24, 4096, 1024, 64, C.GQ_W4, sm_count=152)["path"] == 4
    assert gq.gq_plan(32, 4096, 1024, 64, C.GQ_W4 | C.GQ_ZP, sm_count=152)["path"] == 4
    for M, K, G in ((1, 320, 64), (65, 4096, 32), (65, 4096, 128)):
        with pytest.raises(C.GqError) as e:
            gq.gq_plan(M, K, 1024, G, gu, sm_count=152)
        assert e.value.status == 2
    # the packed size does not change
    assert gq.gq_packed_bytes(4096, 28672, 128, gu) == gq.gq_packed_bytes(4096, 28672, 128, C.GQ_W4)


def test_int8_activation_variant_validation_and_plan():
    a8 = C.GQ_ACT_I8 | C.GQ_SC_F32 | C.GQ_OUT_F32
    # up to four rows with N a multiple of 64 and G <= 128: the warp-specialized decode kernel
    # (dp4a group dots); otherwise the W8A8 block kernel
    for M in (1, 2, 3, 4):
        assert gq.gq_plan(M, 2048, 12288, 32, a8, sm_count=152)["path"] == 9
    assert gq.gq_plan(5, 2048, 12288, 32, a8, sm_count=152)["path"] == 7
    assert gq.gq_plan(1, 2048, 1000, 32, a8, sm_count=152)["path"] == 7
    assert gq.gq_plan(1, 2048, 1024, 256, a8, sm_count=152)["path"] == 7
    p = gq.gq_plan(40, 2048, 1000, 32, a8, sm_count=152)
    assert p["path"] == 7 and p["grid_z"] == 2 and p["m_tile"] == 32
    assert p["grid_x"] % -(-1000 // 64) == 0 and p["smem_bytes"] <= 113 * 1024
    for bad in (C.GQ_ACT_I8 | C.GQ_SC_F32 | C.GQ_W4, C.GQ_ACT_I8 | C.GQ_SC_F32 | C.GQ_ACT_F32,
                C.GQ_ACT_I8):                      # W4, fp32 activations, fp16 scales
        with pytest.raises(C.GqError) as e:
            gq.gq_plan(1, 512, 64, 32, bad, sm_count=152)
        assert e.value.status == 2
    # gq_gemm and the static-scratch entry refuse the flag: the scales need gq_gemm_a8
    assert gq.gq_gemm(1, 512, 64, 32, a8, 16, 16, 16, None, 16, None) == 1
    assert gq.gq_gemm_static_scratch(1, 512, 64, 32, a8, 16, 16, 16, None, 16, None) == 1
    # gq_gemm_a8 without the flag, a NULL activation scale, a misaligned code pointer
    assert gq.gq_gemm_a8(1, 512, 64, 32, C.GQ_SC_F32, 16, 16, 16, 16, 16, None) == 1
    assert gq.gq_gemm_a8(1, 512, 64, 32, a8, 16, None, 16, 16, 16, None) == 1
    assert gq.gq_gemm_a8(1, 512, 64, 32, a8, 8, 16, 16, 16, 16, None) == 3
    # the quantizer: shape and flag checks before any launch
    assert gq.gq_quantize_act(1, 100, 32, 0, 16, 16, 16, None) == 1
    assert gq.gq_quantize_act(1, 512, 32, C.GQ_W4, 16, 16, 16, None) == 1
    assert gq.gq_quantize_act(1, 512, 32, 0, 16, 8, 16, None) == 3
    assert gq.gq_quantize_act(0, 512, 32, 0, None, None, None, None) == 0


def test_float_zero_points_validation_and_plan():
    zf = C.GQ_W4 | C.GQ_ZP_FLOAT | C.GQ_SC_BF16
    # one zero-point form at a time; W4 only; no fused epilogue; the zeros pointer is required
    assert gq.gq_gemm(1, 512, 64, 128, zf | C.GQ_ZP, 16, 16, 16, 16, 16, None) == 1
    assert gq.gq_gemm(1, 512, 64, 32, C.GQ_ZP_FLOAT | C.GQ_ACT_F32 | C.GQ_SC_F32,
                      16, 16, 16, 16, 16, None) == 2
    assert gq.gq_gemm(1, 512, 64, 128, zf | C.GQ_GATE_UP, 16, 16, 16, 16, 16, None) == 2
    assert gq.gq_gemm(1, 512, 64, 128, zf, 16, 16, 16, None, 16, None) == 1
    # every M up to 64 runs on the small-batch kernel (not the striped or prefill ones), with
    # room for the slice's activation group sums
    for M, K, N, G in ((1, 4096, 28672, 128), (16, 8192, 28672, 128), (40, 2048, 264, 128),
                       (64, 1024, 128, 32)):
        p = gq.gq_plan(M, K, N, G, zf, sm_count=152)
        assert p["path"] == 4
        assert p["smem_bytes"] <= 226 * 1024
    for M, K in ((65, 1024), (4096, 4096), (1, 320)):
        with pytest.raises(C.GqError) as e:
            gq.gq_plan(M, K, 512, 64, zf, sm_count=152)
        assert e.value.status == 2
    # bytes: one float zero point per group and column in the scales' format
    assert C.algorithmic_bytes(1, 4096, 1024, 128, True, False, "bf16", "bf16", "bf16", zf=True) == \
        C.algorithmic_bytes(1, 4096, 1024, 128, True, False, "bf16", "bf16", "bf16") + 32 * 1024 * 2


def test_fp8_block_gemm_validation():
    f = gq.gq_gemm_fp8_block
    assert f(4, 192, 128, 0, 16, 16, 16, 16, 16, None) == 1      # K % 128 != 0
    assert f(4, 256, 120, 0, 16, 16, 16, 16, 16, None) == 1      # N % 16 != 0
    assert f(4, 256, 128, C.GQ_W4, 16, 16, 16, 16, 16, None) == 1
    assert f(4, 256, 128, 0, 16, None, 16, 16, 16, None) == 1
    assert f(4, 256, 128, 0, 8, 16, 16, 16, 16, None) == 3       # misaligned
    assert f(0, 256, 128, 0, None, None, None, None, None, None) == 0


def test_fp8_activation_quantizer_validation():
    f = gq.gq_quantize_act_fp8
    assert f(2, 192, 0, 16, 16, 16, None) == 1                # K % 128 != 0
    assert f(2, 256, C.GQ_W4, 16, 16, 16, None) == 1
    assert f(2, 256, 0, 16, 8, 16, None) == 3
    assert f(0, 256, 0, None, None, None, None) == 0


def test_split_override_forces_the_slice_count_and_rejects_counts_a_path_cannot_take():
    """gq_set_split_override: n slices exactly, -1 the largest count, 0 the planner's own
    choice again; the path never changes; a count the path cannot take is GQ_ERR_UNSUPPORTED."""
    from group_quantized_weight_gb300.constants import GqError
    W4ZP = C.GQ_W4 | C.GQ_ZP | C.GQ_SC_BF16
    W8 = C.GQ_ACT_F32 | C.GQ_SC_F32 | C.GQ_OUT_F32
    shapes = [((16, 2048, 1032, 128, W4ZP), 4, 8),     # K / 256 slots
              ((3, 1088, 264, 64, C.GQ_W4), 0, 17),    # K / 64 units
              ((2, 2048, 1000, 32, W8), 5, 8),         # groups / 8 warps
              ((40, 512, 264, 32, W8), 1, 16)]         # K / G units
    try:
        for args, path, largest in shapes:
            base = gq.gq_plan(*args, sm_count=152)
            assert base["path"] == path
            for n, want in ((1, 1), (2, 2), (-1, largest)):
                assert gq.gq_set_split_override(n) in (0, 1, 2, -1)
                p = gq.gq_plan(*args, sm_count=152)
                assert p["path"] == path and p["nsplit"] == want, (args, n, p)
                assert (p["workspace_bytes"] > 0) == (want > 1)
            gq.gq_set_split_override(largest + 1)
            with pytest.raises(GqError) as e:
                gq.gq_plan(*args, sm_count=152)
            assert e.value.status == 2
            gq.gq_set_split_override(0)
            assert gq.gq_plan(*args, sm_count=152) == base
        # the batch kernel needs K / n to be a whole number of 256-k slots
        gq.gq_set_split_override(3)
        with pytest.raises(GqError):
            gq.gq_plan(16, 2048, 1032, 128, W4ZP, sm_count=152)
        assert gq.gq_set_split_override(-5) == -2                  # rejected, unchanged
        assert gq.gq_set_split_override(0) == 3
    finally:
        gq.gq_set_split_override(0)


def test_config_benchmark_validates_its_arguments_before_touching_a_device():
    """gq_bench(config, json_out, cap): an unknown workload name or a NULL buffer is
    GQ_ERR_INVALID_ARG; a known name needs a device (GQ_ERR_NO_DEVICE here, on a machine
    without one).  The buffer holds "" after any error."""
    import ctypes
    lib = gq._lib
    buf = ctypes.create_string_buffer(64)
    buf.value = b"junk"
    assert lib.gq_bench(b"no_such_workload", buf, 64) == 1
    assert buf.value == b""
    assert lib.gq_bench(b"tiny_gemv", None, 64) == 1
    assert lib.gq_bench(None, buf, 64) == 1
    assert lib.gq_bench(b"tiny_gemv", buf, 0) == 1
    import torch
    if not torch.cuda.is_available():
        assert lib.gq_bench(b"tiny_gemv", buf, 64) == 7
        assert lib.gq_bench(b"all", buf, 64) == 7


def test_fault_injection_and_wait_limit_settings_are_validated():
    """gq_set_fault_injection takes the four documented values (returning the previous one)
    and refuses others; gq_set_wait_limit refuses limits outside [1e4, 1e11] cycles before it
    touches a device."""
    lib = gq._lib
    assert lib.gq_set_fault_injection(7) == -1 and lib.gq_set_fault_injection(-1) == -1
    try:
        assert lib.gq_set_fault_injection(2) == 0
        assert lib.gq_set_fault_injection(1) == 2
        assert lib.gq_set_fault_injection(0) == 1
    finally:
        lib.gq_set_fault_injection(0)
    import ctypes
    f = lib.gq_set_wait_limit
    f.argtypes = [ctypes.c_longlong]
    assert f(5) == 1 and f(10 ** 12) == 1 and f(-3) == 1
    import torch
    if not torch.cuda.is_available():
        assert f(0) == 7 and f(2_000_000) == 7            # no device: GQ_ERR_NO_DEVICE


def test_prefill_plan_tiles_and_split_follow_the_rows():
    """Few rows: 64-row activation tiles, one K slice (112 tiles on 112 SMs; every measured
    split was slower) and no scratch; a forced split of whole groups gets its partial sums;
    from 65 rows 128-row tiles, from 129 rows 256."""
    W4 = C.GQ_W4
    p = gq.gq_plan(64, 4096, 14336, 128, W4, sm_count=152)
    assert (p["path"], p["m_tile"], p["nsplit"], p["grid_x"], p["workspace_bytes"]) == \
        (2, 64, 1, 112, 0)
    prev = gq.gq_set_split_override(4)
    try:
        p = gq.gq_plan(64, 4096, 14336, 128, W4, sm_count=152)
    finally:
        gq.gq_set_split_override(prev)
    assert (p["path"], p["m_tile"], p["nsplit"], p["grid_x"]) == (2, 64, 4, 152)
    assert p["workspace_bytes"] >= 4 * 64 * 14336 * 4
    p = gq.gq_plan(128, 4096, 14336, 128, W4, sm_count=152)
    assert (p["path"], p["m_tile"], p["nsplit"]) == (2, 128, 1)
    p = gq.gq_plan(4096, 4096, 14336, 128, W4, sm_count=152)
    assert (p["path"], p["m_tile"], p["nsplit"], p["workspace_bytes"]) == (2, 256, 1, 0)
