"""Host model of the warp-specialized INT8 decode kernel's work partition (plan path 9), CPU
only.  The kernel's index arithmetic is restated here from its description in gq_q8_gemv.cu:
units (64-column block b, group g) in the packed byte order u = b (K / G) + g, CTA ranges from
the z-split of the plan's split_count (times split_mult), sixteen consumer ranges per CTA,
2 KB slots per consumer, per-warp pieces of a first and a last block, per-CTA partial sums of
the blocks shared with other CTAs, and a last arriver per block.  For each shape the plan that
libgq makes is checked against that model: every unit belongs to exactly one consumer, every
copy and load stays inside its buffer and the plan's shared memory and workspace, and every
output block is stored exactly once."""
import pytest

from helpers import load

gq = load()
from group_quantized_weight_gb300 import constants as C  # noqa: E402

NC, STAGES, SLOT, COLS = 16, 3, 2048, 64


def zsplit(units, n, z):
    base, rem = divmod(units, n)
    b = z * base + min(z, rem)
    return b, b + base + (1 if z < rem else 0)


def _prec(a8, gate_up):
    p = (C.GQ_ACT_I8 if a8 else C.GQ_ACT_F32) | C.GQ_SC_F32 | C.GQ_OUT_F32
    return p | (C.GQ_GATE_UP if gate_up else 0)


def _model(M, K, N, G, a8, gate_up, sms=152):
    p = gq.gq_plan(M, K, N, G, _prec(a8, gate_up), sm_count=sms)
    assert p["path"] == 9, p
    grid = p["grid_x"]
    NB, GPB = N // COLS, K // G
    units = NB * GPB
    per = -(-NB // sms)
    whole = NB >= sms and NB >= 0.9 * sms * per
    sc, sm = (NB, GPB) if whole else (units, 1)
    assert grid == (sms if whole else min(sms, -(-units // 32)))
    assert (p["workspace_bytes"] == 0) == whole
    SPU, MR = G // 32, (1 if M <= 1 else 2 if M <= 2 else 4)
    # shared memory: activations, ring, tables, pieces (plus 128 for the base alignment)
    act = (((MR * K + 15) & ~15) + MR * GPB * 4) if a8 else MR * K * 4
    act = (act + 127) & ~127
    table = -(-(-(-sc // grid) * sm) // NC) * COLS * 4
    assert p["smem_bytes"] == 128 + act + STAGES * NC * SLOT + NC * table + NC * 2 * MR * COLS * 4
    assert p["smem_bytes"] + 256 <= 227 * 1024 - 1024
    part_floats = grid * 2 * 4 * COLS
    if not whole:
        assert p["workspace_bytes"] >= part_floats * 4 + NB * 4

    owner = [0] * units
    stored = [0] * NB
    arrived = [0] * NB
    written = {}                                   # (cta, region) -> block
    for c in range(grid):
        cb, ce = zsplit(sc, grid, c)
        cb, ce = cb * sm, ce * sm
        warps = []
        for w in range(NC):
            wb, we = zsplit(ce - cb, NC, w)
            warps.append((wb + cb, we + cb))
        pieces = {}
        for w, (wb, we) in enumerate(warps):
            nu = we - wb
            assert nu * COLS * 4 <= table
            for j in range(nu * SPU):              # the producer lane's bulk copies
                src = wb * COLS * G + j * SLOT
                assert src % 16 == 0 and src + SLOT <= K * N
            for iu in range(nu):
                u = wb + iu
                owner[u] += 1
                b, g = divmod(u, GPB)
                for pc in range(16):               # the scale table's 16-byte copies
                    if gate_up:
                        col = 32 * b + pc * 4 if pc < 8 else N // 2 + 32 * b + (pc - 8) * 4
                    else:
                        col = b * COLS + pc * 4
                    assert 0 <= g * N + col and g * N + col + 4 <= GPB * N
            if nu == 0:
                continue
            t_first, first_j = divmod(wb, GPB)
            bcur, j0, gcur = t_first, first_j, first_j
            for _ in range(nu):                    # flushes: whole blocks stored, else a piece
                gcur += 1
                if gcur == GPB:
                    if j0 == 0:
                        stored[bcur] += 1
                    else:
                        pieces[(w, 0 if bcur == t_first else 1)] = bcur
                    bcur, gcur, j0 = bcur + 1, 0, 0
            if gcur != 0:
                key = (w, 0 if bcur == t_first else 1)
                assert key not in pieces
                pieces[key] = bcur
        for w, (wb, we) in enumerate(warps):       # the reductions
            if we <= wb:
                continue
            t_first = wb // GPB
            for pas in range(2):
                tt = t_first if pas == 0 else (we - 1) // GPB
                if pas == 1 and tt == t_first:
                    break
                tb, te = tt * GPB, tt * GPB + GPB
                if max(tb, wb) == tb and min(te, we) == te:
                    continue
                if pas == 0 and wb > cb and wb % GPB != 0:
                    continue
                for w2 in range(w, NC):
                    b2, e2 = warps[w2]
                    if e2 <= b2 or b2 >= te:
                        break
                    assert pieces.get((w2, 0 if b2 // GPB == tt else 1)) == tt
                if tb >= cb and te <= ce:
                    stored[tt] += 1
                    continue
                region = 0 if tb < cb else 1
                assert (c, region) not in written and (c * 2 + region + 1) * 4 * COLS <= part_floats
                written[(c, region)] = tt
                arrived[tt] += min(te, ce) - max(tb, cb)
    # the last arriver of each shared block reads the regions the CTAs holding it wrote
    for tt in range(NB):
        tb, te = tt * GPB, tt * GPB + GPB
        holders = [c for c in range(grid)
                   if zsplit(sc, grid, c)[0] * sm < te and zsplit(sc, grid, c)[1] * sm > tb]
        if any(written.get((c, r)) == tt for c in holders for r in (0, 1)):
            assert arrived[tt] == GPB
            for c in holders:
                b2 = zsplit(sc, grid, c)[0] * sm
                assert written.get((c, 0 if tb < b2 else 1)) == tt
            stored[tt] += 1
    assert owner == [1] * units
    assert stored == [1] * NB


@pytest.mark.parametrize("M,K,N,G,a8,gate_up", [
    (1, 2048, 12288, 32, False, False),      # the Q8_0 projection: equal unit ranges
    (4, 2048, 12288, 32, False, False),
    (1, 2048, 12288, 32, True, False),       # the same with int8 activations
    (3, 2048, 12288, 64, True, False),
    (2, 1024, 304 * 64, 64, False, False),   # whole blocks per CTA, no scratch
    (4, 512, 19456, 32, True, False),
    (1, 2048, 1024, 32, False, True),        # gate+up, blocks split between CTAs
    (3, 2048, 128, 32, False, True),
    (2, 256, 64, 32, False, False),          # one CTA, later warps without a unit
    (1, 96, 64, 32, False, False),
    (1, 4096, 4096, 128, False, False),
    (4, 2048, 448, 128, False, False),
])
def test_plan_matches_the_kernel_partition(M, K, N, G, a8, gate_up):
    _model(M, K, N, G, a8, gate_up)
