"""The streaming shrink's shared-memory operand arithmetic, restated on the CPU.

The shrink stages A columns as [ks/8][R][8] and the tile's x rows as [ks/8][n_pad][8] in one 32 KB ring
stage and feeds both to tcgen05 MMAs: the A block's rows as the 128-row M operand (blocks of 128 rows when
R > 128; an A block of fewer rows is read as a full 128-row block), the tile's rows rounded up to 16 as N.
These checks restate that arithmetic (stream.cu: group_plan's stage width, x_gather, the producers'
zero-filled K tail, shrink_mma's descriptors) for every stored-rank width and tile height the plan allows:

* the x gather writes every (row, piece) of a stage exactly once, inside the stage's x region;
* every byte an MMA reads lies inside the ring stage (rows past R come from later A columns or the x rows of
  the same stage), so no read leaves the block's shared memory;
* the zero-filled K tail lies inside the stage, past the copied columns;
* descriptor start addresses stay below 2^18 bytes (their 14-bit field in 16-byte units).
"""
import os
import re

import pytest

SRC = os.path.join(os.path.dirname(__file__), "..", "segmented_rank_gemm_lora_gb300", "csrc", "stream.cu")


def _const(name):
    m = re.search(r"constexpr (?:int|uint32_t) %s = ([0-9* ]+);" % name, open(SRC).read())
    assert m, name
    return int(eval(m.group(1)))


STAGE = _const("kShStageBytes")
STAGES = _const("kShStages")
PROD = _const("kShProd")
TILE_ROWS = _const("kTileRows")


def npad16(m):
    return (m + 15) // 16 * 16


def stage_k(R, m_max):
    """group_plan's stage width: A and x columns of one stage fill at most one ring stage."""
    return min(512, STAGE // 2 // (R + npad16(m_max))) // 16 * 16


def x_gather(m, P, n_pad):
    """(byte offset in the x region, row, piece) of every cp.async piece the producer group issues."""
    out = []
    warps = PROD // 32
    for gt in range(PROD):
        lane, w = gt & 31, gt >> 5
        l8, q = lane & 7, lane >> 3
        nrb, npq = (m + 7) >> 3, (P + 3) >> 2
        rb, pq = w, 0
        while rb >= nrb and pq < npq:
            rb -= nrb
            pq += 1
        while pq < npq:
            r, c = rb * 8 + l8, pq * 4 + q
            if r < m and c < P:
                out.append(((c * n_pad + r) * 16, r, c))
            rb += warps
            while rb >= nrb and pq < npq:
                rb -= nrb
                pq += 1
    return out


RANKS = [16 * i for i in range(1, 17)]          # stored A rows R = n_a * rpad, 16 .. 256
HEIGHTS = list(range(1, TILE_ROWS + 1))


@pytest.mark.parametrize("m", HEIGHTS)
def test_x_gather_covers_every_piece_once(m):
    n_pad = npad16(m)
    for P in range(1, 65):
        pieces = x_gather(m, P, n_pad)
        assert sorted((r, c) for _, r, c in pieces) == [(r, c) for r in range(m) for c in range(P)]
        assert all(0 <= off and off + 16 <= P * n_pad * 16 for off, _, _ in pieces)


def test_gather_lanes_fill_contiguous_shared_memory():
    """Every 8 consecutive lanes of a warp write 128 contiguous bytes (one bank-conflict-free wavefront)."""
    m, P, n_pad = 64, 64, 64
    warps = PROD // 32
    for w in range(warps):
        for q in range(4):
            lanes = [w * 32 + q * 8 + l8 for l8 in range(8)]
            # the first item of this warp: row block w, piece quad 0
            offs = [((q * n_pad) + (w * 8 + l8)) * 16 for l8 in range(8)]
            assert offs == list(range(offs[0], offs[0] + 128, 16)), lanes


@pytest.mark.parametrize("R", RANKS)
def test_mma_reads_and_zero_fill_stay_inside_the_stage(R):
    for m in HEIGHTS:
        n_pad = npad16(m)
        ks = stage_k(R, m)
        assert ks >= 16 and ks % 16 == 0
        a_bytes, x_bytes = R * ks * 2, n_pad * ks * 2
        assert a_bytes + x_bytes <= STAGE
        x_off = a_bytes
        for kk in sorted({ks, ks - 8, 8, 16, 24} - {0}):
            if kk > ks or kk < 8:
                continue
            nk = (kk + 15) // 16
            hi = 0
            for k in range(nk):
                for mb in range((R + 127) // 128):
                    start = (k * 2 * R + mb * 128) * 16
                    # two core-matrix columns along K (lbo = 16 R), sixteen 8-row groups (sbo = 128)
                    for kg in range(2):
                        for rg in range(16):
                            hi = max(hi, start + kg * R * 16 + rg * 128 + 128)
                # the x operand: n_pad rows, two K groups
                assert x_off + k * 2 * n_pad * 16 + n_pad * 16 + n_pad * 16 <= x_off + x_bytes
            assert hi <= STAGE, (R, m, ks, kk, hi)
            if kk & 8:
                # zero-filled A rows and x rows of the K group after the copied ones
                assert (kk >> 3) * R * 16 + R * 16 <= a_bytes
                assert x_off + ((kk >> 3) * n_pad + n_pad) * 16 <= x_off + x_bytes


def test_descriptor_start_fields_fit():
    """A descriptor's start address is 14 bits of 16-byte units: every stage byte must lie below 2^18."""
    assert STAGES * STAGE + 2048 < (1 << 18)
