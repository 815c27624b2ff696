"""The FP8 direct-K operand mapping of the unit kernel, restated on the CPU.

From head dim 128 up, the kernel reads K's E4M3 codes straight from the
128-byte-swizzled TMA tile into the A operand of mma m16n8k16 (lane = 4*tq +
qd holds rows tq and tq + 8): for block kb of 32 codes, quad positions 0-1
read the two halves of 16-byte chunk 2*kb' of the 128-code box and positions
2-3 those of chunk (2*kb' + 1) ^ 4 (kb' = kb mod 4), and the codes are used as
columns 2qd, 2qd+1 | 2qd+8, 2qd+9 of k-steps 2kb and 2kb + 1.  q is staged in
the matching column order.  These tests check, with the formulas written as
the kernel's comments state them, that

* the A operand so assembled and the reordered q give exactly K . q^T (the
  same dot product over a permutation of d), for head dims 128 and 256;
* the q reordering is a permutation;
* each half-warp's 8-byte shared loads touch the 32 banks once (no conflict).

The same is checked for the direct V operand (below).  No GPU: the GPU
parity tests cover the kernel itself."""

import numpy as np
import pytest


def chunk_of(kbp: int, qd: int) -> int:
    return 2 * kbp if qd < 2 else ((2 * kbp + 1) ^ 4)


def q_dest_pair(P: int) -> int:
    """Logical pair index (k-step * 8 + pair within it) of q's column pair P."""
    box, Pb = P // 64, P % 64
    c, half, j = Pb // 8, (Pb // 4) & 1, Pb & 3
    if c % 2 == 0:
        kbp, qd = c // 2, half
    else:
        kbp, qd = ((c ^ 4) - 1) // 2, 2 + half
    kb = box * 4 + kbp
    return (2 * kb + (j >> 1)) * 8 + qd + 4 * (j & 1)


def swizzled_tile(K: np.ndarray) -> np.ndarray:
    """The bytes a 128-byte-swizzled TMA load of K (16 rows) leaves in shared memory."""
    rows, D = K.shape
    smem = np.zeros(D // 128 * rows * 128, dtype=K.dtype)
    for b in range(D // 128):
        for t in range(rows):
            for c in range(8):
                dst = b * rows * 128 + t * 128 + (c ^ (t & 7)) * 16
                smem[dst:dst + 16] = K[t, b * 128 + c * 16: b * 128 + c * 16 + 16]
    return smem


def lane_address(kb: int, lane: int) -> int:
    """Byte offset of lane's 8-code read of row tq (row tq + 8 is 8 * 128 further)."""
    tq, qd = lane >> 2, lane & 3
    ch = chunk_of(kb & 3, qd) ^ (tq & 7)
    return (kb >> 2) * 2048 + tq * 128 + ch * 16 + (qd & 1) * 8


@pytest.mark.parametrize("D", [128, 256])
def test_direct_operand_gives_k_qt_exactly(D):
    rng = np.random.default_rng(D)
    K = rng.integers(0, 256, size=(16, D)).astype(np.int64)
    q = rng.integers(-64, 64, size=(8, D)).astype(np.int64)
    smem = swizzled_tile(K)
    qs = np.zeros_like(q)
    for P in range(D // 2):
        d2 = 2 * q_dest_pair(P)
        qs[:, d2:d2 + 2] = q[:, 2 * P:2 * P + 2]
    A = np.full((16, D), -1, dtype=np.int64)
    for kb in range(D // 32):
        for lane in range(32):
            tq, qd = lane >> 2, lane & 3
            a = lane_address(kb, lane)
            for row, base in ((tq, a), (tq + 8, a + 8 * 128)):
                codes = smem[base:base + 8]
                for h in range(2):
                    ks = 2 * kb + h
                    A[row, ks * 16 + 2 * qd: ks * 16 + 2 * qd + 2] = codes[4 * h: 4 * h + 2]
                    A[row, ks * 16 + 2 * qd + 8: ks * 16 + 2 * qd + 10] = codes[4 * h + 2: 4 * h + 4]
    assert (A >= 0).all(), "every operand element is written"
    assert np.array_equal(A @ qs.T, K @ q.T)


@pytest.mark.parametrize("D", [128, 256])
def test_q_order_is_a_permutation(D):
    assert sorted(q_dest_pair(P) for P in range(D // 2)) == list(range(D // 2))


@pytest.mark.parametrize("D", [128, 256])
def test_each_half_warp_covers_every_bank_once(D):
    for kb in range(D // 32):
        for half in range(2):
            for row_off in (0, 8 * 128):
                banks = []
                for lane in range(16 * half, 16 * half + 16):
                    a = lane_address(kb, lane) + row_off
                    banks += [(a // 4) % 32, (a // 4 + 1) % 32]
                assert sorted(banks) == list(range(32)), (D, kb, half)


def test_the_first_mapping_had_a_two_way_conflict():
    # quad positions 2-3 reading chunk 2*kb' + 1 (same aligned group of four
    # chunks as positions 0-1): two lanes per bank in a half-warp
    banks = []
    for lane in range(16):
        tq, qd = lane >> 2, lane & 3
        ch = (0 * 2 + (qd >> 1)) ^ (tq & 7)
        a = tq * 128 + ch * 16 + (qd & 1) * 8
        banks += [(a // 4) % 32, (a // 4 + 1) % 32]
    assert max(np.bincount(banks, minlength=32)) == 2


# ---- the direct V operand (V^T . P^T) -----------------------------------------------------
# From head dim 128 up V's codes also go straight from the 128-byte-swizzled
# tile into the A operand V^T (rows d, columns t) of mma m16n8k16.  Row r of
# m-tile mt stands for d = 128*(mt//8) + 16*(r%8) + 2*(mt%8) + r//8; the lane
# (tq, qd) reads, per 128-code box, 16-byte chunk tq of token rows 2qd, 2qd+1,
# 2qd+8, 2qd+9 (at chunk tq ^ (t & 7)), and builds its four registers from
# byte permutes of those words with selector 0x5140 (even mt) or 0x7362 (odd).


def v_row_d(mt: int, r: int) -> int:
    return 128 * (mt // 8) + 16 * (r % 8) + 2 * (mt % 8) + r // 8


def prmt(a: int, b: int, sel: int) -> int:
    """PTX prmt.b32 (default mode): byte i of the result is byte (sel >> 4i) & 7
    of the eight bytes {b, a}."""
    src = [(a >> (8 * i)) & 0xFF for i in range(4)] + [(b >> (8 * i)) & 0xFF for i in range(4)]
    return sum(src[(sel >> (4 * i)) & 7] << (8 * i) for i in range(4))


def v_direct_operands(smem: np.ndarray, D: int, lane: int):
    """The A registers lane builds for each m-tile: {mt: (a0, a1, a2, a3)}, each
    register a (low, high) pair of codes."""
    tq, qd = lane >> 2, lane & 3
    regs = {}
    for bx in range(D // 128):
        R = []
        for j in range(4):
            t = 2 * qd + (j & 1) + (j >> 1) * 8
            base = bx * 2048 + t * 128 + ((tq ^ (t & 7)) << 4)
            chunk = smem[base:base + 16]
            R.append([int(chunk[4 * w]) | int(chunk[4 * w + 1]) << 8 | int(chunk[4 * w + 2]) << 16
                      | int(chunk[4 * w + 3]) << 24 for w in range(4)])
        for m8 in range(8):
            sel = 0x7362 if m8 & 1 else 0x5140
            x01 = prmt(R[0][m8 >> 1], R[1][m8 >> 1], sel)
            x89 = prmt(R[2][m8 >> 1], R[3][m8 >> 1], sel)
            split = lambda x: ((x & 0xFF, (x >> 8) & 0xFF), ((x >> 16) & 0xFF, (x >> 24) & 0xFF))
            (a0, a1), (a2, a3) = split(x01), split(x89)
            regs[bx * 8 + m8] = (a0, a1, a2, a3)
    return regs


@pytest.mark.parametrize("D", [128, 256])
def test_direct_v_operand_is_v_transposed_on_permuted_rows(D):
    rng = np.random.default_rng(D + 7)
    V = rng.integers(0, 256, size=(16, D)).astype(np.int64)
    smem = swizzled_tile(V)
    KS = D // 16
    A = np.full((KS, 16, 16), -1, dtype=np.int64)   # [mt][row][token]
    for lane in range(32):
        tq, qd = lane >> 2, lane & 3
        for mt, (a0, a1, a2, a3) in v_direct_operands(smem, D, lane).items():
            # m16n8k16 A fragment: a0 (row tq, k 2qd..+1), a1 (row tq+8, k 2qd..),
            # a2 (row tq, k 2qd+8..), a3 (row tq+8, k 2qd+8..); low half = lower k
            for reg, row, k0 in ((a0, tq, 2 * qd), (a1, tq + 8, 2 * qd), (a2, tq, 2 * qd + 8),
                                 (a3, tq + 8, 2 * qd + 8)):
                A[mt, row, k0], A[mt, row, k0 + 1] = reg
    assert (A >= 0).all(), "every operand element is written"
    for mt in range(KS):
        for r in range(16):
            assert np.array_equal(A[mt, r], V[:, v_row_d(mt, r)]), (mt, r)


@pytest.mark.parametrize("D", [128, 256])
def test_direct_v_rows_are_a_permutation_of_d(D):
    ds = sorted(v_row_d(mt, r) for mt in range(D // 16) for r in range(16))
    assert ds == list(range(D))


def test_direct_v_loads_cover_every_bank_once_per_quarter_warp():
    # a 16-byte load is served a quarter-warp (8 lanes) at a time
    for j in range(4):
        for quarter in range(4):
            banks = []
            for lane in range(8 * quarter, 8 * quarter + 8):
                tq, qd = lane >> 2, lane & 3
                t = 2 * qd + (j & 1) + (j >> 1) * 8
                a = t * 128 + ((tq ^ (t & 7)) << 4)
                banks += [(a // 4 + i) % 32 for i in range(4)]
            assert sorted(banks) == list(range(32)), (j, quarter)


@pytest.mark.parametrize("D", [128, 256])
def test_combine_slot_map_undoes_the_v_row_permutation(D):
    """The warps store their accumulators by slot mt*16 + r and the part's sum
    writes slot sl to d = 128*(sl>>7) + 16*(sl&7) + 2*((sl>>4)&7) + ((sl>>3)&1):
    that must be the row map of the direct V operand, slot by slot."""
    for sl in range(D):
        d = 128 * (sl >> 7) + 16 * (sl & 7) + 2 * ((sl >> 4) & 7) + ((sl >> 3) & 1)
        assert d == v_row_d(sl // 16, sl % 16)


def test_slot_order_stores_cover_distinct_banks():
    # the warp-merge stores of one (m-tile, accumulator) for the 16 lanes of the
    # first 4 groups (HL: columns 0..3): row (warp*8 + g) of stride DPAD + 4
    # floats, column slot = mt*16 + tq + 8*(c>>1) -- distinct banks
    OST = 128 + 4
    for mt in range(8):
        for c in range(4):
            banks = []
            for lane in range(32):
                tq, qd = lane >> 2, lane & 3
                g = 2 * qd + (c & 1)
                if g < 4:
                    banks.append((g * OST + mt * 16 + tq + 8 * (c >> 1)) % 32)
            assert len(set(banks)) == len(banks), (mt, c)
