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

No GPU: the GPU parity tests cover the kernel itself."""

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
