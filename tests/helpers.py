"""Shared helpers of the GPU tests: oracle comparison and sub-batch slicing."""

import numpy as np

import oracle
from paged_kv_decode_splitk_gb300 import workloads as W


def assert_within_tolerance(got_bf16_f64: np.ndarray, ref: np.ndarray, what: str = "") -> float:
    """|gpu - ref| <= ulp_bf16(ref) + 1e-3 elementwise; returns the worst error / bound ratio."""
    got = np.asarray(got_bf16_f64, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    tol = oracle.tolerance(ref)
    ratio = err / tol
    worst = float(ratio.max()) if ratio.size else 0.0
    if worst > 1.0:
        i = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
        raise AssertionError(f"{what}: |gpu-ref| exceeds ulp_bf16(ref)+1e-3 at {i}: gpu {got[i]!r} "
                             f"ref {ref[i]!r} err {err[i]:.3g} bound {tol[i]:.3g}; "
                             f"{int((ratio > 1).sum())} of {ratio.size} elements over")
    return worst


def oracle_rows(w: W.PagedWorkload, seqs) -> np.ndarray:
    """Oracle output for a subset of the workload's sequences, [len(seqs), Hq, D]."""
    seqs = np.asarray(seqs)
    return oracle.decode_attn(w.q[seqs], w.k_cache, w.v_cache, w.block_table[seqs],
                              w.context_lens[seqs], w.inv_sqrt_d)
