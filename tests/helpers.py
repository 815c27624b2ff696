"""Shared helpers of the GPU tests: oracle comparison and sub-batch slicing."""

import os
from concurrent.futures import ThreadPoolExecutor

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


def oracle_all_rows(w: W.PagedWorkload) -> np.ndarray:
    """Oracle output for every sequence of a paged workload (BF16 or FP8 cache),
    [S, Hq, D]: the sequences are dealt round-robin to one thread per host core.
    The C oracle runs outside the GIL and keeps no state, and each sequence's
    output depends on its own rows only, so the result is the one-call result."""
    oracle._load()  # build / load once, before the threads
    S = w.num_seqs
    nthr = max(1, min(os.cpu_count() or 1, S))
    chunks = [np.arange(i, S, nthr) for i in range(nthr)]
    fp8 = getattr(w, "kv_dtype", "bf16") == "e4m3"

    def one(seqs):
        if fp8:
            return oracle.decode_attn_fp8(w.q[seqs], w.k_cache, w.v_cache, w.k_scale, w.v_scale,
                                          w.block_table[seqs], w.context_lens[seqs], w.inv_sqrt_d)
        return oracle.decode_attn(w.q[seqs], w.k_cache, w.v_cache, w.block_table[seqs],
                                  w.context_lens[seqs], w.inv_sqrt_d)

    out = np.zeros((S, w.num_q_heads, w.head_dim), dtype=np.float64)
    with ThreadPoolExecutor(nthr) as ex:
        for seqs, part in zip(chunks, ex.map(one, chunks)):
            out[seqs] = part
    return out
