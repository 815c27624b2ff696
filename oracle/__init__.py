"""FP64 CPU oracle for paged-decode attention.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and the
benchmark's CPU-baseline / reference legs may import this package.  The product
library never links, loads or calls it, and it imports nothing from the
product package: the two share no code.

`pd_oracle.c` states the attention itself (definition, split-K replay, tiled
token set); `policy.py` restates the launch-geometry rules.  This module
compiles the C file with the host compiler on first use and marshals numpy
arrays into it.

Parity status: every function here is pinned by `tests/test_oracle.py`
(library routine, high-precision brute force, closed forms, invariants and
the pages' worked values); none is "parity unpinned".
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import policy  # noqa: F401  (re-export)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pd_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile pd_oracle.c into a shared object (plain C11, -O2, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p = ctypes.c_void_p
            i32 = ctypes.c_int
            i64 = ctypes.c_int64
            lib.orc_decode_attn.argtypes = [p, p, p, p, i64, p, i32, i32, i32, i32, i32, i64,
                                            ctypes.c_float, p]
            lib.orc_split_replay.argtypes = [p, p, p, p, i64, p, p, i32, i32, i32, i32, i32, i64,
                                             ctypes.c_float, p]
            lib.orc_tiled_attn.argtypes = [p, p, p, i64, p, p, p, i32, i32, i32, i32, i32, i32,
                                           i32, i64, i64, i64, p]
            lib.orc_tiled_attn_multi.argtypes = [p, p, p, p, p, p, p, p, p, i32, i32, i32, i32,
                                                 i32, i32, p]
            lib.orc_decode_attn_fp8.argtypes = [p, p, p, ctypes.c_float, ctypes.c_float, p, i64, p,
                                                i32, i32, i32, i32, i32, i64, ctypes.c_float, p]
            lib.orc_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_value.restype = ctypes.c_double
            for f in (lib.orc_decode_attn, lib.orc_split_replay, lib.orc_tiled_attn,
                      lib.orc_tiled_attn_multi, lib.orc_decode_attn_fp8):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"BF16 data must be passed as uint16 bit patterns, got {a.dtype}")
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"{what}: oracle rejected the inputs (code {rc})")


def decode_attn(q, k_cache, v_cache, block_table, context_lens, inv_sqrt_d: float) -> np.ndarray:
    """Paged-decode attention by definition, FP64.

    q [S, Hq, D], k_cache / v_cache [num_blocks, block_size, Hkv, D] as BF16 bit
    patterns (uint16); block_table [S, max_blocks] and context_lens [S] int32.
    Returns out [S, Hq, D] float64.
    """
    q, k_cache, v_cache = _u16(q), _u16(k_cache), _u16(v_cache)
    bt, cl = _i32(block_table), _i32(context_lens)
    S, Hq, D = q.shape
    nb, bs, Hkv, D2 = k_cache.shape
    assert D2 == D and v_cache.shape == k_cache.shape and bt.shape[0] == S and cl.shape == (S,)
    out = np.zeros((S, Hq, D), dtype=np.float64)
    rc = _load().orc_decode_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), bt.shape[1],
                                 _ptr(cl), S, Hq, Hkv, D, bs, nb, float(inv_sqrt_d), _ptr(out))
    _check(rc, "decode_attn")
    return out


def split_replay(q, k_cache, v_cache, block_table, context_lens, inv_sqrt_d: float,
                 chunk_tokens) -> np.ndarray:
    """The split-K fold and merge replayed in FP64 with per-sequence chunk sizes."""
    q, k_cache, v_cache = _u16(q), _u16(k_cache), _u16(v_cache)
    bt, cl = _i32(block_table), _i32(context_lens)
    S, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    ch = np.ascontiguousarray(np.broadcast_to(np.asarray(chunk_tokens, dtype=np.int64), (S,)))
    out = np.zeros((S, Hq, D), dtype=np.float64)
    rc = _load().orc_split_replay(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), bt.shape[1],
                                  _ptr(cl), _ptr(ch), S, Hq, Hkv, D, bs, nb, float(inv_sqrt_d),
                                  _ptr(out))
    _check(rc, "split_replay")
    return out


def tiled_attn(q, k_pool, v_pool, tile_blocks, tile_block_counts, last_block_valid_slots,
               num_kv_heads: int, block_size: int, strides) -> np.ndarray:
    """Result of begin_step, one step_tile per call and finalize, FP64.

    q [S, Hq, D] uint16; k_pool / v_pool: flat uint16 arrays (any layout) that
    the (blk, tok, kvh) element strides address; tile_blocks [T, S, tcap],
    tile_block_counts [T, S], last_block_valid_slots [T] int32.
    """
    q = _u16(q)
    kp = _u16(np.asarray(k_pool).reshape(-1))
    vp = _u16(np.asarray(v_pool).reshape(-1))
    tb, tc = _i32(tile_blocks), _i32(tile_block_counts)
    lb = _i32(last_block_valid_slots)
    T, S, tcap = tb.shape
    _, Hq, D = q.shape
    assert tc.shape == (T, S) and lb.shape == (T,) and q.shape[0] == S
    blk, tok, kvh = (int(x) for x in strides)
    out = np.zeros((S, Hq, D), dtype=np.float64)
    rc = _load().orc_tiled_attn(_ptr(q), _ptr(kp), _ptr(vp), min(kp.size, vp.size), _ptr(tb),
                                _ptr(tc), _ptr(lb), T, S, Hq, num_kv_heads, D, block_size, tcap,
                                blk, tok, kvh, _ptr(out))
    _check(rc, "tiled_attn")
    return out


def e4m3_values() -> np.ndarray:
    """The value of every FP8 E4M3 code 0..255 (NaN for the two NaN codes), FP64."""
    lib = _load()
    return np.array([lib.orc_e4m3_value(c) for c in range(256)], dtype=np.float64)


def decode_attn_fp8(q, k_cache, v_cache, k_scale: float, v_scale: float, block_table, context_lens,
                    inv_sqrt_d: float) -> np.ndarray:
    """Paged-decode attention by definition over an FP8 E4M3 KV cache, FP64.

    k_cache / v_cache [num_blocks, block_size, Hkv, D] uint8 E4M3 codes; K and V
    are code value * k_scale / v_scale (per-tensor FP32 scales); q BF16 bits.
    """
    q = _u16(q)
    kc = np.ascontiguousarray(k_cache, dtype=np.uint8)
    vc = np.ascontiguousarray(v_cache, dtype=np.uint8)
    bt, cl = _i32(block_table), _i32(context_lens)
    S, Hq, D = q.shape
    nb, bs, Hkv, D2 = kc.shape
    assert D2 == D and vc.shape == kc.shape and bt.shape[0] == S and cl.shape == (S,)
    out = np.zeros((S, Hq, D), dtype=np.float64)
    rc = _load().orc_decode_attn_fp8(_ptr(q), _ptr(kc), _ptr(vc), float(k_scale), float(v_scale),
                                     _ptr(bt), bt.shape[1], _ptr(cl), S, Hq, Hkv, D, bs, nb,
                                     float(inv_sqrt_d), _ptr(out))
    _check(rc, "decode_attn_fp8")
    return out


def tiled_attn_multi(q, calls, num_kv_heads: int, block_size: int) -> np.ndarray:
    """Result of begin_step, one step_tile per call and finalize, FP64, where each
    call names its own source (tiled_attention.rs page: step_tile takes the pools
    and the strides per call).

    calls: sequence of dicts with k_pool, v_pool (flat uint16 arrays the strides
    address), tile_blocks [S, tcap] int32, tile_block_counts [S] int32,
    last_block_valid_slots (int) and strides (blk, tok, kvh).
    """
    q = _u16(q)
    S, Hq, D = q.shape
    T = len(calls)
    kp = [_u16(np.asarray(c["k_pool"]).reshape(-1)) for c in calls]
    vp = [_u16(np.asarray(c["v_pool"]).reshape(-1)) for c in calls]
    tb = [_i32(c["tile_blocks"]) for c in calls]
    tc = [_i32(c["tile_block_counts"]) for c in calls]
    for c in range(T):
        assert tb[c].ndim == 2 and tb[c].shape[0] == S and tc[c].shape == (S,)
    P = ctypes.c_void_p
    k_arr = (P * max(1, T))(*[_ptr(a) for a in kp])
    v_arr = (P * max(1, T))(*[_ptr(a) for a in vp])
    tb_arr = (P * max(1, T))(*[_ptr(a) for a in tb])
    tc_arr = (P * max(1, T))(*[_ptr(a) for a in tc])
    elems = np.array([min(kp[c].size, vp[c].size) for c in range(T)] or [0], dtype=np.int64)
    strides = np.array([int(x) for c in calls for x in c["strides"]] or [0, 0, 0], dtype=np.int64)
    tcap = np.array([tb[c].shape[1] for c in range(T)] or [0], dtype=np.int32)
    lb = np.array([int(c["last_block_valid_slots"]) for c in calls] or [0], dtype=np.int32)
    out = np.zeros((S, Hq, D), dtype=np.float64)
    rc = _load().orc_tiled_attn_multi(_ptr(q), ctypes.cast(k_arr, P), ctypes.cast(v_arr, P),
                                      _ptr(elems), _ptr(strides), ctypes.cast(tb_arr, P),
                                      ctypes.cast(tc_arr, P), _ptr(tcap), _ptr(lb), T, S, Hq,
                                      num_kv_heads, D, block_size, _ptr(out))
    _check(rc, "tiled_attn_multi")
    return out


def paged_strides(num_kv_heads: int, head_dim: int, block_size: int) -> tuple[int, int, int]:
    """(blk, tok, kvh) element strides of [num_blocks, block_size, Hkv, D]
    (tiled_attention.rs page, TiledAttention::paged_strides)."""
    return (block_size * num_kv_heads * head_dim, num_kv_heads * head_dim, head_dim)


def scratch_pool_strides(num_kv_heads: int, head_dim: int, block_size: int) -> tuple[int, int, int]:
    """(blk, tok, kvh) element strides of [slot, K|V, Hkv, block_size, D]
    (tiled_attention.rs page, TiledAttention::scratch_pool_strides)."""
    stripe = num_kv_heads * block_size * head_dim
    return (2 * stripe, head_dim, block_size * head_dim)


def bf16_ulp(x) -> np.ndarray:
    """Spacing of BF16 numbers at |x|: 2**(floor(log2|x|) - 7) for normal x, 0 at x = 0."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    out = np.zeros_like(x)
    nz = x > 0
    e = np.floor(np.log2(x[nz]))
    out[nz] = np.exp2(np.maximum(e, -126.0) - 7.0)
    return out


def tolerance(ref) -> np.ndarray:
    """Per-element bound |gpu - ref| <= ulp_bf16(ref) + 1e-3."""
    return bf16_ulp(ref) + 1e-3
