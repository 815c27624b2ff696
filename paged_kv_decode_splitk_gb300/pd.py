"""ctypes binding of libpd (include/pd.h), argument marshalling only.

Every function keeps the C name.  Tensors are torch tensors on the device;
their data pointers, sizes and the current CUDA stream go to the library
unchanged.  Every step of the computation runs in libpd's kernels: there is
no Python or CPU fallback, and a missing library raises `PdLibraryError`.

Negative return codes raise `PdError` (with pd_last_error()'s message);
PD_NOT_APPLICABLE is returned as the value 1 so that the caller can take
another path, like the C convention.
"""

from __future__ import annotations

import ctypes
import os
import re
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libpd.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "pd.h")

PD_OK = 0
PD_NOT_APPLICABLE = 1
PD_ERR_INVALID = -1
PD_ERR_CAPACITY = -2
PD_ERR_WORKSPACE = -3
PD_ERR_CUDA = -4
PD_ERR_ALLOC = -5
PD_ERR_UNSUPPORTED = -6

PD_GQA_PACK_OFF = 0
PD_GQA_PACK_ON = 1
PD_GQA_PACK_SPLITK = 2

PD_POLICY_LEGACY = 0
PD_POLICY_AUTO = 1
PD_POLICY_PINNED = 2

PD_DEV_BAD_BLOCK_ID = 1
PD_DEV_BAD_CONTEXT_LEN = 2
PD_DEV_BAD_TILE_COUNT = 4
PD_DEV_WAIT_TIMEOUT = 8

POLICY_NAMES = {"legacy": PD_POLICY_LEGACY, "auto": PD_POLICY_AUTO, "pinned": PD_POLICY_PINNED}


class PdLibraryError(RuntimeError):
    """libpd.so is missing or unloadable."""


class PdError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"libpd error {code}: {message}")
        self.code = code


class pd_tiled_dims(ctypes.Structure):
    _fields_ = [("max_seqs", ctypes.c_int), ("num_q_heads", ctypes.c_int),
                ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("block_size", ctypes.c_int), ("tile_capacity", ctypes.c_int)]


class pd_tiled_source(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("tile_blocks", ctypes.c_void_p), ("tile_block_counts", ctypes.c_void_p),
                ("blk_stride", ctypes.c_int64), ("tok_stride", ctypes.c_int64),
                ("kvh_stride", ctypes.c_int64), ("last_block_valid_slots", ctypes.c_int)]


_lock = threading.Lock()
_lib = None

_VP = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_SIGS = {
    "pd_last_error": (ctypes.c_char_p, []),
    "pd_build_info": (_I, [_VP, _VP, _VP, _VP]),
    "pd_parse_policy": (_I, [ctypes.c_char_p, _VP, _VP]),
    "pd_parse_gqa_pack": (_I, [ctypes.c_char_p, _VP]),
    "pd_resolve_policy": (_I, [ctypes.c_char_p, ctypes.c_char_p, _VP, _VP]),
    "pd_policy_from_env": (_I, [ctypes.c_char_p, _VP, _VP]),
    "pd_gqa_pack_enabled": (_I, []),
    "pd_split_ref_seqs": (_I, [_I, _I]),
    "pd_legacy_splits": (_I, [_I, _I, _I]),
    "pd_auto_splits": (_I, [_I, _I]),
    "pd_num_splits": (_I, [_I, _I, _I, _I, _I, _I]),
    "pd_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "pd_gqa_pack_shape_ok": (_I, [_I, _I, _I]),
    "pd_gqa_pack_ctas": (_I, [_I, _I]),
    "pd_split_chunk_tokens": (_I, [_I, _I, _I]),
    "pd_decode_attn": (_I, [_VP, _VP, _VP, _VP, _I, _VP, _VP, _I, _I, _I, _I, _I, _I,
                            ctypes.c_float, _I, _VP, _SZ, _I, _VP]),
    "pd_decode_attn_fp8": (_I, [_VP, _VP, _VP, ctypes.c_float, ctypes.c_float, _VP, _I, _VP, _VP, _I, _I,
                                _I, _I, _I, _I, ctypes.c_float, _I, _VP, _SZ, _I, _VP]),
    "pd_decode_attn_noalloc": (_I, [_VP, _VP, _VP, _VP, _I, _VP, _VP, _I, _I, _I, _I, _I, _I,
                                    ctypes.c_float, _I, _I, _VP]),
    "pd_tiled_validate": (_I, [_VP]),
    "pd_tiled_state_bytes": (_I, [_VP, _VP, _VP, _VP, _VP]),
    "pd_tiled_create": (_I, [_VP, _VP]),
    "pd_tiled_destroy": (None, [_VP]),
    "pd_tiled_get_dims": (_I, [_VP, _VP]),
    "pd_tiled_state": (_I, [_VP, _VP, _VP, _VP]),
    "pd_tiled_paged_strides": (None, [_VP, _VP]),
    "pd_tiled_scratch_pool_strides": (None, [_VP, _VP]),
    "pd_tiled_begin": (_I, [_VP, _I, _VP]),
    "pd_tiled_step": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _I, _I64, _I64, _I64, _I, _VP]),
    "pd_tiled_finalize": (_I, [_VP, _VP, _I, _VP]),
    "pd_tiled_run": (_I, [_VP, _VP, _VP, _I, _VP, _I, _VP]),
    "pd_device_status": (_I, [_VP]),
    "pd_debug_fail_next_allocs": (None, [_I]),
    "pd_debug_set_tuning": (None, [_I, _I, _I]),
}


def lib():
    """Load libpd.so (built by `__graft_entry__.build()` / `build.py`)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise PdLibraryError(f"{LIB_PATH} is missing: build it with "
                                     "`python -m paged_kv_decode_splitk_gb300.build`")
            try:
                L = ctypes.CDLL(LIB_PATH)
            except OSError as e:
                raise PdLibraryError(f"cannot load {LIB_PATH}: {e}") from e
            for name, (res, args) in _SIGS.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def header_symbols() -> list[str]:
    """Function names include/pd.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pd_[a-z0-9_]+)\s*\(", text)))


def last_error() -> str:
    return lib().pd_last_error().decode(errors="replace")


def _check(rc: int) -> int:
    if rc < 0:
        raise PdError(rc, last_error())
    return rc


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


# ---- policy -----------------------------------------------------------------

def pd_build_info() -> dict:
    v = [ctypes.c_int() for _ in range(4)]
    _check(lib().pd_build_info(*[ctypes.byref(x) for x in v]))
    return {"max_splits": v[0].value, "pack_width": v[1].value, "pack_head_dim": v[2].value,
            "min_kv_per_split": v[3].value}


def pd_parse_policy(text: str) -> tuple[int, int]:
    pol, pin = ctypes.c_int(), ctypes.c_int()
    _check(lib().pd_parse_policy(text.encode(), ctypes.byref(pol), ctypes.byref(pin)))
    return pol.value, pin.value


def pd_parse_gqa_pack(text: str) -> bool:
    e = ctypes.c_int()
    _check(lib().pd_parse_gqa_pack(text.encode(), ctypes.byref(e)))
    return bool(e.value)


def pd_resolve_policy(declared: str | None, override: str | None) -> tuple[int, int]:
    pol, pin = ctypes.c_int(), ctypes.c_int()
    _check(lib().pd_resolve_policy(None if declared is None else declared.encode(),
                                   None if override is None else override.encode(),
                                   ctypes.byref(pol), ctypes.byref(pin)))
    return pol.value, pin.value


def pd_policy_from_env(declared: str | None) -> tuple[int, int]:
    pol, pin = ctypes.c_int(), ctypes.c_int()
    _check(lib().pd_policy_from_env(None if declared is None else declared.encode(),
                                    ctypes.byref(pol), ctypes.byref(pin)))
    return pol.value, pin.value


def pd_gqa_pack_enabled() -> bool:
    return bool(lib().pd_gqa_pack_enabled())


def pd_split_ref_seqs(num_seqs: int, max_decode_seqs: int) -> int:
    return lib().pd_split_ref_seqs(num_seqs, max_decode_seqs)


def pd_legacy_splits(sm_count: int, num_q_heads: int, ref_seqs: int) -> int:
    return _check(lib().pd_legacy_splits(sm_count, num_q_heads, ref_seqs))


def pd_auto_splits(sm_count: int, num_q_heads: int) -> int:
    return _check(lib().pd_auto_splits(sm_count, num_q_heads))


def pd_num_splits(policy, pin: int, sm_count: int, num_q_heads: int, num_seqs: int,
                  max_decode_seqs: int) -> int:
    if isinstance(policy, str):
        policy = POLICY_NAMES[policy]
    return _check(lib().pd_num_splits(policy, pin, sm_count, num_q_heads, num_seqs, max_decode_seqs))


def pd_workspace_bytes(rows: int, num_q_heads: int, head_dim: int, num_splits: int) -> int:
    return lib().pd_workspace_bytes(rows, num_q_heads, head_dim, num_splits)


def pd_gqa_pack_shape_ok(num_q_heads: int, num_kv_heads: int, head_dim: int) -> bool:
    return bool(lib().pd_gqa_pack_shape_ok(num_q_heads, num_kv_heads, head_dim))


def pd_gqa_pack_ctas(num_kv_heads: int, num_seqs: int) -> int:
    return lib().pd_gqa_pack_ctas(num_kv_heads, num_seqs)


def pd_split_chunk_tokens(context_len: int, num_splits: int, block_size: int) -> int:
    return _check(lib().pd_split_chunk_tokens(context_len, num_splits, block_size))


# ---- paged decode -----------------------------------------------------------------

def pd_decode_attn(q, k_cache, v_cache, block_table, context_lens, out, inv_sqrt_d: float,
                   num_splits: int, workspace=None, gqa_pack: int = 0, stream=None,
                   num_blocks: int | None = None) -> int:
    """out[S, Hq, D] <- paged-decode attention (see pd.h).  Shapes come from the tensors:
    q [S, Hq, D]; k_cache / v_cache [num_blocks, block_size, Hkv, D] BF16; block_table
    [S, max_blocks] int32; context_lens [S] int32; workspace a byte/float tensor or None."""
    S, Hq, D = q.shape
    nb, bs, Hkv, D2 = k_cache.shape
    assert D2 == D, "head_dim mismatch"
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().pd_decode_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                              int(block_table.shape[1]), _ptr(context_lens), _ptr(out), S, Hq, Hkv,
                              D, bs, nb if num_blocks is None else num_blocks, float(inv_sqrt_d),
                              int(num_splits), _ptr(workspace), ws_bytes, int(gqa_pack),
                              _stream(stream))
    return _check(rc)


def pd_decode_attn_fp8(q, k_cache, v_cache, k_scale: float, v_scale: float, block_table, context_lens,
                       out, inv_sqrt_d: float, num_splits: int, workspace=None, gqa_pack: int = 0,
                       stream=None, num_blocks: int | None = None) -> int:
    """pd_decode_attn over an FP8 E4M3 cache: k_cache / v_cache uint8 tensors
    [num_blocks, block_size, Hkv, D] of E4M3 codes, K = value * k_scale, V = value * v_scale."""
    S, Hq, D = q.shape
    nb, bs, Hkv, D2 = k_cache.shape
    assert D2 == D, "head_dim mismatch"
    assert k_cache.element_size() == 1 and v_cache.element_size() == 1, "FP8 caches are 1-byte codes"
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().pd_decode_attn_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), float(k_scale), float(v_scale),
                                  _ptr(block_table), int(block_table.shape[1]), _ptr(context_lens), _ptr(out),
                                  S, Hq, Hkv, D, bs, nb if num_blocks is None else num_blocks,
                                  float(inv_sqrt_d), int(num_splits), _ptr(workspace), ws_bytes,
                                  int(gqa_pack), _stream(stream))
    return _check(rc)


def pd_decode_attn_noalloc(q, k_cache, v_cache, block_table, context_lens, out, inv_sqrt_d: float,
                           num_splits: int, gqa_pack: int = 0, stream=None,
                           num_blocks: int | None = None) -> int:
    """pd_decode_attn with the split-K workspace held by the library (see pd.h): for
    callers that cannot allocate device memory.  Same tensors, shapes and gqa_pack
    modes (0 off, 1 packed non-split, 2 packed with splits), no workspace."""
    S, Hq, D = q.shape
    nb, bs, Hkv, D2 = k_cache.shape
    assert D2 == D, "head_dim mismatch"
    rc = lib().pd_decode_attn_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                      int(block_table.shape[1]), _ptr(context_lens), _ptr(out), S, Hq,
                                      Hkv, D, bs, nb if num_blocks is None else num_blocks,
                                      float(inv_sqrt_d), int(num_splits), int(gqa_pack),
                                      _stream(stream))
    return _check(rc)


# ---- tiled ---------------------------------------------------------------------------

def pd_tiled_validate(dims: pd_tiled_dims) -> None:
    _check(lib().pd_tiled_validate(ctypes.byref(dims)))


def pd_tiled_state_bytes(dims: pd_tiled_dims) -> dict:
    v = [ctypes.c_size_t() for _ in range(4)]
    _check(lib().pd_tiled_state_bytes(ctypes.byref(dims), *[ctypes.byref(x) for x in v]))
    return {"m": v[0].value, "l": v[1].value, "o": v[2].value, "output": v[3].value}


class Tiled:
    """Owner of a pd_tiled handle (TiledAttention): create / begin / step / finalize."""

    def __init__(self, max_seqs, num_q_heads, num_kv_heads, head_dim, block_size, tile_capacity):
        self.dims = pd_tiled_dims(max_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                  tile_capacity)
        self.handle = pd_tiled_create(self.dims)

    def close(self):
        if self.handle:
            pd_tiled_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def paged_strides(self):
        return pd_tiled_paged_strides(self.handle)

    def scratch_pool_strides(self):
        return pd_tiled_scratch_pool_strides(self.handle)

    def begin(self, num_seqs, stream=None):
        return pd_tiled_begin(self.handle, num_seqs, stream)

    def step(self, q, k_pool, v_pool, tile_blocks, tile_block_counts, num_seqs, strides,
             last_block_valid_slots, stream=None):
        return pd_tiled_step(self.handle, q, k_pool, v_pool, tile_blocks, tile_block_counts,
                             num_seqs, strides, last_block_valid_slots, stream)

    def finalize(self, out, num_seqs, stream=None):
        return pd_tiled_finalize(self.handle, out, num_seqs, stream)

    def run(self, q, sources, out, num_seqs, stream=None):
        return pd_tiled_run(self.handle, q, sources, out, num_seqs, stream)

    def state(self):
        return pd_tiled_state(self.handle)


def pd_tiled_create(dims: pd_tiled_dims) -> int:
    h = ctypes.c_void_p()
    _check(lib().pd_tiled_create(ctypes.byref(dims), ctypes.byref(h)))
    return h.value


def pd_tiled_destroy(handle: int) -> None:
    lib().pd_tiled_destroy(handle)


def pd_tiled_get_dims(handle: int) -> pd_tiled_dims:
    d = pd_tiled_dims()
    _check(lib().pd_tiled_get_dims(handle, ctypes.byref(d)))
    return d


def pd_tiled_state(handle: int) -> tuple[int, int, int]:
    m, l_, o = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
    _check(lib().pd_tiled_state(handle, ctypes.byref(m), ctypes.byref(l_), ctypes.byref(o)))
    return m.value, l_.value, o.value


def pd_tiled_paged_strides(handle: int) -> tuple[int, int, int]:
    s = (ctypes.c_int64 * 3)()
    lib().pd_tiled_paged_strides(handle, s)
    return tuple(s)


def pd_tiled_scratch_pool_strides(handle: int) -> tuple[int, int, int]:
    s = (ctypes.c_int64 * 3)()
    lib().pd_tiled_scratch_pool_strides(handle, s)
    return tuple(s)


def pd_tiled_begin(handle: int, num_seqs: int, stream=None) -> int:
    return _check(lib().pd_tiled_begin(handle, num_seqs, _stream(stream)))


def pd_tiled_step(handle: int, q, k_pool, v_pool, tile_blocks, tile_block_counts, num_seqs: int,
                  strides, last_block_valid_slots: int, stream=None) -> int:
    blk, tok, kvh = (int(x) for x in strides)
    return _check(lib().pd_tiled_step(handle, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(tile_blocks),
                                      _ptr(tile_block_counts), num_seqs, blk, tok, kvh,
                                      int(last_block_valid_slots), _stream(stream)))


def pd_tiled_run(handle: int, q, sources, out, num_seqs: int, stream=None) -> int:
    """begin, one step per source, finalize.  sources: sequence of
    (k_pool, v_pool, tile_blocks, tile_block_counts, strides, last_block_valid_slots)."""
    arr = (pd_tiled_source * max(1, len(sources)))()
    for i, (k, v, tb, tc, strides, lbvs) in enumerate(sources):
        blk, tok, kvh = (int(x) for x in strides)
        arr[i] = pd_tiled_source(_ptr(k), _ptr(v), _ptr(tb), _ptr(tc), blk, tok, kvh, int(lbvs))
    return _check(lib().pd_tiled_run(handle, _ptr(q), ctypes.cast(arr, _VP) if sources else None,
                                     len(sources), _ptr(out), num_seqs, _stream(stream)))


def pd_tiled_finalize(handle: int, out, num_seqs: int, stream=None) -> int:
    return _check(lib().pd_tiled_finalize(handle, _ptr(out), num_seqs, _stream(stream)))


# ---- diagnostics -------------------------------------------------------------------

def pd_device_status() -> int:
    f = ctypes.c_int()
    _check(lib().pd_device_status(ctypes.byref(f)))
    return f.value


def pd_debug_fail_next_allocs(count: int) -> None:
    lib().pd_debug_fail_next_allocs(count)


def pd_debug_set_tuning(stages_per_warp: int = 0, cluster: int = 0, longest_first: int = -1) -> None:
    lib().pd_debug_set_tuning(stages_per_warp, cluster, longest_first)
