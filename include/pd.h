/*
 * pd.h -- C ABI of libpd, paged-decode split-K attention for GB300 (sm_103a).
 *
 * The library computes, for every sequence s and query head h,
 *
 *     out[s,h,:] = softmax(q[s,h,:] . K[s,kvh,:,:]^T * inv_sqrt_d) . V[s,kvh,:,:]
 *
 * over a BF16 KV cache paged in blocks (or one of FP8 E4M3 codes with
 * per-tensor scales, pd_decode_attn_fp8), with grouped-query sharing
 * (kvh = h / (num_q_heads / num_kv_heads)), and writes BF16; a sequence with
 * no token gets 0.  Sources: the "Module attn_splitk" documentation page
 * (split-K launch geometry, the split-K workspace of [o, m, l] slots, the
 * GQA-packed gate) and the "metrale_storage/tiled_attention.rs" page (the
 * begin_step / step_tile / finalize fold and its two K/V layouts).
 *
 * Conventions for every entry point:
 *   - Ownership: the caller owns every buffer it passes (device memory for
 *     tensors, host memory for scalars and out-parameters).  The library owns
 *     only the tiled state it allocates in pd_tiled_create.
 *   - Asynchrony: launches are enqueued on `stream` (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream) and return without waiting.
 *     Nothing on the compute path synchronises or allocates.
 *   - Errors: functions return PD_OK (0), PD_NOT_APPLICABLE (1: nothing was
 *     launched, the caller should take another path; the "launcher returns
 *     Ok(false)" convention of the prefill_attn_fa128.rs page), or a negative
 *     PD_ERR_* code.  pd_last_error() then holds a message (thread-local).
 *     Launch failures are reported as PD_ERR_CUDA.  Faults inside a kernel
 *     (a block id outside the cache, a context length larger than the block
 *     table, a tile count above the capacity, a bounded wait that ran out)
 *     never trap: the kernel records a PD_DEV_* flag, reads zeros in place
 *     of the bad data, and pd_device_status() reports the flags.
 *   - There is no CPU fallback: without a CUDA device the compute entry
 *     points return PD_ERR_CUDA.
 */
#ifndef PD_H
#define PD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

/* ---- build constants ------------------------------------------------------
 * PD_MAX_DECODE_SPLITS: ceiling on the split count under every policy but
 *   Legacy (Module attn_splitk page, constant MAX_DECODE_SPLITS; the page
 *   prints no value and implies at least 13; this build uses 16).
 * PD_SPLITK_TARGET_WAVES: waves of CTAs Auto aims for (constant
 *   SPLITK_TARGET_WAVES; 2, from "2 * sm_count / num_q_heads").
 * PD_GQA_PACK_WIDTH / PD_GQA_PACK_HEAD_DIM: query heads one packed unit
 *   serves and the head dim it is compiled for (constants
 *   DECODE_GQA_PACK_WIDTH and DECODE_GQA_PACK_HEAD_DIM: PD_GQA and PD_HDIM).
 * PD_MIN_KV_PER_SPLIT: floor on a sequence's split size in tokens (module
 *   description: PD_MIN_KV_PER_SPLIT; value not printed, this build uses 256).
 * PD_MAX_HEAD_DIM: largest head dim (TiledAttentionDims::validate, 256).
 */
#define PD_MAX_DECODE_SPLITS 16
#define PD_SPLITK_TARGET_WAVES 2
#define PD_GQA_PACK_WIDTH 8
#define PD_GQA_PACK_HEAD_DIM 256

/* Values of pd_decode_attn's gqa_pack argument. */
#define PD_GQA_PACK_OFF 0
#define PD_GQA_PACK_ON 1
#define PD_GQA_PACK_SPLITK 2
#define PD_MIN_KV_PER_SPLIT 256
#define PD_MAX_HEAD_DIM 256

/* ---- status codes ---- */
#define PD_OK 0
#define PD_NOT_APPLICABLE 1
#define PD_ERR_INVALID (-1)     /* an argument is out of range or inconsistent */
#define PD_ERR_CAPACITY (-2)    /* num_seqs above the tiled state's max_seqs */
#define PD_ERR_WORKSPACE (-3)   /* split-K workspace missing or too small */
#define PD_ERR_CUDA (-4)        /* a CUDA call failed (no device, launch error) */
#define PD_ERR_ALLOC (-5)       /* pd_tiled_create could not allocate its state */
#define PD_ERR_UNSUPPORTED (-6) /* a legal shape this build has no kernel for */

/* ---- device status flags (pd_device_status) ---- */
#define PD_DEV_BAD_BLOCK_ID 1    /* a block id outside [0, num_blocks): zeros were read */
#define PD_DEV_BAD_CONTEXT_LEN 2 /* a context length < 0 or > max_blocks_per_seq*block_size: clamped */
#define PD_DEV_BAD_TILE_COUNT 4  /* a tile_block_counts entry < 0 or > tile_capacity: clamped */
#define PD_DEV_WAIT_TIMEOUT 8    /* a bounded wait on a copy ran out: that output is garbage */

/* Split-count policies (Module attn_splitk page, enum SplitkPolicy). */
typedef enum { PD_POLICY_LEGACY = 0, PD_POLICY_AUTO = 1, PD_POLICY_PINNED = 2 } pd_policy;

/* Message of the last failing call on this thread ("" if none).  Owned by the
 * library, valid until the next call on the same thread. */
const char *pd_last_error(void);

/* The build constants above, as compiled into the kernels (each pointer may
 * be NULL).  The kernels' own compile-time pack width and head dim are the
 * values reported, so a header/kernel mismatch is detectable.  Returns PD_OK. */
int pd_build_info(int *max_splits, int *pack_width, int *pack_head_dim, int *min_kv_per_split);

/* ---- policy (pure host functions; no CUDA) ------------------------------ */

/* Parse a split-K policy word (Module attn_splitk page, function parse):
 * "legacy" | "auto" | "0"/"off"/"false"/"no" (split-K off: Pinned(1)) |
 * a decimal count, clamped to 1..PD_MAX_DECODE_SPLITS; surrounding white
 * space ignored, case-insensitive.  On success writes *policy (a pd_policy)
 * and *pin (0 unless Pinned) and returns PD_OK; else PD_ERR_INVALID. */
int pd_parse_policy(const char *text, int *policy, int *pin);

/* Parse a GQA-pack switch (function parse_gqa_pack): "1"/"on"/"true"/"yes"
 * -> 1, "0"/"off"/"false"/"no" -> 0, trimmed and case-insensitive.
 * Returns PD_OK or PD_ERR_INVALID. */
int pd_parse_gqa_pack(const char *text, int *enabled);

/* Resolve a target's declared policy against an override (function
 * resolve_policy): a parseable override wins; else the declaration; an
 * unparseable (or NULL) declaration is Legacy.  Returns PD_OK. */
int pd_resolve_policy(const char *declared, const char *override_text, int *policy, int *pin);

/* pd_resolve_policy against the environment variable PD_ATTN_DECODE_SPLITK
 * (function policy_from_env).  Reads the environment on every call. */
int pd_policy_from_env(const char *declared, int *policy, int *pin);

/* Whether the GQA-packed pass is armed in this process (function
 * gqa_pack_enabled): declared off, overridden by a parseable
 * PD_ATTN_DECODE_GQA_PACK.  Resolved once, on the first call, and fixed for
 * the life of the process so that captured CUDA graphs stay consistent
 * with later launches.  Returns 0 or 1. */
int pd_gqa_pack_enabled(void);

/* max(max_decode_seqs, num_seqs) (function legacy_splits). */
int pd_split_ref_seqs(int num_seqs, int max_decode_seqs);

/* Legacy rule (module description): ctas = num_q_heads*ref_seqs;
 * 1 if ctas >= sm_count, else sm_count / ctas.  Not clamped.
 * Returns >= 1, or PD_ERR_INVALID for non-positive arguments. */
int pd_legacy_splits(int sm_count, int num_q_heads, int ref_seqs);

/* Auto rule (function auto_splits):
 * clamp(ceil(PD_SPLITK_TARGET_WAVES*sm_count/num_q_heads), 1, PD_MAX_DECODE_SPLITS).
 * Returns >= 1, or PD_ERR_INVALID. */
int pd_auto_splits(int sm_count, int num_q_heads);

/* Split count of a launch (function num_splits).  Auto and Pinned read only
 * (sm_count, num_q_heads) and pin; only Legacy reads num_seqs and
 * max_decode_seqs.  A pin is clamped to 1..PD_MAX_DECODE_SPLITS.
 * Returns >= 1, or PD_ERR_INVALID. */
int pd_num_splits(int policy, int pin, int sm_count, int num_q_heads, int num_seqs,
                  int max_decode_seqs);

/* Bytes of the split-K workspace (constant MAX_DECODE_SPLITS and function
 * workspace_slots): rows * num_q_heads * num_splits * (head_dim + 2) FP32
 * values, one [o[head_dim], m, l] slot per (row, q head, split).
 * Returns 0 for non-positive arguments. */
size_t pd_workspace_bytes(int rows, int num_q_heads, int head_dim, int num_splits);

/* GQA-pack shape gate (function gqa_pack_shape_ok): 1 iff num_kv_heads > 0,
 * num_q_heads == num_kv_heads * PD_GQA_PACK_WIDTH and
 * head_dim == PD_GQA_PACK_HEAD_DIM; else 0. */
int pd_gqa_pack_shape_ok(int num_q_heads, int num_kv_heads, int head_dim);

/* Units a packed launch serves (function gqa_pack_ctas): num_kv_heads * num_seqs. */
int pd_gqa_pack_ctas(int num_kv_heads, int num_seqs);

/* Tokens per split for one sequence: the split size floored at
 * PD_MIN_KV_PER_SPLIT (module description), i.e.
 * roundup(max(ceil(context_len/num_splits), PD_MIN_KV_PER_SPLIT), block_size).
 * Split i covers [i*chunk, min((i+1)*chunk, context_len)).  This is the
 * function the kernels use.  Returns > 0, or PD_ERR_INVALID. */
int pd_split_chunk_tokens(int context_len, int num_splits, int block_size);

/* ---- paged decode --------------------------------------------------------
 * pd_decode_attn: one decode step of paged attention.
 *   q            [num_seqs, num_q_heads, head_dim] BF16, contiguous, 16-B aligned.
 *   k_cache,
 *   v_cache      [num_blocks, block_size, num_kv_heads, head_dim] BF16, contiguous,
 *                16-B aligned.
 *   block_table  [num_seqs, max_blocks_per_seq] int32: physical block of each
 *                sequence's j-th block of block_size tokens.
 *   context_lens [num_seqs] int32: tokens of each sequence (0 allowed).
 *   out          [num_seqs, num_q_heads, head_dim] BF16, written in full.
 *   inv_sqrt_d   the softmax scale applied to q.k.
 *   num_splits   split count (pd_num_splits); each sequence's range is cut into
 *                pd_split_chunk_tokens-sized chunks; >= 1.
 *   workspace    device buffer of >= pd_workspace_bytes(num_seqs, num_q_heads,
 *                head_dim, num_splits) bytes, 16-B aligned; may be NULL when
 *                num_splits == 1.  Contents on entry are ignored; on return they
 *                are scratch.
 *   gqa_pack     PD_GQA_PACK_OFF (0): split-K path.  PD_GQA_PACK_ON (1): the
 *                GQA-packed pass; it applies only when num_splits == 1 and
 *                pd_gqa_pack_shape_ok(), otherwise the call returns
 *                PD_NOT_APPLICABLE and launches nothing.  PD_GQA_PACK_SPLITK (2):
 *                the packed pass with any split count (no counterpart on the
 *                pages, which gate packing to non-split launches): same shape
 *                gate, and with num_splits > 1 each (sequence, KV head, split)
 *                writes its partial to the workspace and the merge pass folds
 *                them, exactly as on the split-K path.
 * Shape limits: num_q_heads a positive multiple of num_kv_heads; head_dim a
 * multiple of 8 in [8, 256]; block_size a multiple of 16 in [16, 256].
 * Every path serves a whole group of query heads from one read of K and V,
 * and a sequence's output bits depend only on its own data and num_splits,
 * never on the other sequences of the batch.
 * Returns PD_OK, PD_NOT_APPLICABLE, PD_ERR_INVALID, PD_ERR_WORKSPACE,
 * PD_ERR_UNSUPPORTED or PD_ERR_CUDA. */
int pd_decode_attn(const void *q, const void *k_cache, const void *v_cache,
                   const int32_t *block_table, int max_blocks_per_seq,
                   const int32_t *context_lens, void *out, int num_seqs, int num_q_heads,
                   int num_kv_heads, int head_dim, int block_size, int num_blocks,
                   float inv_sqrt_d, int num_splits, void *workspace, size_t workspace_bytes,
                   int gqa_pack, void *stream);

/* Paged-decode attention over an FP8 KV cache (Module attn_splitk page: the
 * dispatch serves "BF16 and FP8" paged-decode launches; the page gives no
 * format or scale, so this build reads it as OCP FP8 E4M3 codes with one FP32
 * scale per tensor).
 *   k_cache, v_cache  [num_blocks, block_size, num_kv_heads, head_dim] E4M3
 *                     codes (1 byte each), 16-B aligned; the keys and values
 *                     are code value * k_scale and code value * v_scale.
 *   k_scale, v_scale  finite FP32 scales.
 * Every other argument, the split geometry, the packed modes, the workspace
 * and the output are those of pd_decode_attn (q stays BF16, out is BF16).
 * head_dim must be a multiple of 16 (PD_ERR_UNSUPPORTED otherwise).  The two
 * E4M3 NaN codes are not valid cache contents.
 * Returns PD_OK, PD_NOT_APPLICABLE, PD_ERR_INVALID, PD_ERR_WORKSPACE,
 * PD_ERR_UNSUPPORTED or PD_ERR_CUDA. */
int pd_decode_attn_fp8(const void *q, const void *k_cache, const void *v_cache, float k_scale,
                       float v_scale, const int32_t *block_table, int max_blocks_per_seq,
                       const int32_t *context_lens, void *out, int num_seqs, int num_q_heads,
                       int num_kv_heads, int head_dim, int block_size, int num_blocks, float inv_sqrt_d,
                       int num_splits, void *workspace, size_t workspace_bytes, int gqa_pack, void *stream);

/* Size of the library-owned split-K workspace behind pd_decode_attn_noalloc. */
#define PD_NOALLOC_WORKSPACE_BYTES 16777216u /* 16 MiB */

/* pd_decode_attn_noalloc: pd_decode_attn for callers that cannot allocate
 * device memory.  The pages this library follows describe no counterpart; it
 * exists for code that must not call cudaMalloc on the decode path: an
 * application whose device memory is all reserved up front by its own pool
 * allocator, or a plug-in that may not grow the host program's footprint,
 * and any caller for whom the implicit device synchronisation and locking of
 * cudaMalloc / cudaFree are not acceptable there.
 *
 * Arguments, shapes, results and error codes are those of pd_decode_attn
 * without workspace / workspace_bytes: the split-K workspace is a fixed
 * PD_NOALLOC_WORKSPACE_BYTES array in libpd's device code, which a GPU holds
 * from the moment that code is loaded on it until the process exits.  A
 * launch whose workspace (pd_workspace_bytes(num_seqs, num_q_heads, head_dim,
 * num_splits), 0 when num_splits == 1) would exceed that size is rejected
 * with PD_ERR_WORKSPACE and launches nothing.  The call itself allocates
 * nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 *
 * Set-up: the first call with num_splits > 1 on a device looks up that
 * device's address of the array (cudaGetSymbolAddress, with the device
 * current).  Under the CUDA driver's lazy module loading (the default since
 * CUDA 12) that lookup is also what loads the array into the device's memory,
 * so the 16 MiB are taken then, not when the library is opened.  Make that
 * first call at start-up, while the memory is still free and before any
 * stream capture; later calls only read the cached address.  All calls on a
 * device share the one array and
 * it keeps the previous call's contents; no part of it needs to start at zero
 * (every value a call reads is written earlier in the same call), but two
 * calls whose kernels overlap on the GPU, on different streams or from
 * different threads, race on it and may produce garbage: serialise them. */
int pd_decode_attn_noalloc(const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *block_table, int max_blocks_per_seq,
                           const int32_t *context_lens, void *out, int num_seqs,
                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           int num_blocks, float inv_sqrt_d, int num_splits, int gqa_pack,
                           void *stream);

/* ---- tiled decode (tiled_attention.rs page) ------------------------------ */

/* TiledAttentionDims: the state is sized for max_seqs sequences. */
typedef struct pd_tiled_dims {
    int max_seqs;
    int num_q_heads;
    int num_kv_heads;
    int head_dim;      /* multiple of 8, <= 256 */
    int block_size;    /* multiple of 16, <= 256 */
    int tile_capacity; /* blocks one step_tile call may fold per sequence */
} pd_tiled_dims;

typedef struct pd_tiled pd_tiled;

/* TiledAttentionDims::validate: num_kv_heads > 0 dividing num_q_heads,
 * head_dim <= 256, plus this build's shape limits.  Returns PD_OK or
 * PD_ERR_INVALID / PD_ERR_UNSUPPORTED. */
int pd_tiled_validate(const pd_tiled_dims *dims);

/* Byte sizes of the state (TiledAttentionDims m_bytes, l_bytes, o_bytes,
 * output_bytes): max_seqs*Hq*4, the same, *head_dim*4, *head_dim*2.
 * Any pointer may be NULL.  Returns PD_OK or PD_ERR_INVALID. */
int pd_tiled_state_bytes(const pd_tiled_dims *dims, size_t *m_bytes, size_t *l_bytes,
                         size_t *o_bytes, size_t *output_bytes);

/* TiledAttention::new: validate and allocate, once, on the current device, the
 * FP32 running state (m, l, o) and the buffer pd_tiled_run keeps the per-call
 * partials of one step in (max_seqs * num_q_heads * 8 * (head_dim + 2)
 * floats: one [o, m, l] slot per row for each of up to 8 calls), so that no
 * later call on the handle allocates.  *out receives the handle.  Returns
 * PD_OK, PD_ERR_INVALID, PD_ERR_UNSUPPORTED, PD_ERR_ALLOC or PD_ERR_CUDA. */
int pd_tiled_create(const pd_tiled_dims *dims, pd_tiled **out);

/* Free the state (NULL is a no-op).  Synchronises the device first. */
void pd_tiled_destroy(pd_tiled *t);

/* The dims the handle was created with.  Returns PD_OK or PD_ERR_INVALID. */
int pd_tiled_get_dims(const pd_tiled *t, pd_tiled_dims *dims);

/* Device addresses of the running state: m [max_seqs, Hq], l [max_seqs, Hq],
 * o [max_seqs, Hq, head_dim], FP32, owned by the handle (for inspection). */
int pd_tiled_state(const pd_tiled *t, void **m, void **l, void **o);

/* TiledAttention::paged_strides: (blk, tok, kvh) element strides of
 * [num_blocks, block_size, Hkv, head_dim]. */
void pd_tiled_paged_strides(const pd_tiled *t, int64_t strides[3]);

/* TiledAttention::scratch_pool_strides: (blk, tok, kvh) element strides of
 * the scratch pool [slot, K|V, Hkv, block_size, head_dim]; V of a slot
 * starts Hkv*block_size*head_dim elements after its K. */
void pd_tiled_scratch_pool_strides(const pd_tiled *t, int64_t strides[3]);

/* TiledAttention::begin_step: set (m, l, o) of the first num_seqs sequences to
 * (-inf, 0, 0) on `stream`.  Returns PD_OK, PD_ERR_CAPACITY
 * (num_seqs > max_seqs), PD_ERR_INVALID or PD_ERR_CUDA. */
int pd_tiled_begin(pd_tiled *t, int num_seqs, void *stream);

/* TiledAttention::step_tile: fold one tile of KV blocks per sequence into the
 * running state.
 *   q                 [num_seqs, Hq, head_dim] BF16, 16-B aligned.
 *   k_pool, v_pool    bases of K and V (16-B aligned); the K row of token tok
 *                     of block blk for KV head kvh starts at element
 *                     blk*blk_stride + tok*tok_stride + kvh*kvh_stride.
 *                     The strides must be multiples of 8 elements (16 B).
 *   tile_blocks       [num_seqs, tile_capacity] int32 block ids.
 *   tile_block_counts [num_seqs] int32, each in 0..tile_capacity.
 *   last_block_valid_slots  tokens held by the last block of each sequence's
 *                     tile (1..block_size-1); any other value means full.
 * The scale is 1/sqrt(head_dim) rounded to FP32 (step_tile has no scale).
 * Returns PD_OK, PD_ERR_CAPACITY, PD_ERR_INVALID or PD_ERR_CUDA. */
int pd_tiled_step(pd_tiled *t, const void *q, const void *k_pool, const void *v_pool,
                  const int32_t *tile_blocks, const int32_t *tile_block_counts, int num_seqs,
                  int64_t blk_stride, int64_t tok_stride, int64_t kvh_stride,
                  int last_block_valid_slots, void *stream);

/* TiledAttention::finalize: out [num_seqs, Hq, head_dim] BF16 = o / l, and 0
 * where l is 0.  Returns PD_OK, PD_ERR_CAPACITY, PD_ERR_INVALID or PD_ERR_CUDA. */
int pd_tiled_finalize(pd_tiled *t, void *out, int num_seqs, void *stream);

/* One step_tile call of a multi-call step: the pools, tile list and strides
 * that call reads (tiled_attention.rs page: step_tile takes them per call, so
 * one step may mix sources, e.g. resident blocks in the paged cache and
 * swapped-in blocks in the scratch pool).  Fields as for pd_tiled_step. */
typedef struct pd_tiled_source {
    const void *k_pool;
    const void *v_pool;
    const int32_t *tile_blocks;        /* [num_seqs, tile_capacity] int32 */
    const int32_t *tile_block_counts;  /* [num_seqs] int32 */
    int64_t blk_stride;
    int64_t tok_stride;
    int64_t kvh_stride;
    int last_block_valid_slots;
} pd_tiled_source;

/* A whole tiled decode step in one call: begin_step, one step_tile per source
 * in array order, finalize into out [num_seqs, Hq, head_dim] BF16 (the
 * tiled_attention.rs page's per-step sequence, driven from one place).  Every
 * source is checked before anything launches, so an invalid argument leaves
 * the running state and `out` untouched.  The result equals one begin, the
 * steps and one finalize made separately (same kernels, same order).
 * num_sources may be 0 (out = 0).  With 1..8 sources the step runs as two
 * launches (every call's tile at once, writing each call's partial to the
 * handle's partials buffer, then the in-order fold and finalize) instead of
 * 2 + num_sources.  Nothing is allocated: any call, the first included, may
 * be captured in a CUDA graph.
 * Returns PD_OK, PD_ERR_CAPACITY, PD_ERR_INVALID or PD_ERR_CUDA. */
int pd_tiled_run(pd_tiled *t, const void *q, const pd_tiled_source *sources, int num_sources,
                 void *out, int num_seqs, void *stream);

/* ---- diagnostics ---- */

/* Synchronise the current device, then read and clear the PD_DEV_* flags the
 * kernels recorded on it since the last call.  Not for the hot path.
 * Returns PD_OK or PD_ERR_CUDA. */
int pd_device_status(int *flags);

/* ---- test hooks ----
 * Not part of the decode interface: the test suite and launch-shape
 * experiments use them.  A program that serves decode steps never needs to
 * call either. */

/* TEST HOOK.  Make the next `count` device allocations of pd_tiled_create
 * (state m, l, o, then the run partials) fail as if the device were out of
 * memory (host-side fault injection). */
void pd_debug_fail_next_allocs(int count);

/* TEST HOOK.  Tuning for launch-shape experiments, applied to the following launches
 * in this process: pipeline stages per warp (1..8; 0 = built-in), where the
 * parts of a unit run (0 = chosen from occupancy, 1 = one CTA per unit, > 1 =
 * one CTA per part in a thread-block cluster) and longest-first service order
 * of small batches (0/1; -1 = built-in).  None of them changes the output
 * bits: the parts and their fold order depend only on each sequence. */
void pd_debug_set_tuning(int stages_per_warp, int cluster, int longest_first);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif

#ifdef __cplusplus
}
#endif

#endif /* PD_H */
