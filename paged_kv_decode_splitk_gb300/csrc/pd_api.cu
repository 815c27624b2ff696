// pd_api.cu -- the C ABI of libpd (declared in include/pd.h): argument
// validation, the split-K launch-geometry policy, TMA tensor-map encoding,
// kernel dispatch and the tiled state.  Host code; the kernels live in
// pd_unit_d*.cu and pd_small.cu.
#include <cudaTypedefs.h>
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cctype>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "pd.h"
#include "pd_internal.h"

namespace {

// ---- errors -------------------------------------------------------------------
thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int ok() {
    g_err[0] = '\0';
    return PD_OK;
}

int cuda_fail(cudaError_t e, const char *what) {
    (void)cudaGetLastError();  // reported here: do not leave it for the next launch check
    return fail(PD_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Largest dynamic shared memory a block may opt in to on the current device.
int max_smem_optin() {
    static std::mutex mu;
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!cached[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            (void)cudaGetLastError();
        cached[dev] = v;
    }
    return cached[dev];
}

// ---- text -----------------------------------------------------------------------
std::string trim_lower(const char *text) {
    std::string s = text ? text : "";
    size_t a = 0, b = s.size();
    while (a < b && std::isspace(static_cast<unsigned char>(s[a]))) ++a;
    while (b > a && std::isspace(static_cast<unsigned char>(s[b - 1]))) --b;
    std::string out = s.substr(a, b - a);
    for (char &c : out) c = static_cast<char>(std::tolower(static_cast<unsigned char>(c)));
    return out;
}

bool is_off_word(const std::string &w) { return w == "0" || w == "off" || w == "false" || w == "no"; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- device status word ------------------------------------------------------------
__device__ unsigned int g_status;

std::mutex g_status_mu;
unsigned int *g_status_ptr[64] = {nullptr};

unsigned int *status_ptr(int *err) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        *err = cuda_fail(e == cudaSuccess ? cudaErrorInvalidDevice : e, "cudaGetDevice");
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_status_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_status);
        if (e != cudaSuccess) {
            *err = cuda_fail(e, "cudaGetSymbolAddress(status)");
            return nullptr;
        }
        g_status_ptr[dev] = static_cast<unsigned int *>(p);
    }
    *err = PD_OK;
    return g_status_ptr[dev];
}

// ---- TMA tensor maps -------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                        cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else if (g_encode_err == cudaSuccess)
            g_encode_err = cudaErrorSymbolNotFound;
    });
    return g_encode;
}

// A 4-D view of one K (or V) pool: dim 0 the head_dim columns, then the token
// and KV-head axes in increasing stride order, then the block axis.  Box: 64
// columns x 16 tokens x 1 head x 1 block, 128-byte swizzle; out-of-range
// coordinates read zeros.  *tok_dim receives the dimension holding tokens.
// Encoded maps are cached by their full description (a map depends on nothing
// else), so repeated launches over the same cache skip the host-side encode.
struct KvMapKey {
    const void *base;
    int head_dim, block_size, num_kv_heads, elem, box_cols, swz128;
    long long num_blocks, blk_stride, tok_stride, kvh_stride;
    bool operator==(const KvMapKey &o) const {
        return base == o.base && head_dim == o.head_dim && block_size == o.block_size &&
               num_kv_heads == o.num_kv_heads && elem == o.elem && box_cols == o.box_cols && swz128 == o.swz128 &&
               num_blocks == o.num_blocks && blk_stride == o.blk_stride && tok_stride == o.tok_stride &&
               kvh_stride == o.kvh_stride;
    }
};
struct KvMapEntry {
    KvMapKey key;
    CUtensorMap map;
    int tok_dim;
    unsigned long long stamp;
};
constexpr int kMapCache = 32;
std::mutex g_map_mu;
KvMapEntry g_maps[kMapCache];
unsigned long long g_map_clock = 0;

int encode_kv_map_uncached(CUtensorMap *map, int *tok_dim, const void *base, int head_dim,
                           int block_size, int num_kv_heads, long long num_blocks,
                           long long blk_stride, long long tok_stride, long long kvh_stride, int elem,
                           int box_cols, int swz128);

// 4-D tensor map of a K or V view (strides in elements), boxes of box_cols
// columns x 16 tokens.  elem 2: BF16, 64 columns with the 128-byte swizzle;
// elem 1: FP8 E4M3 codes, either 128 columns with the 128-byte swizzle (the K
// operand read straight from the tile) or one unswizzled box of the padded head
// dim (V, converted to f16 first; every FP8 tile at head dim 64).
int encode_kv_map(CUtensorMap *map, int *tok_dim, const void *base, int head_dim, int block_size,
                  int num_kv_heads, long long num_blocks, long long blk_stride, long long tok_stride,
                  long long kvh_stride, int elem = 2, int box_cols = pd::kBoxCols, int swz128 = 1) {
    const KvMapKey key = {base, head_dim, block_size, num_kv_heads, elem, box_cols, swz128, num_blocks,
                          blk_stride, tok_stride, kvh_stride};
    std::lock_guard<std::mutex> lock(g_map_mu);
    int victim = 0;
    for (int i = 0; i < kMapCache; ++i) {
        if (g_maps[i].stamp != 0 && g_maps[i].key == key) {
            g_maps[i].stamp = ++g_map_clock;
            *map = g_maps[i].map;
            *tok_dim = g_maps[i].tok_dim;
            return PD_OK;
        }
        if (g_maps[i].stamp < g_maps[victim].stamp) victim = i;
    }
    int rc = encode_kv_map_uncached(map, tok_dim, base, head_dim, block_size, num_kv_heads, num_blocks,
                                    blk_stride, tok_stride, kvh_stride, elem, box_cols, swz128);
    if (rc != PD_OK) return rc;
    g_maps[victim].key = key;
    g_maps[victim].map = *map;
    g_maps[victim].tok_dim = *tok_dim;
    g_maps[victim].stamp = ++g_map_clock;
    return PD_OK;
}

int encode_kv_map_uncached(CUtensorMap *map, int *tok_dim, const void *base, int head_dim,
                           int block_size, int num_kv_heads, long long num_blocks,
                           long long blk_stride, long long tok_stride, long long kvh_stride, int elem,
                           int box_cols, int swz128) {
    auto enc = encoder();
    if (!enc) return cuda_fail(g_encode_err, "cuTensorMapEncodeTiled entry point");
    const bool tok_first = tok_stride <= kvh_stride;
    cuuint64_t dims[4];
    cuuint64_t strides[3];
    cuuint32_t box[4];
    cuuint32_t estr[4] = {1, 1, 1, 1};
    dims[0] = static_cast<cuuint64_t>(head_dim);
    box[0] = static_cast<cuuint32_t>(box_cols);
    if (tok_first) {
        dims[1] = block_size;
        strides[0] = static_cast<cuuint64_t>(tok_stride) * elem;
        box[1] = pd::kTileTokens;
        dims[2] = num_kv_heads;
        strides[1] = static_cast<cuuint64_t>(kvh_stride) * elem;
        box[2] = 1;
    } else {
        dims[1] = num_kv_heads;
        strides[0] = static_cast<cuuint64_t>(kvh_stride) * elem;
        box[1] = 1;
        dims[2] = block_size;
        strides[1] = static_cast<cuuint64_t>(tok_stride) * elem;
        box[2] = pd::kTileTokens;
    }
    dims[3] = static_cast<cuuint64_t>(num_blocks);
    strides[2] = static_cast<cuuint64_t>(blk_stride) * elem;
    box[3] = 1;
    CUresult r = enc(map, elem == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                     const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swz128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PD_ERR_INVALID,
                    "cuTensorMapEncodeTiled rejected the K/V view (error %d): base %p, strides "
                    "(blk %lld, tok %lld, kvh %lld) elements",
                    static_cast<int>(r), base, blk_stride, tok_stride, kvh_stride);
    *tok_dim = tok_first ? 1 : 2;
    return PD_OK;
}

// ---- launch choices ----------------------------------------------------------------
// Stages per warp of the unit pipeline.  A single-wave launch keeps about
// 32-64 KB of K/V in flight per CTA so that three or four CTAs share an SM.  A
// launch of several waves of one-CTA units keeps one stage at D = 128 too, so
// that four CTAs share an SM (measured A/B on the large-batch workload: 494 us
// at one stage against 512 us at two and 615 us at three); at D = 64 it
// doubles the ring, and over an FP8 cache two stages and one run alike.
int g_debug_stages = 0;
int g_debug_cluster = 0;
int g_debug_lpt = -1;

int default_stages(int dpad, bool kv8 = false) {
    if (g_debug_stages > 0) return g_debug_stages;
    if (kv8) return dpad <= 128 ? 2 : 1;  // an FP8 tile is half a BF16 one
    return dpad <= 64 ? 2 : 1;
}

int default_stages_seq(int dpad, bool kv8 = false) {
    if (g_debug_stages > 0) return g_debug_stages;
    if (kv8) return 2;  // measured: 4 stages cost a CTA per SM at D = 128
    return dpad <= 64 ? 2 : 1;
}

// Longest-first service order for small batches (a scheduling choice only).
int default_lpt(int num_seqs) {
    const int on = g_debug_lpt >= 0 ? g_debug_lpt : 1;
    return on && num_seqs > 1 && num_seqs <= pd::kLptMaxSeqs ? 1 : 0;
}

// A unit's range (one split of a sequence, or one tile of it) is cut into up
// to max_parts parts of about pd::kPartTiles 16-token tiles, by its own
// length; the parts fold in order.  Build constants: they fix the summation
// order.
// K/V tiles at the start of its part that a paged-mode CTA of a one-wave launch
// prefetches into L2 before it waits for the previous kernel (a scheduling
// hint: it changes no result): as many tiles as 128 KB of a BF16 cache holds
// (a 16-token K+V tile is 64 * dpad bytes), for an FP8 cache the same number
// of tiles.  Measured on one box, A/B: 64 / 192 / 256 / 384 / 512 KB of BF16
// tiles were slower on the long-context, packed and packed-with-splits steps
// (up to 15%); over an FP8 cache, the same tile count (64 KB) beat 128 KB by 4%
// on the packed step and 1% on the long-context one.
constexpr int kPrefetchBytes = 128 * 1024;
// Cluster sizes (every unit of a cluster launch gets max_parts ranks, and the
// ranks beyond its parts only hold a slot until they see its length):
// * D <= 128: five for BF16 (a 158-tile split in 5 CTAs of 4 warps still fits
//   one wave at 4 CTAs per SM: measured 27.3 -> 26.9 us on the long-context
//   workload; 3 and 4 were slower), four for FP8 (3 CTAs per SM there; 3 and
//   5 slower).
// * D = 256: seven, so that 64 packed units x 7 CTAs fit the 456 slots of one
//   wave (measured on the packed step against 8: BF16 31.9 -> 30.9 us, FP8
//   27.6 -> 26.2 us; 6 and 4 slower); four for the packed pass with splits
//   (the splits already supply the parallelism: 33.0 -> 30.1 us on two
//   32768-token sequences at 16 splits).  A launch with one split keeps the
//   packed pass's seven, so both packed modes give the same bits there.
int max_parts_for(int dpad, bool tiled, bool kv8 = false, bool packed_splits = false) {
    if (tiled) return 2;
    if (dpad >= 256) return packed_splits ? 4 : 7;
    return kv8 ? 4 : 5;
}

int dpad_for(int head_dim) { return head_dim <= 64 ? 64 : (head_dim <= 128 ? 128 : 256); }

template <int MODE, bool KV8>
cudaError_t dispatch_unit(int dpad, int gn, bool hl, bool packed, const CUtensorMap *tk,
                          const CUtensorMap *tv, const pd::UnitParams &p, long long units,
                          int stages_seq, cudaStream_t st) {
    using namespace pd;
    const int layout = g_debug_cluster == 1 ? 1 : (g_debug_cluster > 1 ? 2 : 0);
    if constexpr (MODE == kModePaged) {
        if (packed)
            return launch_unit<256, 1, false, kModePaged, true, KV8>(tk, tv, p, units, stages_seq, st, layout);
    }
#define PD_DISPATCH_D(DP)                                                                              \
    if (dpad == DP) {                                                                                  \
        if (gn == 2) return launch_unit<DP, 2, false, MODE, false, KV8>(tk, tv, p, units, stages_seq, st, layout); \
        if (hl) return launch_unit<DP, 1, true, MODE, false, KV8>(tk, tv, p, units, stages_seq, st, layout);       \
        return launch_unit<DP, 1, false, MODE, false, KV8>(tk, tv, p, units, stages_seq, st, layout);              \
    }
    PD_DISPATCH_D(64)
    PD_DISPATCH_D(128)
    PD_DISPATCH_D(256)
#undef PD_DISPATCH_D
    return cudaErrorInvalidValue;
}

int check_shape(int num_q_heads, int num_kv_heads, int head_dim, int block_size) {
    if (num_kv_heads <= 0 || num_q_heads <= 0)
        return fail(PD_ERR_INVALID, "num_q_heads (%d) and num_kv_heads (%d) must be positive",
                    num_q_heads, num_kv_heads);
    if (num_q_heads % num_kv_heads != 0)
        return fail(PD_ERR_INVALID, "num_kv_heads (%d) must divide num_q_heads (%d)", num_kv_heads,
                    num_q_heads);
    if (head_dim > PD_MAX_HEAD_DIM)
        return fail(PD_ERR_INVALID, "head_dim %d exceeds PD_MAX_HEAD_DIM=%d", head_dim, PD_MAX_HEAD_DIM);
    if (head_dim < 8 || head_dim % 8 != 0)
        return fail(PD_ERR_UNSUPPORTED, "head_dim %d: this build needs a positive multiple of 8",
                    head_dim);
    if (block_size < 16 || block_size > 256 || block_size % 16 != 0)
        return fail(PD_ERR_UNSUPPORTED,
                    "block_size %d: this build needs a multiple of 16 in [16, 256]", block_size);
    return PD_OK;
}

}  // namespace

namespace pd {
int report_error(int code, const char *message) { return fail(code, "%s", message); }
}  // namespace pd

struct pd_tiled {
    pd_tiled_dims dims;
    float *m;
    float *l;
    float *o;
    int device;
    float *run_ws;  // per-call partials of a fused pd_tiled_run [max_seqs*Hq, kMaxRunSources, D + 2]
};

namespace {
// Floats of a handle's fused-run partials: one [o[D], m, l] slot per (row, call)
// for up to kMaxRunSources calls.
size_t run_partials_floats(const pd_tiled_dims &d) {
    return static_cast<size_t>(d.max_seqs) * d.num_q_heads * pd::kMaxRunSources *
           (static_cast<size_t>(d.head_dim) + 2);
}
}  // namespace

namespace {
std::atomic<int> g_fail_allocs{0};
}

extern "C" {

const char *pd_last_error(void) { return g_err; }

int pd_build_info(int *max_splits, int *pack_width, int *pack_head_dim, int *min_kv_per_split) {
    if (max_splits) *max_splits = PD_MAX_DECODE_SPLITS;
    if (pack_width) *pack_width = pd::kernel_pack_width();
    if (pack_head_dim) *pack_head_dim = pd::kernel_pack_head_dim();
    if (min_kv_per_split) *min_kv_per_split = PD_MIN_KV_PER_SPLIT;
    return ok();
}

// ---- policy -------------------------------------------------------------------------

int pd_parse_policy(const char *text, int *policy, int *pin) {
    if (!text || !policy || !pin) return fail(PD_ERR_INVALID, "pd_parse_policy: null argument");
    const std::string w = trim_lower(text);
    if (w == "legacy") {
        *policy = PD_POLICY_LEGACY;
        *pin = 0;
        return ok();
    }
    if (w == "auto") {
        *policy = PD_POLICY_AUTO;
        *pin = 0;
        return ok();
    }
    if (is_off_word(w)) {
        *policy = PD_POLICY_PINNED;
        *pin = 1;
        return ok();
    }
    if (!w.empty() && w.find_first_not_of("0123456789") == std::string::npos) {
        // A decimal count, clamped to 1..MAX (saturating: long strings are large counts).
        long long v = 0;
        for (char c : w) {
            v = v * 10 + (c - '0');
            if (v > PD_MAX_DECODE_SPLITS) {
                v = PD_MAX_DECODE_SPLITS;
                break;
            }
        }
        *policy = PD_POLICY_PINNED;
        *pin = static_cast<int>(v < 1 ? 1 : v);
        return ok();
    }
    return fail(PD_ERR_INVALID, "not a split-K policy: '%s'", text);
}

int pd_parse_gqa_pack(const char *text, int *enabled) {
    if (!text || !enabled) return fail(PD_ERR_INVALID, "pd_parse_gqa_pack: null argument");
    const std::string w = trim_lower(text);
    if (w == "1" || w == "on" || w == "true" || w == "yes") {
        *enabled = 1;
        return ok();
    }
    if (is_off_word(w)) {
        *enabled = 0;
        return ok();
    }
    return fail(PD_ERR_INVALID, "not a GQA-pack switch: '%s'", text);
}

int pd_resolve_policy(const char *declared, const char *override_text, int *policy, int *pin) {
    if (!policy || !pin) return fail(PD_ERR_INVALID, "pd_resolve_policy: null argument");
    int pol = 0, pn = 0;
    if (override_text && pd_parse_policy(override_text, &pol, &pn) == PD_OK) {
        *policy = pol;
        *pin = pn;
        return ok();
    }
    if (declared && pd_parse_policy(declared, &pol, &pn) == PD_OK) {
        *policy = pol;
        *pin = pn;
        return ok();
    }
    *policy = PD_POLICY_LEGACY;
    *pin = 0;
    return ok();
}

int pd_policy_from_env(const char *declared, int *policy, int *pin) {
    return pd_resolve_policy(declared, std::getenv("PD_ATTN_DECODE_SPLITK"), policy, pin);
}

int pd_gqa_pack_enabled(void) {
    static std::once_flag once;
    static int enabled = 0;  // declared state: off
    std::call_once(once, [] {
        const char *v = std::getenv("PD_ATTN_DECODE_GQA_PACK");
        int e = 0;
        if (v && pd_parse_gqa_pack(v, &e) == PD_OK) enabled = e;
    });
    return enabled;
}

int pd_split_ref_seqs(int num_seqs, int max_decode_seqs) {
    return num_seqs > max_decode_seqs ? num_seqs : max_decode_seqs;
}

int pd_legacy_splits(int sm_count, int num_q_heads, int ref_seqs) {
    if (sm_count <= 0 || num_q_heads <= 0 || ref_seqs <= 0)
        return fail(PD_ERR_INVALID, "legacy_splits: sm_count %d, num_q_heads %d, ref_seqs %d",
                    sm_count, num_q_heads, ref_seqs);
    const long long ctas = static_cast<long long>(num_q_heads) * ref_seqs;
    ok();
    return ctas >= sm_count ? 1 : static_cast<int>(sm_count / ctas);
}

int pd_auto_splits(int sm_count, int num_q_heads) {
    if (sm_count <= 0 || num_q_heads <= 0)
        return fail(PD_ERR_INVALID, "auto_splits: sm_count %d, num_q_heads %d", sm_count, num_q_heads);
    const long long want =
        (static_cast<long long>(PD_SPLITK_TARGET_WAVES) * sm_count + num_q_heads - 1) / num_q_heads;
    ok();
    return static_cast<int>(want < 1 ? 1 : (want > PD_MAX_DECODE_SPLITS ? PD_MAX_DECODE_SPLITS : want));
}

int pd_num_splits(int policy, int pin, int sm_count, int num_q_heads, int num_seqs,
                  int max_decode_seqs) {
    switch (policy) {
        case PD_POLICY_LEGACY:
            if (num_seqs < 0 || max_decode_seqs < 0)
                return fail(PD_ERR_INVALID, "num_splits: negative batch");
            return pd_legacy_splits(sm_count, num_q_heads, pd_split_ref_seqs(num_seqs, max_decode_seqs));
        case PD_POLICY_AUTO:
            return pd_auto_splits(sm_count, num_q_heads);
        case PD_POLICY_PINNED:
            ok();
            return pin < 1 ? 1 : (pin > PD_MAX_DECODE_SPLITS ? PD_MAX_DECODE_SPLITS : pin);
        default:
            return fail(PD_ERR_INVALID, "unknown split-K policy %d", policy);
    }
}

size_t pd_workspace_bytes(int rows, int num_q_heads, int head_dim, int num_splits) {
    if (rows <= 0 || num_q_heads <= 0 || head_dim <= 0 || num_splits <= 0) return 0;
    return static_cast<size_t>(rows) * num_q_heads * num_splits * (head_dim + 2) * sizeof(float);
}

int pd_gqa_pack_shape_ok(int num_q_heads, int num_kv_heads, int head_dim) {
    return num_kv_heads > 0 && num_q_heads == num_kv_heads * PD_GQA_PACK_WIDTH &&
           head_dim == PD_GQA_PACK_HEAD_DIM;
}

int pd_gqa_pack_ctas(int num_kv_heads, int num_seqs) { return num_kv_heads * num_seqs; }

int pd_split_chunk_tokens(int context_len, int num_splits, int block_size) {
    if (context_len < 0 || num_splits <= 0 || block_size <= 0)
        return fail(PD_ERR_INVALID, "split_chunk_tokens: context_len %d, num_splits %d, block_size %d",
                    context_len, num_splits, block_size);
    ok();
    return pd::split_chunk_tokens(context_len, num_splits, block_size, PD_MIN_KV_PER_SPLIT);
}

// ---- paged decode ----------------------------------------------------------------------

namespace {
// pd_decode_attn over a BF16 cache (kv8 false) or an FP8 E4M3 cache with
// per-tensor scales (kv8 true); one body so that both take the same checks,
// split geometry, launch choices and merge.
int decode_impl(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
                int max_blocks_per_seq, const int32_t *context_lens, void *out, int num_seqs,
                int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                float inv_sqrt_d, int num_splits, void *workspace, size_t workspace_bytes, int gqa_pack,
                void *stream, bool kv8, float k_scale, float v_scale) {
    if (gqa_pack < PD_GQA_PACK_OFF || gqa_pack > PD_GQA_PACK_SPLITK)
        return fail(PD_ERR_INVALID, "gqa_pack must be 0, 1 or 2");
    if (gqa_pack) {
        if (gqa_pack == PD_GQA_PACK_ON && num_splits != 1)
            return fail(PD_NOT_APPLICABLE, "GQA-packed pass serves non-split launches only (num_splits=%d)",
                        num_splits);
        if (!pd_gqa_pack_shape_ok(num_q_heads, num_kv_heads, head_dim))
            return fail(PD_NOT_APPLICABLE,
                        "GQA-packed pass needs num_q_heads == %d*num_kv_heads and head_dim == %d "
                        "(got %d, %d, %d)",
                        PD_GQA_PACK_WIDTH, PD_GQA_PACK_HEAD_DIM, num_q_heads, num_kv_heads, head_dim);
    }
    int rc = check_shape(num_q_heads, num_kv_heads, head_dim, block_size);
    if (rc != PD_OK) return rc;
    if (kv8) {
        if (head_dim % 16 != 0)
            return fail(PD_ERR_UNSUPPORTED, "FP8 cache: head_dim %d must be a multiple of 16", head_dim);
        if (!std::isfinite(k_scale) || !std::isfinite(v_scale))
            return fail(PD_ERR_INVALID, "FP8 cache: k_scale and v_scale must be finite");
    }
    if (num_seqs < 0) return fail(PD_ERR_INVALID, "num_seqs %d < 0", num_seqs);
    if (num_splits < 1 || num_splits > 4096)
        return fail(PD_ERR_INVALID, "num_splits %d outside 1..4096", num_splits);
    if (!std::isfinite(inv_sqrt_d)) return fail(PD_ERR_INVALID, "inv_sqrt_d is not finite");
    if (num_seqs == 0) return ok();
    if (!q || !k_cache || !v_cache || !block_table || !context_lens || !out)
        return fail(PD_ERR_INVALID, "null tensor pointer");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return fail(PD_ERR_INVALID, "q, k_cache, v_cache and out must be 16-byte aligned");
    if (max_blocks_per_seq <= 0 || num_blocks <= 0)
        return fail(PD_ERR_INVALID, "max_blocks_per_seq (%d) and num_blocks (%d) must be positive",
                    max_blocks_per_seq, num_blocks);
    if (static_cast<long long>(max_blocks_per_seq) * block_size > 0x7fffffffLL)
        return fail(PD_ERR_INVALID, "max_blocks_per_seq * block_size overflows int32");
    if (num_splits > 1) {
        const size_t need = pd_workspace_bytes(num_seqs, num_q_heads, head_dim, num_splits);
        if (!workspace || workspace_bytes < need)
            return fail(PD_ERR_WORKSPACE, "split-K workspace of %zu bytes needed, %zu given%s", need,
                        workspace ? workspace_bytes : static_cast<size_t>(0), workspace ? "" : " (null)");
        if (!aligned16(workspace)) return fail(PD_ERR_INVALID, "workspace must be 16-byte aligned");
    }

    const int G = num_q_heads / num_kv_heads;
    const bool packed = gqa_pack != PD_GQA_PACK_OFF;
    const int dpad = packed ? PD_GQA_PACK_HEAD_DIM : dpad_for(head_dim);
    const int gn = packed ? 1 : (G <= 8 ? 1 : 2);
    const int rows = 8 * gn;
    const int qtiles = (G + rows - 1) / rows;
    const int stages = default_stages(dpad, kv8);
    const long long units = static_cast<long long>(num_seqs) * num_kv_heads * qtiles * num_splits;
    const bool packed_splits = gqa_pack == PD_GQA_PACK_SPLITK && num_splits > 1;
    if (units * max_parts_for(dpad, false, kv8, packed_splits) > 0x7fffffffLL)
        return fail(PD_ERR_INVALID, "launch too large (%lld units)", units);

    int err = PD_OK;
    unsigned int *status = status_ptr(&err);
    if (!status) return err;

    CUtensorMap tk, tv;
    int tok_dim = 1;
    const long long kvh_s = head_dim, tok_s = static_cast<long long>(num_kv_heads) * head_dim;
    const long long blk_s = tok_s * block_size;
    const int elem = kv8 ? 1 : 2;
    // FP8 from head dim 128 up: K and V in 128-code swizzled boxes (read
    // straight into the mma operands); at head dim 64 one unswizzled box of the
    // padded row each (converted to f16 tiles first)
    const bool k_direct = kv8 && dpad >= 128;
    const int box_k = !kv8 ? pd::kBoxCols : (k_direct ? 128 : dpad);
    const int box_v = box_k;
    rc = encode_kv_map(&tk, &tok_dim, k_cache, head_dim, block_size, num_kv_heads, num_blocks, blk_s,
                       tok_s, kvh_s, elem, box_k, !kv8 || k_direct);
    if (rc != PD_OK) return rc;
    rc = encode_kv_map(&tv, &tok_dim, v_cache, head_dim, block_size, num_kv_heads, num_blocks, blk_s,
                       tok_s, kvh_s, elem, box_v, !kv8 || k_direct);
    if (rc != PD_OK) return rc;

    pd::UnitParams p = {};
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.block_table = block_table;
    p.context_lens = context_lens;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.num_splits = num_splits;
    p.min_kv_per_split = PD_MIN_KV_PER_SPLIT;
    p.out = static_cast<__nv_bfloat16 *>(out);
    float *ws = static_cast<float *>(workspace);
    p.ws_o = num_splits > 1 ? ws : nullptr;
    p.ws_ml = num_splits > 1 ? ws + static_cast<size_t>(num_seqs) * num_q_heads * num_splits * head_dim
                             : nullptr;
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = G;
    p.head_dim = head_dim;
    p.block_size = block_size;
    p.qtiles = qtiles;
    p.cluster = 1;
    p.fd_bs = pd::make_fastdiv(p.block_size);
    p.fd_kvh = pd::make_fastdiv(p.num_kv_heads);
    p.fd_split = pd::make_fastdiv(num_splits);
    p.max_parts = max_parts_for(dpad, false, kv8, packed_splits);
    p.stages = stages;
    p.lpt = default_lpt(num_seqs);
    p.prefetch_tiles = kPrefetchBytes / (2 * pd::kTileTokens * dpad * 2);
    p.tok_dim = tok_dim;
    // An FP8 cache's K scale multiplies every score: fold it into the softmax scale.
    p.scale_log2 = static_cast<float>(static_cast<double>(inv_sqrt_d) * (kv8 ? static_cast<double>(k_scale) : 1.0) *
                                      1.4426950408889634);
    p.v_scale = kv8 ? v_scale : 1.f;
    p.status = status;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int smem = pd::unit_smem_bytes(dpad, rows, stages, kv8);
    if (smem > max_smem_optin())
        return fail(PD_ERR_INVALID, "launch shape needs %d bytes of shared memory, the device allows %d",
                    smem, max_smem_optin());
    int stages_seq = default_stages_seq(dpad, kv8);
    if (pd::unit_smem_bytes(dpad, rows, stages_seq, kv8) > max_smem_optin()) stages_seq = stages;
    const bool hl = !packed && G <= 4;
    cudaError_t e = kv8 ? dispatch_unit<pd::kModePaged, true>(dpad, gn, hl, packed, &tk, &tv, p, units, stages_seq, st)
                        : dispatch_unit<pd::kModePaged, false>(dpad, gn, hl, packed, &tk, &tv, p, units, stages_seq, st);
    if (e != cudaSuccess) return cuda_fail(e, "unit kernel launch");
    if (num_splits > 1) {
        pd::MergeParams mp = {};
        mp.context_lens = context_lens;
        mp.ws_o = p.ws_o;
        mp.ws_ml = p.ws_ml;
        mp.out = p.out;
        mp.num_seqs = num_seqs;
        mp.num_q_heads = num_q_heads;
        mp.head_dim = head_dim;
        mp.num_splits = num_splits;
        mp.block_size = block_size;
        mp.min_kv_per_split = PD_MIN_KV_PER_SPLIT;
        mp.max_tokens = max_blocks_per_seq * block_size;
        mp.fd_hq = pd::make_fastdiv(num_q_heads);
        mp.fd_split = pd::make_fastdiv(num_splits);
        mp.fd_bs = pd::make_fastdiv(block_size);
        e = pd::launch_merge(mp, st, true);
        if (e != cudaSuccess) return cuda_fail(e, "merge kernel launch");
    }
    return ok();
}
}  // namespace

int pd_decode_attn(const void *q, const void *k_cache, const void *v_cache,
                   const int32_t *block_table, int max_blocks_per_seq,
                   const int32_t *context_lens, void *out, int num_seqs, int num_q_heads,
                   int num_kv_heads, int head_dim, int block_size, int num_blocks,
                   float inv_sqrt_d, int num_splits, void *workspace, size_t workspace_bytes,
                   int gqa_pack, void *stream) {
    return decode_impl(q, k_cache, v_cache, block_table, max_blocks_per_seq, context_lens, out, num_seqs,
                       num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, inv_sqrt_d, num_splits,
                       workspace, workspace_bytes, gqa_pack, stream, false, 1.f, 1.f);
}

int pd_decode_attn_fp8(const void *q, const void *k_cache, const void *v_cache, float k_scale,
                       float v_scale, const int32_t *block_table, int max_blocks_per_seq,
                       const int32_t *context_lens, void *out, int num_seqs, int num_q_heads,
                       int num_kv_heads, int head_dim, int block_size, int num_blocks, float inv_sqrt_d,
                       int num_splits, void *workspace, size_t workspace_bytes, int gqa_pack, void *stream) {
    return decode_impl(q, k_cache, v_cache, block_table, max_blocks_per_seq, context_lens, out, num_seqs,
                       num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, inv_sqrt_d, num_splits,
                       workspace, workspace_bytes, gqa_pack, stream, true, k_scale, v_scale);
}

// ---- tiled ----------------------------------------------------------------------------------

int pd_tiled_validate(const pd_tiled_dims *d) {
    if (!d) return fail(PD_ERR_INVALID, "null dims");
    if (d->max_seqs < 0 || d->tile_capacity < 0)
        return fail(PD_ERR_INVALID, "max_seqs (%d) and tile_capacity (%d) must be >= 0", d->max_seqs,
                    d->tile_capacity);
    int rc = check_shape(d->num_q_heads, d->num_kv_heads, d->head_dim, d->block_size);
    if (rc != PD_OK) return rc;
    return ok();
}

int pd_tiled_state_bytes(const pd_tiled_dims *d, size_t *m_bytes, size_t *l_bytes, size_t *o_bytes,
                         size_t *output_bytes) {
    if (!d || d->max_seqs < 0 || d->num_q_heads < 0 || d->head_dim < 0)
        return fail(PD_ERR_INVALID, "bad dims");
    const size_t nq = static_cast<size_t>(d->max_seqs) * d->num_q_heads;
    if (m_bytes) *m_bytes = nq * 4;
    if (l_bytes) *l_bytes = nq * 4;
    if (o_bytes) *o_bytes = nq * d->head_dim * 4;
    if (output_bytes) *output_bytes = nq * d->head_dim * 2;
    return ok();
}

int pd_tiled_create(const pd_tiled_dims *dims, pd_tiled **out) {
    if (!out) return fail(PD_ERR_INVALID, "null out");
    *out = nullptr;
    int rc = pd_tiled_validate(dims);
    if (rc != PD_OK) return rc;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    size_t mb = 0, lb = 0, ob = 0;
    pd_tiled_state_bytes(dims, &mb, &lb, &ob, nullptr);
    pd_tiled *t = new pd_tiled();
    t->dims = *dims;
    t->device = dev;
    float **bufs[4] = {&t->m, &t->l, &t->o, &t->run_ws};
    size_t sizes[4] = {mb, lb, ob, run_partials_floats(*dims) * sizeof(float)};
    for (int i = 0; i < 4; ++i) {
        void *p = nullptr;
        int inject = g_fail_allocs.load();
        while (inject > 0 && !g_fail_allocs.compare_exchange_weak(inject, inject - 1)) {
        }
        if (inject > 0) {
            e = cudaErrorMemoryAllocation;
        } else {
            e = cudaMalloc(&p, sizes[i] > 0 ? sizes[i] : 16);
        }
        if (e != cudaSuccess) {
            cudaFree(t->m);
            cudaFree(t->l);
            cudaFree(t->o);
            cudaFree(t->run_ws);
            delete t;
            return fail(PD_ERR_ALLOC, "tiled state allocation of %zu bytes failed: %s", sizes[i],
                        cudaGetErrorString(e));
        }
        *bufs[i] = static_cast<float *>(p);
    }
    *out = t;
    return ok();
}

void pd_tiled_destroy(pd_tiled *t) {
    if (!t) return;
    int cur = 0;
    cudaGetDevice(&cur);
    cudaSetDevice(t->device);
    cudaDeviceSynchronize();
    cudaFree(t->m);
    cudaFree(t->l);
    cudaFree(t->o);
    cudaFree(t->run_ws);
    cudaSetDevice(cur);
    delete t;
}

int pd_tiled_get_dims(const pd_tiled *t, pd_tiled_dims *dims) {
    if (!t || !dims) return fail(PD_ERR_INVALID, "null argument");
    *dims = t->dims;
    return ok();
}

int pd_tiled_state(const pd_tiled *t, void **m, void **l, void **o) {
    if (!t) return fail(PD_ERR_INVALID, "null handle");
    if (m) *m = t->m;
    if (l) *l = t->l;
    if (o) *o = t->o;
    return ok();
}

void pd_tiled_paged_strides(const pd_tiled *t, int64_t s[3]) {
    if (!t || !s) return;
    const pd_tiled_dims &d = t->dims;
    s[0] = static_cast<int64_t>(d.block_size) * d.num_kv_heads * d.head_dim;
    s[1] = static_cast<int64_t>(d.num_kv_heads) * d.head_dim;
    s[2] = d.head_dim;
}

void pd_tiled_scratch_pool_strides(const pd_tiled *t, int64_t s[3]) {
    if (!t || !s) return;
    const pd_tiled_dims &d = t->dims;
    const int64_t stripe = static_cast<int64_t>(d.num_kv_heads) * d.block_size * d.head_dim;
    s[0] = 2 * stripe;
    s[1] = d.head_dim;
    s[2] = static_cast<int64_t>(d.block_size) * d.head_dim;
}

int pd_tiled_begin(pd_tiled *t, int num_seqs, void *stream) {
    if (!t) return fail(PD_ERR_INVALID, "null handle");
    if (num_seqs < 0) return fail(PD_ERR_INVALID, "num_seqs %d < 0", num_seqs);
    if (num_seqs > t->dims.max_seqs)
        return fail(PD_ERR_CAPACITY, "begin_step num_seqs %d > max_seqs %d", num_seqs, t->dims.max_seqs);
    cudaError_t e = pd::launch_tiled_begin(t->m, t->l, t->o, num_seqs * t->dims.num_q_heads,
                                           t->dims.head_dim, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tiled begin launch");
    return ok();
}

// Block extent of a tiled K/V view: the tiled interface passes no pool size,
// so block ids are bounded by this constant (ids outside read zeros and raise
// PD_DEV_BAD_BLOCK_ID).
constexpr long long kTiledBlockExtent = 1LL << 24;

namespace {
// Argument checks of one step_tile call.  PD_OK with *skip set when the call
// has nothing to fold (no sequence, or a zero tile capacity).
int check_step(const pd_tiled *t, const void *q, const void *k_pool, const void *v_pool,
               const int32_t *tile_blocks, const int32_t *tile_block_counts, int num_seqs,
               int64_t blk_stride, int64_t tok_stride, int64_t kvh_stride, bool *skip) {
    *skip = true;
    if (!t) return fail(PD_ERR_INVALID, "null handle");
    if (num_seqs < 0) return fail(PD_ERR_INVALID, "num_seqs %d < 0", num_seqs);
    if (num_seqs > t->dims.max_seqs)
        return fail(PD_ERR_CAPACITY, "step_tile num_seqs %d > max_seqs %d", num_seqs, t->dims.max_seqs);
    if (num_seqs == 0 || t->dims.tile_capacity == 0) return PD_OK;
    if (!q || !k_pool || !v_pool || !tile_blocks || !tile_block_counts)
        return fail(PD_ERR_INVALID, "null pointer");
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
        return fail(PD_ERR_INVALID, "q, k_pool and v_pool must be 16-byte aligned");
    if (blk_stride <= 0 || tok_stride <= 0 || kvh_stride <= 0 || blk_stride % 8 || tok_stride % 8 ||
        kvh_stride % 8)
        return fail(PD_ERR_INVALID,
                    "strides (blk %lld, tok %lld, kvh %lld) must be positive multiples of 8 elements",
                    static_cast<long long>(blk_stride), static_cast<long long>(tok_stride),
                    static_cast<long long>(kvh_stride));
    *skip = false;
    return PD_OK;
}
}  // namespace

int pd_tiled_step(pd_tiled *t, const void *q, const void *k_pool, const void *v_pool,
                  const int32_t *tile_blocks, const int32_t *tile_block_counts, int num_seqs,
                  int64_t blk_stride, int64_t tok_stride, int64_t kvh_stride,
                  int last_block_valid_slots, void *stream) {
    bool skip = true;
    const int crc = check_step(t, q, k_pool, v_pool, tile_blocks, tile_block_counts, num_seqs,
                               blk_stride, tok_stride, kvh_stride, &skip);
    if (crc != PD_OK) return crc;
    if (skip) return ok();
    const pd_tiled_dims &d = t->dims;
    const int G = d.num_q_heads / d.num_kv_heads;
    const int dpad = dpad_for(d.head_dim);
    const int gn = G <= 8 ? 1 : 2;
    const int rows = 8 * gn;
    const int qtiles = (G + rows - 1) / rows;
    const int stages = default_stages(dpad);
    const long long units = static_cast<long long>(num_seqs) * d.num_kv_heads * qtiles;
    if (units * max_parts_for(dpad, true) > 0x7fffffffLL) return fail(PD_ERR_INVALID, "launch too large");

    int err = PD_OK;
    unsigned int *status = status_ptr(&err);
    if (!status) return err;
    CUtensorMap tk, tv;
    int tok_dim = 1;
    int rc = encode_kv_map(&tk, &tok_dim, k_pool, d.head_dim, d.block_size, d.num_kv_heads,
                           kTiledBlockExtent, blk_stride, tok_stride, kvh_stride);
    if (rc != PD_OK) return rc;
    rc = encode_kv_map(&tv, &tok_dim, v_pool, d.head_dim, d.block_size, d.num_kv_heads,
                       kTiledBlockExtent, blk_stride, tok_stride, kvh_stride);
    if (rc != PD_OK) return rc;

    pd::UnitParams p = {};
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.num_blocks = static_cast<int>(kTiledBlockExtent);
    p.tile_blocks = tile_blocks;
    p.tile_counts = tile_block_counts;
    p.tile_capacity = d.tile_capacity;
    p.last_valid = last_block_valid_slots;
    p.st_m = t->m;
    p.st_l = t->l;
    p.st_o = t->o;
    p.num_seqs = num_seqs;
    p.num_q_heads = d.num_q_heads;
    p.num_kv_heads = d.num_kv_heads;
    p.group = G;
    p.head_dim = d.head_dim;
    p.block_size = d.block_size;
    p.qtiles = qtiles;
    p.cluster = 1;
    p.fd_bs = pd::make_fastdiv(p.block_size);
    p.fd_kvh = pd::make_fastdiv(p.num_kv_heads);
    p.fd_split = pd::make_fastdiv(1);
    p.max_parts = max_parts_for(dpad, true);
    p.stages = stages;
    p.lpt = 0;
    // No early prefetch in the tiled step: measured no gain (the begin pass or
    // the previous step ahead of it leaves no idle tail to fill).
    p.prefetch_tiles = 0;
    p.tok_dim = tok_dim;
    // step_tile carries no scale: 1/sqrt(head_dim), rounded to FP32 first.
    const float inv_sqrt_d = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d.head_dim)));
    p.scale_log2 = static_cast<float>(static_cast<double>(inv_sqrt_d) * 1.4426950408889634);
    p.status = status;
    const int smem = pd::unit_smem_bytes(dpad, rows, stages, false);
    if (smem > max_smem_optin())
        return fail(PD_ERR_INVALID, "launch shape needs %d bytes of shared memory, the device allows %d",
                    smem, max_smem_optin());
    int stages_seq = default_stages_seq(dpad);
    if (pd::unit_smem_bytes(dpad, rows, stages_seq, false) > max_smem_optin()) stages_seq = stages;
    cudaError_t e = dispatch_unit<pd::kModeTiled, false>(dpad, gn, G <= 4, false, &tk, &tv, p, units, stages_seq,
                                                         static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tiled step launch");
    return ok();
}

int pd_tiled_finalize(pd_tiled *t, void *out, int num_seqs, void *stream) {
    if (!t) return fail(PD_ERR_INVALID, "null handle");
    if (num_seqs < 0) return fail(PD_ERR_INVALID, "num_seqs %d < 0", num_seqs);
    if (num_seqs > t->dims.max_seqs)
        return fail(PD_ERR_CAPACITY, "finalize num_seqs %d > max_seqs %d", num_seqs, t->dims.max_seqs);
    if (num_seqs == 0) return ok();
    if (!out) return fail(PD_ERR_INVALID, "null out");
    cudaError_t e = pd::launch_tiled_finalize(t->l, t->o, static_cast<__nv_bfloat16 *>(out),
                                              num_seqs * t->dims.num_q_heads, t->dims.head_dim,
                                              static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tiled finalize launch");
    return ok();
}

}  // extern "C"

namespace {
// pd_tiled_run for 1..kMaxRunSources calls in two launches: the unit pass over
// every (sequence, KV head, call) writes one partial [o, m, l] per call, and
// the fold pass replays step_tile's fold of those partials in call order from
// begin's (-inf, 0, 0), then finalizes.  Same arithmetic, same bits, as the
// calls made one by one.  The partials live in the buffer pd_tiled_create
// allocated with the state (kMaxRunSources slots per row), so a run allocates
// nothing.
int tiled_run_fused(pd_tiled *t, const void *q, const pd_tiled_source *sources, int num_sources, void *out,
                    int num_seqs, void *stream) {
    const pd_tiled_dims &d = t->dims;
    const int G = d.num_q_heads / d.num_kv_heads;
    const int dpad = dpad_for(d.head_dim);
    const int gn = G <= 8 ? 1 : 2;
    const int rows = 8 * gn;
    const int qtiles = (G + rows - 1) / rows;
    const int stages = default_stages(dpad);
    const long long units = static_cast<long long>(num_seqs) * d.num_kv_heads * qtiles * num_sources;
    if (units * max_parts_for(dpad, true) > 0x7fffffffLL) return fail(PD_ERR_INVALID, "launch too large");

    int err = PD_OK;
    unsigned int *status = status_ptr(&err);
    if (!status) return err;
    CUtensorMap tk[pd::kMaxRunSources], tv[pd::kMaxRunSources];
    pd::UnitParams p = {};
    for (int c = 0; c < num_sources; ++c) {
        const pd_tiled_source &src = sources[c];
        int tok_dim = 1;
        int rc = encode_kv_map(&tk[c], &tok_dim, src.k_pool, d.head_dim, d.block_size, d.num_kv_heads,
                               kTiledBlockExtent, src.blk_stride, src.tok_stride, src.kvh_stride);
        if (rc != PD_OK) return rc;
        rc = encode_kv_map(&tv[c], &tok_dim, src.v_pool, d.head_dim, d.block_size, d.num_kv_heads,
                           kTiledBlockExtent, src.blk_stride, src.tok_stride, src.kvh_stride);
        if (rc != PD_OK) return rc;
        p.src_blocks[c] = src.tile_blocks;
        p.src_counts[c] = src.tile_block_counts;
        p.src_last_valid[c] = src.last_block_valid_slots;
        p.src_tok_dim[c] = tok_dim;
    }
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.num_blocks = static_cast<int>(kTiledBlockExtent);
    p.tile_capacity = d.tile_capacity;
    p.num_sources = num_sources;
    p.num_splits = num_sources;  // partial slots per row
    p.ws_o = t->run_ws;
    p.ws_ml = t->run_ws + static_cast<size_t>(num_seqs) * d.num_q_heads * num_sources * d.head_dim;
    p.num_seqs = num_seqs;
    p.num_q_heads = d.num_q_heads;
    p.num_kv_heads = d.num_kv_heads;
    p.group = G;
    p.head_dim = d.head_dim;
    p.block_size = d.block_size;
    p.qtiles = qtiles;
    p.cluster = 1;
    p.fd_bs = pd::make_fastdiv(p.block_size);
    p.fd_kvh = pd::make_fastdiv(p.num_kv_heads);
    p.fd_split = pd::make_fastdiv(1);
    p.max_parts = max_parts_for(dpad, true);
    p.stages = stages;
    p.lpt = 0;
    p.prefetch_tiles = 0;
    p.tok_dim = p.src_tok_dim[0];
    const float inv_sqrt_d = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d.head_dim)));
    p.scale_log2 = static_cast<float>(static_cast<double>(inv_sqrt_d) * 1.4426950408889634);
    p.v_scale = 1.f;
    p.status = status;
    const int smem = pd::unit_smem_bytes(dpad, rows, stages, false);
    if (smem > max_smem_optin())
        return fail(PD_ERR_INVALID, "launch shape needs %d bytes of shared memory, the device allows %d",
                    smem, max_smem_optin());
    int stages_seq = default_stages_seq(dpad);
    if (pd::unit_smem_bytes(dpad, rows, stages_seq, false) > max_smem_optin()) stages_seq = stages;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = dispatch_unit<pd::kModeTiledRun, false>(dpad, gn, G <= 4, false, tk, tv, p, units, stages_seq, st);
    if (e != cudaSuccess) return cuda_fail(e, "fused tiled run: unit launch");
    pd::RunMergeParams mp = {};
    mp.ws_o = p.ws_o;
    mp.ws_ml = p.ws_ml;
    for (int c = 0; c < num_sources; ++c) mp.src_counts[c] = sources[c].tile_block_counts;
    mp.st_m = t->m;
    mp.st_l = t->l;
    mp.st_o = t->o;
    mp.out = static_cast<__nv_bfloat16 *>(out);
    mp.num_seqs = num_seqs;
    mp.num_q_heads = d.num_q_heads;
    mp.head_dim = d.head_dim;
    mp.num_sources = num_sources;
    mp.tile_capacity = d.tile_capacity;
    e = pd::launch_tiled_run_merge(mp, st);
    if (e != cudaSuccess) return cuda_fail(e, "fused tiled run: fold launch");
    return ok();
}
}  // namespace

extern "C" {

int pd_tiled_run(pd_tiled *t, const void *q, const pd_tiled_source *sources, int num_sources,
                 void *out, int num_seqs, void *stream) {
    if (!t) return fail(PD_ERR_INVALID, "null handle");
    if (num_sources < 0) return fail(PD_ERR_INVALID, "num_sources %d < 0", num_sources);
    if (num_sources > 0 && !sources) return fail(PD_ERR_INVALID, "null sources");
    if (num_seqs < 0) return fail(PD_ERR_INVALID, "num_seqs %d < 0", num_seqs);
    if (num_seqs > t->dims.max_seqs)
        return fail(PD_ERR_CAPACITY, "num_seqs %d > max_seqs %d", num_seqs, t->dims.max_seqs);
    if (num_seqs > 0 && !out) return fail(PD_ERR_INVALID, "null out");
    for (int i = 0; i < num_sources; ++i) {
        const pd_tiled_source &src = sources[i];
        bool skip = true;
        const int crc = check_step(t, q, src.k_pool, src.v_pool, src.tile_blocks, src.tile_block_counts,
                                   num_seqs, src.blk_stride, src.tok_stride, src.kvh_stride, &skip);
        if (crc != PD_OK) {
            char msg[512];
            snprintf(msg, sizeof msg, "source %d: %s", i, pd_last_error());
            return fail(crc, "%s", msg);
        }
    }
    if (num_sources >= 1 && num_sources <= pd::kMaxRunSources && num_seqs > 0 && t->dims.tile_capacity > 0)
        return tiled_run_fused(t, q, sources, num_sources, out, num_seqs, stream);
    int rc = pd_tiled_begin(t, num_seqs, stream);
    if (rc != PD_OK) return rc;
    for (int i = 0; i < num_sources; ++i) {
        const pd_tiled_source &src = sources[i];
        rc = pd_tiled_step(t, q, src.k_pool, src.v_pool, src.tile_blocks, src.tile_block_counts, num_seqs,
                           src.blk_stride, src.tok_stride, src.kvh_stride, src.last_block_valid_slots,
                           stream);
        if (rc != PD_OK) return rc;
    }
    return pd_tiled_finalize(t, out, num_seqs, stream);
}

// ---- diagnostics ------------------------------------------------------------------------------

int pd_device_status(int *flags) {
    if (!flags) return fail(PD_ERR_INVALID, "null flags");
    int err = PD_OK;
    unsigned int *sp = status_ptr(&err);
    if (!sp) return err;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    unsigned int v = 0;
    e = cudaMemcpy(&v, sp, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read status");
    const unsigned int zero = 0;
    e = cudaMemcpy(sp, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clear status");
    *flags = static_cast<int>(v);
    return ok();
}

void pd_debug_fail_next_allocs(int count) { g_fail_allocs.store(count < 0 ? 0 : count); }

void pd_debug_set_tuning(int stages_per_warp, int cluster, int longest_first) {
    g_debug_stages = stages_per_warp > 0 && stages_per_warp <= pd::kMaxStagesPerWarp ? stages_per_warp : 0;
    g_debug_cluster = cluster == 1 ? 1 : (cluster > 1 ? 2 : 0);
    g_debug_lpt = longest_first == 0 || longest_first == 1 ? longest_first : -1;
}

}  // extern "C"
