// pd_noalloc.cu -- pd_decode_attn_noalloc: paged-decode attention for callers
// that cannot allocate device memory (see include/pd.h).  The split-K
// workspace is a fixed array in the library's device memory instead of a
// buffer the caller allocates; the launch itself is pd_decode_attn's.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "pd.h"
#include "pd_internal.h"

// The workspace every call on a device shares.  Loaded with the library's
// kernels, kept until the process exits.
static __device__ __align__(256) float g_noalloc_workspace[PD_NOALLOC_WORKSPACE_BYTES / sizeof(float)];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_workspace_ptr[kMaxDevices] = {nullptr};

// Device address of the array on the current device, looked up once per
// device.  In host code `g_noalloc_workspace` names a host-side shadow, not
// device memory, so it must never be passed to a kernel directly.
int workspace_on_current_device(void **ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return pd::report_error(PD_ERR_CUDA, "pd_decode_attn_noalloc: no usable current CUDA device");
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_workspace_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_workspace);
        if (e != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();
            char msg[256];
            snprintf(msg, sizeof msg, "pd_decode_attn_noalloc: cudaGetSymbolAddress failed on device %d: %s",
                     dev, cudaGetErrorString(e));
            return pd::report_error(PD_ERR_CUDA, msg);
        }
        g_workspace_ptr[dev] = p;
    }
    *ptr = g_workspace_ptr[dev];
    return PD_OK;
}

}  // namespace

extern "C" int pd_decode_attn_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                      const int32_t *block_table, int max_blocks_per_seq,
                                      const int32_t *context_lens, void *out, int num_seqs,
                                      int num_q_heads, int num_kv_heads, int head_dim,
                                      int block_size, int num_blocks, float inv_sqrt_d,
                                      int num_splits, int gqa_pack, void *stream) {
    const size_t need =
        num_splits > 1 ? pd_workspace_bytes(num_seqs, num_q_heads, head_dim, num_splits) : 0;
    if (need > PD_NOALLOC_WORKSPACE_BYTES) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "pd_decode_attn_noalloc: this launch needs a %zu-byte split-K workspace, more than "
                 "the library's fixed %u bytes; use pd_decode_attn with a caller workspace, or fewer "
                 "sequences or splits per call",
                 need, PD_NOALLOC_WORKSPACE_BYTES);
        return pd::report_error(PD_ERR_WORKSPACE, msg);
    }
    void *ws = nullptr;
    if (num_splits > 1) {
        const int rc = workspace_on_current_device(&ws);
        if (rc != PD_OK) return rc;
    }
    return pd_decode_attn(q, k_cache, v_cache, block_table, max_blocks_per_seq, context_lens, out,
                          num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                          inv_sqrt_d, num_splits, ws, ws ? PD_NOALLOC_WORKSPACE_BYTES : 0, gqa_pack,
                          stream);
}
