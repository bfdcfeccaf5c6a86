// decode_noalloc.cu -- paged_attn_decode_noalloc: the decode entry point for
// callers that cannot allocate device memory.
//
// paged_attn_decode needs a caller-provided workspace when a context is cut
// into several splits (it holds each split's partial output, running max and
// running sum until the merge kernel combines them).  Some callers cannot
// produce that buffer on demand: a serving loop that reserved all of HBM for
// the KV pool at start-up and may not call cudaMalloc afterwards (cudaMalloc
// can also wait for the whole device, which a per-token decode loop cannot
// afford), or a host framework / plugin that owns the allocator and forbids
// allocations outside it.  This variant takes the same inputs and outputs but
// uses a fixed scratch array compiled into the library instead of a
// workspace argument, and allocates nothing itself.
//
// Limits and sharing rules (stated in pagedkv.h as well):
//   * The scratch is PKV_NOALLOC_SCRATCH_BYTES (16 MiB) per device that loads
//     the library, held until the process exits.  A problem whose split
//     partials need more (see pkv_decode_workspace_bytes) is rejected with
//     PKV_ERR_WORKSPACE before anything is launched.
//   * All calls on a device share the one array.  Two calls whose kernels
//     can overlap on the GPU (different streams, no ordering between them)
//     race on it; order them on one stream or by events.
//   * Nothing in the array needs to start at zero: every partial the merge
//     kernel reads is written earlier in the same call.  The array keeps the
//     last call's contents.
//   * The first call on each device looks up the array's device address
//     (cudaGetSymbolAddress) with that device current; make that first call
//     before any stream capture begins.  The address is cached for the life
//     of the process: it does not survive cudaDeviceReset, after which the
//     library must not be called on that device again.
#include <mutex>

#include "../../include/pagedkv.h"
#include <cuda_runtime.h>

namespace pkv {
void record_detail(const char* msg);
}

namespace {

// The scratch itself.  Host code must not pass `g_noalloc_scratch` to a
// kernel directly: on the host that name is only a stand-in for the device
// symbol; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of the scratch on the current device (looked up once per
// device, with that device current).
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" PKV_API pkv_status paged_attn_decode_noalloc(
    void* out, pkv_dtype out_dtype, const void* q, const void* k_pool, const void* v_pool,
    pkv_dtype kv_dtype, const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int num_seqs, int n_heads, int n_kv_heads, int head_dim,
    int block_size, int num_blocks, float scale, int max_context_len, int split_tokens,
    void* stream) {
    const size_t need = pkv_decode_workspace_bytes(num_seqs, n_heads, n_kv_heads, head_dim,
                                                   block_size, max_context_len, split_tokens);
    if (need > (size_t)PKV_NOALLOC_SCRATCH_BYTES) {
        pkv::record_detail(
            "paged_attn_decode_noalloc: the split partials of this problem need more than the "
            "16 MiB built-in scratch; use a larger split_tokens, fewer sequences per call, or "
            "paged_attn_decode with a caller workspace");
        return PKV_ERR_WORKSPACE;
    }
    void* scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        pkv::record_detail(cudaGetErrorString(e));
        return PKV_ERR_CUDA;
    }
    return paged_attn_decode(out, out_dtype, q, k_pool, v_pool, kv_dtype, block_tables,
                             max_blocks_per_seq, context_lens, num_seqs, n_heads, n_kv_heads,
                             head_dim, block_size, num_blocks, scale, max_context_len,
                             split_tokens, scratch, (size_t)PKV_NOALLOC_SCRATCH_BYTES, stream);
}
