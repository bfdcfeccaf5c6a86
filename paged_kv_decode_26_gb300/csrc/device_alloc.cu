// device_alloc.cu -- the physical block manager on the GPU.
//
// Page "大模型长文本推理基座从 FlashAttention 硬件加速机制到 vLLM 核心
// PagedAttention 显存物理布局深度剖析", section 三 (KVBlockManager,
// PagedAttentionScheduler.append_token) with the same semantics as the host
// manager (block_manager.cpp): blocks carry reference counts, the lowest free
// id is handed out first, sequences are served in order, an append opens a
// new block when the token count is a multiple of the block size.
//
// Device state (caller-owned device memory):
//   ref_counts  int32 [num_blocks]
//   free_ids    int32 [num_blocks]: the free ids in increasing order, from
//               state[0] (head) for state[1] (count) entries
//   state       int32 [4]: head, count, sequences that got no block in the
//               last append, spare
// Keeping the free ids sorted makes "lowest id first" for S sequences at
// once a prefix sum: the k-th sequence that needs a block takes
// free_ids[head + k].
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pagedkv.h"
#include "pkv_device.cuh"

namespace pkv {
void record_detail(const char* msg);
}

namespace {

constexpr int kAllocThreads = 1024;

// Exclusive prefix sum of one int per thread across the CTA; returns the
// exclusive sum and writes the total to *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += y;
        }
        warp_sums[lane] = w;  // inclusive sums of the warps
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
    *total = warp_sums[(blockDim.x >> 5) - 1];
    __syncthreads();
    return before;
}

// One step's append for every sequence, in sequence order (one CTA).
__global__ void __launch_bounds__(kAllocThreads)
    device_append_kernel(int32_t* __restrict__ ref_counts, const int32_t* __restrict__ free_ids,
                         int32_t* __restrict__ state, int32_t* __restrict__ block_tables,
                         int max_blocks, int32_t* __restrict__ context_lens,
                         int64_t* __restrict__ slot_mapping, int num_seqs, int block_size,
                         int num_blocks) {
    __shared__ int warp_sums[32];
    const int head = state[0];
    const int count = state[1];
    int used = 0;      // blocks handed out so far (uniform)
    int failed = 0;    // sequences without a slot (thread 0's tally)
    for (int base = 0; base < num_seqs; base += blockDim.x) {
        const int s = base + threadIdx.x;
        int n = 0, j = 0;
        bool ok = false, need = false;
        if (s < num_seqs) {
            n = context_lens[s];
            j = n / block_size;
            ok = n >= 0 && j < max_blocks;
            need = ok && (n % block_size == 0);
        }
        int total = 0;
        const int rank = block_exclusive_scan(need ? 1 : 0, warp_sums, &total);
        int32_t* row = block_tables + (size_t)s * max_blocks;
        if (s < num_seqs) {
            if (need) {
                if (used + rank < count) {
                    const int b = free_ids[head + used + rank];
                    if (b >= 0 && b < num_blocks) {
                        ref_counts[b] = 1;
                        row[j] = b;
                    } else {
                        ok = false;  // corrupt free list: leave the sequence alone
                    }
                } else {
                    ok = false;      // pool exhausted
                }
            }
            if (ok) {
                const int b = row[j];
                slot_mapping[s] = (int64_t)b * block_size + n % block_size;
                context_lens[s] = n + 1;
            } else {
                slot_mapping[s] = -1;
            }
        }
        int nfail = 0;
        const int fail_before = block_exclusive_scan((s < num_seqs && !ok) ? 1 : 0, warp_sums,
                                                     &nfail);
        (void)fail_before;
        failed += nfail;
        used = min(count, used + total);
    }
    if (threadIdx.x == 0) {
        state[0] = head + used;
        state[1] = count - used;
        state[2] = failed;
    }
}

// Drop one reference per listed id (an id listed twice is dropped twice).
__global__ void __launch_bounds__(256)
    device_unref_kernel(int32_t* __restrict__ ref_counts, const int32_t* __restrict__ ids, int n,
                        int num_blocks, unsigned int* errors) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const int b = ids[i];
        if (b < 0 || b >= num_blocks) {
            pkv::raise_error(errors, PKV_DEVERR_PAIR);
            continue;
        }
        // decrement unless already 0 (a free block stays free)
        int cur = ref_counts[b];
        while (cur > 0) {
            const int seen = atomicCAS(&ref_counts[b], cur, cur - 1);
            if (seen == cur) break;
            cur = seen;
        }
    }
}

// free_ids = every id with reference count 0, increasing; head = 0 (one CTA).
__global__ void __launch_bounds__(kAllocThreads)
    device_rebuild_kernel(const int32_t* __restrict__ ref_counts, int32_t* __restrict__ free_ids,
                          int32_t* __restrict__ state, int num_blocks) {
    __shared__ int warp_sums[32];
    int written = 0;
    for (int base = 0; base < num_blocks; base += blockDim.x) {
        const int b = base + threadIdx.x;
        const bool is_free = b < num_blocks && ref_counts[b] == 0;
        int total = 0;
        const int rank = block_exclusive_scan(is_free ? 1 : 0, warp_sums, &total);
        if (is_free) free_ids[written + rank] = b;
        written += total;
    }
    if (threadIdx.x == 0) {
        state[0] = 0;
        state[1] = written;
        state[2] = 0;
    }
}

bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

pkv_status fail_invalid(const char* why) {
    pkv::record_detail(why);
    return PKV_ERR_INVALID;
}

pkv_status launch_status(const char* where) {
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) return PKV_OK;
    pkv::record_detail(cudaGetErrorString(e));
    (void)where;
    return PKV_ERR_CUDA;
}

}  // namespace

namespace pkv {
unsigned int* device_error_word();
}

extern "C" {

PKV_API pkv_status pkv_device_rebuild_free_list(const int32_t* ref_counts, int32_t* free_ids,
                                                int32_t* state, int num_blocks, void* stream) {
    if (num_blocks < 0) return fail_invalid("num_blocks < 0");
    if (!ref_counts || !free_ids || !state) return fail_invalid("NULL pointer");
    if (!al4(ref_counts) || !al4(free_ids) || !al4(state)) return fail_invalid("alignment");
    device_rebuild_kernel<<<1, kAllocThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        ref_counts, free_ids, state, num_blocks);
    return launch_status("pkv_device_rebuild_free_list");
}

PKV_API pkv_status pkv_device_append_slots(int32_t* ref_counts, const int32_t* free_ids,
                                           int32_t* state, int32_t* block_tables,
                                           int max_blocks_per_seq, int32_t* context_lens,
                                           int num_seqs, int block_size, int num_blocks,
                                           int64_t* slot_mapping, void* stream) {
    if (num_seqs < 0 || max_blocks_per_seq < 0 || block_size <= 0 || num_blocks < 0)
        return fail_invalid("sizes");
    if (num_seqs == 0) return PKV_OK;
    if (!ref_counts || !free_ids || !state || !block_tables || !context_lens || !slot_mapping)
        return fail_invalid("NULL pointer");
    if (!al4(ref_counts) || !al4(free_ids) || !al4(state) || !al4(block_tables) ||
        !al4(context_lens) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return fail_invalid("alignment");
    device_append_kernel<<<1, kAllocThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        ref_counts, free_ids, state, block_tables, max_blocks_per_seq, context_lens, slot_mapping,
        num_seqs, block_size, num_blocks);
    return launch_status("pkv_device_append_slots");
}

PKV_API pkv_status pkv_device_free_blocks(int32_t* ref_counts, int32_t* free_ids, int32_t* state,
                                          const int32_t* block_ids, int n_ids, int num_blocks,
                                          void* stream) {
    if (n_ids < 0 || num_blocks < 0) return fail_invalid("sizes");
    if (!ref_counts || !free_ids || !state || (n_ids > 0 && !block_ids))
        return fail_invalid("NULL pointer");
    if (!al4(ref_counts) || !al4(free_ids) || !al4(state) || (n_ids > 0 && !al4(block_ids)))
        return fail_invalid("alignment");
    unsigned int* errors = pkv::device_error_word();
    if (!errors) return PKV_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (n_ids > 0) {
        const int grid = (n_ids + 255) / 256 < 1024 ? (n_ids + 255) / 256 : 1024;
        device_unref_kernel<<<grid, 256, 0, st>>>(ref_counts, block_ids, n_ids, num_blocks,
                                                  errors);
        const pkv_status s1 = launch_status("pkv_device_free_blocks");
        if (s1 != PKV_OK) return s1;
    }
    device_rebuild_kernel<<<1, kAllocThreads, 0, st>>>(ref_counts, free_ids, state, num_blocks);
    return launch_status("pkv_device_free_blocks");
}

}  // extern "C"
