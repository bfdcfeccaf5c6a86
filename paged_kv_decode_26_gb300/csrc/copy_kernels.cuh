// copy_kernels.cuh -- the two bit-exact copy companions of paged decode.
//
//   kv_append: one new token per sequence written into its page
//     (reshape-and-cache).  Page "大模型长文本推理基座从 FlashAttention 硬件加速
//     机制到 vLLM 核心 PagedAttention 显存物理布局深度剖析", section 三
//     append_token: the token lands in the last block, a new block having
//     been allocated when the previous one was full.
//   swap_blocks: dst[j] = src[i] for (i, j) pairs.  Page "vLLM 中
//     FlashAttention 与 KVCache 交换机制深度解析", swap_blocks(src_kv_cache,
//     dst_kv_cache, src_to_dst) with src_to_dst[i] = j; page "vLLM中
//     FlashAttention与KVCache优化解析", "Swap Blocks 机制": Key and Value caches
//     copied by separate calls.
//
// Both move 16-byte vectors; a row of one token (all kv heads) and a whole
// block are contiguous in the [num_blocks, B, Hk, D] pool, so every warp
// access is a fully coalesced 512-byte run.
#pragma once

#include "pkv_device.cuh"

namespace pkv {

// Threads = num_seqs * row_vec (16-byte vectors per token row) for K and V.
__global__ void __launch_bounds__(256)
    kv_append_kernel(uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                     const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                     const int64_t* __restrict__ slots, int num_seqs, int row_vec,
                     int64_t num_slots, unsigned int* errors) {
    const int64_t total = (int64_t)num_seqs * row_vec;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int s = (int)(i / row_vec);
        const int v = (int)(i - (int64_t)s * row_vec);
        const int64_t slot = slots[s];
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (v == 0) raise_error(errors, PKV_DEVERR_SLOT);
            continue;
        }
        const int64_t src = (int64_t)s * row_vec + v;
        const int64_t dst = slot * row_vec + v;
        k_pool[dst] = k_new[src];
        v_pool[dst] = v_new[src];
    }
}

constexpr int kSwapThreads = 256;
constexpr int kSwapUnroll = 8;

// Up to two caches (Key and Value) copied by one launch with the same pairs.
struct SwapPools {
    uint4* dst[2];
    const uint4* src[2];
};

// One CTA per (pair, cache) (grid-strided over pairs, blockIdx.y = cache),
// each thread moving up to kSwapUnroll 16-byte vectors per round with all
// loads issued before the stores.  The data is touched once: loads and
// stores use the streaming (evict-first) cache policy.
__global__ void __launch_bounds__(kSwapThreads)
    swap_blocks_kernel(const SwapPools pools, int64_t block_vec,
                       const int64_t* __restrict__ pairs, int n_pairs, int64_t num_src,
                       int64_t num_dst, unsigned int* errors) {
    uint4* __restrict__ dst = pools.dst[blockIdx.y];
    const uint4* __restrict__ src = pools.src[blockIdx.y];
    for (int k = blockIdx.x; k < n_pairs; k += gridDim.x) {
        const int64_t i = pairs[2 * (int64_t)k];
        const int64_t j = pairs[2 * (int64_t)k + 1];
        if (i < 0 || j < 0) continue;
        if (i >= num_src || j >= num_dst) {
            if (threadIdx.x == 0 && blockIdx.y == 0) raise_error(errors, PKV_DEVERR_PAIR);
            continue;
        }
        const uint4* s = src + i * block_vec;
        uint4* d = dst + j * block_vec;
        for (int64_t base = 0; base < block_vec; base += (int64_t)kSwapThreads * kSwapUnroll) {
            uint4 r[kSwapUnroll];
#pragma unroll
            for (int u = 0; u < kSwapUnroll; ++u) {
                const int64_t e = base + (int64_t)u * kSwapThreads + threadIdx.x;
                if (e < block_vec) r[u] = __ldcs(s + e);
            }
#pragma unroll
            for (int u = 0; u < kSwapUnroll; ++u) {
                const int64_t e = base + (int64_t)u * kSwapThreads + threadIdx.x;
                if (e < block_vec) __stcs(d + e, r[u]);
            }
        }
    }
}

}  // namespace pkv
