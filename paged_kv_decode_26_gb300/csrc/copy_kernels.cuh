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
// A row of one token (all kv heads) and a whole block are contiguous in the
// [num_blocks, B, Hk, D] pool.  The append and the block copy move 16-byte
// vectors (every warp access a coalesced 512-byte run; a pinned-host source
// is reached through unified addressing).  A second block-copy kernel
// moves whole blocks between device pools with bulk copies through shared
// memory; it measured a few percent behind the vector kernel on GB300 and
// runs only when asked for (see capi.cu).
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
constexpr int kMaxBulkStages = 8;
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

// ------------------------------------------------------- bulk block copy
//
// swap_blocks between two device pools through the copy engine of each SM
// (cp.async.bulk): a block (or a chunk of it) moves global -> shared with
// one bulk load that completes on an mbarrier, then shared -> global with
// one bulk store; no thread touches the bytes.  One warp per CTA: its lanes
// look up the pairs of the CTA's items in batches, then lane 0 keeps
// `stages` chunks in flight: the store of chunk n is issued as soon as its
// load lands, and the slot of chunk n - 1 is refilled with chunk n - 1 +
// stages once that chunk's store has finished reading it.  The grid is a
// whole number of CTAs per SM; CTA b takes a contiguous range of the
// (pair, cache, chunk) items, so the ranges differ by one item at most.

constexpr int kBulkBatch = 128;   // item descriptors looked up at once

struct BulkSwapParams {
    SwapPools pools;
    const int64_t* pairs;
    int64_t n_pairs;
    int64_t num_src;
    int64_t num_dst;
    uint64_t block_bytes;
    uint32_t chunk_bytes;   // multiple of 16; the last chunk of a block may be shorter
    int chunks;             // per block
    int n_pools;
    int stages;
    int hint;               // 1: loads and stores carry the L2 evict-first hint
    unsigned int* errors;
};

struct BulkItem {
    const char* src;
    char* dst;
    uint32_t bytes;   // 0: skipped pair
};

__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst_smem)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_store(void* dst, const void* src_smem, uint32_t bytes,
                                           uint64_t policy) {
    asm volatile(
        "cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(
            reinterpret_cast<uint64_t>(dst)),
        "r"(smem_addr(src_smem)), "r"(bytes), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_load_plain(void* dst_smem, const void* src, uint32_t bytes,
                                                uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst_smem)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_store_plain(void* dst, const void* src_smem,
                                                 uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                     reinterpret_cast<uint64_t>(dst)),
                 "r"(smem_addr(src_smem)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Every bulk store group but the newest `1` has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all_but_one() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// Every bulk store group has completed (its writes are performed).
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__global__ void __launch_bounds__(32)
    swap_blocks_bulk_kernel(const BulkSwapParams p) {
    extern __shared__ __align__(128) unsigned char bulk_smem[];
    __shared__ __align__(8) uint64_t full[kMaxBulkStages];
    __shared__ BulkItem items[kBulkBatch];
    const int lane = threadIdx.x;
    const int S = p.stages;
    if (S < 2 || S > kMaxBulkStages) {
        if (lane == 0) raise_error(p.errors, PKV_DEVERR_CONFIG);
        return;
    }
    const int64_t per_pair = (int64_t)p.n_pools * p.chunks;
    const int64_t total = p.n_pairs * per_pair;
    const int64_t begin = total * blockIdx.x / gridDim.x;
    const int64_t end = total * (blockIdx.x + 1) / gridDim.x;
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    __syncwarp();
    const uint64_t policy = l2_policy_evict_first();
    uint32_t phase_bits = 0;   // lane 0: parity of each slot's next wait
    bool ok = true;
    for (int64_t b0 = begin; b0 < end && ok; b0 += kBulkBatch) {
        const int nb = (int)(end - b0 < kBulkBatch ? end - b0 : kBulkBatch);
        // ---- look up the batch's pairs (all lanes)
        for (int t = lane; t < nb; t += 32) {
            const int64_t u = b0 + t;
            const int64_t k = u / per_pair;
            const int r = (int)(u - k * per_pair);
            const int pool = r / p.chunks;
            const int c = r - pool * p.chunks;
            const int64_t i = p.pairs[2 * k];
            const int64_t j = p.pairs[2 * k + 1];
            BulkItem it;
            it.src = nullptr;
            it.dst = nullptr;
            it.bytes = 0;
            if (i >= 0 && j >= 0) {
                if (i >= p.num_src || j >= p.num_dst) {
                    if (pool == 0 && c == 0) raise_error(p.errors, PKV_DEVERR_PAIR);
                } else {
                    const uint64_t off = (uint64_t)c * p.chunk_bytes;
                    const uint64_t left = p.block_bytes - off;
                    it.bytes = (uint32_t)(left < p.chunk_bytes ? left : p.chunk_bytes);
                    it.src = reinterpret_cast<const char*>(p.pools.src[pool]) +
                             (uint64_t)i * p.block_bytes + off;
                    it.dst = reinterpret_cast<char*>(p.pools.dst[pool]) +
                             (uint64_t)j * p.block_bytes + off;
                }
            }
            items[t] = it;
        }
        __syncwarp();
        if (lane == 0) {
            // ---- pipeline over the batch: slot n % S holds item n
            const int pre = nb < S ? nb : S;
            for (int n = 0; n < pre; ++n) {
                if (items[n].bytes) {
                    mbar_arrive_expect_tx(&full[n], items[n].bytes);
                    if (p.hint)
                        bulk_load(bulk_smem + (size_t)n * p.chunk_bytes, items[n].src,
                                  items[n].bytes, &full[n], policy);
                    else
                        bulk_load_plain(bulk_smem + (size_t)n * p.chunk_bytes, items[n].src,
                                        items[n].bytes, &full[n]);
                } else {
                    mbar_arrive(&full[n]);
                }
            }
            int n = 0;
            for (; n < nb; ++n) {
                const int slot = n % S;
                if (!mbar_wait(&full[slot], (phase_bits >> slot) & 1u, p.errors)) {
                    ok = false;
                    break;
                }
                phase_bits ^= 1u << slot;
                if (items[n].bytes) {
                    fence_proxy_async_smem();
                    if (p.hint)
                        bulk_store(items[n].dst, bulk_smem + (size_t)slot * p.chunk_bytes,
                                   items[n].bytes, policy);
                    else
                        bulk_store_plain(items[n].dst, bulk_smem + (size_t)slot * p.chunk_bytes,
                                         items[n].bytes);
                }
                bulk_commit();
                // refill the slot of item n - 1 with item n - 1 + S once the
                // store of item n - 1 has read it
                const int m = n - 1 + S;
                if (n >= 1 && m < nb) {
                    bulk_wait_read_all_but_one();
                    const int ms = m % S;
                    if (items[m].bytes) {
                        mbar_arrive_expect_tx(&full[ms], items[m].bytes);
                        if (p.hint)
                            bulk_load(bulk_smem + (size_t)ms * p.chunk_bytes, items[m].src,
                                      items[m].bytes, &full[ms], policy);
                        else
                            bulk_load_plain(bulk_smem + (size_t)ms * p.chunk_bytes, items[m].src,
                                            items[m].bytes, &full[ms]);
                    } else {
                        mbar_arrive(&full[ms]);
                    }
                }
            }
            if (!ok) {
                // item n never landed: wait once more (bounded) for it and
                // for the loads issued after it, so that no copy still
                // writes shared memory when the CTA leaves
                const int issued = min(nb, S + max(0, n - 1));
                for (int q = n; q < issued; ++q) {
                    const int slot = q % S;
                    if (!mbar_wait(&full[slot], (phase_bits >> slot) & 1u, p.errors)) break;
                    phase_bits ^= 1u << slot;
                }
            }
            bulk_wait_all();
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        __syncwarp();
    }
}

}  // namespace pkv
