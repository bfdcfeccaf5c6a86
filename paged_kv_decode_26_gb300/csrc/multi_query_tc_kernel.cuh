// multi_query_tc_kernel.cuh -- causal attention of several new tokens per
// sequence over the paged KV cache on Blackwell's 5th-generation tensor
// cores (tcgen05: MMAs issued by one thread from shared-memory descriptors,
// fp32 accumulators in tensor memory), sm_103a.  Same operation, inputs and
// outputs as paged_multi_query_kernel; taken for chunks of at least 48 rows
// (tokens x group, groups of 1 and 2) or 16 rows (groups of 4 and 8), where
// it measured faster.
//
// Pages followed (cited by title and section):
//   [SWAP]   "vLLM 中 FlashAttention 与 KVCache 交换机制深度解析": FlashAttention
//            (Kernel Fusion + Tiling + OnlineSoftmax: Q, K, V tiles through
//            on-chip memory, the running max M and sum L, O rescaled) and the
//            serving loop's prefill step.
//   [LAYOUT] "大模型长文本推理基座从 FlashAttention 硬件加速机制到 vLLM 核心
//            PagedAttention 显存物理布局深度剖析", section 二.2: block table.
//
// One CTA per (pair of query tiles, kv head, sequence).  A query tile is 128
// rows: 128/G consecutive query tokens x the G query heads of the kv head
// (row r: token r / G, head r % G); the pair shares every K/V page it loads.
// Warps 0-3 and 4-7 run the softmax of tile 0 and tile 1, one thread per row
// (thread r of a group owns tensor-memory lane r).  Lane 0 of warp 8 issues
// every MMA of tile 0 and lane 0 of warp 10 those of tile 1 (a thread issues
// one tcgen05.mma per ~100 cycles, so two issuers double the MMA rate;
// keeping each tile's products in one thread keeps them in order); warp 8
// also owns the tensor memory.  Warp 9 loads K/V by TMA and zeroes V rows
// that must not reach a product.  Per key tile j of 64 keys and query tile t:
//   K_j, V_j            pages by TMA into a ring of `stages` slots, per head
//                       64-element boxes with 128-byte swizzle
//   S_tj = Q_t K_j^T    M=128 N=64, A = Q_t (K-major), B = K_j (K-major), into
//                       one of two S buffers of tile t in tensor memory
//   P_tj                2^(x - m) as hi + lo 16-bit parts, written by the
//                       softmax threads into the S buffer they just read
//   O_t += P_tj V_j     M=128 N=D, A = P from tensor memory, B = V_j
//                       (MN-major: D contiguous), O_t in tensor memory
// S_t,j+1 is ready while the softmax works on tile j, so the tensor core
// alternates between the groups' products.  Rescaling O costs a
// tensor-memory round trip, so a row keeps an older maximum until a new
// score exceeds it by more than 2^8 (P <= 256 meanwhile; O and the sum L
// share the maximum they were built with, so the quotient is unchanged).
// V rows past the context, on a missing page or never loaded are zeroed by
// the loading warp before the tile is marked full (P is 0 there, but 0 * NaN
// is not).
#pragma once

#include <type_traits>

#include "multi_query_kernel.cuh"

namespace pkv {

constexpr int kTcKeys = 64;          // keys per tile (N of S = Q K^T)
constexpr int kTcRows = 128;         // query rows per query tile (M)
constexpr int kTcQTiles = 2;         // query tiles per CTA
constexpr int kTcThreads = 352;      // 8 softmax warps, 2 MMA warps, 1 TMA warp
constexpr float kTcRescale = 8.0f;   // log2 of the growth tolerated before O is rescaled

// ---------------------------------------------------------------- tcgen05

// Shared-memory matrix descriptor, 128-byte swizzle: start, leading and
// stride byte offsets (>> 4), descriptor version 1.
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// kind::f16 instruction descriptor: fp32 accumulator, A and B both of type
// T, A K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1), shape M x N.
template <typename T>
__device__ __forceinline__ uint32_t tc_idesc(int M, int N, int b_mn) {
    const uint32_t fmt = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
    return (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// Same with A read from tensor memory: row i of A in lane i, 16-bit
// elements k = 2c, 2c + 1 in the low and high half of column c (one K=16
// step spans 8 columns).
__device__ __forceinline__ void tc_mma_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// `bar` completes once every MMA this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Makes this thread's ordinary shared-memory stores visible to the tensor
// core (async proxy) once a barrier orders them.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

#define PKV_TC_REGS32(r)                                                                       \
    "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),         \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), \
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),          \
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),          \
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])

// 32 consecutive 32-bit columns of one tensor-memory lane per thread
// (32x32b shape: thread i of warp w reads lane 32 (w % 4) + i).
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : PKV_TC_REGS32(r)
        : "r"(taddr));
}

__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tc_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared memory of one CTA: 1 KB alignment slack, the two Q tiles, the K/V
// ring, barriers, block ids, one word.
inline size_t multi_query_tc_smem_bytes(int D, int stages, int max_pages, int lpt_seqs = 0) {
    const size_t q = (size_t)kTcQTiles * kTcRows * D * 2;
    const size_t kv = (size_t)stages * 2 * kTcKeys * D * 2;
    return 1024 + q + kv + (size_t)(3 * stages + 15) * sizeof(uint64_t) +
           (size_t)max_pages * sizeof(int) + sizeof(int) +
           (lpt_seqs > 0 ? (size_t)(lpt_seqs + 1) * sizeof(int) : 0);
}

// Longest context first.  A CTA's work grows with its sequence's context,
// and with lengths spread over orders of magnitude the longest sequences'
// CTAs, dispatched in index order, can start last and form the tail.  With
// p.lpt_seqs the sequences are ranked by context length (ties: lower index
// first) and CTA u (grid order) takes the sequence of rank u / (kv heads x
// query tiles), the kv head fastest and the query tiles from the last (the
// one that sees the most keys).  s_len: p.lpt_seqs + 1 ints of shared
// memory that nothing else uses.
__device__ __forceinline__ void longest_first(const MultiQueryParams& p, int* s_len, int& tile,
                                              int& kvh, int& s) {
    const int S = p.lpt_seqs;
    int* s_pick = s_len + S;
    const long long u =
        blockIdx.x + (long long)gridDim.x * (blockIdx.y + (long long)gridDim.y * blockIdx.z);
    const int per_seq = (int)(gridDim.x * gridDim.y);
    const int r = (int)(u / per_seq);
    const int rem = (int)(u % per_seq);
    kvh = rem % (int)gridDim.y;
    tile = (int)gridDim.x - 1 - rem / (int)gridDim.y;
    for (int i = threadIdx.x; i < S; i += blockDim.x) s_len[i] = p.context_lens[i];
    __syncthreads();
    // the ranks are a permutation of 0 .. S-1: exactly one sequence has rank r
    for (int i = threadIdx.x; i < S; i += blockDim.x) {
        const int ni = s_len[i];
        int rank = 0;
        for (int j = 0; j < S; ++j) {
            const int nj = s_len[j];
            rank += (nj > ni || (nj == ni && j < i)) ? 1 : 0;
        }
        if (rank == r) *s_pick = i;
    }
    __syncthreads();
    s = *s_pick;
}

template <int D, int BS, typename T>
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_multi_query_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                                const __grid_constant__ CUtensorMap tm_k,
                                const __grid_constant__ CUtensorMap tm_v,
                                const MultiQueryParams p) {
    constexpr int HALVES = D / 64;
    constexpr int PAGES = kTcKeys / BS;                 // pages per key tile
    constexpr uint32_t KV_HALF = kTcKeys * 128;         // [64 keys x 64 elements]
    constexpr uint32_t KV_BYTES = HALVES * KV_HALF;     // one K (or V) tile
    constexpr uint32_t Q_HALF = kTcRows * 128;          // [128 rows x 64 elements]
    constexpr uint32_t Q_BYTES = HALVES * Q_HALF;       // one query tile
    constexpr uint32_t TMEM_COLS = 512;
    constexpr uint32_t TILE_COLS = 256;                 // per query tile: O, then two S buffers
    constexpr uint32_t S_COL = D;
    constexpr int ALL_PAGES = (1 << PAGES) - 1;
    static_assert(kTcKeys % BS == 0 && D % 64 == 0 && D + 2 * kTcKeys <= TILE_COLS, "shape");

    extern __shared__ __align__(1024) unsigned char smem_raw[];

    const int G = p.group;
    if (blockDim.x != kTcThreads || G < 1 || G > 8 || kTcRows % G != 0 || p.stages < 2) {
        if (threadIdx.x == 0) raise_error(p.errors, PKV_DEVERR_CONFIG);
        return;
    }

    // ---- shared memory (1024-byte aligned for the swizzle)
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char* sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    unsigned char* sQ = sm;                                         // 2 x HALVES x [128 x 128 B]
    unsigned char* sKV = sQ + kTcQTiles * Q_BYTES;                  // stages x (K, V)
    uint64_t* kv_full = reinterpret_cast<uint64_t*>(sKV + (size_t)p.stages * 2 * KV_BYTES);
    uint64_t* kv_free = kv_full + p.stages;      // [stages]: both issuers done with the slot
    uint64_t* kv_land = kv_free + p.stages;      // [stages]: loads landed (tiles to zero)
    uint64_t* q_full = kv_land + p.stages;
    uint64_t* s_full = q_full + 1;               // [tile][buffer]: S ready
    uint64_t* p_full = s_full + 4;               // [tile][buffer]: P written (128 arrivals)
    uint64_t* o_done = p_full + 4;               // [tile][parity of key tile]: P V done
    uint64_t* fin = o_done + 4;                  // [tile]: every MMA of the tile's issuer done
    int* s_bid = reinterpret_cast<int*>(fin + 2);
    int* s_tmem = s_bid + p.max_pages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    int tile = blockIdx.x, kvh = blockIdx.y, s = blockIdx.z;
    if (p.lpt_seqs > 0) longest_first(p, s_tmem + 1, tile, kvh, s);
    const int QT = kTcRows / G;                  // query tokens per query tile
    const int qs0 = p.q_start[s], qs1 = p.q_start[s + 1];
    const int n = p.context_lens[s];
    const int q_len = qs1 - qs0;
    if (q_len < 0 || q_len > n || qs0 < 0 || qs1 > p.total_q || q_len > p.max_q_len ||
        n > p.max_blocks_per_seq * BS || (n + BS - 1) / BS > p.max_pages) {
        if (tile == 0 && kvh == 0 && threadIdx.x == 0) raise_error(p.errors, PKV_DEVERR_CONTEXT);
        return;
    }
    const int tok_lo = tile * kTcQTiles * QT;
    if (tok_lo >= q_len) return;
    const int first_pos = n - q_len;                 // position of query token 0
    // key tiles each query tile needs (0: the tile has no token)
    const int nt0 = (first_pos + min(q_len, tok_lo + QT) + kTcKeys - 1) / kTcKeys;
    const int nt1 = tok_lo + QT < q_len
                        ? (first_pos + min(q_len, tok_lo + 2 * QT) + kTcKeys - 1) / kTcKeys
                        : 0;
    auto ntiles = [&](int t) { return t ? nt1 : nt0; };
    const int n_tiles = max(nt0, nt1);
    const int n_keys = first_pos + min(q_len, tok_lo + kTcQTiles * QT);
    const int n_pages = (n_keys + BS - 1) / BS;
    const int zero_from = min(n, n_pages * BS);      // V rows from here on are zeroed

    int missing = 0;
    for (int i = threadIdx.x; i < n_pages; i += blockDim.x) {
        int b = p.block_tables[(size_t)s * p.max_blocks_per_seq + i];
        if (b < 0 || b >= p.num_blocks) {
            raise_error(p.errors, PKV_DEVERR_BLOCK_ID);
            b = -1;
            missing = 1;
        }
        s_bid[i] = b;
    }
    if (warp == 8) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(s_tmem)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (threadIdx.x == 0) {
        for (int st = 0; st < p.stages; ++st) {
            mbar_init(&kv_full[st], 1);
            mbar_init(&kv_free[st], kTcQTiles);
            mbar_init(&kv_land[st], 1);
        }
        mbar_init(q_full, 1);
        for (int b = 0; b < 4; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&p_full[b], kTcRows);
            mbar_init(&o_done[b], 1);
        }
        mbar_init(&fin[0], 1);
        mbar_init(&fin[1], 1);
        fence_barrier_init();
    }
    tc_fence_before();
    const bool any_missing = __syncthreads_or(missing) != 0;   // a page of the context is absent
    tc_fence_after();
    const uint32_t tmem = (uint32_t)*s_tmem;

    // pages of key tile j that are present: bit pg for page j * PAGES + pg
    // (all bits where no page is absent: pages past n_pages hold only keys
    // that every row masks by position)
    auto page_mask = [&](int j) -> int {
        if (!any_missing) return ALL_PAGES;
        int m = 0;
#pragma unroll
        for (int pg = 0; pg < PAGES; ++pg) {
            const int page = j * PAGES + pg;
            if (page < n_pages && s_bid[page] >= 0) m |= 1 << pg;
        }
        return m;
    };
    // V rows of key tile j that must be zeroed before P V: past the context,
    // never loaded, or on a missing page
    auto needs_zero = [&](int j) -> bool {
        return (j + 1) * kTcKeys > zero_from || page_mask(j) != ALL_PAGES;
    };
    // (with every page present, a tile ending at or before zero_from lies
    // wholly on pages below n_pages)

    if (warp == 9) {
        // ================= TMA producer (the whole warp zeroes V rows) =================
        if (lane == 0) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
            uint32_t q_bytes = 0;
#pragma unroll
            for (int t = 0; t < kTcQTiles; ++t) q_bytes += ntiles(t) > 0 ? Q_BYTES : 0;
            mbar_arrive_expect_tx(q_full, q_bytes);
            const uint64_t once = l2_policy_evict_first();
#pragma unroll
            for (int t = 0; t < kTcQTiles; ++t) {
                if (ntiles(t) == 0) continue;
                for (int h = 0; h < HALVES; ++h)
                    tma_load_4d(sQ + t * Q_BYTES + h * Q_HALF, &tm_q, q_full, 0, h, kvh * G,
                                qs0 + tok_lo + t * QT, once);
            }
        }
        const uint64_t keep = l2_policy_evict_normal();   // pages serve other query tiles
        int issued = 0;
        int st = 0, round = 0;               // slot of tile j, times the ring wrapped
        uint32_t land_par = 0;               // bit st: phase of kv_land[st] to wait for next
        for (int j = 0; j < n_tiles; ++j) {
            const bool w = round == 0 || mbar_wait(&kv_free[st], (round - 1) & 1, p.errors);
            if (!__all_sync(0xffffffffu, w)) break;
            const bool zero = needs_zero(j);
            // a tile with rows to zero lands on kv_land; kv_full follows the zeroing
            uint64_t* bar = zero ? &kv_land[st] : &kv_full[st];
            unsigned char* dk = sKV + (size_t)st * 2 * KV_BYTES;
            if (lane == 0) {
                uint32_t bytes = 0;
                for (int pg = 0; pg < PAGES; ++pg) {
                    const int page = j * PAGES + pg;
                    if (page < n_pages && s_bid[page] >= 0) bytes += 2 * HALVES * BS * 128;
                }
                if (bytes == 0) {
                    mbar_arrive(bar);
                } else {
                    mbar_arrive_expect_tx(bar, bytes);
                    for (int pg = 0; pg < PAGES; ++pg) {
                        const int page = j * PAGES + pg;
                        if (page >= n_pages || s_bid[page] < 0) continue;
                        for (int h = 0; h < HALVES; ++h) {
                            tma_load_4d(dk + h * KV_HALF + pg * BS * 128, &tm_k, bar, 0,
                                        kvh * HALVES + h, 0, s_bid[page], keep);
                            tma_load_4d(dk + KV_BYTES + h * KV_HALF + pg * BS * 128, &tm_v, bar,
                                        0, kvh * HALVES + h, 0, s_bid[page], keep);
                        }
                    }
                }
            }
            issued = j + 1;
            if (zero) {
                const bool w2 = mbar_wait(&kv_land[st], (land_par >> st) & 1u, p.errors);
                land_par ^= 1u << st;
                if (!__all_sync(0xffffffffu, w2)) break;
                const int pm = page_mask(j);
                unsigned char* sv = dk + KV_BYTES;
                for (int idx = lane; idx < kTcKeys * HALVES; idx += 32) {
                    const int row = idx % kTcKeys, h = idx / kTcKeys;
                    const int key = j * kTcKeys + row;
                    if (key >= zero_from || !((pm >> (row / BS)) & 1)) {
                        uint4* z = reinterpret_cast<uint4*>(sv + h * KV_HALF + row * 128);
#pragma unroll
                        for (int c = 0; c < 8; ++c) z[c] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&kv_full[st]);
            }
            if (++st == p.stages) {
                st = 0;
                ++round;
            }
        }
        // every load issued has landed before the CTA may exit (earlier
        // tiles of a slot were consumed before the slot was refilled)
        if (lane == 0)
            for (int j = max(0, issued - p.stages); j < issued; ++j)
                mbar_wait(&kv_full[j % p.stages], (j / p.stages) & 1, p.errors);
        __syncwarp();
    } else if (warp == 8 || warp == 10) {
        // ================= MMA issuer of query tile t =================
        const int t = warp == 8 ? 0 : 1;
        const int ntt = ntiles(t);
        if (lane == 0) {
            const uint32_t id_s = tc_idesc<T>(kTcRows, kTcKeys, 0);
            const uint32_t id_o = tc_idesc<T>(kTcRows, D, 1);
            // Descriptors of Q tile t, K and V of slot 0; other operands add
            // their byte offset >> 4 to the start-address field (shared
            // addresses stay below 2^18, so the 14-bit field never carries).
            const uint64_t dq = tc_desc_sw128(smem_addr(sQ + t * Q_BYTES), 16, 1024);
            const uint64_t dk = tc_desc_sw128(smem_addr(sKV), 16, 1024);
            const uint64_t dv = tc_desc_sw128(smem_addr(sKV + KV_BYTES), KV_HALF, 1024);
            constexpr uint32_t SLOT16 = (2 * KV_BYTES) >> 4;
            const uint32_t base = tmem + t * TILE_COLS;      // O of tile t, then its S buffers
            int s_st = 0;          // slot of the next tile whose S is issued
            uint32_t s_ph = 0;     // and the phase of its kv_full
            // S_tj = Q_t K_j^T into S buffer j & 1
            auto issue_s = [&](int j) -> bool {
                if (!mbar_wait(&kv_full[s_st], s_ph, p.errors)) return false;
                tc_fence_after();
                const uint64_t kd = dk + (uint64_t)(s_st * SLOT16);
                const uint32_t d = base + S_COL + (j & 1) * kTcKeys;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t qo = ((ks / 4) * Q_HALF + (ks % 4) * 32) >> 4;
                    const uint32_t ko = ((ks / 4) * KV_HALF + (ks % 4) * 32) >> 4;
                    tc_mma(d, dq + qo, kd + ko, id_s, ks > 0 ? 1u : 0u);
                }
                tc_commit(&s_full[t * 2 + (j & 1)]);
                if (++s_st == p.stages) {
                    s_st = 0;
                    s_ph ^= 1u;
                }
                return true;
            };
            bool ok = ntt == 0 || mbar_wait(q_full, 0, p.errors);
            for (int j = 0; ok && j < 2 && j < ntt; ++j) ok = issue_s(j);
            int v_st = 0, v_round = 0;     // slot of tile j, times the ring wrapped
            for (int j = 0; ok && j < n_tiles; ++j) {
                if (j < ntt) {
                    if (!mbar_wait(&p_full[t * 2 + (j & 1)], (j >> 1) & 1, p.errors)) {
                        ok = false;
                        break;
                    }
                    // O_t += P_tj V_j (hi part, then lo part; P in tensor memory)
                    tc_fence_after();
                    const uint64_t vd = dv + (uint64_t)(v_st * SLOT16);
                    const uint32_t pa = base + S_COL + (j & 1) * kTcKeys;
#pragma unroll
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int ks = 0; ks < kTcKeys / 16; ++ks)
                            tc_mma_tmem_a(base, pa + part * (kTcKeys / 2) + ks * 8,
                                          vd + (uint64_t)((ks * 16 * 128) >> 4), id_o,
                                          (j > 0 || part > 0 || ks > 0) ? 1u : 0u);
                    tc_commit(&o_done[t * 2 + (j & 1)]);
                    tc_commit(&kv_free[v_st]);
                    if (j + 2 < ntt) ok = issue_s(j + 2);
                } else {
                    // this tile's rows never see key tile j: release the slot
                    // once it is loaded (keeps kv_free's phases in step)
                    if (!mbar_wait(&kv_full[v_st], v_round & 1, p.errors)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive(&kv_free[v_st]);
                }
                if (++v_st == p.stages) {
                    v_st = 0;
                    ++v_round;
                }
            }
            // every MMA of this issuer complete before the tensor memory is released
            if (ntt > 0) {
                tc_commit(&fin[t]);
                mbar_wait(&fin[t], 0, p.errors);
            }
        }
        __syncwarp();
    } else {
        // ================= softmax: group t, thread r owns row r of tile t =================
        const int t = warp >> 2;
        const int r = (warp & 3) * 32 + lane;            // tensor-memory lane
        if (ntiles(t) > 0) {
            const int tok = tok_lo + t * QT + r / G;
            const bool real = tok < q_len;
            const int pos = real ? first_pos + tok : -1;     // last key of this row
            const uint32_t t_lane = tmem + t * TILE_COLS + ((uint32_t)((warp & 3) * 32) << 16);
            const float sc = p.scale_log2;
            const bool pos_sc = sc > 0.f;                    // the usual case
            float m_used = -INFINITY;
            float2 l4[4];                                  // row sum as 8 partial sums
#pragma unroll
            for (int i = 0; i < 4; ++i) l4[i] = make_float2(0.f, 0.f);
            bool ok = true;
            const int ntt = ntiles(t);
            for (int j = 0; j < ntt; ++j) {
                const int b = j & 1;
                const bool w = mbar_wait(&s_full[t * 2 + b], (j >> 1) & 1, p.errors);
                if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                tc_fence_after();
                uint32_t sr[kTcKeys];
                tc_ld32(t_lane + S_COL + b * kTcKeys, sr);
                tc_ld32(t_lane + S_COL + b * kTcKeys + 32, sr + 32);
                tc_wait_ld();
                const int key0 = j * kTcKeys;
                const int pm = page_mask(j);
                const bool full = key0 + kTcKeys - 1 <= pos && pm == ALL_PAGES;
                // y: raw scores (scaled ones if the scale is not positive),
                // -inf where a key is hidden from this row
                float y[kTcKeys];
                if (full && pos_sc) {
#pragma unroll
                    for (int c = 0; c < kTcKeys; ++c) y[c] = __uint_as_float(sr[c]);
                } else {
#pragma unroll
                    for (int c = 0; c < kTcKeys; ++c) {
                        const bool keep = key0 + c <= pos && ((pm >> (c / BS)) & 1);
                        const float v = pos_sc ? __uint_as_float(sr[c]) : __uint_as_float(sr[c]) * sc;
                        y[c] = keep ? v : -INFINITY;
                    }
                }
                // row maximum as 8 independent chains
                float m8[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) m8[c] = y[c];
#pragma unroll
                for (int c = 8; c < kTcKeys; ++c) m8[c & 7] = fmaxf(m8[c & 7], y[c]);
                const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                       fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
                const float a = pos_sc ? sc : 1.f;           // exponent = y * a - m
                const float tmax = mx * a;
                const bool first = m_used == -INFINITY;
                const bool grow = tmax > m_used + kTcRescale;
                float alpha = 1.f;
                if (grow) {
                    alpha = first ? 1.f : exp2f(m_used - tmax);
                    m_used = tmax;
                }
                if (__any_sync(0xffffffffu, grow && !first)) {
                    // O of this warp's rows holds P V up to key tile j-1 first
                    const bool w2 = mbar_wait(&o_done[t * 2 + ((j - 1) & 1)], ((j - 1) >> 1) & 1,
                                              p.errors);
                    if (!__all_sync(0xffffffffu, w2)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t ov[32];
                        tc_ld32(t_lane + c0, ov);
                        tc_wait_ld();
                        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                        for (int c = 0; c < 32; c += 2) {
                            const float2 v = __fmul2_rn(
                                make_float2(__uint_as_float(ov[c]), __uint_as_float(ov[c + 1])), a2);
                            ov[c] = __float_as_uint(v.x);
                            ov[c + 1] = __float_as_uint(v.y);
                        }
                        tc_st32(t_lane + c0, ov);
                    }
                }
                if (j >= 2) {
                    // keeps this barrier's phases in step with the waits above
                    const bool w2 = mbar_wait(&o_done[t * 2 + b], ((j - 2) >> 1) & 1, p.errors);
                    if (!__all_sync(0xffffffffu, w2)) { ok = false; break; }
                }
                l4[0] = __fmul2_rn(l4[0], make_float2(alpha, alpha));
                l4[1] = __fmul2_rn(l4[1], make_float2(alpha, alpha));
                l4[2] = __fmul2_rn(l4[2], make_float2(alpha, alpha));
                l4[3] = __fmul2_rn(l4[3], make_float2(alpha, alpha));
                const float mu = m_used == -INFINITY ? 0.f : m_used;
                const float2 a2 = make_float2(a, a), nmu2 = make_float2(-mu, -mu);
                const float2 neg1 = make_float2(-1.f, -1.f);
                // P = 2^(y a - m) as hi + lo over the S buffer just read: hi in
                // its columns [0, 32), lo in [32, 64), keys 2i and 2i+1 in column i
                uint32_t ph[kTcKeys / 2], pl[kTcKeys / 2];
#pragma unroll
                for (int i = 0; i < kTcKeys / 2; ++i) {
                    const float2 e = __ffma2_rn(make_float2(y[2 * i], y[2 * i + 1]), a2, nmu2);
                    const float2 pv = make_float2(exp2f(e.x), exp2f(e.y));
                    l4[i & 3] = __fadd2_rn(l4[i & 3], pv);
                    ph[i] = pack2<T>(pv.x, pv.y);
                    const float2 lo = __ffma2_rn(unpack2<T>(ph[i]), neg1, pv);
                    pl[i] = pack2<T>(lo.x, lo.y);
                }
                tc_st32(t_lane + S_COL + b * kTcKeys, ph);
                tc_st32(t_lane + S_COL + b * kTcKeys + 32, pl);
                tc_wait_st();
                tc_fence_before();
                mbar_arrive(&p_full[t * 2 + b]);
            }
            // ---- O / L of this row
            const int jl = ntt - 1;
            const bool w4 = ok && mbar_wait(&o_done[t * 2 + (jl & 1)], (jl >> 1) & 1, p.errors);
            if (__all_sync(0xffffffffu, w4)) {
                tc_fence_after();
                const float2 la = __fadd2_rn(l4[0], l4[1]), lb = __fadd2_rn(l4[2], l4[3]);
                const float l = (la.x + lb.x) + (la.y + lb.y);
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const int qh = kvh * G + r % G;
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t ov[32];
                    tc_ld32(t_lane + c0, ov);
                    tc_wait_ld();
                    if (!real) continue;
                    const size_t e = ((size_t)(qs0 + tok) * p.n_heads + qh) * D + c0;
                    if (p.out_dtype == PKV_F32) {
                        float4* o4 = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + e);
#pragma unroll
                        for (int c = 0; c < 32; c += 4)
                            o4[c / 4] = make_float4(__uint_as_float(ov[c]) * inv,
                                                    __uint_as_float(ov[c + 1]) * inv,
                                                    __uint_as_float(ov[c + 2]) * inv,
                                                    __uint_as_float(ov[c + 3]) * inv);
                    } else {
                        uint4* o4 =
                            reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out) + e);
#pragma unroll
                        for (int c = 0; c < 32; c += 8)
                            o4[c / 8] = make_uint4(
                                pack_out(__uint_as_float(ov[c]) * inv,
                                         __uint_as_float(ov[c + 1]) * inv, p.out_dtype),
                                pack_out(__uint_as_float(ov[c + 2]) * inv,
                                         __uint_as_float(ov[c + 3]) * inv, p.out_dtype),
                                pack_out(__uint_as_float(ov[c + 4]) * inv,
                                         __uint_as_float(ov[c + 5]) * inv, p.out_dtype),
                                pack_out(__uint_as_float(ov[c + 6]) * inv,
                                         __uint_as_float(ov[c + 7]) * inv, p.out_dtype));
                    }
                }
            }
        }
    }

    // ---- tensor memory is released after every thread is done with it
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 8)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TMEM_COLS)
                     : "memory");
}

}  // namespace pkv
