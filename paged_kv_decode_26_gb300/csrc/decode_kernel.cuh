// decode_kernel.cuh -- paged single-query attention for sm_103a.
//
// Pages followed (cited by title and section):
//   [SWAP]   "vLLM 中 FlashAttention 与 KVCache 交换机制深度解析": the attention
//            formula softmax(Q K^T / sqrt(d_k)) V, Tiling (K/V loaded block by
//            block into on-chip SRAM), Kernel Fusion (scores, softmax and PV in
//            one kernel, nothing intermediate in HBM), and the OnlineSoftmax
//            recurrence M_new = max(M_old, max X_i),
//            L_new = L_old e^{M_old - M_new} + sum e^{X_i - M_new}, with O
//            rescaled by the same factor.
//   [LAYOUT] "大模型长文本推理基座从 FlashAttention 硬件加速机制到 vLLM 核心
//            PagedAttention 显存物理布局深度剖析", section 二.2: logical
//            blocks mapped to scattered physical blocks by a block table.
//
// Design (GB300): one CTA per (sequence, group of HPC kv heads, context
// split).  Warp 0 is the producer: one lane walks the split's block ids
// (prefetched into shared memory) and issues one 4-D TMA tile load per page
// for K and one for V, covering the HPC heads of the group
// ([B, HPC, D] boxes out of the [num_blocks, B, Hk, D] pool), into a ring of
// `stages` shared-memory buffers guarded by full/empty mbarriers.  The other
// warps are consumers.  A consumer owns QPW query heads of one kv head and
// every WPT-th page of the split (WPT warps share a head and merge their
// states in shared memory at the end).  Inside a warp, LPR = D/8 lanes cover
// one K/V row (8 dims, 16 bytes each) and the warp walks TPI = 32/LPR rows
// at a time; per chunk of 16 tokens each lane forms its partial dot
// products, a transpose-reduce across the LPR lanes of a row completes them
// (each halving step trades half of the values with the partner lane), the
// running max M and per-lane sum L are updated with exp2 (scores pre-scaled
// by log2 e), the weights are broadcast through shared memory and P V is
// accumulated with packed fp32x2 FMAs.  O is normalised once at the end
// (algebraically the same as the pages' per-step normalisation).  A context
// longer than one split leaves a normalised partial state (O, M, L) in the
// workspace; a second kernel merges them with the same recurrence.
#pragma once

#include "pkv_device.cuh"

namespace pkv {

constexpr int kChunk = 16;        // tokens per softmax update
constexpr int kMaxConsumerWarps = 8;
constexpr int kMaxThreads = 32 * (1 + kMaxConsumerWarps);

struct DecodeParams {
    void* out;
    int out_dtype;  // pkv_dtype
    const void* q;
    const int32_t* block_tables;
    int max_blocks_per_seq;
    const int32_t* context_lens;
    int num_seqs;
    int n_heads;
    int n_kv_heads;
    int group;  // n_heads / n_kv_heads
    int num_blocks;
    float scale_log2;  // scale * log2(e)
    int split_tokens;  // a multiple of the block size
    int max_splits;    // grid extent over splits
    int heads_per_cta;  // HPC
    int warps_per_kv;   // consumer warps sharing a kv head's pages by query heads
    int warps_per_tok;  // consumer warps sharing a kv head's query heads by pages
    int stages;
    int max_pages_per_split;
    float* ws_o;   // [num_seqs, n_heads, max_splits, D]
    float* ws_ml;  // [num_seqs, n_heads, max_splits, 2]
    int4* ws_desc; // stream decode: the runs its share boundaries cut [grid] (see there)
    unsigned int* errors;
    // Fused append (paged_attn_decode_append; NULL slot_mapping: none):
    // row k_new[s] / v_new[s] ([num_seqs, n_kv_heads, D]) goes to pool row
    // slot_mapping[s] before the decode reads the context.
    void* k_pool;
    void* v_pool;
    const void* k_new;
    const void* v_new;
    const int64_t* slot_mapping;
    // How a CTA finds its (split, head group, sequence): 0 = its grid
    // coordinates, 1 = the dense unit list (dense_unit), 2 = grid order
    // with the head group fastest (decode_unit).
    int dense;
};

// Fused append: the CTA of a sequence's last split writes the new token's K
// and V rows for its kv heads (hg * HPC ...) into pool row slot_mapping[s]
// (skipped for -1, flagged when outside the pool), then makes the stores
// visible to the TMA loads that follow the CTA barrier.  The last split is
// the only one whose pages hold the new token's position (splits are
// page-aligned), so no other CTA of the sequence reads that row.
//
// The slot and the rows depend on the sequence only, so every CTA loads them
// together with the context length (append_load: the slot and this thread's
// 16-byte vector of the rows -- 2 * HPC * D / 8 vectors, never more than the
// CTA's threads at D <= 128), and the last split's CTA stores them once it
// knows it is the last (append_store): no memory round trip of its own.
struct AppendRow {
    int64_t slot;   // -1: nothing to append
    uint4 v;        // this thread's vector of the new K then V rows
};

template <int D, int BS, typename T>
__device__ __forceinline__ AppendRow append_load(const DecodeParams& p, int s, int hg, int HPC) {
    AppendRow a;
    a.slot = -1;
    a.v = make_uint4(0u, 0u, 0u, 0u);
    if (p.slot_mapping == nullptr) return a;
    a.slot = p.slot_mapping[s];
    constexpr int VEC = 16 / (int)sizeof(T);           // elements per 16-byte vector
    const int per_row = HPC * D / VEC;                  // vectors of this CTA's heads
    const int i = (int)threadIdx.x;
    if (i < 2 * per_row) {
        const bool is_v = i >= per_row;
        const int j = (is_v ? i - per_row : i) * VEC;
        const T* src = static_cast<const T*>(is_v ? p.v_new : p.k_new) +
                       (size_t)s * p.n_kv_heads * D + (size_t)hg * HPC * D + j;
        a.v = *reinterpret_cast<const uint4*>(src);
    }
    return a;
}

template <int D, int BS, typename T>
__device__ __forceinline__ void append_store(const DecodeParams& p, const AppendRow& a, int s,
                                             int hg, int HPC, bool last_split) {
    if (p.slot_mapping == nullptr || !last_split || a.slot < 0) return;
    if (a.slot >= (int64_t)p.num_blocks * BS) {
        if (threadIdx.x == 0 && hg == 0) raise_error(p.errors, PKV_DEVERR_SLOT);
        return;
    }
    constexpr int VEC = 16 / (int)sizeof(T);
    const int per_row = HPC * D / VEC;
    const size_t row = (size_t)p.n_kv_heads * D;        // elements of one token row
    const size_t off_new = (size_t)s * row + (size_t)hg * HPC * D;
    const size_t off_pool = (size_t)a.slot * row + (size_t)hg * HPC * D;
    for (int i = threadIdx.x; i < 2 * per_row; i += blockDim.x) {
        const bool is_v = i >= per_row;
        const int j = (is_v ? i - per_row : i) * VEC;
        T* dst = static_cast<T*>(is_v ? p.v_pool : p.k_pool) + off_pool + j;
        // the vector loaded with the length; any beyond one a thread (not
        // the case for the launch shapes used) copied here
        const uint4 v = i == (int)threadIdx.x
                            ? a.v
                            : *reinterpret_cast<const uint4*>(
                                  static_cast<const T*>(is_v ? p.v_new : p.k_new) + off_new + j);
        *reinterpret_cast<uint4*>(dst) = v;
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Shared-memory bytes of one CTA (must match the carve-up in the kernel).
// The ring doubles as the buffer of the end-of-CTA merge between the WPT
// warps of a kv head.
inline size_t decode_smem_bytes(int D, int BS, int QPW, int elem_bytes, int hpc, int wpk,
                                int wpt, int stages, int max_pages_per_split) {
    size_t tile = (size_t)BS * hpc * D * elem_bytes;
    size_t ring = (size_t)stages * 2 * tile;
    size_t merge = (size_t)(wpt - 1) * hpc * wpk * QPW * (D + 2) * sizeof(float);
    size_t bytes = ring > merge ? ring : merge;
    bytes = (bytes + 15) / 16 * 16;
    bytes += (size_t)stages * 2 * sizeof(uint64_t);
    bytes += (size_t)hpc * wpk * wpt * QPW * kChunk * sizeof(float);
    bytes += (size_t)max_pages_per_split * sizeof(int);
    bytes += 2 * sizeof(int);  // abort flag, pages issued
    return bytes;
}

// ------------------------------------------------------------ warp helpers

// Transpose-reduce over the lanes that differ in bits O, O/2, ..., 1: every
// lane holds N partial sums v[0..N); each halving step keeps one half and
// adds the partner lane's copy of it, so the complete sums end up spread
// over the lanes (lane-index bits select which values a lane keeps) at a
// cost of one shuffle per value instead of one per value per step.  When
// the values run out before the lanes do, the remaining steps are plain
// butterflies and neighbouring lanes hold duplicates.
template <int N, int O>
__device__ __forceinline__ void transpose_reduce(float* v, int lane) {
    if constexpr (O >= 1) {
        if constexpr (N > 1) {
            constexpr int H = N / 2;
            const bool upper = (lane & O) != 0;
#pragma unroll
            for (int i = 0; i < H; ++i) {
                const float send = upper ? v[i] : v[i + H];
                const float keep = upper ? v[i + H] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
            }
            transpose_reduce<H, O / 2>(v, lane);
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
            transpose_reduce<1, O / 2>(v, lane);
        }
    }
}

// 8 consecutive 16-bit elements (16 bytes) -> 4 fp32 pairs (exact widening);
// with ok == false the row counts as zeros.
template <typename T>
__device__ __forceinline__ void load8(const T* p, float2 (&f)[4], bool ok = true) {
    uint4 w = *reinterpret_cast<const uint4*>(p);
    if (!ok) w = make_uint4(0u, 0u, 0u, 0u);
    f[0] = unpack2<T>(w.x);
    f[1] = unpack2<T>(w.y);
    f[2] = unpack2<T>(w.z);
    f[3] = unpack2<T>(w.w);
}

__device__ __forceinline__ uint32_t pack_out(float a, float b, int out_dtype) {
    if (out_dtype == PKV_BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Store 8 fp32 values as out_dtype at base + elem_off (16/32-byte aligned).
__device__ __forceinline__ void store8(void* base, size_t elem_off, int out_dtype,
                                       const float2 (&v)[4]) {
    if (out_dtype == PKV_F32) {
        float4* p = reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + elem_off);
        p[0] = make_float4(v[0].x, v[0].y, v[1].x, v[1].y);
        p[1] = make_float4(v[2].x, v[2].y, v[3].x, v[3].y);
    } else {
        uint4 w;
        w.x = pack_out(v[0].x, v[0].y, out_dtype);
        w.y = pack_out(v[1].x, v[1].y, out_dtype);
        w.z = pack_out(v[2].x, v[2].y, out_dtype);
        w.w = pack_out(v[3].x, v[3].y, out_dtype);
        *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(base) + elem_off) = w;
    }
}

// Named barrier over the consumer warps only (the producer does not join).
__device__ __forceinline__ void consumer_sync(int n_threads) {
    asm volatile("bar.sync 1, %0;" ::"r"(n_threads) : "memory");
}

// ------------------------------------------------------------ the kernel

// One CTA's work: (sequence s, kv-head group hg, context split `split`) of
// the problem described by p, its K/V pools seen through tm_k / tm_v (and
// tm_kh / tm_vh, boxes of half a block, for a last block whose tokens fit
// its first half).
template <int D, int BS, int QPW, typename T>
__device__ __forceinline__ void decode_cta(const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                           const CUtensorMap* tm_kh, const CUtensorMap* tm_vh,
                                           const DecodeParams& p, int split, int hg, int s) {
    constexpr int LPR = D / 8;                   // lanes per K/V row (8 dims each)
    constexpr int TPI = 32 / LPR;                // rows per warp iteration
    constexpr int IPC = kChunk / TPI;            // iterations per 16-token chunk
    constexpr int N = QPW * IPC;                 // partial dots per lane per chunk
    constexpr int NL = N >= LPR ? N / LPR : 1;   // complete dots per lane after reduce
    constexpr int DUP = N >= LPR ? 1 : LPR / N;  // lanes holding the same dot
    constexpr int GL = LPR / QPW;                // lanes of a row sharing a query head
    static_assert(BS % kChunk == 0, "block size must be a multiple of 16");
    static_assert(LPR % QPW == 0 && IPC % 4 == 0, "lane layout");

    extern __shared__ __align__(128) unsigned char smem[];

    const int HPC = p.heads_per_cta;
    const int per_sub = HPC * p.warps_per_kv;   // consumer warps per page
    const int n_cons = per_sub * p.warps_per_tok;
    // Each ring slot must belong to one warp subset (see the host-side
    // configuration); refuse an inconsistent launch before any barrier.
    if (p.stages % p.warps_per_tok != 0 || (int)blockDim.x != 32 * (1 + n_cons)) {
        if (threadIdx.x == 0) raise_error(p.errors, PKV_DEVERR_CONFIG);
        return;
    }

    // ---- this CTA's token range (clamped to what the grid and table cover)
    int n = p.context_lens[s];
    const AppendRow app = append_load<D, BS, T>(p, s, hg, HPC);   // same round trip
    const int cap = min(p.max_blocks_per_seq * BS, p.max_splits * p.split_tokens);
    if (n < 0 || n > cap) {
        if (split == 0 && hg == 0 && threadIdx.x == 0) raise_error(p.errors, PKV_DEVERR_CONTEXT);
        n = n < 0 ? 0 : cap;
    }
    const int n_splits = max(1, (n + p.split_tokens - 1) / p.split_tokens);
    if (split >= n_splits) return;
    const int tok_begin = split * p.split_tokens;
    const int tok_end = min(n, tok_begin + p.split_tokens);
    const int n_pages = (tok_end - tok_begin + BS - 1) / BS;  // 0 for an empty context
    const int page0 = tok_begin / BS;

    // ---- shared-memory carve-up
    const uint32_t tile_bytes = (uint32_t)(BS * HPC * D * sizeof(T));
    size_t ring = (size_t)p.stages * 2 * tile_bytes;
    const size_t merge =
        (size_t)(p.warps_per_tok - 1) * per_sub * QPW * (D + 2) * sizeof(float);
    ring = ((ring > merge ? ring : merge) + 15) / 16 * 16;
    unsigned char* tiles = smem;
    float* merge_buf = reinterpret_cast<float*>(smem);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + ring);
    uint64_t* empty = full + p.stages;
    float* ps_all = reinterpret_cast<float*>(empty + p.stages);
    int* s_bid = reinterpret_cast<int*>(ps_all + n_cons * QPW * kChunk);
    int* s_abort = s_bid + p.max_pages_per_split;
    int* s_issued = s_abort + 1;

    for (int i = threadIdx.x; i < n_pages; i += blockDim.x) {
        int b = p.block_tables[(size_t)s * p.max_blocks_per_seq + page0 + i];
        if (b < 0 || b >= p.num_blocks) {
            raise_error(p.errors, PKV_DEVERR_BLOCK_ID);
            b = -1;
        }
        s_bid[i] = b;
    }
    append_store<D, BS, T>(p, app, s, hg, HPC, split == n_splits - 1);
    if (threadIdx.x == 0) {
        for (int st = 0; st < p.stages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], per_sub);
        }
        *s_abort = 0;
        *s_issued = 0;
        fence_barrier_init();
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (warp == 0) {
        // ================= producer =================
        if (lane == 0) {
            prefetch_tensormap(tm_k);
            prefetch_tensormap(tm_v);
            prefetch_tensormap(tm_kh);
            prefetch_tensormap(tm_vh);
            const uint64_t policy = l2_policy_evict_first();
            int i = 0;
            for (; i < n_pages; ++i) {
                const int st = i % p.stages;
                if (i >= p.stages) {
                    if (!mbar_wait(&empty[st], ((i / p.stages) - 1) & 1, p.errors)) {
                        atomicExch(s_abort, 1);
                        break;
                    }
                }
                if (*reinterpret_cast<volatile int*>(s_abort)) break;
                const int b = s_bid[i];
                if (b >= 0) {
                    // a last block holding at most half a block of tokens:
                    // only its first half is loaded (the consumers mask the
                    // rows past the context, whatever the slot holds there)
                    const bool half = tok_end - (tok_begin + i * BS) <= BS / 2;
                    unsigned char* dst = tiles + (size_t)st * 2 * tile_bytes;
                    mbar_arrive_expect_tx(&full[st], half ? tile_bytes : 2 * tile_bytes);
                    tma_load_4d(dst, half ? tm_kh : tm_k, &full[st], 0, hg * HPC, 0, b, policy);
                    tma_load_4d(dst + tile_bytes, half ? tm_vh : tm_v, &full[st], 0, hg * HPC, 0,
                                b, policy);
                } else {
                    mbar_arrive(&full[st]);
                }
            }
            *s_issued = i;
        }
        __syncwarp();
    } else {
        // ================= consumers =================
        const int c = warp - 1;
        const int sub = c / per_sub;          // pages i with i % WPT == sub
        const int r = c % per_sub;            // role within one page
        const int kv_local = r / p.warps_per_kv;
        const int qh0 = (hg * HPC + kv_local) * p.group + (r % p.warps_per_kv) * QPW;
        float* ps = ps_all + c * QPW * kChunk;
        const int tq = lane / LPR;            // row of the iteration this lane reads
        const int dl = lane % LPR;            // dims [8 dl, 8 dl + 8)

        float2 q2[QPW][4];
#pragma unroll
        for (int g = 0; g < QPW; ++g) {
            const T* qrow = reinterpret_cast<const T*>(p.q) + ((size_t)s * p.n_heads + qh0 + g) * D;
            float2 f[4];
            load8<T>(qrow + dl * 8, f);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                q2[g][k] = make_float2(f[k].x * p.scale_log2, f[k].y * p.scale_log2);
        }

        float2 o2[QPW][4];
        float m[QPW];
#pragma unroll
        for (int g = 0; g < QPW; ++g) {
            m[g] = -INFINITY;
#pragma unroll
            for (int k = 0; k < 4; ++k) o2[g][k] = make_float2(0.f, 0.f);
        }
        float l_part = 0.f;

        const int idx0 = ((lane & (LPR - 1)) * N) / LPR;
        const int g_own = idx0 / IPC;
        const bool counts = (DUP == 1) || ((lane & (DUP - 1)) == 0);
        const int row_stride = HPC * D;

        for (int i = sub; i < n_pages; i += p.warps_per_tok) {
            const int st = i % p.stages;
            if (!mbar_wait(&full[st], (i / p.stages) & 1, p.errors)) {
                atomicExch(s_abort, 1);
                break;
            }
            if (s_bid[i] >= 0) {
                const T* sK = reinterpret_cast<const T*>(tiles + (size_t)st * 2 * tile_bytes);
                const T* sV = reinterpret_cast<const T*>(tiles + (size_t)st * 2 * tile_bytes +
                                                         tile_bytes);
                const int page_tok = tok_begin + i * BS;
#pragma unroll
                for (int ch = 0; ch < BS / kChunk; ++ch) {
                    const int tok0 = page_tok + ch * kChunk;
                    const int valid = min(kChunk, tok_end - tok0);
                    if (valid <= 0) break;
                    const size_t row0 = ((size_t)(ch * kChunk + tq) * HPC + kv_local) * D + dl * 8;
                    const T* kbase = sK + row0;
                    const T* vbase = sV + row0;

                    // -- partial scores: IPC rows x QPW heads, 8 dims each
                    float acc[N];
#pragma unroll
                    for (int it = 0; it < IPC; ++it) {
                        float2 k2[4];
                        load8<T>(kbase + it * TPI * row_stride, k2);
#pragma unroll
                        for (int g = 0; g < QPW; ++g) {
                            float2 a = __fmul2_rn(q2[g][0], k2[0]);
                            a = __ffma2_rn(q2[g][1], k2[1], a);
                            a = __ffma2_rn(q2[g][2], k2[2], a);
                            a = __ffma2_rn(q2[g][3], k2[3], a);
                            acc[g * IPC + it] = a.x + a.y;
                        }
                    }
                    transpose_reduce<N, LPR / 2>(acc, lane);

                    // -- mask, chunk max per query head
                    float cmax = -INFINITY;
#pragma unroll
                    for (int j = 0; j < NL; ++j) {
                        const int t = ((idx0 + j) % IPC) * TPI + tq;
                        if (t >= valid) acc[j] = -INFINITY;
                        cmax = fmaxf(cmax, acc[j]);
                    }
#pragma unroll
                    for (int off = 1; off < GL; off <<= 1)
                        cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, off));
#pragma unroll
                    for (int off = LPR; off < 32; off <<= 1)
                        cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, off));

                    float m_own = m[0];
#pragma unroll
                    for (int g = 1; g < QPW; ++g)
                        if (g == g_own) m_own = m[g];
                    const float mnew_own = fmaxf(m_own, cmax);

                    float alpha[QPW];
                    float alpha_own = 1.f;
#pragma unroll
                    for (int g = 0; g < QPW; ++g) {
                        const float mn = __shfl_sync(0xffffffffu, mnew_own, g * GL);
                        const float mu = (mn == -INFINITY) ? 0.f : mn;
                        alpha[g] = exp2f(m[g] - mu);
                        m[g] = mn;
                        if (g == g_own) alpha_own = alpha[g];
                    }
                    const float mu_own = (mnew_own == -INFINITY) ? 0.f : mnew_own;
                    float psum = 0.f;
#pragma unroll
                    for (int j = 0; j < NL; ++j) {
                        const float pj = exp2f(acc[j] - mu_own);
                        psum += pj;
                        ps[g_own * kChunk + tq * IPC + (idx0 + j) % IPC] = pj;
                    }
                    l_part = l_part * alpha_own + (counts ? psum : 0.f);
#pragma unroll
                    for (int g = 0; g < QPW; ++g) {
                        const float2 a2 = make_float2(alpha[g], alpha[g]);
#pragma unroll
                        for (int k = 0; k < 4; ++k) o2[g][k] = __fmul2_rn(o2[g][k], a2);
                    }
                    __syncwarp();

                    // -- O += P V over this lane's rows (rows past the context add 0)
                    float pw[QPW][IPC];
#pragma unroll
                    for (int g = 0; g < QPW; ++g)
#pragma unroll
                        for (int it = 0; it < IPC; it += 4) {
                            const float4 x = *reinterpret_cast<const float4*>(
                                ps + g * kChunk + tq * IPC + it);
                            pw[g][it] = x.x;
                            pw[g][it + 1] = x.y;
                            pw[g][it + 2] = x.z;
                            pw[g][it + 3] = x.w;
                        }
#pragma unroll
                    for (int it = 0; it < IPC; ++it) {
                        float2 v2[4];
                        load8<T>(vbase + it * TPI * row_stride, v2, it * TPI + tq < valid);
#pragma unroll
                        for (int g = 0; g < QPW; ++g) {
                            const float2 w2 = make_float2(pw[g][it], pw[g][it]);
#pragma unroll
                            for (int k = 0; k < 4; ++k) o2[g][k] = __ffma2_rn(w2, v2[k], o2[g][k]);
                        }
                    }
                    __syncwarp();
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
        }

        // ---- combine the rows of the warp: O over tq, L over the head's lanes
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1)
#pragma unroll
            for (int g = 0; g < QPW; ++g)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    o2[g][k].x += __shfl_xor_sync(0xffffffffu, o2[g][k].x, off);
                    o2[g][k].y += __shfl_xor_sync(0xffffffffu, o2[g][k].y, off);
                }
        float lsum = l_part;
#pragma unroll
        for (int off = 1; off < GL; off <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
        float lg[QPW];
#pragma unroll
        for (int g = 0; g < QPW; ++g) lg[g] = __shfl_sync(0xffffffffu, lsum, g * GL);

        // ---- merge the WPT warps that took turns on this kv head's pages
        if (p.warps_per_tok > 1) {
            consumer_sync(n_cons * 32);  // every warp is done with the ring
            if (sub > 0) {
                float* st = merge_buf + ((size_t)(sub - 1) * per_sub + r) * QPW * (D + 2);
#pragma unroll
                for (int g = 0; g < QPW; ++g) {
                    float* e = st + g * (D + 2);
                    if (tq == 0) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            e[2 + dl * 8 + 2 * k] = o2[g][k].x;
                            e[2 + dl * 8 + 2 * k + 1] = o2[g][k].y;
                        }
                    }
                    if (lane == 0) {
                        e[0] = m[g];
                        e[1] = lg[g];
                    }
                }
            }
            consumer_sync(n_cons * 32);
            if (sub == 0) {
                for (int w = 1; w < p.warps_per_tok; ++w) {
                    const float* st = merge_buf + ((size_t)(w - 1) * per_sub + r) * QPW * (D + 2);
#pragma unroll
                    for (int g = 0; g < QPW; ++g) {
                        const float* e = st + g * (D + 2);
                        const float mo = e[0];
                        const float mx = fmaxf(m[g], mo);
                        const float mu = (mx == -INFINITY) ? 0.f : mx;
                        const float a_self = exp2f(m[g] - mu);
                        const float a_other = exp2f(mo - mu);
                        lg[g] = lg[g] * a_self + e[1] * a_other;
                        m[g] = mx;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            o2[g][k].x = o2[g][k].x * a_self + e[2 + dl * 8 + 2 * k] * a_other;
                            o2[g][k].y = o2[g][k].y * a_self + e[2 + dl * 8 + 2 * k + 1] * a_other;
                        }
                    }
                }
            }
        }

        // ---- epilogue: normalise, write
        if (sub == 0 && tq == 0) {
#pragma unroll
            for (int g = 0; g < QPW; ++g) {
                const float inv = lg[g] > 0.f ? 1.f / lg[g] : 0.f;
                float2 v[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) v[k] = make_float2(o2[g][k].x * inv, o2[g][k].y * inv);
                const int qh = qh0 + g;
                if (n_splits == 1) {
                    store8(p.out, ((size_t)s * p.n_heads + qh) * D + dl * 8, p.out_dtype, v);
                } else {
                    const size_t unit = ((size_t)s * p.n_heads + qh) * p.max_splits + split;
                    store8(p.ws_o, unit * D + dl * 8, PKV_F32, v);
                    if (lane == 0)
                        *reinterpret_cast<float2*>(p.ws_ml + unit * 2) = make_float2(m[g], lg[g]);
                }
            }
        }
    }

    // ---- leave only when no TMA load is still writing this CTA's smem
    __syncthreads();
    if (*reinterpret_cast<volatile int*>(s_abort) && threadIdx.x == 0) {
        // Some wait gave up.  Wait (bounded) for every ring slot's most
        // recently issued load so that nothing lands after the CTA exits.
        const int issued = *reinterpret_cast<volatile int*>(s_issued);
        for (int st = 0; st < p.stages && st < issued; ++st) {
            const int last = st + ((issued - 1 - st) / p.stages) * p.stages;
            mbar_wait(&full[st], (last / p.stages) & 1, p.errors);
        }
    }
}

template <int DL>
__device__ __forceinline__ void store_row(void* base, size_t elem_off, int out_dtype,
                                          const float (&v)[DL]) {
    if (out_dtype == PKV_F32) {
        float* q = reinterpret_cast<float*>(base) + elem_off;
#pragma unroll
        for (int i = 0; i < DL; ++i) q[i] = v[i];
    } else {
        uint32_t* q = reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(base) + elem_off);
#pragma unroll
        for (int i = 0; i < DL; i += 2) q[i / 2] = pack_out(v[i], v[i + 1], out_dtype);
    }
}

// ------------------------------------------------------------ dense order

// The grid holds one CTA per (split, kv-head group, sequence) of the longest
// context, but a sequence of n tokens has only max(1, ceil(n / split_tokens))
// splits.  Taken in grid order, the CTAs of missing splits sit between the
// working ones; each holds an SM slot for the time it takes to read its
// context length, and the dispatcher waits for slots.  With p.dense == 1, CTA u
// (in grid order, the head group fastest) takes the u-th entry of a dense
// list instead: every sequence's full splits (sequence by sequence), then
// every sequence's shorter last split.  The CTAs without an entry all come at
// the end of the grid and the short units run in the tail.  Lengths are
// clamped as decode_cta clamps them.  Uses the first 136 bytes of dynamic
// shared memory before decode_cta does; returns false for a CTA without work.
template <int BS>
__device__ __forceinline__ bool dense_unit(const DecodeParams& p, int& split, int& hg, int& s) {
    extern __shared__ __align__(16) int dense_scratch[];
    int* s_full = dense_scratch;          // per-warp sums of full splits
    int* s_last = dense_scratch + 16;     // per-warp sums of short last splits
    int* s_pick = dense_scratch + 32;     // (sequence, split) of this CTA
    const int groups = (int)gridDim.y;
    const long long u =
        blockIdx.x + (long long)gridDim.x * (blockIdx.y + (long long)gridDim.y * blockIdx.z);
    hg = (int)(u % groups);
    const long long want = u / groups;
    const int S = p.num_seqs;
    const int nt = (int)blockDim.x;
    const int per = (S + nt - 1) / nt;
    const int lo = min(S, (int)threadIdx.x * per);
    const int hi = min(S, lo + per);
    const int st = p.split_tokens;
    const int cap = min(p.max_blocks_per_seq * BS, p.max_splits * st);
    int f = 0, r = 0;  // full splits and short last splits of this thread's sequences
    for (int i = lo; i < hi; ++i) {
        int n = p.context_lens[i];
        n = n < 0 ? 0 : (n > cap ? cap : n);
        f += n / st;
        r += (n == 0 || n % st != 0) ? 1 : 0;
    }
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int fi = f, ri = r;  // inclusive scans within the warp
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, fi, d);
        const int b = __shfl_up_sync(0xffffffffu, ri, d);
        if (lane >= d) {
            fi += a;
            ri += b;
        }
    }
    if (lane == 31) {
        s_full[w] = fi;
        s_last[w] = ri;
    }
    if (threadIdx.x == 0) s_pick[0] = -1;
    __syncthreads();
    int fo = fi - f, ro = ri - r, F = 0, R = 0;
    for (int k = 0; k < (nt >> 5); ++k) {
        const int a = s_full[k], b = s_last[k];
        if (k < w) {
            fo += a;
            ro += b;
        }
        F += a;
        R += b;
    }
    if (want < F) {
        if (want >= fo && want < fo + f) {
            int cum = fo;
            for (int i = lo; i < hi; ++i) {
                int n = p.context_lens[i];
                n = n < 0 ? 0 : (n > cap ? cap : n);
                if (want < cum + n / st) {
                    s_pick[0] = i;
                    s_pick[1] = (int)(want - cum);
                    break;
                }
                cum += n / st;
            }
        }
    } else if (want - F < R) {
        const int t = (int)(want - F);
        if (t >= ro && t < ro + r) {
            int cum = ro;
            for (int i = lo; i < hi; ++i) {
                int n = p.context_lens[i];
                n = n < 0 ? 0 : (n > cap ? cap : n);
                if (n == 0 || n % st != 0) {
                    if (t == cum) {
                        s_pick[0] = i;
                        s_pick[1] = n / st;
                        break;
                    }
                    ++cum;
                }
            }
        }
    }
    __syncthreads();
    // The scratch lies in the ring, which only TMA writes, and only after
    // the CTA barrier that follows the mbarrier setup: no barrier is needed
    // between these reads and the kernel body.
    s = s_pick[0];
    split = s_pick[1];
    return s >= 0;
}

// The CTA's (split, head group, sequence): dense list (p.dense == 1), grid
// order with the head group fastest (2), or the grid coordinates (0).
template <int BS>
__device__ __forceinline__ bool decode_unit(const DecodeParams& p, int& split, int& hg, int& s) {
    split = blockIdx.x;
    hg = blockIdx.y;
    s = blockIdx.z;
    if (p.dense == 1) return dense_unit<BS>(p, split, hg, s);
    if (p.dense == 2) {
        const long long u =
            blockIdx.x + (long long)gridDim.x * (blockIdx.y + (long long)gridDim.y * blockIdx.z);
        hg = (int)(u % gridDim.y);
        const long long rest = u / gridDim.y;
        split = (int)(rest % gridDim.x);
        s = (int)(rest / gridDim.x);
    }
    return true;
}

template <int D, int BS, int QPW, typename T>
__global__ void __launch_bounds__(kMaxThreads, 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_kh,
                        const __grid_constant__ CUtensorMap tm_vh,
                        const __grid_constant__ DecodeParams p) {
    launch_dependents();  // the split merge may start its CTAs (they wait)
    int split, hg, s;
    if (!decode_unit<BS>(p, split, hg, s)) return;
    decode_cta<D, BS, QPW, T>(&tm_k, &tm_v, &tm_kh, &tm_vh, p, split, hg, s);
}

// ------------------------------------------------------------ split merge

struct ReduceParams {
    void* out;
    int out_dtype;
    const int32_t* context_lens;
    int num_seqs;
    int n_heads;
    int split_tokens;
    int max_splits;
    int cap_tokens;  // same clamp as the decode kernel
    const float* ws_o;
    const float* ws_ml;
};

// One warp merges n partial states of one (sequence, query head): state k
// has its (M_k, L_k) at ml + k * ml_step floats and its normalised output
// row at o + k * o_step floats.  O = sum_k w_k O_k / sum_k w_k with
// w_k = L_k 2^{M_k - M*}, M* the largest M_k of a state with L_k > 0;
// written to out (element offset out_off, out_dtype).
template <int D>
__device__ __forceinline__ void merge_states(const float* ml, size_t ml_step, const float* o,
                                             size_t o_step, int n, void* out, size_t out_off,
                                             int out_dtype, int lane) {
    constexpr int DL = D / 32;
    float mx = -INFINITY;
    for (int k = lane; k < n; k += 32) {
        const float2 v = *reinterpret_cast<const float2*>(ml + (size_t)k * ml_step);
        if (v.y > 0.f) mx = fmaxf(mx, v.x);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));

    float acc[DL];
#pragma unroll
    for (int d = 0; d < DL; ++d) acc[d] = 0.f;
    float wsum = 0.f;
    // States in batches of RB: the batch's loads are all issued before its
    // accumulation, so a warp waits one memory round trip per batch rather
    // than per state; the accumulation order (k ascending) is unchanged.
    constexpr int RB = 8;
    for (int k0 = 0; k0 < n; k0 += RB) {
        float2 mlv[RB];
        float x[RB][DL];
#pragma unroll
        for (int u = 0; u < RB; ++u) {
            const int k = k0 + u;
            mlv[u] = make_float2(0.f, 0.f);
            if (k < n) {
                mlv[u] = *reinterpret_cast<const float2*>(ml + (size_t)k * ml_step);
                const float* ok = o + (size_t)k * o_step + lane * DL;
                if constexpr (DL == 4) {
                    const float4 t = *reinterpret_cast<const float4*>(ok);
                    x[u][0] = t.x;
                    x[u][1] = t.y;
                    x[u][2] = t.z;
                    x[u][3] = t.w;
                } else {
                    const float2 t = *reinterpret_cast<const float2*>(ok);
                    x[u][0] = t.x;
                    x[u][1] = t.y;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < RB; ++u) {
            if (k0 + u >= n || !(mlv[u].y > 0.f)) continue;
            const float w = mlv[u].y * exp2f(mlv[u].x - mx);
            wsum += w;
#pragma unroll
            for (int d = 0; d < DL; ++d) acc[d] = fmaf(w, x[u][d], acc[d]);
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    float v[DL];
#pragma unroll
    for (int d = 0; d < DL; ++d) v[d] = acc[d] * inv;
    store_row<DL>(out, out_off + lane * DL, out_dtype, v);
}

// One warp per (sequence, query head): merges the partial states of its
// splits ([unit][split] in the workspace).
template <int D>
__device__ __forceinline__ void reduce_unit(const ReduceParams& p, int unit, int lane) {
    if (unit >= p.num_seqs * p.n_heads) return;
    const int s = unit / p.n_heads;
    int n = p.context_lens[s];
    n = n < 0 ? 0 : min(n, p.cap_tokens);
    const int n_splits = max(1, (n + p.split_tokens - 1) / p.split_tokens);
    if (n_splits == 1) return;  // the decode kernel wrote this row itself
    merge_states<D>(p.ws_ml + (size_t)unit * p.max_splits * 2, 2,
                    p.ws_o + (size_t)unit * p.max_splits * D, D, n_splits, p.out,
                    (size_t)unit * D, p.out_dtype, lane);
}

template <int D>
__global__ void __launch_bounds__(128) paged_decode_reduce_kernel(const __grid_constant__ ReduceParams p) {
    dependency_wait();  // the decode kernel's partials (launched as its dependent)
    reduce_unit<D>(p, blockIdx.x * 4 + (threadIdx.x >> 5), threadIdx.x & 31);
}

}  // namespace pkv
