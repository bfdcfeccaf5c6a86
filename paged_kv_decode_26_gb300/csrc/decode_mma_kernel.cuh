// decode_mma_kernel.cuh -- paged single-query attention for grouped-query
// heads on the tensor cores (sm_103a), same inputs and outputs as
// paged_decode_kernel.
//
// Pages followed (cited by title and section):
//   [SWAP]   "vLLM 中 FlashAttention 与 KVCache 交换机制深度解析": the attention
//            formula, Tiling + Kernel Fusion + the OnlineSoftmax recurrence
//            (M_new, L_new, O rescaled), and MQA/GQA: several query heads
//            share one KV head by indexing, without copying K/V.
//   [LAYOUT] "大模型长文本推理基座从 FlashAttention 硬件加速机制到 vLLM 核心
//            PagedAttention 显存物理布局深度剖析", section 二.2: block table.
//
// With G query heads per kv head, one page of one kv head is a small dense
// contraction.  One warp per kv head computes it with mma.sync m16n8k16
// (bf16/fp16 in, fp32 accumulate) with the tokens as the 16 rows and the
// query heads as the 8 columns: S^T = K Q^T (A = 16 tokens x 16 dims of K,
// B = Q^T, column n = query head n) and O^T += V^T P^T (A = 16 dims x 16
// tokens of V, B = P^T).  A group of 4 then fills half of each product's
// columns, a group of 8 all of them -- against a quarter / half with the
// query heads as rows -- so a 16-token chunk costs head_dim/16 score
// products and head_dim/16 x 2 value products.  The score accumulators hold
// P^T by token rows; a lane needs it by head columns for the B operand of
// the value product, which eight warp shuffles per chunk provide.  P enters
// that product as two 16-bit parts (hi + lo) so that its rounding stays at
// fp32 level.
//
// Staging: per page and kv head, K and V arrive as head_dim/64 TMA boxes of
// [B tokens x 64 elements] with 128-byte swizzle: token t's 16-byte chunk c
// sits at chunk c ^ (t % 8) of its 128-byte row, so the 8 rows an ldmatrix
// reads fall in 8 different bank groups.  Producer, ring, bounded waits,
// splits and partial states work as in paged_decode_kernel.
#pragma once

#include "decode_kernel.cuh"

namespace pkv {

constexpr int kMmaMaxWarps = 8;
constexpr int kMmaMaxThreads = 32 * (1 + kMmaMaxWarps);

// Shared-memory bytes of one CTA of the tensor-core kernel: 1 KB alignment
// slack + ring + barriers + block ids + flags.
inline size_t decode_mma_smem_bytes(int D, int BS, int elem_bytes, int hpc, int stages,
                                    int max_pages_per_split) {
    size_t ring = (size_t)stages * 2 * hpc * D * BS * elem_bytes;
    return 1024 + ring + (size_t)stages * 2 * sizeof(uint64_t) +
           (size_t)max_pages_per_split * sizeof(int) + 2 * sizeof(int);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D = A(16x16) * B(16x8) + D, fp32 accumulate.
template <typename T>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1);

template <>
__device__ __forceinline__ void mma16816<__nv_bfloat16>(float (&d)[4], const uint32_t (&a)[4],
                                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <>
__device__ __forceinline__ void mma16816<__half>(float (&d)[4], const uint32_t (&a)[4],
                                                 uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two fp32 -> one packed pair of T (low half = first).
template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Byte offset of (token row t, 16-byte chunk c) inside one swizzled
// [rows x 128 B] box whose base is 1024-byte aligned.
__device__ __forceinline__ uint32_t swz(int t, int c) {
    return (uint32_t)(t * 128 + ((c ^ (t & 7)) << 4));
}

// Running state of one kv head's G query heads in one warp (lane = 4 gid +
// tig): Q^T as B fragments, O^T accumulators (m-tile j: dims 16j..16j+15,
// columns = query heads; this lane holds dims 16j + gid and 16j + gid + 8 of
// heads 2 tig and 2 tig + 1), and the running maximum (log2 domain) and this
// lane's share of the sum of heads 2 tig and 2 tig + 1.
template <int D>
struct MmaHeads {
    uint32_t qb[D / 16][2];
    float o[D / 16][4];
    float m[2];
    float l[2];
};

// Query rows qrow0 + h * D (h < G; the rest zero) as the B operand.
template <int D, typename T>
__device__ __forceinline__ void mma_heads_start(MmaHeads<D>& st, const T* qrow0, int G, int lane) {
    const int gid = lane >> 2, tig = lane & 3;
    const bool real = gid < G;
    const T* qrow = qrow0 + (size_t)(real ? gid : 0) * D;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t lo = *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + tig * 2);
        const uint32_t hi = *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + tig * 2);
        st.qb[ks][0] = real ? lo : 0u;
        st.qb[ks][1] = real ? hi : 0u;
    }
#pragma unroll
    for (int j = 0; j < D / 16; ++j) st.o[j][0] = st.o[j][1] = st.o[j][2] = st.o[j][3] = 0.f;
    st.m[0] = st.m[1] = -INFINITY;
    st.l[0] = st.l[1] = 0.f;
}

// One 16-token chunk (`valid` of its tokens inside the context, 1..16) of
// one kv head's K and V, swizzled [rows x 128 B] boxes at kbase / vbase,
// token rows t0 .. t0 + 15 of the boxes.
template <int D, typename T>
__device__ __forceinline__ void mma_heads_chunk(MmaHeads<D>& st, uint32_t kbase, uint32_t vbase,
                                                uint32_t box_bytes, int t0, int valid,
                                                float scale_log2, int lane) {
    constexpr int KSTEPS = D / 16;
    const int gid = lane >> 2, tig = lane & 3;
    const int mat = lane >> 3, mrow = lane & 7;
    // ldmatrix matrices: K (tokens 0-7, c), (0-7, c+1), (8-15, c), (8-15, c+1);
    // V transposed: (tokens 0-7, c), (8-15, c), (0-7, c+1), (8-15, c+1)
    const int k_tok = t0 + (mat >> 1) * 8 + mrow, k_dc = mat & 1;
    const int v_tok = t0 + (mat & 1) * 8 + mrow, v_dc = mat >> 1;

    // ---- S^T = K Q^T: rows = tokens, columns = query heads
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
        const int h = ks / 4;
        const int c = (ks % 4) * 2 + k_dc;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + h * box_bytes + swz(k_tok, c), b0, b1, b2, b3);
        const uint32_t a[4] = {b0, b2, b1, b3};
        mma16816<T>(s, a, st.qb[ks][0], st.qb[ks][1]);
    }
    // this lane: tokens gid (s0, s1) and gid + 8 (s2, s3) of heads 2 tig, 2 tig + 1
    const bool v0 = gid < valid, v1 = gid + 8 < valid;
    const float x0 = v0 ? s[0] * scale_log2 : -INFINITY;
    const float x1 = v0 ? s[1] * scale_log2 : -INFINITY;
    const float x2 = v1 ? s[2] * scale_log2 : -INFINITY;
    const float x3 = v1 ? s[3] * scale_log2 : -INFINITY;
    float c0 = fmaxf(x0, x2), c1 = fmaxf(x1, x3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        c0 = fmaxf(c0, __shfl_xor_sync(0xffffffffu, c0, off));
        c1 = fmaxf(c1, __shfl_xor_sync(0xffffffffu, c1, off));
    }
    const float mn0 = fmaxf(st.m[0], c0), mn1 = fmaxf(st.m[1], c1);
    const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = exp2f(st.m[0] - mu0), al1 = exp2f(st.m[1] - mu1);
    st.m[0] = mn0;
    st.m[1] = mn1;
    const float p0 = exp2f(x0 - mu0), p1 = exp2f(x1 - mu1);
    const float p2 = exp2f(x2 - mu0), p3 = exp2f(x3 - mu1);
    st.l[0] = st.l[0] * al0 + (p0 + p2);
    st.l[1] = st.l[1] * al1 + (p1 + p3);
    // P in two 16-bit parts (hi = round(p), lo = round(p - hi)), packed by
    // token: (head 2 tig, head 2 tig + 1) of token gid and of token gid + 8
    const uint32_t hA = pack2<T>(p0, p1), hB = pack2<T>(p2, p3);
    const float2 fA = unpack2<T>(hA), fB = unpack2<T>(hB);
    const uint32_t lA = pack2<T>(p0 - fA.x, p1 - fA.y), lB = pack2<T>(p2 - fB.x, p3 - fB.y);
    // ---- P^T as the B operand: this lane (column = head gid) needs tokens
    // 2 tig, 2 tig + 1 (k 0-7) and 2 tig + 8, 2 tig + 9 (k 8-15), which lanes
    // 4 (2 tig) + gid / 2 and 4 (2 tig + 1) + gid / 2 hold (half gid % 2)
    const int srcA = 4 * (2 * tig) + (gid >> 1), srcB = srcA + 4;
    const uint32_t sel = (gid & 1) ? 0x7632u : 0x5410u;   // the half of this lane's head
    const uint32_t hAa = __shfl_sync(0xffffffffu, hA, srcA), hAb = __shfl_sync(0xffffffffu, hA, srcB);
    const uint32_t hBa = __shfl_sync(0xffffffffu, hB, srcA), hBb = __shfl_sync(0xffffffffu, hB, srcB);
    const uint32_t lAa = __shfl_sync(0xffffffffu, lA, srcA), lAb = __shfl_sync(0xffffffffu, lA, srcB);
    const uint32_t lBa = __shfl_sync(0xffffffffu, lB, srcA), lBb = __shfl_sync(0xffffffffu, lB, srcB);
    // (keys 2 tig, 2 tig + 1) -> low / high half of one register
    const uint32_t bh0 = __byte_perm(hAa, hAb, sel);
    const uint32_t bh1 = __byte_perm(hBa, hBb, sel);
    const uint32_t bl0 = __byte_perm(lAa, lAb, sel);
    const uint32_t bl1 = __byte_perm(lBa, lBb, sel);
    // ---- O^T = O^T * alpha + V^T P^T; V rows past the context may hold
    // anything (NaN included): P is 0 there, but 0 * NaN is not, so those
    // rows are cleared in the A fragments (tokens 2 tig, 2 tig + 1 in a0/a1,
    // 2 tig + 8, 2 tig + 9 in a2/a3)
    uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
    if (valid < 16) {
        vm0 = (tig * 2 < valid ? 0x0000ffffu : 0u) | (tig * 2 + 1 < valid ? 0xffff0000u : 0u);
        vm1 = (8 + tig * 2 < valid ? 0x0000ffffu : 0u) | (8 + tig * 2 + 1 < valid ? 0xffff0000u : 0u);
    }
#pragma unroll
    for (int j = 0; j < D / 16; ++j) {
        st.o[j][0] *= al0;
        st.o[j][1] *= al1;
        st.o[j][2] *= al0;
        st.o[j][3] *= al1;
        const int h = j / 4;
        const int c = (j % 4) * 2 + v_dc;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_trans(vbase + h * box_bytes + swz(v_tok, c), b0, b1, b2, b3);
        const uint32_t a[4] = {b0 & vm0, b2 & vm0, b1 & vm1, b3 & vm1};
        mma16816<T>(st.o[j], a, bh0, bh1);
        mma16816<T>(st.o[j], a, bl0, bl1);
    }
}

// Sum of each query head's softmax weights over the warp: lane (gid, tig)
// holds heads 2 tig and 2 tig + 1 for its token rows; the other token rows
// sit in the lanes of the same tig.
template <int D>
__device__ __forceinline__ void mma_heads_sums(const MmaHeads<D>& st, float& l0, float& l1) {
    l0 = st.l[0];
    l1 = st.l[1];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
}

// A partial state (normalised O, M, L) per real query head hh < G: row
// row0 + hh * row_step of ws_o ([rows, D]) and ws_ml ([rows, 2]).
template <int D>
__device__ __forceinline__ void mma_heads_partial(const MmaHeads<D>& st, float* ws_o,
                                                  float* ws_ml, size_t row0, size_t row_step,
                                                  int G, int lane) {
    const int gid = lane >> 2, tig = lane & 3;
    float l0, l1;
    mma_heads_sums<D>(st, l0, l1);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int hh = 2 * tig + e;
        if (hh >= G) continue;
        const float l = e ? l1 : l0;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const size_t unit = row0 + (size_t)hh * row_step;
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
            ws_o[unit * D + j * 16 + gid] = st.o[j][e] * inv;
            ws_o[unit * D + j * 16 + gid + 8] = st.o[j][2 + e] * inv;
        }
        if (gid == 0) *reinterpret_cast<float2*>(ws_ml + unit * 2) = make_float2(st.m[e], l);
    }
}

// The unit's result: normalised rows of the real query heads qh0 .. qh0+G-1
// to the output (one split) or to the split partials.
template <int D>
__device__ __forceinline__ void mma_heads_finish(const MmaHeads<D>& st, const DecodeParams& p,
                                                 int s, int qh0, int G, int n_splits, int split,
                                                 int lane) {
    if (n_splits != 1) {
        mma_heads_partial<D>(st, p.ws_o, p.ws_ml,
                             ((size_t)s * p.n_heads + qh0) * p.max_splits + split, p.max_splits,
                             G, lane);
        return;
    }
    const int gid = lane >> 2, tig = lane & 3;
    float l0, l1;
    mma_heads_sums<D>(st, l0, l1);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int hh = 2 * tig + e;
        if (hh >= G) continue;
        const float l = e ? l1 : l0;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const size_t row = ((size_t)s * p.n_heads + qh0 + hh) * D;
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
            const float a = st.o[j][e] * inv, b = st.o[j][2 + e] * inv;
            const size_t d0 = row + j * 16 + gid, d1 = d0 + 8;
            if (p.out_dtype == PKV_F32) {
                reinterpret_cast<float*>(p.out)[d0] = a;
                reinterpret_cast<float*>(p.out)[d1] = b;
            } else {
                const uint32_t w = pack_out(a, b, p.out_dtype);
                reinterpret_cast<uint16_t*>(p.out)[d0] = (uint16_t)(w & 0xffffu);
                reinterpret_cast<uint16_t*>(p.out)[d1] = (uint16_t)(w >> 16);
            }
        }
    }
}

// One CTA's work (sequence s, kv-head group hg, split) of the problem p
// (tm_kh / tm_vh: boxes of half a block, for a last block whose tokens fit
// its first half).
template <int D, int BS, typename T>
__device__ __forceinline__ void decode_mma_cta(const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                               const CUtensorMap* tm_kh, const CUtensorMap* tm_vh,
                                               const DecodeParams& p, int split, int hg, int s) {
    constexpr int HALVES = D / 64;        // 128-byte boxes per token row
    constexpr uint32_t BOX = BS * 128;    // bytes of one [BS x 64] box
    static_assert(BS % 16 == 0 && D % 64 == 0, "shape");

    extern __shared__ __align__(1024) unsigned char smem_raw[];

    const int HPC = p.heads_per_cta;
    const int G = p.group;
    if ((int)blockDim.x != 32 * (1 + HPC) || G > 8 || p.warps_per_tok != 1) {
        if (threadIdx.x == 0) raise_error(p.errors, PKV_DEVERR_CONFIG);
        return;
    }

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
    const int n_pages = (tok_end - tok_begin + BS - 1) / BS;
    const int page0 = tok_begin / BS;

    // ---- shared memory: ring (1024-byte aligned), barriers, block ids
    const uint32_t raw_addr = smem_addr(smem_raw);
    unsigned char* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const uint32_t head_bytes = HALVES * BOX;              // one kv head's K (or V) page
    const uint32_t stage_bytes = 2 * HPC * head_bytes;     // K then V for HPC heads
    unsigned char* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)p.stages * stage_bytes);
    uint64_t* empty = full + p.stages;
    int* s_bid = reinterpret_cast<int*>(empty + p.stages);
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
            mbar_init(&empty[st], HPC);
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
                    // rows past the context)
                    const bool half = tok_end - (tok_begin + i * BS) <= BS / 2;
                    const CUtensorMap* mk = half ? tm_kh : tm_k;
                    const CUtensorMap* mv = half ? tm_vh : tm_v;
                    unsigned char* dst = ring + (size_t)st * stage_bytes;
                    mbar_arrive_expect_tx(&full[st], half ? stage_bytes / 2 : stage_bytes);
                    for (int hh = 0; hh < HPC; ++hh) {
                        const int row = (hg * HPC + hh) * HALVES;
                        for (int h = 0; h < HALVES; ++h) {
                            tma_load_4d(dst + hh * head_bytes + h * BOX, mk, &full[st], 0,
                                        row + h, 0, b, policy);
                            tma_load_4d(dst + (HPC + hh) * head_bytes + h * BOX, mv,
                                        &full[st], 0, row + h, 0, b, policy);
                        }
                    }
                } else {
                    mbar_arrive(&full[st]);
                }
            }
            *s_issued = i;
        }
        __syncwarp();
    } else {
        // ================= consumers: one warp per kv head =================
        const int kv_local = warp - 1;
        const int qh0 = (hg * HPC + kv_local) * G;
        MmaHeads<D> st;
        mma_heads_start<D, T>(st, reinterpret_cast<const T*>(p.q) + ((size_t)s * p.n_heads + qh0) * D,
                              G, lane);
        for (int i = 0; i < n_pages; ++i) {
            const int slot = i % p.stages;
            if (!mbar_wait(&full[slot], (i / p.stages) & 1, p.errors)) {
                atomicExch(s_abort, 1);
                break;
            }
            if (s_bid[i] >= 0) {
                const uint32_t kbase = smem_addr(ring + (size_t)slot * stage_bytes +
                                                 kv_local * head_bytes);
                const uint32_t vbase = smem_addr(ring + (size_t)slot * stage_bytes +
                                                 (HPC + kv_local) * head_bytes);
                const int page_tok = tok_begin + i * BS;
#pragma unroll
                for (int ch = 0; ch < BS / 16; ++ch) {
                    const int valid = min(16, tok_end - (page_tok + ch * 16));
                    if (valid <= 0) break;
                    mma_heads_chunk<D, T>(st, kbase, vbase, BOX, ch * 16, valid, p.scale_log2,
                                          lane);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
        mma_heads_finish<D>(st, p, s, qh0, G, n_splits, split, lane);
    }

    __syncthreads();
    if (*reinterpret_cast<volatile int*>(s_abort) && threadIdx.x == 0) {
        const int issued = *reinterpret_cast<volatile int*>(s_issued);
        for (int st = 0; st < p.stages && st < issued; ++st) {
            const int last = st + ((issued - 1 - st) / p.stages) * p.stages;
            mbar_wait(&full[st], (last / p.stages) & 1, p.errors);
        }
    }
}

template <int D, int BS, typename T>
__global__ void __launch_bounds__(kMmaMaxThreads, 1)
    paged_decode_mma_kernel(const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v,
                            const __grid_constant__ CUtensorMap tm_kh,
                            const __grid_constant__ CUtensorMap tm_vh,
                            const __grid_constant__ DecodeParams p) {
    launch_dependents();  // the split merge may start its CTAs (they wait)
    int split, hg, s;
    if (!decode_unit<BS>(p, split, hg, s)) return;
    decode_mma_cta<D, BS, T>(&tm_k, &tm_v, &tm_kh, &tm_vh, p, split, hg, s);
}

}  // namespace pkv
