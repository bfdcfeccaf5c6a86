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
// contraction: S = Q K^T is [G x 16 tokens x head_dim] and O += P V is
// [G x head_dim x 16 tokens].  One warp per kv head computes both with
// mma.sync m16n8k16 (bf16/fp16 in, fp32 accumulate), the G query heads
// being rows 0..G-1 of the 16-row tile.  The scores' accumulator layout is
// the A-operand layout of P, so P never leaves registers; P enters the P V
// product as two 16-bit parts (hi + lo) so that its rounding stays at fp32
// level.
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

// One CTA's work (sequence s, kv-head group hg, split) of the problem p.
template <int D, int BS, typename T>
__device__ __forceinline__ void decode_mma_cta(const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                               const DecodeParams& p, int split, int hg, int s) {
    constexpr int HALVES = D / 64;        // 128-byte boxes per token row
    constexpr int KSTEPS = D / 16;        // k-steps of the score MMA
    constexpr int NT = D / 8;             // n-tiles of the P V MMA
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
    fused_append<D, BS, T>(p, s, hg, HPC, split == n_splits - 1);
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
                    unsigned char* dst = ring + (size_t)st * stage_bytes;
                    mbar_arrive_expect_tx(&full[st], stage_bytes);
                    for (int hh = 0; hh < HPC; ++hh) {
                        const int row = (hg * HPC + hh) * HALVES;
                        for (int h = 0; h < HALVES; ++h) {
                            tma_load_4d(dst + hh * head_bytes + h * BOX, tm_k, &full[st], 0,
                                        row + h, 0, b, policy);
                            tma_load_4d(dst + (HPC + hh) * head_bytes + h * BOX, tm_v,
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
        const int gid = lane >> 2;     // fragment row (query head) of this lane
        const int tig = lane & 3;      // pair of columns of this lane
        const bool row_real = gid < G;

        // Q as the A operand: rows = query heads (rows >= G and 8..15 zero)
        uint32_t qa[KSTEPS][4];
        {
            const T* qrow = reinterpret_cast<const T*>(p.q) +
                            ((size_t)s * p.n_heads + qh0 + (row_real ? gid : 0)) * D;
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
                const uint32_t lo = *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + tig * 2);
                const uint32_t hi = *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + tig * 2);
                qa[ks][0] = row_real ? lo : 0u;
                qa[ks][1] = 0u;
                qa[ks][2] = row_real ? hi : 0u;
                qa[ks][3] = 0u;
            }
        }

        float o[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
        float m_row = -INFINITY;   // running max of this lane's row
        float l_part = 0.f;        // this lane's share of the row's sum

        // ldmatrix row addresses (lane-dependent parts)
        const int mat = lane >> 3;          // which 8x8 matrix this lane addresses
        const int mrow = lane & 7;          // row inside it
        // scores: matrices (tokens 0-7, c), (tokens 0-7, c+1), (8-15, c), (8-15, c+1)
        const int k_tok = (mat >> 1) * 8 + mrow;
        const int k_dc = mat & 1;
        // P V: matrices (tokens 0-7, n), (8-15, n), (0-7, n+1), (8-15, n+1)
        const int v_tok = (mat & 1) * 8 + mrow;
        const int v_dc = mat >> 1;

        for (int i = 0; i < n_pages; ++i) {
            const int st = i % p.stages;
            if (!mbar_wait(&full[st], (i / p.stages) & 1, p.errors)) {
                atomicExch(s_abort, 1);
                break;
            }
            if (s_bid[i] >= 0) {
                const uint32_t kbase = smem_addr(ring + (size_t)st * stage_bytes +
                                                 kv_local * head_bytes);
                const uint32_t vbase = smem_addr(ring + (size_t)st * stage_bytes +
                                                 (HPC + kv_local) * head_bytes);
                const int page_tok = tok_begin + i * BS;
#pragma unroll
                for (int ch = 0; ch < BS / 16; ++ch) {
                    const int valid = min(16, tok_end - (page_tok + ch * 16));
                    if (valid <= 0) break;
                    // ---- S = Q K^T for 16 tokens (two n-tiles of 8)
                    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                    for (int ks = 0; ks < KSTEPS; ++ks) {
                        const int h = ks / 4;                  // which 64-wide half
                        const int c = (ks % 4) * 2 + k_dc;     // 16-byte chunk in the row
                        const int t = ch * 16 + k_tok;
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(kbase + h * BOX + swz(t, c), b0, b1, b2, b3);
                        mma16816<T>(sc[0], qa[ks], b0, b1);
                        mma16816<T>(sc[1], qa[ks], b2, b3);
                    }
                    // ---- online softmax on this lane's row (4 of its 16 scores)
                    float x[4];
                    x[0] = sc[0][0] * p.scale_log2;
                    x[1] = sc[0][1] * p.scale_log2;
                    x[2] = sc[1][0] * p.scale_log2;
                    x[3] = sc[1][1] * p.scale_log2;
                    if (tig * 2 >= valid) x[0] = -INFINITY;
                    if (tig * 2 + 1 >= valid) x[1] = -INFINITY;
                    if (8 + tig * 2 >= valid) x[2] = -INFINITY;
                    if (8 + tig * 2 + 1 >= valid) x[3] = -INFINITY;
                    float cmax = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
                    cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 1));
                    cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 2));
                    const float m_new = fmaxf(m_row, cmax);
                    const float mu = (m_new == -INFINITY) ? 0.f : m_new;
                    const float alpha = exp2f(m_row - mu);
                    m_row = m_new;
                    const float p0 = exp2f(x[0] - mu), p1 = exp2f(x[1] - mu);
                    const float p2 = exp2f(x[2] - mu), p3 = exp2f(x[3] - mu);
                    l_part = l_part * alpha + ((p0 + p1) + (p2 + p3));
                    // V rows past the context may hold anything (NaN included):
                    // P is 0 there, but 0 * NaN is not, so those rows are
                    // cleared in the B fragments of the last chunk.  Lane
                    // fragments hold tokens 2*tig, 2*tig+1 (low / high half)
                    // and 8 more in the second register.
                    uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
                    if (valid < 16) {
                        vm0 = (tig * 2 < valid ? 0x0000ffffu : 0u) |
                              (tig * 2 + 1 < valid ? 0xffff0000u : 0u);
                        vm1 = (8 + tig * 2 < valid ? 0x0000ffffu : 0u) |
                              (8 + tig * 2 + 1 < valid ? 0xffff0000u : 0u);
                    }
                    // P in two parts of the input type (hi = round(p), lo =
                    // round(p - hi)): one 16-bit rounding of the weights would
                    // cost ~2^-9 relative in O; hi + lo leaves ~2^-17.
                    uint32_t pa[4], pl[4];
                    pa[0] = pack2<T>(p0, p1);
                    pa[2] = pack2<T>(p2, p3);
                    {
                        const float2 h01 = unpack2<T>(pa[0]), h23 = unpack2<T>(pa[2]);
                        pl[0] = pack2<T>(p0 - h01.x, p1 - h01.y);
                        pl[2] = pack2<T>(p2 - h23.x, p3 - h23.y);
                    }
                    pa[1] = pa[3] = pl[1] = pl[3] = 0u;
                    // ---- O = O * alpha + P V (n-tiles of 8 dims, two per ldmatrix)
#pragma unroll
                    for (int j = 0; j < NT; j += 2) {
                        o[j][0] *= alpha;
                        o[j][1] *= alpha;
                        o[j + 1][0] *= alpha;
                        o[j + 1][1] *= alpha;
                        const int h = j / 8;
                        const int c = (j % 8) + v_dc;
                        const int t = ch * 16 + v_tok;
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_trans(vbase + h * BOX + swz(t, c), b0, b1, b2, b3);
                        b0 &= vm0;
                        b1 &= vm1;
                        b2 &= vm0;
                        b3 &= vm1;
                        mma16816<T>(o[j], pa, b0, b1);
                        mma16816<T>(o[j + 1], pa, b2, b3);
                        mma16816<T>(o[j], pl, b0, b1);
                        mma16816<T>(o[j + 1], pl, b2, b3);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
        }

        // ---- L of each row: the 4 lanes of a row hold its parts
        float l_row = l_part;
        l_row += __shfl_xor_sync(0xffffffffu, l_row, 1);
        l_row += __shfl_xor_sync(0xffffffffu, l_row, 2);
        if (row_real) {
            const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
            const int qh = qh0 + gid;
            if (n_splits == 1) {
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const size_t e = ((size_t)s * p.n_heads + qh) * D + j * 8 + tig * 2;
                    if (p.out_dtype == PKV_F32) {
                        *reinterpret_cast<float2*>(reinterpret_cast<float*>(p.out) + e) =
                            make_float2(o[j][0] * inv, o[j][1] * inv);
                    } else {
                        *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(p.out) + e) =
                            pack_out(o[j][0] * inv, o[j][1] * inv, p.out_dtype);
                    }
                }
            } else {
                const size_t unit = ((size_t)s * p.n_heads + qh) * p.max_splits + split;
#pragma unroll
                for (int j = 0; j < NT; ++j)
                    *reinterpret_cast<float2*>(p.ws_o + unit * D + j * 8 + tig * 2) =
                        make_float2(o[j][0] * inv, o[j][1] * inv);
                if (tig == 0)
                    *reinterpret_cast<float2*>(p.ws_ml + unit * 2) = make_float2(m_row, l_row);
            }
        }
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
                            const __grid_constant__ DecodeParams p) {
    launch_dependents();  // the split merge may start its CTAs (they wait)
    int split, hg, s;
    if (!decode_unit<BS>(p, split, hg, s)) return;
    decode_mma_cta<D, BS, T>(&tm_k, &tm_v, p, split, hg, s);
}

}  // namespace pkv
