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
// `stages` shared-memory buffers guarded by full/empty mbarriers.  Every
// other warp is a consumer owning QPW query heads of one kv head: lane l
// holds head dims [l*D/32, (l+1)*D/32) of q and of the fp32 accumulator O,
// computes 16 partial dot products per chunk of 16 tokens, reduces them
// across the warp with a transpose-reduce (one shuffle per score), updates
// the running max M and per-lane sum L with exp2 (scores pre-scaled by
// log2 e), broadcasts the 16 weights through shared memory and accumulates
// P V.  O is normalised once at the end (algebraically the same as the
// pages' per-step normalisation).  A context longer than one split leaves a
// normalised partial state (O, M, L) in the workspace; a second kernel
// merges them with the same recurrence.
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
    int warps_per_kv;   // consumer warps per kv head
    int stages;
    int max_pages_per_split;
    float* ws_o;   // [num_seqs, n_heads, max_splits, D]
    float* ws_ml;  // [num_seqs, n_heads, max_splits, 2]
    unsigned int* errors;
};

// Shared-memory bytes of one CTA (must match the carve-up in the kernel).
inline size_t decode_smem_bytes(int D, int BS, int QPW, int elem_bytes, int hpc, int wpk,
                                int stages, int max_pages_per_split) {
    size_t tile = (size_t)BS * hpc * D * elem_bytes;
    size_t bytes = (size_t)stages * 2 * tile;
    bytes += (size_t)stages * 2 * sizeof(uint64_t);
    bytes += (size_t)hpc * wpk * QPW * kChunk * sizeof(float);
    bytes += (size_t)max_pages_per_split * sizeof(int);
    bytes += 2 * sizeof(int);  // abort flag, pages issued
    return bytes;
}

// ------------------------------------------------------------ warp helpers

// Transpose-reduce: every lane holds N partial sums v[0..N); afterwards lane
// l holds the complete (32-lane) sums of indices [idx0, idx0 + max(1,N/32))
// in v[0..), with idx0 = l * N / 32 for N >= 32 and l / 2 for N == 16
// (lanes 2k and 2k+1 then hold the same sum).  Each halving step trades
// half of the values with the partner lane, so the whole reduction costs
// N - 1 shuffles for N >= 32 instead of 5 N.
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

template <int D, typename T>
struct RowLoad {
    static constexpr int DL = D / 32;
    // Loads this lane's DL elements of a row and widens them to fp32.
    __device__ __forceinline__ static void load(const T* row, int lane, float (&f)[DL]) {
        if constexpr (DL == 4) {
            const uint2 w = *reinterpret_cast<const uint2*>(row + lane * 4);
            const float2 a = unpack2<T>(w.x), b = unpack2<T>(w.y);
            f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
        } else {
            static_assert(DL == 2, "head_dim 64 or 128");
            const uint32_t w = *reinterpret_cast<const uint32_t*>(row + lane * 2);
            const float2 a = unpack2<T>(w);
            f[0] = a.x; f[1] = a.y;
        }
    }
};

template <int DL>
__device__ __forceinline__ void store_row(void* base, size_t elem_off, int out_dtype,
                                          const float (&v)[DL]) {
    if (out_dtype == PKV_F32) {
        float* p = reinterpret_cast<float*>(base) + elem_off;
        if constexpr (DL == 4) {
            *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
            *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
        }
    } else if (out_dtype == PKV_BF16) {
        __nv_bfloat16* p = reinterpret_cast<__nv_bfloat16*>(base) + elem_off;
#pragma unroll
        for (int i = 0; i < DL; i += 2)
            *reinterpret_cast<__nv_bfloat162*>(p + i) = __floats2bfloat162_rn(v[i], v[i + 1]);
    } else {
        __half* p = reinterpret_cast<__half*>(base) + elem_off;
#pragma unroll
        for (int i = 0; i < DL; i += 2)
            *reinterpret_cast<__half2*>(p + i) = __floats2half2_rn(v[i], v[i + 1]);
    }
}

// ------------------------------------------------------------ the kernel

template <int D, int BS, int QPW, typename T>
__global__ void __launch_bounds__(kMaxThreads, 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
    constexpr int DL = D / 32;
    constexpr int N = QPW * kChunk;            // partial sums per lane per chunk
    constexpr int NL = N >= 32 ? N / 32 : 1;   // complete sums per lane after reduce
    constexpr int LANES_PER_Q = 32 / QPW;      // lanes sharing one query head's sums
    static_assert(BS % kChunk == 0, "block size must be a multiple of 16");

    extern __shared__ __align__(128) unsigned char smem[];

    const int split = blockIdx.x;
    const int hg = blockIdx.y;
    const int s = blockIdx.z;
    const int HPC = p.heads_per_cta;
    const int n_cons = HPC * p.warps_per_kv;

    // ---- this CTA's token range (clamped to what the grid and table cover)
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
    const int n_pages = (tok_end - tok_begin + BS - 1) / BS;  // 0 for an empty context
    const int page0 = tok_begin / BS;

    // ---- shared-memory carve-up
    const uint32_t tile_bytes = (uint32_t)(BS * HPC * D * sizeof(T));
    unsigned char* tiles = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)p.stages * 2 * tile_bytes);
    uint64_t* empty = full + p.stages;
    float* ps_all = reinterpret_cast<float*>(empty + p.stages);
    int* s_bid = reinterpret_cast<int*>(ps_all + n_cons * N);
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
    if (threadIdx.x == 0) {
        for (int st = 0; st < p.stages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], n_cons);
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
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
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
                    unsigned char* dst = tiles + (size_t)st * 2 * tile_bytes;
                    mbar_arrive_expect_tx(&full[st], 2 * tile_bytes);
                    tma_load_4d(dst, &tm_k, &full[st], 0, hg * HPC, 0, b, policy);
                    tma_load_4d(dst + tile_bytes, &tm_v, &full[st], 0, hg * HPC, 0, b, policy);
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
        const int kv_local = c / p.warps_per_kv;
        const int qh0 = (hg * HPC + kv_local) * p.group + (c % p.warps_per_kv) * QPW;
        float* ps = ps_all + c * N;

        float qf[QPW][DL];
#pragma unroll
        for (int g = 0; g < QPW; ++g) {
            const T* qrow = reinterpret_cast<const T*>(p.q) + ((size_t)s * p.n_heads + qh0 + g) * D;
            float f[DL];
            RowLoad<D, T>::load(qrow, lane, f);
#pragma unroll
            for (int i = 0; i < DL; ++i) qf[g][i] = f[i] * p.scale_log2;
        }

        float o[QPW][DL];
        float m[QPW];
#pragma unroll
        for (int g = 0; g < QPW; ++g) {
            m[g] = -INFINITY;
#pragma unroll
            for (int i = 0; i < DL; ++i) o[g][i] = 0.f;
        }
        float l_part = 0.f;

        const int idx0 = (N >= 32) ? lane * NL : (lane >> 1);
        const int g_own = idx0 / kChunk;
        const bool counts = (N >= 32) || ((lane & 1) == 0);  // de-duplicate N == 16
        const int row_stride = HPC * D;

        for (int i = 0; i < n_pages; ++i) {
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
                    const T* kbase = sK + ((size_t)ch * kChunk * HPC + kv_local) * D;
                    const T* vbase = sV + ((size_t)ch * kChunk * HPC + kv_local) * D;

                    // -- partial scores of 16 tokens x QPW heads
                    float acc[N];
#pragma unroll
                    for (int t = 0; t < kChunk; ++t) {
                        float kf[DL];
                        RowLoad<D, T>::load(kbase + t * row_stride, lane, kf);
#pragma unroll
                        for (int g = 0; g < QPW; ++g) {
                            float a = qf[g][0] * kf[0];
#pragma unroll
                            for (int d = 1; d < DL; ++d) a = fmaf(qf[g][d], kf[d], a);
                            acc[g * kChunk + t] = a;
                        }
                    }
                    transpose_reduce<N, 16>(acc, lane);

                    // -- mask, chunk max per query head
                    float r[NL];
                    float cmax = -INFINITY;
#pragma unroll
                    for (int j = 0; j < NL; ++j) {
                        const int t = (idx0 + j) % kChunk;
                        r[j] = (t < valid) ? acc[j] : -INFINITY;
                        cmax = fmaxf(cmax, r[j]);
                    }
#pragma unroll
                    for (int off = LANES_PER_Q / 2; off >= 1; off >>= 1)
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
                        const float mn = __shfl_sync(0xffffffffu, mnew_own, g * LANES_PER_Q);
                        const float mu = (mn == -INFINITY) ? 0.f : mn;
                        alpha[g] = exp2f(m[g] - mu);
                        m[g] = mn;
                        if (g == g_own) alpha_own = alpha[g];
                    }
                    const float mu_own = (mnew_own == -INFINITY) ? 0.f : mnew_own;
                    float psum = 0.f;
#pragma unroll
                    for (int j = 0; j < NL; ++j) {
                        const float pj = exp2f(r[j] - mu_own);
                        psum += pj;
                        ps[idx0 + j] = pj;
                    }
                    l_part = l_part * alpha_own + (counts ? psum : 0.f);
#pragma unroll
                    for (int g = 0; g < QPW; ++g)
#pragma unroll
                        for (int d = 0; d < DL; ++d) o[g][d] *= alpha[g];
                    __syncwarp();

                    // -- O += P V over the valid rows
#pragma unroll
                    for (int t4 = 0; t4 < kChunk; t4 += 4) {
                        float4 pw[QPW];
#pragma unroll
                        for (int g = 0; g < QPW; ++g)
                            pw[g] = *reinterpret_cast<const float4*>(ps + g * kChunk + t4);
#pragma unroll
                        for (int tt = 0; tt < 4; ++tt) {
                            if (t4 + tt < valid) {
                                float vf[DL];
                                RowLoad<D, T>::load(vbase + (t4 + tt) * row_stride, lane, vf);
#pragma unroll
                                for (int g = 0; g < QPW; ++g) {
                                    const float w = tt == 0 ? pw[g].x
                                                  : tt == 1 ? pw[g].y
                                                  : tt == 2 ? pw[g].z
                                                            : pw[g].w;
#pragma unroll
                                    for (int d = 0; d < DL; ++d) o[g][d] = fmaf(w, vf[d], o[g][d]);
                                }
                            }
                        }
                    }
                    __syncwarp();
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
        }

        // ---- epilogue: L per query head, normalise, write
        float lsum = l_part;
#pragma unroll
        for (int off = LANES_PER_Q / 2; off >= 1; off >>= 1)
            lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
#pragma unroll
        for (int g = 0; g < QPW; ++g) {
            const float lg = __shfl_sync(0xffffffffu, lsum, g * LANES_PER_Q);
            const float inv = lg > 0.f ? 1.f / lg : 0.f;
            float v[DL];
#pragma unroll
            for (int d = 0; d < DL; ++d) v[d] = o[g][d] * inv;
            const int qh = qh0 + g;
            if (n_splits == 1) {
                store_row<DL>(p.out, ((size_t)s * p.n_heads + qh) * D + lane * DL, p.out_dtype, v);
            } else {
                const size_t unit = ((size_t)s * p.n_heads + qh) * p.max_splits + split;
                store_row<DL>(p.ws_o, unit * D + lane * DL, PKV_F32, v);
                if (lane == 0)
                    *reinterpret_cast<float2*>(p.ws_ml + unit * 2) = make_float2(m[g], lg);
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

// One warp per (sequence, query head): merges the partial states of its
// splits, O = sum_k w_k O_k / sum_k w_k with w_k = L_k 2^{M_k - M*}.
template <int D>
__global__ void __launch_bounds__(128) paged_decode_reduce_kernel(const ReduceParams p) {
    constexpr int DL = D / 32;
    const int unit = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (unit >= p.num_seqs * p.n_heads) return;
    const int s = unit / p.n_heads;
    int n = p.context_lens[s];
    n = n < 0 ? 0 : min(n, p.cap_tokens);
    const int n_splits = max(1, (n + p.split_tokens - 1) / p.split_tokens);
    if (n_splits == 1) return;  // the decode kernel wrote this row itself

    const float2* ml = reinterpret_cast<const float2*>(p.ws_ml) + (size_t)unit * p.max_splits;
    const float* os = p.ws_o + (size_t)unit * p.max_splits * D;

    float mx = -INFINITY;
    for (int k = lane; k < n_splits; k += 32) {
        const float2 v = ml[k];
        if (v.y > 0.f) mx = fmaxf(mx, v.x);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));

    float acc[DL];
#pragma unroll
    for (int d = 0; d < DL; ++d) acc[d] = 0.f;
    float wsum = 0.f;
    for (int k = 0; k < n_splits; ++k) {
        const float2 v = ml[k];
        if (!(v.y > 0.f)) continue;
        const float w = v.y * exp2f(v.x - mx);
        wsum += w;
        const float* ok = os + (size_t)k * D + lane * DL;
        if constexpr (DL == 4) {
            const float4 x = *reinterpret_cast<const float4*>(ok);
            acc[0] = fmaf(w, x.x, acc[0]);
            acc[1] = fmaf(w, x.y, acc[1]);
            acc[2] = fmaf(w, x.z, acc[2]);
            acc[3] = fmaf(w, x.w, acc[3]);
        } else {
            const float2 x = *reinterpret_cast<const float2*>(ok);
            acc[0] = fmaf(w, x.x, acc[0]);
            acc[1] = fmaf(w, x.y, acc[1]);
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    float v[DL];
#pragma unroll
    for (int d = 0; d < DL; ++d) v[d] = acc[d] * inv;
    store_row<DL>(p.out, (size_t)unit * D + lane * DL, p.out_dtype, v);
}

}  // namespace pkv
