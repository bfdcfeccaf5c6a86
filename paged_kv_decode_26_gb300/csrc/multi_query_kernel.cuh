// multi_query_kernel.cuh -- causal attention of several new tokens per
// sequence (a prefill chunk, or tokens to verify) over the paged KV cache,
// on the tensor cores (sm_103a).
//
// Pages followed (cited by title and section):
//   [SWAP]   "vLLM 中 FlashAttention 与 KVCache 交换机制深度解析": the attention
//            formula and FlashAttention's tiling of Q, K, V blocks through
//            on-chip memory with the OnlineSoftmax recurrence; the serving
//            loop's prefill step ("Prefill: 使用FlashAttention计算全部KV并写入
//            Pages") followed by decode.
//   [LAYOUT] "大模型长文本推理基座从 FlashAttention 硬件加速机制到 vLLM 核心
//            PagedAttention 显存物理布局深度剖析", section 二.2: block table.
//
// Sequence s owns query rows q_start[s] .. q_start[s+1]-1, its last q_len
// tokens: row i sits at position p_i = n - q_len + i and attends to keys
// t <= p_i.  One CTA per (query tile, kv head, sequence).  Each consumer
// warp owns 16 mma rows = 16/G consecutive query tokens x the G query heads
// of the kv head (row r: token r / G, head r % G), so every page of K and V
// loaded once serves 16 x W rows of the CTA.  Pages arrive as in the decode
// tensor-core kernel (per-head [B x 64] TMA boxes, 128-byte swizzle), and
// S = Q K^T, the online softmax and O += P V (P as hi + lo parts) are the
// same per 16-token chunk, with the causal mask per row.
#pragma once

#include "decode_mma_kernel.cuh"

namespace pkv {

struct MultiQueryParams {
    void* out;          // [total_q, n_heads, D]
    int out_dtype;
    const void* q;      // [total_q, n_heads, D]
    const int32_t* q_start;  // [num_seqs + 1]
    int total_q;
    int max_q_len;
    const int32_t* block_tables;
    int max_blocks_per_seq;
    const int32_t* context_lens;
    int num_seqs;
    int n_heads;
    int n_kv_heads;
    int group;
    int num_blocks;
    float scale_log2;
    int stages;
    int max_pages;      // block ids prefetched per CTA (ceil(max_context_len / B))
    unsigned int* errors;
    // tcgen05 kernel: 0 = CTAs take sequences in index order; else num_seqs,
    // and CTAs take them longest context first (see longest_first).
    int lpt_seqs;
};

inline size_t multi_query_smem_bytes(int D, int BS, int elem_bytes, int stages, int max_pages) {
    return 1024 + (size_t)stages * 2 * D * BS * elem_bytes + (size_t)stages * 2 * sizeof(uint64_t) +
           (size_t)max_pages * sizeof(int) + 2 * sizeof(int);
}

template <int D, int BS, typename T>
__global__ void __launch_bounds__(kMmaMaxThreads, 1)
    paged_multi_query_kernel(const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v, const MultiQueryParams p) {
    constexpr int HALVES = D / 64;
    constexpr int KSTEPS = D / 16;
    constexpr int NT = D / 8;
    constexpr uint32_t BOX = BS * 128;
    static_assert(BS % 16 == 0 && D % 64 == 0, "shape");

    extern __shared__ __align__(1024) unsigned char smem_raw[];

    const int tile = blockIdx.x;
    const int kvh = blockIdx.y;
    const int s = blockIdx.z;
    const int G = p.group;
    const int QT = 16 / G;                      // query tokens per warp
    const int W = (int)(blockDim.x >> 5) - 1;   // consumer warps
    if (G < 1 || G > 16 || 16 % G != 0 || W < 1) {
        if (threadIdx.x == 0) raise_error(p.errors, PKV_DEVERR_CONFIG);
        return;
    }

    // ---- this CTA's query tokens and the keys they need
    const int qs0 = p.q_start[s], qs1 = p.q_start[s + 1];
    const int n = p.context_lens[s];
    const int q_len = qs1 - qs0;
    if (q_len < 0 || q_len > n || qs0 < 0 || qs1 > p.total_q || q_len > p.max_q_len ||
        n > p.max_blocks_per_seq * BS || (n + BS - 1) / BS > p.max_pages) {
        if (tile == 0 && kvh == 0 && threadIdx.x == 0) raise_error(p.errors, PKV_DEVERR_CONTEXT);
        return;
    }
    const int tok_lo = tile * W * QT;           // first query token (0-based in the sequence)
    if (tok_lo >= q_len) return;
    const int tok_hi = min(q_len, tok_lo + W * QT);
    const int first_pos = n - q_len;            // position of query token 0
    const int n_keys = first_pos + tok_hi;      // keys 0 .. first_pos + tok_hi - 1
    const int n_pages = (n_keys + BS - 1) / BS;

    const uint32_t raw_addr = smem_addr(smem_raw);
    unsigned char* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const uint32_t head_bytes = HALVES * BOX;
    const uint32_t stage_bytes = 2 * head_bytes;
    unsigned char* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)p.stages * stage_bytes);
    uint64_t* empty = full + p.stages;
    int* s_bid = reinterpret_cast<int*>(empty + p.stages);
    int* s_abort = s_bid + p.max_pages;
    int* s_issued = s_abort + 1;

    for (int i = threadIdx.x; i < n_pages; i += blockDim.x) {
        int b = p.block_tables[(size_t)s * p.max_blocks_per_seq + i];
        if (b < 0 || b >= p.num_blocks) {
            raise_error(p.errors, PKV_DEVERR_BLOCK_ID);
            b = -1;
        }
        s_bid[i] = b;
    }
    if (threadIdx.x == 0) {
        for (int st = 0; st < p.stages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], W);
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
            const uint64_t policy = l2_policy_evict_normal();  // pages are re-read by other tiles
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
                    for (int h = 0; h < HALVES; ++h) {
                        tma_load_4d(dst + h * BOX, &tm_k, &full[st], 0, kvh * HALVES + h, 0, b,
                                    policy);
                        tma_load_4d(dst + head_bytes + h * BOX, &tm_v, &full[st], 0,
                                    kvh * HALVES + h, 0, b, policy);
                    }
                } else {
                    mbar_arrive(&full[st]);
                }
            }
            *s_issued = i;
        }
        __syncwarp();
    } else {
        // ================= consumers: 16 rows = QT tokens x G heads =================
        const int c = warp - 1;
        const int gid = lane >> 2;
        const int tig = lane & 3;
        const int wtok0 = tok_lo + c * QT;     // this warp's first query token
        // the two rows of this lane: gid and gid + 8
        int pos[2];
        const T* qrow[2];
        bool real[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int r = gid + 8 * h2;
            const int tok = wtok0 + r / G;
            const int g = r % G;
            real[h2] = tok < tok_hi;
            pos[h2] = real[h2] ? first_pos + tok : -1;
            qrow[h2] = reinterpret_cast<const T*>(p.q) +
                       ((size_t)(qs0 + (real[h2] ? tok : 0)) * p.n_heads + kvh * G + g) * D;
        }
        // last key any row of this warp may see (-1: the warp has no token)
        const int warp_last_pos = wtok0 < tok_hi ? first_pos + min(tok_hi, wtok0 + QT) - 1 : -1;

        uint32_t qa[KSTEPS][4];
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const uint32_t lo = *reinterpret_cast<const uint32_t*>(qrow[h2] + ks * 16 + tig * 2);
                const uint32_t hi =
                    *reinterpret_cast<const uint32_t*>(qrow[h2] + ks * 16 + 8 + tig * 2);
                qa[ks][h2] = real[h2] ? lo : 0u;       // a0 (row gid), a1 (row gid + 8)
                qa[ks][2 + h2] = real[h2] ? hi : 0u;   // a2, a3
            }
        }

        float o[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
        float m_row[2] = {-INFINITY, -INFINITY};
        float l_part[2] = {0.f, 0.f};

        const int mat = lane >> 3, mrow = lane & 7;
        const int k_tok = (mat >> 1) * 8 + mrow, k_dc = mat & 1;
        const int v_tok = (mat & 1) * 8 + mrow, v_dc = mat >> 1;

        for (int i = 0; i < n_pages; ++i) {
            const int st = i % p.stages;
            if (!mbar_wait(&full[st], (i / p.stages) & 1, p.errors)) {
                atomicExch(s_abort, 1);
                break;
            }
            const int page_tok = i * BS;
            if (s_bid[i] >= 0 && page_tok <= warp_last_pos) {
                const uint32_t kbase = smem_addr(ring + (size_t)st * stage_bytes);
                const uint32_t vbase = kbase + head_bytes;
#pragma unroll
                for (int ch = 0; ch < BS / 16; ++ch) {
                    const int key0 = page_tok + ch * 16;
                    if (key0 > warp_last_pos) break;
                    const int valid = min(16, n - key0);   // keys past the context
                    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                    for (int ks = 0; ks < KSTEPS; ++ks) {
                        const int h = ks / 4;
                        const int cc = (ks % 4) * 2 + k_dc;
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(kbase + h * BOX + swz(ch * 16 + k_tok, cc), b0, b1, b2, b3);
                        mma16816<T>(sc[0], qa[ks], b0, b1);
                        mma16816<T>(sc[1], qa[ks], b2, b3);
                    }
                    // scores of this lane: row h2 (gid / gid + 8), keys
                    // key0 + 8 nt + 2 tig + {0, 1}
                    float x[2][4];
                    float alpha[2];
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int key = key0 + nt * 8 + tig * 2 + e;
                                const float v = sc[nt][h2 * 2 + e] * p.scale_log2;
                                x[h2][nt * 2 + e] = key <= pos[h2] ? v : -INFINITY;
                            }
                        float cmax = fmaxf(fmaxf(x[h2][0], x[h2][1]), fmaxf(x[h2][2], x[h2][3]));
                        cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 1));
                        cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 2));
                        const float m_new = fmaxf(m_row[h2], cmax);
                        const float mu = (m_new == -INFINITY) ? 0.f : m_new;
                        alpha[h2] = exp2f(m_row[h2] - mu);
                        m_row[h2] = m_new;
#pragma unroll
                        for (int e = 0; e < 4; ++e) x[h2][e] = exp2f(x[h2][e] - mu);
                        l_part[h2] = l_part[h2] * alpha[h2] +
                                     ((x[h2][0] + x[h2][1]) + (x[h2][2] + x[h2][3]));
                    }
                    uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
                    if (valid < 16) {
                        vm0 = (tig * 2 < valid ? 0x0000ffffu : 0u) |
                              (tig * 2 + 1 < valid ? 0xffff0000u : 0u);
                        vm1 = (8 + tig * 2 < valid ? 0x0000ffffu : 0u) |
                              (8 + tig * 2 + 1 < valid ? 0xffff0000u : 0u);
                    }
                    // P (rows gid, gid + 8; keys 2 tig.. and 8 + 2 tig..) as hi + lo
                    uint32_t pa[4], pl[4];
                    pa[0] = pack2<T>(x[0][0], x[0][1]);
                    pa[1] = pack2<T>(x[1][0], x[1][1]);
                    pa[2] = pack2<T>(x[0][2], x[0][3]);
                    pa[3] = pack2<T>(x[1][2], x[1][3]);
#pragma unroll
                    for (int a = 0; a < 4; ++a) {
                        const int h2 = a & 1, nt = a >> 1;
                        const float2 hv = unpack2<T>(pa[a]);
                        pl[a] = pack2<T>(x[h2][nt * 2] - hv.x, x[h2][nt * 2 + 1] - hv.y);
                    }
#pragma unroll
                    for (int j = 0; j < NT; j += 2) {
                        o[j][0] *= alpha[0];
                        o[j][1] *= alpha[0];
                        o[j][2] *= alpha[1];
                        o[j][3] *= alpha[1];
                        o[j + 1][0] *= alpha[0];
                        o[j + 1][1] *= alpha[0];
                        o[j + 1][2] *= alpha[1];
                        o[j + 1][3] *= alpha[1];
                        const int h = j / 8;
                        const int cc = (j % 8) + v_dc;
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_trans(vbase + h * BOX + swz(ch * 16 + v_tok, cc), b0, b1, b2, b3);
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

        // ---- normalise and write the two rows of this lane
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            float l = l_part[h2];
            l += __shfl_xor_sync(0xffffffffu, l, 1);
            l += __shfl_xor_sync(0xffffffffu, l, 2);
            if (!real[h2]) continue;
            const int r = gid + 8 * h2;
            const int tok = wtok0 + r / G;
            const int qh = kvh * G + r % G;
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const size_t e = ((size_t)(qs0 + tok) * p.n_heads + qh) * D + j * 8 + tig * 2;
                const float a = o[j][h2 * 2] * inv, b = o[j][h2 * 2 + 1] * inv;
                if (p.out_dtype == PKV_F32) {
                    *reinterpret_cast<float2*>(reinterpret_cast<float*>(p.out) + e) =
                        make_float2(a, b);
                } else {
                    *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(p.out) + e) =
                        pack_out(a, b, p.out_dtype);
                }
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

}  // namespace pkv
