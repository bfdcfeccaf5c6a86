// decode_stream_kernel.cuh -- paged single-query attention for grouped-query
// heads on the tensor cores, one CTA streaming many work units (sm_103a).
// Same inputs, outputs and arithmetic per unit as paged_decode_mma_kernel.
//
// Pages followed (cited by title and section):
//   [SWAP]   "vLLM 中 FlashAttention 与 KVCache 交换机制深度解析": the attention
//            formula, Tiling + Kernel Fusion + the OnlineSoftmax recurrence,
//            MQA/GQA by indexing.
//   [LAYOUT] "大模型长文本推理基座从 FlashAttention 硬件加速机制到 vLLM 核心
//            PagedAttention 显存物理布局深度剖析", section 二.2: block table.
//
// Why: with many short contexts (a continuous-batching step: most sequences
// hold 1-4 pages), a CTA per (sequence, head group, split) spends its life on
// one dependent chain -- context length, block ids, page loads, a few pages
// of work -- and the SMs wait on latency instead of streaming HBM.  Here a
// grid of resident CTAs covers the work instead: the units (sequence s,
// split k, head group h) are laid out one after another, each weighing its
// page count, and CTA c takes the units that start in the c-th equal share
// of the total pages.  Its producer warp walks those units in order and
// keeps the page ring full across unit boundaries: while the consumers
// finish one unit's pages, the next unit's block ids are looked up and its
// pages (and its query rows) are already loading.  Each ring slot carries a
// small record of the unit it belongs to; a consumer starts a unit (query
// fragments from the slot, fresh state) on the unit's first page and writes
// its output (or split partial) after the last.  A record with no pages
// ends the stream.  Sequences with an empty context get their zero rows
// from the CTA whose share holds their (empty) place in the layout.
#pragma once

#include "decode_mma_kernel.cuh"

namespace pkv {

constexpr int kStreamMaxSeqs = 2048;   // context lengths held in shared memory
constexpr int kStreamBatchUnits = 32;  // units whose block ids one lookup fetches
constexpr int kStreamBatchPages = 128; // pages of one lookup (at least one split's)

// A unit queued by the producer: sequence, split, head group, its pages and
// where its block ids start in the batch buffer.
struct StreamUnit {
    int s;
    int k;
    int hg;
    int npk;
    int n_splits;
    int first;
};

// What the producer tells the consumers about the page in one ring slot.
struct StreamSlot {
    int s;          // sequence (-1: end of the stream)
    int hg;         // kv-head group
    int split;      // split of the sequence
    int page;       // page of the unit (0 = first: query rows in the slot)
    int n_pages;    // pages of the unit
    int n_splits;   // splits of the sequence
    int tok_begin;  // first token of the unit
    int tok_end;    // one past its last token
    int valid;      // the page's block id was in range (else the page is skipped)
};

// Shared memory of one CTA (must match the carve-up in the kernel): 1 KB
// alignment slack, the ring of K/V pages, the query rows of each slot,
// barriers, slot records, block ids of one unit, the clamped lengths and
// their page prefix sums, a few words.
inline size_t decode_stream_smem_bytes(int D, int BS, int G, int elem_bytes, int hpc,
                                       int stages, int max_pages_per_split, int num_seqs) {
    const size_t ring = (size_t)stages * 2 * hpc * D * BS * elem_bytes;
    const size_t qs = (size_t)stages * hpc * G * D * elem_bytes;
    const int batch = max_pages_per_split > kStreamBatchPages ? max_pages_per_split
                                                              : kStreamBatchPages;
    return 1024 + ring + qs + (size_t)stages * 2 * sizeof(uint64_t) +
           (size_t)stages * sizeof(StreamSlot) + kStreamBatchUnits * sizeof(StreamUnit) +
           (size_t)batch * sizeof(int) + (size_t)(2 * num_seqs + 2) * sizeof(int) +
           8 * sizeof(int);
}

__device__ __forceinline__ void bulk_load_q(void* dst_smem, const void* src, uint32_t bytes,
                                            uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst_smem)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

template <int D, int BS, typename T>
__global__ void __launch_bounds__(kMmaMaxThreads, 1)
    paged_decode_mma_stream_kernel(const __grid_constant__ CUtensorMap tm_k,
                                   const __grid_constant__ CUtensorMap tm_v,
                                   const __grid_constant__ DecodeParams p) {
    constexpr int HALVES = D / 64;        // 128-byte boxes per token row
    constexpr uint32_t BOX = BS * 128;    // bytes of one [BS x 64] box
    static_assert(BS % 16 == 0 && D % 64 == 0, "shape");

    launch_dependents();  // the split merge may start its CTAs (they wait)

    extern __shared__ __align__(1024) unsigned char smem_raw[];

    const int HPC = p.heads_per_cta;
    const int G = p.group;
    const int S = p.num_seqs;
    const int stages = p.stages;
    const int PPS = p.split_tokens / BS;   // pages per full split
    if ((int)blockDim.x != 32 * (1 + HPC) || G > 8 || p.warps_per_tok != 1 || S > kStreamMaxSeqs ||
        stages < 2 || stages > 16 || PPS > p.max_pages_per_split || PPS < 1) {
        if (threadIdx.x == 0) raise_error(p.errors, PKV_DEVERR_CONFIG);
        return;
    }
    const int HG = p.n_kv_heads / HPC;

    // ---- shared memory
    const uint32_t raw_addr = smem_addr(smem_raw);
    unsigned char* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const uint32_t head_bytes = HALVES * BOX;              // one kv head's K (or V) page
    const uint32_t stage_bytes = 2 * HPC * head_bytes;     // K then V for HPC heads
    const uint32_t q_bytes = (uint32_t)(HPC * G * D * sizeof(T));   // query rows of a unit
    unsigned char* ring = smem;
    unsigned char* qbuf = ring + (size_t)stages * stage_bytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(qbuf + (size_t)stages * q_bytes);
    uint64_t* empty = full + stages;
    StreamSlot* slot = reinterpret_cast<StreamSlot*>(empty + stages);
    StreamUnit* s_unitq = reinterpret_cast<StreamUnit*>(slot + stages);
    int* s_bid = reinterpret_cast<int*>(s_unitq + kStreamBatchUnits);
    int* s_len = s_bid + max(kStreamBatchPages, p.max_pages_per_split);   // clamped lengths [S]
    int* s_pref = s_len + S;                         // page prefix sums [S + 1]
    int* s_var = s_pref + S + 1;   // first sequence, abort, slots issued, queued units

    const int cap = min(p.max_blocks_per_seq * BS, p.max_splits * p.split_tokens);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- layout of the work: W_s = HG x pages of sequence s, prefix sums
    // (one pass: each thread a contiguous run of sequences, then a scan of
    // the per-thread sums through warp shuffles and shared memory)
    {
        const int nt = (int)blockDim.x;
        const int per = (S + nt - 1) / nt;
        const int lo = min(S, (int)threadIdx.x * per);
        const int hi = min(S, lo + per);
        int sum = 0;
        for (int i = lo; i < hi; ++i) {
            int n = p.context_lens[i];
            if (n < 0 || n > cap) {
                if (blockIdx.x == 0) raise_error(p.errors, PKV_DEVERR_CONTEXT);
                n = n < 0 ? 0 : cap;
            }
            s_len[i] = n;
            sum += HG * ((n + BS - 1) / BS);
        }
        int incl = sum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += a;
        }
        __shared__ int warp_tot[kMmaMaxWarps + 1];
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        int before = incl - sum;
        for (int w = 0; w < warp; ++w) before += warp_tot[w];
        int run = before;
        for (int i = lo; i < hi; ++i) {
            s_pref[i] = run;
            run += HG * ((s_len[i] + BS - 1) / BS);
        }
        if (threadIdx.x == nt - 1) s_pref[S] = run;
        __syncthreads();
    }
    const long long P = s_pref[S];
    const long long C = gridDim.x;
    const long long P0 = P * blockIdx.x / C;
    const long long P1 = P * (blockIdx.x + 1) / C;
    const bool last_cta = blockIdx.x == gridDim.x - 1;

    // ---- empty contexts: zero rows, written by the CTA whose share holds
    // the sequence's place (the last CTA for places at the very end)
    for (int i = threadIdx.x; i < S * HG; i += blockDim.x) {
        const int s = i / HG;
        if (s_len[s] != 0) continue;
        const long long at = s_pref[s];
        if (!((at >= P0 && at < P1) || (at >= P && last_cta))) continue;
        const int hg = i - s * HG;
        if (p.slot_mapping != nullptr) {
            // an append into an empty context (its length not counting the
            // token) still writes the row, as the per-unit kernels do
            const int64_t slot_row = p.slot_mapping[s];
            if (slot_row >= (int64_t)p.num_blocks * BS) {
                if (hg == 0) raise_error(p.errors, PKV_DEVERR_SLOT);
            } else if (slot_row >= 0) {
                constexpr int VEC = 16 / (int)sizeof(T);
                const size_t row = (size_t)p.n_kv_heads * D;
                const size_t off_new = (size_t)s * row + (size_t)hg * HPC * D;
                const size_t off_pool = (size_t)slot_row * row + (size_t)hg * HPC * D;
                for (int j = 0; j < HPC * D; j += VEC) {
                    *reinterpret_cast<uint4*>(static_cast<T*>(p.k_pool) + off_pool + j) =
                        *reinterpret_cast<const uint4*>(static_cast<const T*>(p.k_new) + off_new + j);
                    *reinterpret_cast<uint4*>(static_cast<T*>(p.v_pool) + off_pool + j) =
                        *reinterpret_cast<const uint4*>(static_cast<const T*>(p.v_new) + off_new + j);
                }
            }
        }
        const int q0 = hg * HPC * G;
        for (int qh = q0; qh < q0 + HPC * G; ++qh) {
            const size_t e = ((size_t)s * p.n_heads + qh) * D;
            if (p.out_dtype == PKV_F32) {
                float* o = reinterpret_cast<float*>(p.out) + e;
                for (int d = 0; d < D; ++d) o[d] = 0.f;
            } else {
                uint16_t* o = reinterpret_cast<uint16_t*>(p.out) + e;
                for (int d = 0; d < D; ++d) o[d] = 0;
            }
        }
    }

    // first sequence whose pages reach into [P0, P1): the last s with
    // pref[s] <= P0 (binary search; sequences of no pages are skipped later)
    if (threadIdx.x == 0) {
        int a = 0, b = S - 1, f = 0;
        while (a <= b) {
            const int m = (a + b) >> 1;
            if ((long long)s_pref[m] <= P0) {
                f = m;
                a = m + 1;
            } else {
                b = m - 1;
            }
        }
        s_var[0] = f;
        s_var[1] = 0;   // abort
        s_var[2] = 0;   // slots issued
        for (int st = 0; st < stages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], HPC);
        }
        fence_barrier_init();
    }
    __syncthreads();
    volatile int* s_abort = s_var + 1;

    if (warp == 0) {
        // ================= producer =================
        // Units are taken in batches: lane 0 queues the next units (up to
        // kStreamBatchUnits, or until their pages would pass the batch's
        // block-id buffer), the whole warp looks up all their block ids at
        // once (one memory round trip per batch instead of one per unit) and
        // writes the fused appends, then lane 0 issues every page.
        const uint64_t policy = l2_policy_evict_first();
        if (lane == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
        const int cap_pages = max(kStreamBatchPages, PPS);
        int g = 0;                          // slots issued so far (lane 0)
        // walk cursor (lane 0): sequence, its place, split and head group
        int cs = s_var[0], ck = 0, ch = 0;
        bool done = false, stop = false;
        while (!done && !stop) {
            if (lane == 0) {
                int nu = 0, np_batch = 0;
                while (nu < kStreamBatchUnits && cs < S) {
                    const long long Ps = s_pref[cs];
                    if (Ps >= P1) {
                        cs = S;
                        break;
                    }
                    const int n = s_len[cs];
                    const int np = (n + BS - 1) / BS;
                    const int n_splits = max(1, (n + p.split_tokens - 1) / p.split_tokens);
                    if (n == 0 || ck >= n_splits) {
                        ++cs;
                        ck = ch = 0;
                        continue;
                    }
                    const int npk = min(PPS, np - ck * PPS);
                    const long long start = Ps + (long long)HG * ck * PPS + (long long)ch * npk;
                    if (start >= P1) {
                        cs = S;
                        break;
                    }
                    if (start >= P0) {
                        if (np_batch + npk > cap_pages) break;   // the next batch takes it
                        StreamUnit& u = s_unitq[nu++];
                        u.s = cs;
                        u.k = ck;
                        u.hg = ch;
                        u.npk = npk;
                        u.n_splits = n_splits;
                        u.first = np_batch;
                        np_batch += npk;
                    }
                    if (++ch == HG) {
                        ch = 0;
                        ++ck;
                    }
                }
                s_var[3] = nu;
            }
            __syncwarp();
            const int nu = s_var[3];
            if (nu == 0) {
                done = true;
                break;
            }
            // ---- block ids of every queued unit (all lanes, independent loads)
            for (int ui = 0; ui < nu; ++ui) {
                const StreamUnit u = s_unitq[ui];
                const int* row = p.block_tables + (size_t)u.s * p.max_blocks_per_seq + u.k * PPS;
                for (int i = lane; i < u.npk; i += 32) {
                    int b = row[i];
                    if (b < 0 || b >= p.num_blocks) {
                        raise_error(p.errors, PKV_DEVERR_BLOCK_ID);
                        b = -1;
                    }
                    s_bid[u.first + i] = b;
                }
            }
            // ---- fused append: a last split's unit writes the new token's
            // rows of its heads before any of its pages load
            if (p.slot_mapping != nullptr) {
                constexpr int VEC = 16 / (int)sizeof(T);
                const int per_row = HPC * D / VEC;
                const size_t row = (size_t)p.n_kv_heads * D;
                for (int ui = 0; ui < nu; ++ui) {
                    const StreamUnit u = s_unitq[ui];
                    if (u.k != u.n_splits - 1) continue;
                    const int64_t slot_row = p.slot_mapping[u.s];
                    if (slot_row < 0) continue;
                    if (slot_row >= (int64_t)p.num_blocks * BS) {
                        if (u.hg == 0 && lane == 0) raise_error(p.errors, PKV_DEVERR_SLOT);
                        continue;
                    }
                    const size_t off_new = (size_t)u.s * row + (size_t)u.hg * HPC * D;
                    const size_t off_pool = (size_t)slot_row * row + (size_t)u.hg * HPC * D;
                    for (int i = lane; i < 2 * per_row; i += 32) {
                        const bool is_v = i >= per_row;
                        const int j = (is_v ? i - per_row : i) * VEC;
                        const T* src = static_cast<const T*>(is_v ? p.v_new : p.k_new) + off_new + j;
                        T* dst = static_cast<T*>(is_v ? p.v_pool : p.k_pool) + off_pool + j;
                        *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
                    }
                }
                asm volatile("fence.proxy.async.global;" ::: "memory");
            }
            __syncwarp();
            // ---- issue every page of the batch (lane 0)
            if (lane == 0) {
                asm volatile("fence.proxy.async.global;" ::: "memory");
                for (int ui = 0; ui < nu && !stop; ++ui) {
                    const StreamUnit u = s_unitq[ui];
                    const int n = s_len[u.s];
                    const int tok_begin = u.k * p.split_tokens;
                    const int tok_end = min(n, tok_begin + p.split_tokens);
                    const T* qsrc = reinterpret_cast<const T*>(p.q) +
                                    ((size_t)u.s * p.n_heads + (size_t)u.hg * HPC * G) * D;
                    for (int i = 0; i < u.npk; ++i, ++g) {
                        const int st = g % stages;
                        if (g >= stages &&
                            !mbar_wait(&empty[st], ((g / stages) - 1) & 1, p.errors)) {
                            *s_abort = 1;
                            stop = true;
                            break;
                        }
                        if (*s_abort) {
                            stop = true;
                            break;
                        }
                        const int b = s_bid[u.first + i];
                        StreamSlot& r = slot[st];
                        r.s = u.s;
                        r.hg = u.hg;
                        r.split = u.k;
                        r.page = i;
                        r.n_pages = u.npk;
                        r.n_splits = u.n_splits;
                        r.tok_begin = tok_begin;
                        r.tok_end = tok_end;
                        r.valid = b >= 0;
                        const uint32_t bytes =
                            (b >= 0 ? stage_bytes : 0u) + (i == 0 ? q_bytes : 0u);
                        if (bytes == 0) {
                            mbar_arrive(&full[st]);
                            continue;
                        }
                        mbar_arrive_expect_tx(&full[st], bytes);
                        if (i == 0)
                            bulk_load_q(qbuf + (size_t)st * q_bytes, qsrc, q_bytes, &full[st],
                                        policy);
                        if (b >= 0) {
                            unsigned char* dst = ring + (size_t)st * stage_bytes;
                            for (int hh = 0; hh < HPC; ++hh) {
                                const int hrow = (u.hg * HPC + hh) * HALVES;
                                for (int h = 0; h < HALVES; ++h) {
                                    tma_load_4d(dst + hh * head_bytes + h * BOX, &tm_k,
                                                &full[st], 0, hrow + h, 0, b, policy);
                                    tma_load_4d(dst + (HPC + hh) * head_bytes + h * BOX, &tm_v,
                                                &full[st], 0, hrow + h, 0, b, policy);
                                }
                            }
                        }
                    }
                }
            }
            stop = __shfl_sync(0xffffffffu, stop ? 1 : 0, 0) != 0;
            __syncwarp();
        }
        // ---- end of the stream: a record without pages
        if (lane == 0 && !*s_abort) {
            const int st = g % stages;
            if (g < stages || mbar_wait(&empty[st], ((g / stages) - 1) & 1, p.errors)) {
                slot[st].s = -1;
                mbar_arrive(&full[st]);
                ++g;
            } else {
                *s_abort = 1;
            }
        }
        if (lane == 0) s_var[2] = g;
        __syncwarp();
    } else {
        // ================= consumers: one warp per kv head =================
        const int kv_local = warp - 1;
        MmaHeads<D> st;
        for (int g = 0;; ++g) {
            const int slot_i = g % stages;
            if (!mbar_wait(&full[slot_i], (g / stages) & 1, p.errors)) {
                *s_abort = 1;
                break;
            }
            const StreamSlot r = slot[slot_i];
            if (r.s < 0) break;
            if (r.page == 0)
                // query rows of this unit's kv head (loaded into the slot)
                mma_heads_start<D, T>(st, reinterpret_cast<const T*>(qbuf + (size_t)slot_i * q_bytes) +
                                              (size_t)kv_local * G * D,
                                      G, lane);
            if (r.valid) {
                const uint32_t kbase = smem_addr(ring + (size_t)slot_i * stage_bytes +
                                                 kv_local * head_bytes);
                const uint32_t vbase = smem_addr(ring + (size_t)slot_i * stage_bytes +
                                                 (HPC + kv_local) * head_bytes);
                const int page_tok = r.tok_begin + r.page * BS;
#pragma unroll
                for (int ch = 0; ch < BS / 16; ++ch) {
                    const int valid = min(16, r.tok_end - (page_tok + ch * 16));
                    if (valid <= 0) break;
                    mma_heads_chunk<D, T>(st, kbase, vbase, BOX, ch * 16, valid, p.scale_log2,
                                          lane);
                }
            }
            if (r.page == r.n_pages - 1)
                mma_heads_finish<D>(st, p, r.s, (r.hg * HPC + kv_local) * G, G, r.n_splits,
                                    r.split, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot_i]);
        }
    }

    __syncthreads();
    if (*s_abort && threadIdx.x == 0) {
        // loads still in flight land before the CTA's shared memory goes away
        const int issued = s_var[2];
        for (int st = 0; st < stages && st < issued; ++st) {
            const int last = st + ((issued - 1 - st) / stages) * stages;
            mbar_wait(&full[st], (last / stages) & 1, p.errors);
        }
    }
}

}  // namespace pkv
