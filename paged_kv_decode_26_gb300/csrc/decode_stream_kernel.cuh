// decode_stream_kernel.cuh -- paged single-query attention for grouped-query
// heads on the tensor cores, by resident CTAs that each stream an exactly
// equal share of the pages (sm_103a).  Same inputs and outputs as
// paged_decode_mma_kernel, and the same per-page arithmetic.
//
// Pages followed (cited by title and section):
//   [SWAP]   "vLLM 中 FlashAttention 与 KVCache 交换机制深度解析": the attention
//            formula, Tiling + Kernel Fusion + the OnlineSoftmax recurrence
//            (partial states merged by the same recurrence), MQA/GQA by
//            indexing.
//   [LAYOUT] "大模型长文本推理基座从 FlashAttention 硬件加速机制到 vLLM 核心
//            PagedAttention 显存物理布局深度剖析", section 二.2: block table.
//
// Why: with many short contexts (a continuous-batching step: most sequences
// hold 1-4 pages), a CTA per (sequence, head group, split) spends its life on
// one dependent chain -- context length, block ids, page loads, a few pages
// of work -- and the SMs wait on latency instead of streaming HBM.  Cutting
// the work into whole units and handing each CTA the units that start in its
// share still leaves the CTA that drew a long unit working alone at the end.
//
// Layout of the work: the pages of every run (sequence s, kv-head group hg)
// are laid end to end, sequence by sequence and head group by head group:
// run r = s * HG + hg covers positions [a_r, a_r + np_s) with np_s the
// sequence's page count.  With P positions and C shares (one per CTA, at
// most P, see stream_shares), CTA c takes exactly positions
// [P c / C, P (c + 1) / C).  A run that lies inside one share is finished by
// that CTA (its rows go straight to the output); a run that a share boundary
// cuts leaves one partial state (normalised O, M, L) per CTA that holds part
// of it.  A CTA holds at most two such pieces -- one cut at the start of its
// share, one cut at its end -- in workspace slots 2c and 2c + 1 (a piece cut
// at both ends takes 2c), so the workspace does not grow with the number of
// sequences.  The merge kernel below combines them with the OnlineSoftmax
// recurrence; each CTA records the run cut at the end of its share, if the
// run starts in its share, so the merge needs no layout of its own.
//
// Each CTA: a producer warp and one consumer warp per kv head of the group.
// The producer walks the CTA's positions in batches of chunks (pieces of
// runs), looks up all their block ids (and append slots) at once, then keeps
// the page ring full across run boundaries.  Each ring slot carries a record
// of the page's run and whether it starts the CTA's piece of the run (the
// query rows come along in the slot), ends it, and whether the run is whole;
// the slot of a run's last page also brings the step's new K and V rows when
// the call appends, which the consumers put into the page and the pool.  A
// record without pages ends the stream.  Sequences with an empty
// context get their zero rows from the CTA whose share holds their (empty)
// place in the layout.
#pragma once

#include "decode_mma_kernel.cuh"

namespace pkv {

constexpr int kStreamMaxSeqs = 2048;     // context lengths held in shared memory
constexpr int kStreamBatchChunks = 32;   // chunks whose block ids one lookup fetches (one a lane)
static_assert(kStreamBatchChunks <= 32, "the append slots of a batch are read one chunk a lane");
constexpr int kStreamBatchPages = 128;   // pages of one lookup (a multiple of 32)
static_assert(kStreamBatchPages % 32 == 0, "a lookup spreads its pages over a warp");

// Slot record flags.
constexpr int kSlotFirst = 1;   // first page of the CTA's piece of the run (query rows in the slot)
constexpr int kSlotLast = 2;    // last page of the piece: write the result
constexpr int kSlotWhole = 4;   // the run lies inside this CTA's share: result to the output
constexpr int kSlotValid = 8;   // the page's block id was in range (else the page is skipped)
constexpr int kSlotHead = 16;   // the piece starts the CTA's share inside a run begun before it
constexpr int kSlotAppend = 32;  // the page's last token is this step's new row (in the slot's row buffer)

// Consecutive pages of one run queued by the producer, with where their
// block ids start in the batch buffer.
struct StreamChunk {
    int s;
    int hg;
    int i0;     // first page (of the sequence)
    int n;      // pages
    int flags;  // kSlotFirst on its first page / kSlotLast on its last page, kSlotWhole
    int first;  // index of its first block id in the batch buffer
};

// What the producer tells the consumers about the page in one ring slot.
struct StreamSlot {
    long long pool_off;   // kSlotAppend: element offset of the new row of the group's heads
    int s;      // sequence (-1: end of the stream)
    int hg;     // kv-head group
    int page;   // page of the sequence
    int n_tok;  // the sequence's (clamped) context length
    int flags;  // kSlot* bits
};

// Shared memory of one CTA (must match the carve-up in the kernel): 1 KB
// alignment slack, the ring of K/V pages, the query rows of each slot, the
// new token's K and V rows of each slot (fused append), barriers, slot
// records, the chunk queue and block ids of one batch, the clamped lengths
// and their page prefix sums, a few words.
inline size_t decode_stream_smem_bytes(int D, int BS, int G, int elem_bytes, int hpc,
                                       int stages, int num_seqs) {
    const size_t ring = (size_t)stages * 2 * hpc * D * BS * elem_bytes;
    const size_t qs = (size_t)stages * hpc * G * D * elem_bytes;
    const size_t rows = (size_t)stages * 2 * hpc * D * elem_bytes;
    return 1024 + ring + qs + rows + (size_t)stages * 2 * sizeof(uint64_t) +
           (size_t)stages * sizeof(StreamSlot) + kStreamBatchChunks * sizeof(StreamChunk) +
           (size_t)kStreamBatchPages * sizeof(int) + (size_t)(2 * num_seqs + 1) * sizeof(int) +
           8 * sizeof(int);
}

// Partial-state rows the stream decode may write: two slots per CTA (the
// piece of a run cut at the start of its share and the one cut at its
// end), HPC x G query heads each.
inline size_t decode_stream_partial_rows(int ctas, int hpc, int G) {
    return 2 * (size_t)ctas * hpc * G;
}

__device__ __forceinline__ void bulk_load_q(void* dst_smem, const void* src, uint32_t bytes,
                                            uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst_smem)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// The layout of the work, computed by every CTA of both kernels from the
// context lengths: s_len[s] = the clamped length, s_pref[s] = HG x (pages of
// the sequences before s), s_pref[S] = P.  One pass: each thread a
// contiguous run of sequences, then a scan of the per-thread sums through
// warp shuffles and shared memory.  Ends with a CTA barrier.
template <int BS>
__device__ __forceinline__ void stream_layout(const DecodeParams& p, int HG, int* s_len,
                                              int* s_pref, bool flag_errors) {
    __shared__ int warp_tot[kMmaMaxWarps + 1];
    const int S = p.num_seqs;
    const int cap = min(p.max_blocks_per_seq * BS, p.max_splits * p.split_tokens);
    const int nt = (int)blockDim.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per = (S + nt - 1) / nt;
    const int lo = min(S, (int)threadIdx.x * per);
    const int hi = min(S, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; ++i) {
        int n = p.context_lens[i];
        if (n < 0 || n > cap) {
            if (flag_errors) raise_error(p.errors, PKV_DEVERR_CONTEXT);
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
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int run = incl - sum;
    for (int w = 0; w < warp; ++w) run += warp_tot[w];
    for (int i = lo; i < hi; ++i) {
        s_pref[i] = run;
        run += HG * ((s_len[i] + BS - 1) / BS);
    }
    if (threadIdx.x == nt - 1) s_pref[S] = run;
    __syncthreads();
}

// The sequence holding position x: the last s with s_pref[s] <= x (a
// sequence without pages shares its place with the next one and is passed).
__device__ __forceinline__ int stream_seq_at(const int* s_pref, int S, long long x) {
    int a = 0, b = S - 1, f = 0;
    while (a <= b) {
        const int m = (a + b) >> 1;
        if ((long long)s_pref[m] <= x) {
            f = m;
            a = m + 1;
        } else {
            b = m - 1;
        }
    }
    return f;
}

// a * b / c for non-negative operands with a * b < 2^63 (32-bit division
// when everything fits 32 bits, which is the usual case).
__device__ __forceinline__ long long mul_div(long long a, long long b, long long c) {
    const unsigned long long ab = (unsigned long long)a * (unsigned long long)b;
    if (ab <= 0xffffffffull && (unsigned long long)c <= 0xffffffffull)
        return (long long)((unsigned)ab / (unsigned)c);
    return (long long)(ab / (unsigned long long)c);
}

// Number of shares: one per CTA, but never more than the P positions (so
// that no share is empty and every CTA between a run's first and last holds
// part of it), and at least one (the CTA that writes the zero rows when
// every context is empty).  CTAs past the shares have no work.
__device__ __forceinline__ long long stream_shares(long long P, long long ctas) {
    const long long c = P < ctas ? P : ctas;
    return c < 1 ? 1 : c;
}

// The share holding position x (0 <= x < P): the largest c with
// floor(P c / C) <= x.
__device__ __forceinline__ int stream_cta_at(long long x, long long P, long long C) {
    return (int)mul_div((x + 1) * C - 1, 1, P);
}

// The record for the boundary at the end of this CTA's share [P0, P1): the
// run it cuts, if that run starts inside the share -- (s, hg, this CTA,
// number of shares holding the run) -- else s = -1 (no cut, or an earlier
// boundary cut the run and its record names it).
template <int BS>
__device__ __forceinline__ int4 stream_boundary_record(const int* s_len, const int* s_pref, int S,
                                                       int HG, long long P, long long C,
                                                       long long P0, long long P1,
                                                       bool has_share) {
    if (!has_share || P1 >= P) return make_int4(-1, 0, 0, 0);
    const int s = stream_seq_at(s_pref, S, P1);
    const int np = (s_len[s] + BS - 1) / BS;
    const int hg = (int)(P1 - s_pref[s]) / np;
    const long long a = s_pref[s] + (long long)hg * np;
    if (!(a < P1 && a >= P0)) return make_int4(-1, 0, 0, 0);
    const int c0 = (int)blockIdx.x;
    return make_int4(s, hg, c0, stream_cta_at(a + np - 1, P, C) - c0 + 1);
}

// Zero rows (and any fused append) of the sequences with an empty context
// whose place in the layout lies in this share (the last share also takes
// the places at the very end), by `nt` threads numbered from `tid`.
template <int D, int BS, typename T>
__device__ __forceinline__ void stream_zero_rows(const DecodeParams& p, const int* s_len,
                                                 const int* s_pref, int HG, int HPC, int G,
                                                 long long P, long long P0, long long P1,
                                                 bool last_cta, int tid, int nt) {
    const int S = p.num_seqs;
    for (int i = tid; i < S * HG; i += nt) {
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
}

template <int D, int BS, typename T>
__global__ void __launch_bounds__(kMmaMaxThreads, 1)
    paged_decode_mma_stream_kernel(const __grid_constant__ CUtensorMap tm_k,
                                   const __grid_constant__ CUtensorMap tm_v,
                                   const __grid_constant__ CUtensorMap tm_kh,
                                   const __grid_constant__ CUtensorMap tm_vh,
                                   const __grid_constant__ DecodeParams p) {
    constexpr int HALVES = D / 64;        // 128-byte boxes per token row
    constexpr uint32_t BOX = BS * 128;    // bytes of one [BS x 64] box
    static_assert(BS % 16 == 0 && D % 64 == 0, "shape");

    launch_dependents();  // the boundary merge may start its CTAs (they wait)

    extern __shared__ __align__(1024) unsigned char smem_raw[];

    const int HPC = p.heads_per_cta;
    const int G = p.group;
    const int S = p.num_seqs;
    const int stages = p.stages;
    if ((int)blockDim.x != 32 * (1 + HPC) || G > 8 || p.warps_per_tok != 1 || S > kStreamMaxSeqs ||
        stages < 2 || stages > 16) {
        if (threadIdx.x == 0) raise_error(p.errors, PKV_DEVERR_CONFIG);
        return;
    }
    const int HG = p.n_kv_heads / HPC;

    // ---- shared memory
    const uint32_t raw_addr = smem_addr(smem_raw);
    unsigned char* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const uint32_t head_bytes = HALVES * BOX;              // one kv head's K (or V) page
    const uint32_t stage_bytes = 2 * HPC * head_bytes;     // K then V for HPC heads
    const uint32_t q_bytes = (uint32_t)(HPC * G * D * sizeof(T));   // query rows of a run
    const uint32_t row_bytes = (uint32_t)(HPC * D * sizeof(T));      // one token's K (or V) row
    unsigned char* ring = smem;
    unsigned char* qbuf = ring + (size_t)stages * stage_bytes;
    unsigned char* nbuf = qbuf + (size_t)stages * q_bytes;   // new K then V row per slot
    const uint32_t ring_addr = smem_addr(ring), nbuf_addr = smem_addr(nbuf);
    uint64_t* full = reinterpret_cast<uint64_t*>(nbuf + (size_t)stages * 2 * row_bytes);
    uint64_t* empty = full + stages;
    StreamSlot* slot = reinterpret_cast<StreamSlot*>(empty + stages);
    StreamChunk* s_chunk = reinterpret_cast<StreamChunk*>(slot + stages);
    int* s_bid = reinterpret_cast<int*>(s_chunk + kStreamBatchChunks);
    int* s_len = s_bid + kStreamBatchPages;   // clamped lengths [S]
    int* s_pref = s_len + S;                  // page prefix sums [S + 1]
    int* s_var = s_pref + S + 1;   // batch pages, abort, slots issued, queued chunks

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    __shared__ long long s_aslot[kStreamBatchChunks];   // append slot of each chunk (-1: none)

    // barriers and tensor-map prefetches first: they overlap the
    // context-length loads
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_kh);
        prefetch_tensormap(&tm_vh);
        s_var[1] = 0;   // abort
        s_var[2] = 0;   // slots issued
        for (int st = 0; st < stages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], HPC);
        }
        fence_barrier_init();
    }
    stream_layout<BS>(p, HG, s_len, s_pref, blockIdx.x == 0);   // ends with a CTA barrier
    const long long P = s_pref[S];
    const long long C = stream_shares(P, gridDim.x);
    const bool has_share = blockIdx.x < C;
    const long long P0 = has_share ? mul_div(P, blockIdx.x, C) : P;
    const long long P1 = has_share ? mul_div(P, blockIdx.x + 1, C) : P;
    const bool last_cta = blockIdx.x == C - 1;
    volatile int* s_abort = s_var + 1;

    if (warp == 0) {
        // ================= producer =================
        const uint64_t policy = l2_policy_evict_first();
        int g = 0;   // slots issued so far (lane 0)
        // walk cursor (lane 0): position x = sequence cs, head group ch, page ci
        long long x = P0;
        int cs = S, ch = 0, ci = 0;
        if (lane == 0 && P0 < P) {
            cs = stream_seq_at(s_pref, S, P0);
            const int np = (s_len[cs] + BS - 1) / BS;
            const int off = (int)(P0 - s_pref[cs]);   // positions fit 31 bits
            ch = off / np;
            ci = off - ch * np;
        }
        bool stop = false;
        while (!stop) {
            if (lane == 0) {
                int nc = 0, npg = 0;
                while (nc < kStreamBatchChunks && npg < kStreamBatchPages && x < P1) {
                    const int np = (s_len[cs] + BS - 1) / BS;
                    if (np == 0) {   // a sequence without pages (x < P1 <= P: one follows)
                        ++cs;
                        continue;
                    }
                    const long long a = s_pref[cs] + (long long)ch * np;   // the run's start
                    long long take = np - ci;
                    if (take > P1 - x) take = P1 - x;
                    if (take > kStreamBatchPages - npg) take = kStreamBatchPages - npg;
                    StreamChunk& u = s_chunk[nc++];
                    u.s = cs;
                    u.hg = ch;
                    u.i0 = ci;
                    u.n = (int)take;
                    u.flags = (ci == 0 || x == P0 ? kSlotFirst : 0) |
                              (ci + take == np || x + take == P1 ? kSlotLast : 0) |
                              (a >= P0 && a + np <= P1 ? kSlotWhole : 0) |
                              (x == P0 && ci > 0 ? kSlotHead : 0);
                    u.first = npg;
                    npg += (int)take;
                    x += take;
                    ci += (int)take;
                    if (ci == np) {
                        ci = 0;
                        if (++ch == HG) {
                            ch = 0;
                            ++cs;
                        }
                    }
                }
                s_var[3] = nc;
                s_var[0] = npg;
            }
            __syncwarp();
            const int nc = s_var[3];
            if (nc == 0) break;
            // ---- block ids of every queued page and the append slots:
            // lane l takes the batch's pages l, l + 32, ... (its chunk found
            // by a forward scan of the chunks' first offsets) and issues all
            // its loads before any store, so the batch starts after one
            // memory round trip however many chunks it holds
            const int npg = s_var[0];
            constexpr int PER_LANE = kStreamBatchPages / 32;
            int bid[PER_LANE];
            {
                int ci = 0;
#pragma unroll
                for (int j = 0; j < PER_LANE; ++j) {
                    const int f = lane + 32 * j;
                    bid[j] = -1;
                    if (f < npg) {
                        while (ci + 1 < nc && s_chunk[ci + 1].first <= f) ++ci;
                        const int s_of = s_chunk[ci].s, i_of = s_chunk[ci].i0 + (f - s_chunk[ci].first);
                        bid[j] = p.block_tables[(size_t)s_of * p.max_blocks_per_seq + i_of];
                    }
                }
            }
            // ---- fused append: the page holding a run's last token also
            // brings the token's new K and V rows of its heads (bulk copies
            // into the slot's row buffer); its consumers put them into the
            // page and write them to the pool (no other CTA reads that page),
            // so nothing waits for the pool write.  The slot of chunk ui
            // (when it ends its run) loads with the block ids.
            if (lane < nc) {
                long long sl = -1;
                if (p.slot_mapping != nullptr) {
                    const StreamChunk u = s_chunk[lane];
                    if (u.i0 + u.n == (s_len[u.s] + BS - 1) / BS) sl = p.slot_mapping[u.s];
                }
                s_aslot[lane] = sl;
            }
#pragma unroll
            for (int j = 0; j < PER_LANE; ++j) {
                const int f = lane + 32 * j;
                if (f >= npg) continue;
                int b = bid[j];
                if (b < 0 || b >= p.num_blocks) {
                    raise_error(p.errors, PKV_DEVERR_BLOCK_ID);
                    b = -1;
                }
                s_bid[f] = b;
            }
            __syncwarp();
            // ---- issue every page of the batch (lane 0)
            if (lane == 0) {
                const size_t row = (size_t)p.n_kv_heads * D;
                for (int ui = 0; ui < nc && !stop; ++ui) {
                    const StreamChunk u = s_chunk[ui];
                    const int n = s_len[u.s];
                    const T* qsrc = reinterpret_cast<const T*>(p.q) +
                                    ((size_t)u.s * p.n_heads + (size_t)u.hg * HPC * G) * D;
                    long long slot_row = s_aslot[ui];
                    if (slot_row >= (long long)p.num_blocks * BS) {
                        // outside the pool: skipped and flagged (once a sequence)
                        if (u.hg == 0) raise_error(p.errors, PKV_DEVERR_SLOT);
                        slot_row = -1;
                    }
                    for (int i = 0; i < u.n; ++i, ++g) {
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
                        const bool first = i == 0 && (u.flags & kSlotFirst);
                        const bool app = i == u.n - 1 && slot_row >= 0;
                        StreamSlot& r = slot[st];
                        r.pool_off = app ? slot_row * (long long)row + (long long)u.hg * HPC * D : -1;
                        r.s = u.s;
                        r.hg = u.hg;
                        r.page = u.i0 + i;
                        r.n_tok = n;
                        r.flags = (first ? kSlotFirst | (u.flags & kSlotHead) : 0) |
                                  (i == u.n - 1 ? (u.flags & kSlotLast) : 0) |
                                  (u.flags & kSlotWhole) | (b >= 0 ? kSlotValid : 0) |
                                  (app ? kSlotAppend : 0);
                        // a context's last block holding at most half a block
                        // of its tokens: only that half is loaded (the rows
                        // past the context are masked by the consumers)
                        const bool half = n - (u.i0 + i) * BS <= BS / 2;
                        const uint32_t kv_bytes = half ? stage_bytes / 2 : stage_bytes;
                        const uint32_t bytes = (b >= 0 ? kv_bytes : 0u) + (first ? q_bytes : 0u) +
                                               (app ? 2 * row_bytes : 0u);
                        if (bytes == 0) {
                            mbar_arrive(&full[st]);
                            continue;
                        }
                        mbar_arrive_expect_tx(&full[st], bytes);
                        if (first)
                            bulk_load_q(qbuf + (size_t)st * q_bytes, qsrc, q_bytes, &full[st],
                                        policy);
                        if (app) {
                            const size_t off = (size_t)u.s * row + (size_t)u.hg * HPC * D;
                            unsigned char* nb = nbuf + (size_t)st * 2 * row_bytes;
                            bulk_load_q(nb, static_cast<const T*>(p.k_new) + off, row_bytes,
                                        &full[st], policy);
                            bulk_load_q(nb + row_bytes, static_cast<const T*>(p.v_new) + off,
                                        row_bytes, &full[st], policy);
                        }
                        if (b >= 0) {
                            unsigned char* dst = ring + (size_t)st * stage_bytes;
                            const CUtensorMap* mk = half ? &tm_kh : &tm_k;
                            const CUtensorMap* mv = half ? &tm_vh : &tm_v;
                            for (int hh = 0; hh < HPC; ++hh) {
                                const int hrow = (u.hg * HPC + hh) * HALVES;
                                for (int h = 0; h < HALVES; ++h) {
                                    tma_load_4d(dst + hh * head_bytes + h * BOX, mk, &full[st],
                                                0, hrow + h, 0, b, policy);
                                    tma_load_4d(dst + (HPC + hh) * head_bytes + h * BOX, mv,
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
        // first, while the first pages load: the boundary record and the
        // zero rows of empty contexts
        if (threadIdx.x == 32 && p.ws_desc != nullptr && blockIdx.x + 1 < gridDim.x)
            p.ws_desc[blockIdx.x + 1] = stream_boundary_record<BS>(s_len, s_pref, S, HG, P, C,
                                                                   P0, P1, has_share);
        stream_zero_rows<D, BS, T>(p, s_len, s_pref, HG, HPC, G, P, P0, P1, last_cta,
                                   (int)threadIdx.x - 32, (int)blockDim.x - 32);
        const int kv_local = warp - 1;
        MmaHeads<D> st;
        bool head = false;   // the current piece began at the share's start
        for (int g = 0;; ++g) {
            const int slot_i = g % stages;
            if (!mbar_wait(&full[slot_i], (g / stages) & 1, p.errors)) {
                *s_abort = 1;
                break;
            }
            // the producer rewrites the record only after this slot is released
            const StreamSlot& r = slot[slot_i];
            if (r.s < 0) break;
            if (r.flags & kSlotAppend) {
                // the page's last token is this step's new row: this kv
                // head's K and V rows come from the slot's row buffer into
                // the page (row t of each swizzled box) and into the pool
                constexpr int CH = D / 8;   // 16-byte pieces of one row of one head
                if (lane < 2 * CH) {
                    const bool is_v = lane >= CH;
                    const int idx = is_v ? lane - CH : lane;
                    const uint32_t src = nbuf_addr + slot_i * 2 * row_bytes +
                                         (is_v ? row_bytes : 0u) +
                                         (uint32_t)(kv_local * D + idx * 8) * (uint32_t)sizeof(T);
                    uint32_t w0, w1, w2, w3;
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3) : "r"(src));
                    if (r.flags & kSlotValid) {
                        const int t = r.n_tok - 1 - r.page * BS;
                        const uint32_t box = ring_addr + slot_i * stage_bytes +
                                             ((is_v ? HPC : 0) + kv_local) * head_bytes +
                                             (idx >> 3) * BOX + swz(t, idx & 7);
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};"
                                     :: "r"(box), "r"(w0), "r"(w1), "r"(w2), "r"(w3) : "memory");
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    }
                    T* dst = static_cast<T*>(is_v ? p.v_pool : p.k_pool) + r.pool_off +
                             kv_local * D + idx * 8;
                    *reinterpret_cast<uint4*>(dst) = make_uint4(w0, w1, w2, w3);
                }
                __syncwarp();
            }
            if (r.flags & kSlotFirst) {
                head = (r.flags & kSlotHead) != 0;
                // query rows of this run's kv head (loaded into the slot)
                mma_heads_start<D, T>(st, reinterpret_cast<const T*>(qbuf + (size_t)slot_i * q_bytes) +
                                              (size_t)kv_local * G * D,
                                      G, lane);
            }
            if (r.flags & kSlotValid) {
                const uint32_t kbase = smem_addr(ring + (size_t)slot_i * stage_bytes +
                                                 kv_local * head_bytes);
                const uint32_t vbase = smem_addr(ring + (size_t)slot_i * stage_bytes +
                                                 (HPC + kv_local) * head_bytes);
                const int page_tok = r.page * BS;
                // one 16-token chunk at a time (32-token blocks: two chunks
                // interleaved need more than the 168 registers a thread has)
#pragma unroll 1
                for (int c = 0; c < BS / 16; ++c) {
                    const int valid = min(16, r.n_tok - (page_tok + c * 16));
                    if (valid <= 0) break;
                    mma_heads_chunk<D, T>(st, kbase, vbase, BOX, c * 16, valid, p.scale_log2,
                                          lane);
                }
            }
            if (r.flags & kSlotLast) {
                const int qh0 = (r.hg * HPC + kv_local) * G;
                if (r.flags & kSlotWhole)
                    mma_heads_finish<D>(st, p, r.s, qh0, G, 1, 0, lane);
                else
                    // slot 2c (the piece cut at the share's start) or 2c + 1
                    // (the one cut at its end), rows [kv head][query head]
                    mma_heads_partial<D>(
                        st, p.ws_o, p.ws_ml,
                        ((2 * (size_t)blockIdx.x + (head ? 0 : 1)) * HPC + kv_local) * G, 1, G,
                        lane);
            }
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

// merge_states over the pieces of a cut run, in one pass (batches of RB,
// each batch's loads issued together).  Piece 0 sits at ml / o, piece
// k >= 1 at 2k - 1 steps further (the first piece is its CTA's end piece,
// slot 2 c0 + 1; the others are start pieces, slots 2 (c0 + k)).  The
// running maximum M* is raised batch by batch
// and what was summed so far is rescaled by 2^{M*old - M*new}, the
// OnlineSoftmax recurrence applied to partial states.  With at most RB
// states (the usual two or three pieces of a run) the merge waits for one
// memory round trip.
template <int D>
__device__ __forceinline__ void merge_states_one_pass(const float* ml, size_t ml_step,
                                                      const float* o, size_t o_step, int n,
                                                      void* out, size_t out_off, int out_dtype,
                                                      int lane) {
    constexpr int DL = D / 32;
    constexpr int RB = 8;
    float acc[DL];
#pragma unroll
    for (int d = 0; d < DL; ++d) acc[d] = 0.f;
    float wsum = 0.f, mx = -INFINITY;
    for (int k0 = 0; k0 < n; k0 += RB) {
        float2 mlv[RB];
        float x[RB][DL];
#pragma unroll
        for (int u = 0; u < RB; ++u) {
            const int k = k0 + u;
            mlv[u] = make_float2(0.f, 0.f);
            if (k < n) {
                const size_t at = k == 0 ? 0 : 2 * (size_t)k - 1;
                mlv[u] = *reinterpret_cast<const float2*>(ml + at * ml_step);
                const float* ok = o + at * o_step + lane * DL;
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
        float bm = mx;
#pragma unroll
        for (int u = 0; u < RB; ++u)
            if (k0 + u < n && mlv[u].y > 0.f) bm = fmaxf(bm, mlv[u].x);
        if (bm > mx) {
            const float r = exp2f(mx - bm);   // 0 while nothing was summed
            wsum *= r;
#pragma unroll
            for (int d = 0; d < DL; ++d) acc[d] *= r;
            mx = bm;
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

// The boundary merge, launched as the stream decode's programmatic dependent
// on a grid of (C, ceil(HPC G / 4)) CTAs of four warps, C the decode's grid.
// CTA (m, y) reads the record decode CTA m - 1 left for the boundary between
// shares m - 1 and m: a run (s, hg) whose partial states lie in the n CTAs
// from c0 = m - 1 on (slot 2 c0 + 1, then slots 2 (c0 + k)).  Each warp
// merges one of the run's query heads (row 4 y + warp of the HPC x G rows)
// with the OnlineSoftmax recurrence and writes it to the output.
template <int D>
__global__ void __launch_bounds__(128)
    paged_decode_stream_merge_kernel(const __grid_constant__ DecodeParams p) {
    const int m = blockIdx.x;
    if (m == 0) return;
    const int HPC = p.heads_per_cta;
    const int G = p.group;
    const int rows = HPC * G;
    const int row = (int)blockIdx.y * 4 + (int)(threadIdx.x >> 5);
    if (row >= rows) return;
    dependency_wait();  // the decode grid's records and partial states
    const int4 d = p.ws_desc[m];
    if (d.x < 0) return;
    const int s = d.x, hg = d.y, n = d.w;
    // piece 0 in slot 2 c0 + 1, piece k >= 1 in slot 2 (c0 + k); a slot is
    // `rows` rows
    const size_t r0 = (2 * (size_t)d.z + 1) * rows + row;
    merge_states_one_pass<D>(p.ws_ml + r0 * 2, (size_t)rows * 2, p.ws_o + r0 * D,
                             (size_t)rows * D, n, p.out,
                             ((size_t)s * p.n_heads + (size_t)hg * rows + row) * D,
                             p.out_dtype, threadIdx.x & 31);
}

}  // namespace pkv
