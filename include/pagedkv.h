/*
 * pagedkv.h -- C ABI of libpagedkv.so: single-query (decode) attention over a
 * paged KV cache, the append-one-token write into the last page, and batched
 * block copy, for NVIDIA GB300 (sm_103a).
 *
 * Pages the operations come from (cited by title and section):
 *   [SWAP]   "vLLM 中 FlashAttention 与 KVCache 交换机制深度解析":
 *            the attention formula softmax(Q K^T / sqrt(d_k)) V; the
 *            OnlineSoftmax recurrence (M_new, L_new, O_new); PagedAttention
 *            pages addressed through a page table; the swap_blocks signature
 *            (src_kv_cache, dst_kv_cache, src_to_dst) and its mock.
 *   [LAYOUT] "大模型长文本推理基座从 FlashAttention 硬件加速机制到 vLLM 核心
 *            PagedAttention 显存物理布局深度剖析": section 二.2 (logical
 *            blocks of 16 tokens, block table, a new physical block appended
 *            when the last one is full) and section 三 (KVBlockManager,
 *            append_token, ref counts).
 *   [OPT]    "vLLM中FlashAttention与KVCache优化解析": "Block Table 管理",
 *            "Swap Blocks 机制" (Key and Value caches copied by separate
 *            calls) and FlashAttentionMetadata (context_lens_tensor,
 *            block_tables, max_decode_seq_len).
 *
 * Conventions for every entry point:
 *   - Buffers belong to the caller.  The library allocates no device memory
 *     and synchronises nothing unless asked to (paged_attn_decode_append_host
 *     with synchronize set; the pkv_device_errors diagnostic); all work is
 *     enqueued on `stream` (a cudaStream_t passed as void*, NULL = the legacy
 *     default stream).
 *   - "device" pointers must be device memory of the current CUDA device
 *     (or host memory the device can address, where stated).
 *   - Arguments are validated on the host before anything is launched; an
 *     invalid call returns PKV_ERR_INVALID / PKV_ERR_UNSUPPORTED and enqueues
 *     nothing.  The host never reads device arrays (block tables, lengths,
 *     slot maps, pairs); the kernels check those themselves: an out-of-range
 *     index is skipped (never dereferenced) and recorded in the device error
 *     word read by pkv_device_errors().
 *   - Launch failures return PKV_ERR_CUDA (cudaGetLastError after launch).
 *   - Per-device facts (the device error word's address, the SM count, the
 *     no-alloc scratch address) are looked up on a device's first call and
 *     kept for the life of the process.  They do not survive
 *     cudaDeviceReset: a process that resets a device must not call the
 *     library on that device again.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID = 1,      /* bad pointer, shape, alignment or range */
    PKV_ERR_UNSUPPORTED = 2,  /* valid but not compiled (head_dim, block_size, group) */
    PKV_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    PKV_ERR_WORKSPACE = 4,    /* workspace missing or smaller than required */
    PKV_ERR_NO_BLOCKS = 5     /* block manager: no free physical block */
} pkv_status;

typedef enum pkv_dtype { PKV_F16 = 0, PKV_BF16 = 1, PKV_F32 = 2 } pkv_dtype;

/* Bits of the device error word (pkv_device_errors). */
#define PKV_DEVERR_BLOCK_ID 0x1u    /* decode: block table entry outside [0, num_blocks) */
#define PKV_DEVERR_CONTEXT 0x2u     /* decode: context_len < 0, beyond the table, or beyond max_context_len */
#define PKV_DEVERR_SLOT 0x4u        /* append: slot beyond num_blocks * block_size */
#define PKV_DEVERR_PAIR 0x8u        /* copy: pair index beyond its pool */
#define PKV_DEVERR_TIMEOUT 0x10u    /* a pipeline wait gave up (should never happen) */
#define PKV_DEVERR_CONFIG 0x20u     /* inconsistent launch configuration (should never happen) */

/* Human-readable name of a status code (static string). */
PKV_API const char* pkv_status_string(pkv_status status);

/* Text of the last failure on the calling thread (validation reason or
 * CUDA error string); empty when none.  Static thread-local storage. */
PKV_API const char* pkv_last_error_detail(void);

/* Library version: major * 10000 + minor * 100 + patch. */
PKV_API int pkv_version(void);

/*
 * Launch-shape overrides, for tests and tuning sweeps only.  The library
 * picks every launch shape by itself (the values measured best on GB300);
 * nothing but pkv_set_tuning changes that choice (no environment variable
 * is read).  A knob holds PKV_TUNE_AUTO (the automatic choice) until set.
 * Knobs are process-wide and apply to every later call on every thread;
 * out-of-range values are clamped or ignored by the call that reads them,
 * never let through to a kernel.  No page has a counterpart.
 */
#define PKV_TUNE_AUTO (-2147483647 - 1)
typedef enum pkv_tune_knob {
    PKV_TUNE_DECODE_MMA = 0,      /* 0/1: tensor-core decode consumer off/on (any group) */
    PKV_TUNE_DECODE_HPC = 1,      /* kv heads per decode CTA */
    PKV_TUNE_DECODE_STAGES = 2,   /* decode ring depth, 2..8 */
    PKV_TUNE_DECODE_WPT = 3,      /* decode warps taking turns on a head's pages */
    PKV_TUNE_DECODE_QPW = 4,      /* query heads per CUDA-core consumer warp, 1/2/4 */
    PKV_TUNE_DECODE_SPLIT = 5,    /* automatic split length, tokens */
    PKV_TUNE_DECODE_ORDER = 6,    /* 0 grid order, 1 dense unit list, 2 head group fastest */
    PKV_TUNE_DECODE_PDL = 7,      /* 0: launch the split merge without programmatic overlap */
    PKV_TUNE_MQ_TC = 8,           /* 0/1: multi-query on mma.sync / tcgen05 */
    PKV_TUNE_MQ_TC_STAGES = 9,    /* tcgen05 multi-query ring depth */
    PKV_TUNE_MQ_LPT = 10,         /* 0/1: multi-query longest-context-first order off/on */
    PKV_TUNE_MQ_STAGES = 11,      /* mma.sync multi-query ring depth */
    PKV_TUNE_SWAP_BULK = 12,      /* 1: device-to-device block copy by bulk copies (default 0) */
    PKV_TUNE_SWAP_CHUNK = 13,     /* bulk block copy: bytes per copy (multiple of 16) */
    PKV_TUNE_SWAP_STAGES = 14,    /* bulk block copy: copies in flight per CTA, 2..8 */
    PKV_TUNE_SWAP_CTAS = 15,      /* bulk block copy: CTAs per SM */
    PKV_TUNE_SWAP_HINT = 16,      /* bulk block copy L2 hint: 0 none, 1 evict-first */
    PKV_TUNE_DECODE_STREAM = 17,  /* 0/1: tensor-core decode by resident CTAs taking equal
                                     page shares (automatic split only) */
    PKV_TUNE_COUNT = 18
} pkv_tune_knob;

/* Set one knob (value PKV_TUNE_AUTO restores the automatic choice).
 * PKV_ERR_INVALID for an unknown knob. */
PKV_API pkv_status pkv_set_tuning(int knob, int value);

/* Current value of a knob (PKV_TUNE_AUTO when unset or unknown). */
PKV_API int pkv_get_tuning(int knob);

/*
 * Device error word of the current device: OR of PKV_DEVERR_* bits set by
 * kernels since the last clear.  Synchronises the current device (it is a
 * diagnostic, not part of the hot path).  clear != 0 resets it to 0.
 */
PKV_API pkv_status pkv_device_errors(uint32_t* flags, int clear);

/*
 * Workspace bytes paged_attn_decode needs for the given problem and split
 * length (split_tokens = 0 means the automatic choice; the same arguments
 * must then be passed to the decode call).  Returns 0 when no workspace is
 * needed (every sequence fits one split; for the streaming decode, every
 * context fits one block).  The streaming decode's workspace holds two
 * partial states per resident CTA and does not grow with num_seqs.
 */
PKV_API size_t pkv_decode_workspace_bytes(int num_seqs, int n_heads, int n_kv_heads,
                                          int head_dim, int block_size, int max_context_len,
                                          int split_tokens);

/*
 * The split length (tokens per work unit) the automatic choice takes, for
 * the current device: 512 tokens; 1024 when max_context_len is 8192 or more
 * and there are at most 2 x SMs (sequence, kv-head group) units; the whole
 * context (no split, no merge) when the units fill the SMs 16 times over;
 * the whole context when the decode streams through resident CTAs (groups
 * of 4 or 8 query heads, 2 to 2048 sequences, max_context_len at most
 * 4096; or any group size and context length from 256 to 2048 sequences),
 * which cut the work at equal page shares
 * instead of at splits; rounded to whole blocks and capped at the context.
 * Returns 0 for an unsupported shape.
 */
PKV_API int pkv_decode_split_tokens(int num_seqs, int n_heads, int n_kv_heads, int head_dim,
                                    int block_size, int max_context_len);

/*
 * The launch shape the automatic choice (tuning knobs as currently set)
 * takes for a decode problem on a device with sm_count SMs, smem_optin
 * bytes of shared memory a block may use and smem_per_sm bytes an SM holds
 * (GB300: 152, 232448, 233472) -- host arithmetic only, no device is
 * touched, so it serves to inspect and test the choice anywhere.
 * split_tokens 0 asks for the automatic split, as in paged_attn_decode.
 * PKV_ERR_INVALID / PKV_ERR_UNSUPPORTED as paged_attn_decode would return
 * for the shape; *shape is written on PKV_OK.  No page has a counterpart.
 */
typedef struct {
    int kernel;              /* 0 CUDA-core per unit, 1 tensor-core per unit, 2 streaming */
    int split_tokens;        /* tokens per work unit (the whole context when streaming) */
    int max_splits;          /* grid extent over splits (per-unit kernels) */
    int heads_per_cta;       /* kv heads per CTA */
    int stages;              /* pages in each CTA's ring */
    int warps_per_token;     /* consumer warps taking turns on a head's pages */
    int threads;             /* threads per CTA */
    int stream_ctas;         /* streaming: the most CTAs the grid takes (else 0) */
    size_t smem_bytes;       /* dynamic shared memory per CTA */
} pkv_decode_shape;

PKV_API pkv_status pkv_decode_launch_shape(int num_seqs, int n_heads, int n_kv_heads,
                                           int head_dim, int block_size, int max_context_len,
                                           int split_tokens, int sm_count, int smem_optin,
                                           int smem_per_sm, pkv_decode_shape* shape);

/*
 * paged_attn_decode -- for every sequence s and query head h:
 *
 *     out[s,h,:] = sum_t softmax_t(scale * q[s,h,:] . K_t) * V_t,
 *     t < context_lens[s],
 *
 * where token t of sequence s lives in physical block
 * block_tables[s][t / block_size] at row t % block_size ([SWAP]
 * PagedAttention; [LAYOUT] section 二.2; [OPT] "Block Table 管理"), and
 * query head h reads KV head h / (n_heads / n_kv_heads).  Computed in one
 * pass per work unit with the [SWAP] OnlineSoftmax recurrence in fp32; long
 * contexts are cut into splits of split_tokens whose partial (M, L, O)
 * states are merged by the same recurrence in a second kernel.  A work unit
 * is (sequence, group of kv heads, split), one CTA each.  For groups of 4 or
 * 8 query heads with short contexts and split_tokens = 0 (see
 * pkv_decode_split_tokens) a grid of resident CTAs runs instead, each taking
 * an exactly equal share of all (sequence, kv-head group, block) positions;
 * a context that a share boundary cuts leaves one partial state per CTA,
 * merged by the same recurrence in a second kernel.
 *
 *   out          device, [num_seqs, n_heads, head_dim] of out_dtype
 *                (F16, BF16 or F32), written completely.  A sequence with
 *                context_len 0 gets zeros.
 *   q            device, [num_seqs, n_heads, head_dim] of kv_dtype
 *   k_pool,v_pool device, [num_blocks, block_size, n_kv_heads, head_dim] of
 *                kv_dtype (F16 or BF16), 16-byte aligned; num_blocks may be 0
 *                (then the pools may be NULL and every context must be empty)
 *   block_tables device int32 [num_seqs, max_blocks_per_seq]; only the
 *                first ceil(context_lens[s] / block_size) entries of a row
 *                are read
 *   context_lens device int32 [num_seqs]
 *   scale        multiplies q . k (normally 1/sqrt(head_dim))
 *   max_context_len  host-side upper bound of context_lens (sizes the grid;
 *                the metadata's max_decode_seq_len).  A longer context is
 *                clamped and flagged PKV_DEVERR_CONTEXT.
 *   split_tokens tokens per split (a multiple of block_size), 0 = automatic;
 *                an explicit length always selects one CTA per unit
 *   workspace    device, >= pkv_decode_workspace_bytes(...) bytes, 256-byte
 *                aligned; may be NULL when that size is 0.  Scratch only:
 *                contents on entry are ignored.
 * Supported: head_dim 64 or 128; block_size 16 or 32;
 * n_heads / n_kv_heads in {1, 2, 4, 8}.
 */
PKV_API pkv_status paged_attn_decode(void* out, pkv_dtype out_dtype, const void* q,
                                     const void* k_pool, const void* v_pool, pkv_dtype kv_dtype,
                                     const int32_t* block_tables, int max_blocks_per_seq,
                                     const int32_t* context_lens, int num_seqs, int n_heads,
                                     int n_kv_heads, int head_dim, int block_size, int num_blocks,
                                     float scale, int max_context_len, int split_tokens,
                                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * paged_attn_decode_append -- kv_append followed by paged_attn_decode, in
 * one launch: the decode CTA that reads each sequence's last block (of its
 * last split, or of its streaming share) writes k_new[s] and v_new[s]
 * ([num_seqs, n_kv_heads, head_dim] of kv_dtype, 16-byte aligned) into pool
 * row slot_mapping[s] (int64 [num_seqs], 8-byte aligned; -1 skips, a slot
 * outside the pool is skipped and flagged PKV_DEVERR_SLOT) for its kv
 * heads, and attends to them as the context's last token: slot_mapping[s]
 * must be the pool row of token context_lens[s] - 1 through the block table
 * (what the block manager's append_slots gives).  context_lens already
 * counts the appended token ([SWAP] serving loop: append, then attend; the
 * host allocator's append_slots gives both).  Same outputs and pool bytes
 * as the two calls, provided no other sequence of the call reads the page
 * holding a slot (true once shared pages are copied on write), since the
 * other sequences' CTAs do not wait for the append.  Other arguments as
 * paged_attn_decode.
 */
PKV_API pkv_status paged_attn_decode_append(
    void* out, pkv_dtype out_dtype, const void* q, void* k_pool, void* v_pool, pkv_dtype kv_dtype,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int num_seqs, int n_heads, int n_kv_heads, int head_dim, int block_size, int num_blocks,
    float scale, int max_context_len, int split_tokens, void* workspace, size_t workspace_bytes,
    const void* k_new, const void* v_new, const int64_t* slot_mapping, void* stream);

/*
 * One host-to-device copy of paged_attn_decode_append_host: `bytes` bytes
 * from host address `host` (pinned memory gives asynchronous copies) to
 * device address `device`.
 */
typedef struct {
    const void* host;
    void* device;
    size_t bytes;
} pkv_copy;

/*
 * paged_attn_decode_append_host -- one serving step from host memory in one
 * call ([SWAP] serving loop: the step's inputs arrive from the host, the
 * attention output goes back to it): on `stream`, in order,
 *   1. the n_h2d copies h2d[i] (host to device; a copy of 0 bytes is
 *      skipped), which typically move the step's q, k_new, v_new,
 *      block_tables, context_lens and slot_mapping -- packed in one staging
 *      buffer they are one copy;
 *   2. paged_attn_decode_append with the remaining arguments (all device
 *      pointers, as there);
 *   3. a device-to-host copy of the first out_bytes bytes of `out` to
 *      out_host (none when out_bytes is 0);
 *   4. with synchronize nonzero, a wait for the stream, so that out_host
 *      holds the result on return.
 * The caller owns every buffer; the host buffers must stay valid until the
 * copies complete (pinned host memory makes them asynchronous).  Invalid
 * copy arguments (a negative n_h2d, a missing list, a copy without an
 * address, out_bytes larger than `out`, a missing out_host) are refused
 * with PKV_ERR_INVALID before anything is issued; a refusal by
 * paged_attn_decode_append comes after the copies of step 1 were issued and
 * issues nothing more.
 */
PKV_API pkv_status paged_attn_decode_append_host(
    const pkv_copy* h2d, int n_h2d, void* out_host, size_t out_bytes, int synchronize,
    void* out, pkv_dtype out_dtype, const void* q, void* k_pool, void* v_pool, pkv_dtype kv_dtype,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int num_seqs, int n_heads, int n_kv_heads, int head_dim, int block_size, int num_blocks,
    float scale, int max_context_len, int split_tokens, void* workspace, size_t workspace_bytes,
    const void* k_new, const void* v_new, const int64_t* slot_mapping, void* stream);

/*
 * Batched decode -- many independent decode problems (each with its own
 * K/V pools, block tables, lengths, queries and outputs, and optionally a
 * fused append) in one launch.  The problems share the head counts,
 * head_dim, block_size and dtypes.  Plan once, run many times:
 * pkv_decode_batched_plan writes every problem's TMA maps and parameters
 * into the caller's workspace; paged_attn_decode_batched then launches from
 * it.  A plan stays valid while the problems' buffers stay at the same
 * addresses and every context stays within max_context_len; their contents
 * (queries, tables, lengths, pools, new rows) may change between runs.
 * Each problem computes exactly what paged_attn_decode (or, with
 * slot_mapping, paged_attn_decode_append) computes for it.
 */
typedef struct {
    void* out;                    /* device [num_seqs, n_heads, head_dim] of out_dtype */
    const void* q;                /* device [num_seqs, n_heads, head_dim] of kv_dtype */
    void* k_pool;                 /* device [num_blocks, block_size, n_kv_heads, head_dim] */
    void* v_pool;
    const int32_t* block_tables;  /* device int32 [num_seqs, max_blocks_per_seq] */
    const int32_t* context_lens;  /* device int32 [num_seqs] */
    const void* k_new;            /* fused append: device [num_seqs, n_kv_heads, head_dim], */
    const void* v_new;            /*   16-byte aligned, with slot_mapping; else NULL */
    const int64_t* slot_mapping;  /* device int64 [num_seqs] (-1 skips), or NULL: no append */
    int num_seqs;
    int num_blocks;
    int max_blocks_per_seq;
} pkv_decode_problem;

/* Opaque launch plan, filled by pkv_decode_batched_plan (caller-owned). */
typedef struct {
    uint64_t opaque[16];
} pkv_decode_plan;

/* Workspace bytes a batch needs (descriptors, offsets, split partials). */
PKV_API size_t pkv_decode_batched_workspace_bytes(const pkv_decode_problem* problems,
                                                  int num_problems, int n_heads, int n_kv_heads,
                                                  int head_dim, int block_size,
                                                  int max_context_len, int split_tokens);

/*
 * Validates the problems (host-side, as paged_attn_decode does), chooses
 * one launch shape for all of them and copies their descriptors into the
 * workspace (device, 256-byte aligned, >= pkv_decode_batched_workspace_bytes)
 * with cudaMemcpyAsync on `stream` from library-owned host memory (the call
 * returns once the copy is staged; it is not meant for a timed loop).
 * problems is a host array; at most 65535 sequences in total.
 */
PKV_API pkv_status pkv_decode_batched_plan(pkv_decode_plan* plan,
                                           const pkv_decode_problem* problems, int num_problems,
                                           pkv_dtype out_dtype, pkv_dtype kv_dtype, int n_heads,
                                           int n_kv_heads, int head_dim, int block_size,
                                           float scale, int max_context_len, int split_tokens,
                                           void* workspace, size_t workspace_bytes, void* stream);

/* Runs a planned batch on `stream` (one decode launch, plus the split merge
 * when a context is longer than one split). */
PKV_API pkv_status paged_attn_decode_batched(const pkv_decode_plan* plan, void* stream);

/*
 * paged_attn_decode_noalloc -- paged_attn_decode for callers that cannot
 * allocate device memory.  The pages have no counterpart: this is an
 * interface addition of this library.
 *
 * Some callers cannot hand over a workspace buffer: a serving loop that
 * reserved all of HBM for its KV pool at start-up and may not call
 * cudaMalloc again (which can also wait for the whole device), or a host
 * framework or plugin that owns the allocator and forbids allocations
 * outside it.  This entry point computes exactly what paged_attn_decode
 * computes, with the same inputs and outputs, but keeps the split partials
 * in a scratch array compiled into the library (PKV_NOALLOC_SCRATCH_BYTES
 * per device that loads it, held until exit) and allocates nothing.
 *   - A problem whose split partials need more than that
 *     (pkv_decode_workspace_bytes > PKV_NOALLOC_SCRATCH_BYTES) returns
 *     PKV_ERR_WORKSPACE before any launch.
 *   - Every call on a device shares the one array, which keeps the last
 *     call's contents (nothing in it needs to start at zero).  Calls whose
 *     kernels may overlap on the GPU (different streams without ordering)
 *     race on it.
 *   - The first call on each device looks up the array's device address;
 *     make that first call before any stream capture begins.  The address
 *     is kept for the life of the process and does not survive
 *     cudaDeviceReset (see the conventions at the top of this header).
 */
#define PKV_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
PKV_API pkv_status paged_attn_decode_noalloc(void* out, pkv_dtype out_dtype, const void* q,
                                             const void* k_pool, const void* v_pool,
                                             pkv_dtype kv_dtype, const int32_t* block_tables,
                                             int max_blocks_per_seq, const int32_t* context_lens,
                                             int num_seqs, int n_heads, int n_kv_heads,
                                             int head_dim, int block_size, int num_blocks,
                                             float scale, int max_context_len, int split_tokens,
                                             void* stream);

/*
 * paged_attn_multi_query -- several new tokens per sequence attend causally
 * to the paged context: a prefill chunk, or tokens to verify ([SWAP]: the
 * serving loop's prefill step computes attention for all of a request's
 * tokens with FlashAttention and writes their KV into pages; FlashAttention
 * tiles Q, K and V through on-chip memory with the OnlineSoftmax
 * recurrence).  Sequence s owns rows q_start[s] .. q_start[s+1]-1 of q, its
 * last q_len = q_start[s+1] - q_start[s] tokens (their K and V already in
 * the pool, e.g. by kv_append or a cache write); row i sits at position
 * p = context_lens[s] - q_len + i and attends to the keys t <= p:
 *
 *     out[row, h, :] = sum_{t <= p} softmax_t(scale * q[row, h, :] . K_t) V_t
 *
 *   out, q       device [total_q, n_heads, head_dim]; q of kv_dtype, out of
 *                out_dtype (F16, BF16, F32); 16-byte aligned
 *   q_start      device int32 [num_seqs + 1], non-decreasing, q_start[0] >= 0,
 *                q_start[num_seqs] <= total_q
 *   max_q_len    host-side bound of q_len (sizes the grid)
 *   max_context_len host-side bound of context_lens
 *   other arguments as paged_attn_decode.
 * A sequence whose q_len is negative, above its context, above max_q_len or
 * whose context exceeds max_context_len is skipped (its rows are not
 * written) and flagged PKV_DEVERR_CONTEXT.  Tensor cores: query tokens x
 * query heads of one kv head form the tile rows: on tcgen05, two tiles of
 * 128 rows per CTA with S, P and O in tensor memory, when max_q_len x group
 * >= 16 (groups of 4 and 8) or >= 48 (groups of 1 and 2), and total_q >=
 * 128 / group; else 16 rows per warp on mma.sync.
 */
PKV_API pkv_status paged_attn_multi_query(void* out, pkv_dtype out_dtype, const void* q,
                                          const int32_t* q_start, int total_q, int max_q_len,
                                          const void* k_pool, const void* v_pool,
                                          pkv_dtype kv_dtype, const int32_t* block_tables,
                                          int max_blocks_per_seq, const int32_t* context_lens,
                                          int num_seqs, int n_heads, int n_kv_heads,
                                          int head_dim, int block_size, int num_blocks,
                                          float scale, int max_context_len, void* stream);

/*
 * kv_append -- write one new token per sequence into its page
 * (reshape-and-cache; [LAYOUT] section 三 append_token):
 *
 *     k_pool[slot / block_size, slot % block_size, :, :] = k_new[s, :, :]
 *     v_pool[...same...]                                 = v_new[s, :, :]
 *
 * with slot = slot_mapping[s]; a negative slot skips the sequence, a slot
 * >= num_blocks * block_size is skipped and flagged PKV_DEVERR_SLOT.
 *   k_pool, v_pool device [num_blocks, block_size, n_kv_heads, head_dim]
 *   k_new, v_new   device [num_seqs, n_kv_heads, head_dim], same dtype
 *   slot_mapping   device int64 [num_seqs]
 * Bit-exact copy.  dtype F16, BF16 or F32; head_dim * element size must be a
 * multiple of 16 bytes and all four buffers 16-byte aligned.
 */
PKV_API pkv_status kv_append(void* k_pool, void* v_pool, const void* k_new, const void* v_new,
                             pkv_dtype dtype, const int64_t* slot_mapping, int num_seqs,
                             int n_kv_heads, int head_dim, int block_size, int num_blocks,
                             void* stream);

/*
 * swap_blocks -- batched block copy ([SWAP] swap_blocks; [OPT] "Swap Blocks
 * 机制", one call per cache: Key, then Value):
 *
 *     dst_pool[j] = src_pool[i]   for each pair (i, j) = pairs[k]
 *
 *   dst_pool  device memory, num_dst_blocks blocks of block_bytes
 *   src_pool  device memory, or pinned host memory the device can address
 *             (cudaHostAlloc / cudaHostRegister); num_src_blocks blocks
 *   pairs     int64 [n_pairs, 2] (source, destination), device memory or
 *             device-addressable pinned host memory.  A pair with a negative
 *             entry is skipped; one out of range is skipped and flagged
 *             PKV_DEVERR_PAIR.  Destinations must be distinct and must not
 *             be sources of the same call (otherwise the result is
 *             undefined).
 *   block_bytes a positive multiple of 16; both pools 16-byte aligned.
 * Bit-exact copy; bytes outside the destination blocks are not touched.
 */
PKV_API pkv_status swap_blocks(void* dst_pool, const void* src_pool, size_t block_bytes,
                               const int64_t* pairs, int n_pairs, int64_t num_src_blocks,
                               int64_t num_dst_blocks, void* stream);

/*
 * swap_blocks_kv -- swap_blocks on the Key and the Value cache in one
 * launch, with the same pairs: [SWAP] swap_blocks takes the whole KV cache
 * (src_kv_cache, dst_kv_cache) and [OPT] "Swap Blocks 机制" copies its Key
 * half and its Value half with the same src_to_dst map.  Same arguments,
 * rules and errors as swap_blocks, for two pools of equal block size.
 */
PKV_API pkv_status swap_blocks_kv(void* dst_k, void* dst_v, const void* src_k,
                                  const void* src_v, size_t block_bytes, const int64_t* pairs,
                                  int n_pairs, int64_t num_src_blocks, int64_t num_dst_blocks,
                                  void* stream);

/*
 * Host-side physical block manager ([LAYOUT] section 三 KVBlockManager):
 * a pool of num_blocks ids with reference counts.  allocate() hands out the
 * lowest free id and sets its count to 1; free() decrements a held block's
 * count and returns the id to the free set when it reaches 0;
 * add_reference() increments the count of a held block (prefix sharing,
 * [LAYOUT] section 四.2).  Plain host code; not thread-safe.
 */
typedef struct pkv_block_manager pkv_block_manager;

/* A pool with every block free.  NULL on bad arguments or no host memory. */
PKV_API pkv_block_manager* pkv_block_manager_create(int num_blocks, int block_size);
/* A pool where exactly the listed ids are free and every other block is
 * held once (to start from an existing cache state). */
PKV_API pkv_block_manager* pkv_block_manager_create_with_free(int num_blocks, int block_size,
                                                              const int32_t* free_ids,
                                                              int n_free);
PKV_API void pkv_block_manager_destroy(pkv_block_manager* mgr);
/* PKV_ERR_NO_BLOCKS (and *block_id = -1) when the pool is empty. */
PKV_API pkv_status pkv_block_allocate(pkv_block_manager* mgr, int32_t* block_id);
/* PKV_ERR_INVALID for an id outside the pool; a free block is left as is. */
PKV_API pkv_status pkv_block_free(pkv_block_manager* mgr, int32_t block_id);
/* PKV_ERR_INVALID for an id outside the pool or a block that is free. */
PKV_API pkv_status pkv_block_add_reference(pkv_block_manager* mgr, int32_t block_id);
PKV_API int pkv_block_free_count(const pkv_block_manager* mgr);
/* Reference count of a block, -1 for an id outside the pool. */
PKV_API int pkv_block_ref_count(const pkv_block_manager* mgr, int32_t block_id);
/* Writes up to `cap` free ids in increasing order; returns how many exist. */
PKV_API int pkv_block_free_ids(const pkv_block_manager* mgr, int32_t* out, int cap);

/*
 * pkv_append_slots -- one decode step's bookkeeping for every sequence, in
 * sequence order ([LAYOUT] section 三 append_token): when context_lens[s]
 * is a multiple of block_size (the last page is full, or there is none) a
 * block is allocated and written to block_tables[s][context_lens[s] /
 * block_size]; then slot_mapping[s] = block_tables[s][n / B] * B + n % B
 * for the old length n, and context_lens[s] = n + 1.  A sequence whose
 * allocation fails (pool empty) or whose table row is full gets slot -1
 * and keeps its table and length; the call then returns PKV_ERR_NO_BLOCKS
 * after processing every sequence.
 *   block_tables host int32 [num_seqs, max_blocks_per_seq], updated in place
 *   context_lens host int32 [num_seqs], updated in place
 *   slot_mapping host int64 [num_seqs], written
 */
PKV_API pkv_status pkv_append_slots(pkv_block_manager* mgr, int32_t* block_tables,
                                    int max_blocks_per_seq, int32_t* context_lens, int num_seqs,
                                    int64_t* slot_mapping);

/*
 * pkv_append_slots_cow -- pkv_append_slots with copy-on-write ([LAYOUT]
 * section 四.2: requests that share a prompt point at the same physical
 * blocks, and only a request that writes its own next token into a shared
 * block gets a private copy of it).  For a sequence whose token lands in an
 * existing block with reference count > 1, a block is allocated, the
 * sequence's reference to the shared block is dropped, the table is
 * repointed and the pair (shared, private) is appended to copy_pairs.
 * The caller copies those pairs (swap_blocks / swap_blocks_kv) before
 * kv_append writes the new tokens.
 *   copy_pairs   host int64 [num_seqs, 2], written (n_copy_pairs rows used)
 *   n_copy_pairs host int, written
 * Other arguments, updates and errors as pkv_append_slots; a table entry
 * outside the pool gives slot -1 and PKV_ERR_INVALID.
 */
PKV_API pkv_status pkv_append_slots_cow(pkv_block_manager* mgr, int32_t* block_tables,
                                        int max_blocks_per_seq, int32_t* context_lens,
                                        int num_seqs, int64_t* slot_mapping,
                                        int64_t* copy_pairs, int* n_copy_pairs);

/*
 * pkv_defrag -- plan a compaction of the pool ([SWAP]: swap_blocks also
 * serves to rearrange scattered pages into a more compact layout).  With n
 * blocks in use, every used block whose id is >= n is paired with a free
 * id < n (both taken in increasing order); the manager's counts and free set
 * and the given host block tables are updated as if the blocks had moved.
 * The caller then copies the pairs (swap_blocks / swap_blocks_kv; sources
 * and destinations are disjoint) and uploads the tables.  Afterwards the
 * used blocks are exactly [0, n).
 *   block_tables host int32 [num_seqs, max_blocks_per_seq], updated in place
 *   pairs        host int64 [cap, 2], written; *n_pairs rows used
 * PKV_ERR_INVALID if cap is too small (nothing is changed then, *n_pairs =
 * rows needed so far) or the counts are inconsistent.
 */
PKV_API pkv_status pkv_defrag(pkv_block_manager* mgr, int32_t* block_tables,
                              int max_blocks_per_seq, int num_seqs, int64_t* pairs, int cap,
                              int* n_pairs);

/*
 * Block manager on the GPU ([LAYOUT] section 三, same semantics as the host
 * manager above: reference counts, lowest free id first, sequences served in
 * order, a new block when the token count is a multiple of the block size),
 * so that a decode step's bookkeeping runs on the device without a host
 * round trip.  State, all caller-owned device memory:
 *   ref_counts int32 [num_blocks]
 *   free_ids   int32 [num_blocks]: free ids in increasing order, entries
 *              state[0] .. state[0] + state[1] - 1
 *   state      int32 [4]: head, count, sequences left without a slot by the
 *              last pkv_device_append_slots, spare
 * Calls on one state must be ordered (one stream); each is one or two
 * single-CTA kernels.
 */

/* free_ids / state from ref_counts (every id with count 0 is free). */
PKV_API pkv_status pkv_device_rebuild_free_list(const int32_t* ref_counts, int32_t* free_ids,
                                                int32_t* state, int num_blocks, void* stream);

/*
 * pkv_append_slots on the device: block_tables (int32 [num_seqs,
 * max_blocks_per_seq]), context_lens (int32 [num_seqs]) updated in place,
 * slot_mapping (int64 [num_seqs]) written; a sequence that gets no block
 * (pool empty, table row full, negative length) keeps its row and length,
 * gets slot -1 and is counted in state[2].
 */
PKV_API pkv_status pkv_device_append_slots(int32_t* ref_counts, const int32_t* free_ids,
                                           int32_t* state, int32_t* block_tables,
                                           int max_blocks_per_seq, int32_t* context_lens,
                                           int num_seqs, int block_size, int num_blocks,
                                           int64_t* slot_mapping, void* stream);

/*
 * Drop one reference per listed block id (device int32 [n_ids]; an id
 * listed twice is dropped twice, a free block stays free, an id outside the
 * pool is skipped and flagged PKV_DEVERR_PAIR), then rebuild the free list.
 */
PKV_API pkv_status pkv_device_free_blocks(int32_t* ref_counts, int32_t* free_ids, int32_t* state,
                                          const int32_t* block_ids, int n_ids, int num_blocks,
                                          void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
