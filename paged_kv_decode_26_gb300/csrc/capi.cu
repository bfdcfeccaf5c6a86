// capi.cu -- the C ABI of libpagedkv.so: host-side validation, launch
// configuration (split length, heads per CTA, pipeline depth), TMA tensor
// maps, the device error word, and the launches of the decode, split-merge,
// append and block-copy kernels (paged_attn_multi_query: multi_query_capi.cu).
// Declarations and contracts: pagedkv.h.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "capi_host.h"
#include "copy_kernels.cuh"
#include "decode_batched.cuh"
#include "decode_launch.h"
#include "decode_stream_kernel.cuh"

// ----------------------------------------------------------------- errors

// The device error word (PKV_DEVERR_* bits), one per device that loads the
// library.  Kernels get its address as a parameter.
__device__ unsigned int g_pkv_device_errors = 0;

namespace {
thread_local char t_detail[256] = "";
}  // namespace

namespace pkv {
namespace host {

void set_detail(const char* fmt, const char* what) {
    std::snprintf(t_detail, sizeof(t_detail), fmt, what);
}

pkv_status invalid(const char* why) {
    set_detail("invalid argument: %s", why);
    return PKV_ERR_INVALID;
}

pkv_status unsupported(const char* why) {
    set_detail("unsupported: %s", why);
    return PKV_ERR_UNSUPPORTED;
}

pkv_status cuda_fail(cudaError_t e) {
    set_detail("CUDA error: %s", cudaGetErrorString(e));
    return PKV_ERR_CUDA;
}

constexpr int kMaxDevices = 64;

DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

// Per-device facts, looked up once with that device current.
cudaError_t device_info(DeviceInfo** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_pkv_device_errors)) != cudaSuccess) return e;
        d.errors = static_cast<unsigned int*>(p);
        if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)))
            return e;
        if ((e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                        dev)))
            return e;
        if ((e = cudaDeviceGetAttribute(&d.smem_per_sm,
                                        cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)))
            return e;
        d.ready = true;
    }
    *out = &d;
    return cudaSuccess;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

std::atomic<int> g_tuning[PKV_TUNE_COUNT] = {};
std::once_flag g_tuning_once;

void tuning_init() {
    std::call_once(g_tuning_once, [] {
        for (auto& k : g_tuning) k.store(PKV_TUNE_AUTO, std::memory_order_relaxed);
    });
}

int tuning(pkv_tune_knob knob, int fallback) {
    tuning_init();
    const int v = g_tuning[knob].load(std::memory_order_relaxed);
    return v == PKV_TUNE_AUTO ? fallback : v;
}

bool tuned(pkv_tune_knob knob) {
    tuning_init();
    return g_tuning[knob].load(std::memory_order_relaxed) != PKV_TUNE_AUTO;
}

bool table_tokens_fit(int max_blocks_per_seq, int block_size) {
    return (long long)max_blocks_per_seq * block_size <= 0x7fffffffLL;
}

bool supported_shape(int n_heads, int n_kv_heads, int head_dim, int block_size) {
    if (n_kv_heads <= 0 || n_heads <= 0 || n_heads % n_kv_heads) return false;
    const int G = n_heads / n_kv_heads;
    return (head_dim == 64 || head_dim == 128) && (block_size == 16 || block_size == 32) &&
           (G == 1 || G == 2 || G == 4 || G == 8);
}


// The pool [num_blocks, B, Hk, D] as a 4-D tensor for TMA.
//   CUDA-core path: dims (D, Hk, B, blocks), box (D, hpc, B, 1): one page of
//     hpc heads lands as [B][hpc][D], rows unswizzled.
//   Tensor-core path: dims (64, Hk*D/64, B, blocks), box (64, 1, B, 1) with
//     128-byte swizzle: one 64-element half of one head's page per load,
//     landing as [B][64] with each 128-byte row's 16-byte chunks permuted.
cudaError_t encode_pool_map(CUtensorMap* map, const void* pool, pkv_dtype dt, int num_blocks,
                            int block_size, int n_kv_heads, int head_dim, int hpc, bool mma,
                            int box_rows) {
    auto encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t es = 2;
    const cuuint64_t inner = mma ? 64 : (cuuint64_t)head_dim;
    const cuuint64_t rows = mma ? (cuuint64_t)n_kv_heads * head_dim / 64 : (cuuint64_t)n_kv_heads;
    cuuint64_t dims[4] = {inner, rows, (cuuint64_t)block_size, (cuuint64_t)num_blocks};
    cuuint64_t strides[3] = {inner * es, (cuuint64_t)n_kv_heads * head_dim * es,
                             (cuuint64_t)block_size * n_kv_heads * head_dim * es};
    const cuuint32_t rows_per_box = box_rows > 0 ? (cuuint32_t)box_rows : (cuuint32_t)block_size;
    cuuint32_t box[4] = {(cuuint32_t)inner, mma ? 1u : (cuuint32_t)hpc, rows_per_box, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = encode(map, dt == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        4, const_cast<void*>(pool), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        mma ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}


}  // namespace host
}  // namespace pkv

using namespace pkv::host;

namespace {

// ------------------------------------------------------ decode configuration

struct DecodeConfig {
    bool mma;    // tensor-core consumer (one warp per kv head, all its query heads)
    int qpw;     // query heads per consumer warp
    int wpk;     // consumer warps per kv head, splitting its query heads
    int wpt;     // consumer warps per kv head, taking turns on its pages
    int hpc;     // kv heads per CTA
    int stages;  // ring depth
    int split_tokens;
    int max_splits;
    int max_pages;
    size_t smem;
    int threads;
    bool stream;      // tensor-core decode by resident CTAs streaming equal page shares
    int stream_ctas;  // its grid is at most this many CTAs (sizes the workspace)
};

constexpr int kDefaultSplitTokens = 512;
// The streaming decode is chosen (knob PKV_TUNE_DECODE_STREAM unset) for
// tensor-core decodes with the automatic split of two or more sequences
// whose longest context is at most this long, with a two-page ring (three
// where that costs no resident CTA, below).  Its
// equal page shares do not depend on how the lengths are spread, while one
// CTA per unit waits on the longest unit.  GB300, 32 / 8 heads, CUDA graphs
// of L2 flush + decode, streaming against one CTA per unit:
//   continuous-batching step (256 Pareto lengths, longest 1235): 21.9 / 37.5 us
//   768 / 1024 / 2048 Pareto lengths: 44.5 / 83.1, 53.8 / 107.0, 90.9 / 233.0 us
//   8 of U[1500, 3000]: 24.2 / 28.2 us; 2 of U[2000, 4096]: 21.7 / 24.6 us
//   shared-prefix GQA, log-uniform to 2048 / 4096: 57.9 / 64.3, 91.1 / 92.1 us
//   uniform batches: 128 of U[256, 2048] 106.5 / 112.5, 256 of U[2048, 4096]
//   486.7 / 473.6, 2048 of U[1, 4096] 2516 / 2452 us
// Past 4096 tokens the per-unit kernel's three-page ring wins where prefix
// blocks are shared (log-uniform to 8192: 146.7 / 133.6 us; to 32768: 427.9
// / 397.9 us), and so it does for a single sequence (U[3000, 4096]: 25.2 /
// 24.5 us).
constexpr int kStreamMaxContext = 4096;
// From this many sequences the streaming decode is taken for any group size
// (MHA and groups of 2 then run on the tensor-core consumer) and any context
// length.  Large batches are where lengths spread (continuous batching) and
// where one CTA per unit waits longest on its longest unit.  GB300, CUDA
// graphs of flush + decode, streaming against one CTA per unit:
//   GQA 32 / 8, Pareto lengths past 4K tokens: 512 seqs 32.0 / 60.3 us,
//   2048 seqs 93.1 / 226.3 us; uniform 512 of U[4096, 8192] 1888 / 1901 us,
//   1024 of U[1, 16384] 5047 / 5273 us; shared prefixes (512 seqs,
//   log-uniform to 8192) 591 / 529 us
//   MHA 32 / 32, Pareto lengths: 256 seqs 52.1 / 71.6 us, 640 seqs 104.8 /
//   197.9 us; uniform 256 of U[512, 4096] 1348 / 1298 us
constexpr int kStreamManySeqs = 256;
constexpr int kStreamStages = 2;
// Few (sequence, head-group) units with contexts of 8K tokens or more: every
// unit is cut into many pieces anyway, and at 1024 tokens a piece the GPU stays
// as full while each CTA pays its prologue and writes its partials half as
// often (GB300: 32K-token GQA and long-context decodes 1.6 % and 2.5 % faster).
// Shorter contexts lose parallelism (the 4K-token MHA decode: 1.1 % slower).
// With many units the short sequences fill the GPU by themselves and the
// longest sequence's splits set the time, so they keep 512 tokens (a
// continuous-batching decode: 41.7 us at 512, 62.6 us at 1024).
constexpr int kLongSplitTokens = 1024;
constexpr int kLongContextTokens = 8192;
constexpr int kMaxPagesPerSplit = 4096;
constexpr int kDenseMaxSeqs = 1024;


// Heads per CTA, ring depth and warp roles.  A pipeline stage holds one page
// of K and V for the CTA's kv heads: at head_dim 128, HPC = 4 heads are 512
// elements, i.e. 1 KB contiguous per token row and 32 KB (block size 16) or
// 64 KB (block size 32) per stage.  Three stages keep two CTAs (block size
// 16) or one CTA (block size 32) resident per SM with ~192 KB of loads in
// flight per SM, which measured best on GB300 for both block sizes.  At
// head_dim 64 four heads per CTA (16 KB stages, four CTAs per SM) beat
// eight (32 KB stages) on GB300: GQA 32/8 at log-uniform lengths 0.82
// against 0.64 of the copy peak, 32K-token MHA 1.045 against 1.029, the
// tiny workload's 1100 problems in one batched launch 0.89-0.91 against
// 0.87; 4K-token MHA 0.961 against 0.972.  The knobs PKV_TUNE_DECODE_HPC,
// _STAGES, _WPT and _QPW override the choice (for tuning sweeps).
constexpr int kHeadsPerCta = 4;
void shape_config_hpc(int n_heads, int n_kv_heads, int head_dim, int block_size, int hpc_target,
                      DecodeConfig* c, bool prefer_mma = false) {
    const int G = n_heads / n_kv_heads;
    // Groups of four or more query heads per kv head make each page a small
    // dense contraction: the tensor-core consumer takes them (and any group
    // when the streaming decode, which runs on it, is preferred).
    c->mma = tuning(PKV_TUNE_DECODE_MMA, G >= 4 || prefer_mma ? 1 : 0) != 0;
    if (c->mma) {
        c->qpw = G;
        c->wpk = 1;
        c->wpt = 1;
        int target = hpc_target;
        if (target < 1) target = 1;
        int hpc = 1;
        for (int h = 1; h <= n_kv_heads; ++h)
            if (n_kv_heads % h == 0 && h <= target && h <= pkv::kMmaMaxWarps) hpc = h;
        c->hpc = hpc;
        const int stages = tuning(PKV_TUNE_DECODE_STAGES, 3);
        c->stages = stages < 2 ? 2 : (stages > 8 ? 8 : stages);
        c->threads = 32 * (1 + c->hpc);
        return;
    }
    int qpw = tuning(PKV_TUNE_DECODE_QPW, G < 4 ? G : 4);
    if (qpw < 1 || qpw > 4 || (qpw & (qpw - 1)) || G % qpw) qpw = G < 4 ? G : 4;
    c->qpw = qpw;
    c->wpk = G / c->qpw;
    int target = hpc_target;
    if (target < 1) target = 1;
    int hpc = 1;
    for (int h = 1; h <= n_kv_heads; ++h)
        if (n_kv_heads % h == 0 && h <= target && h * c->wpk <= pkv::kMaxConsumerWarps) hpc = h;
    c->hpc = hpc;
    int stages = tuning(PKV_TUNE_DECODE_STAGES, 3);
    c->stages = stages < 2 ? 2 : (stages > 8 ? 8 : stages);
    // Optionally let several warps take turns on the pages of a kv head
    // (merged in shared memory at the end of the CTA).
    int wpt = tuning(PKV_TUNE_DECODE_WPT, 1);
    if (wpt < 1) wpt = 1;
    while (wpt > 1 && c->hpc * c->wpk * wpt > pkv::kMaxConsumerWarps) --wpt;
    c->wpt = wpt;
    // Page i goes to ring slot i % stages and to warp subset i % wpt.  With
    // stages a multiple of wpt every slot belongs to one subset, which then
    // waits on each phase of that slot's barrier in turn; otherwise a subset
    // would skip phases and its parity wait could match an older phase.
    c->stages = c->stages / wpt * wpt;
    if (c->stages < wpt) c->stages = wpt;
    if (c->stages < 2) c->stages = 2;
    c->threads = 32 * (1 + c->hpc * c->wpk * c->wpt);
}

void shape_config(int n_heads, int n_kv_heads, int head_dim, int block_size, DecodeConfig* c,
                  bool prefer_mma = false) {
    shape_config_hpc(n_heads, n_kv_heads, head_dim, block_size,
                     tuning(PKV_TUNE_DECODE_HPC, kHeadsPerCta), c, prefer_mma);
}

int auto_split_tokens(int num_seqs, int n_kv_heads, int hpc, int block_size, int max_context_len,
                      int sm_count) {
    const int full = ((max_context_len > 0 ? max_context_len : 1) + block_size - 1) / block_size *
                     block_size;
    const long long units = (long long)num_seqs * (n_kv_heads / hpc);
    const int sms = sm_count > 0 ? sm_count : 1;
    const int base = max_context_len >= kLongContextTokens && units <= 2LL * sms
                         ? kLongSplitTokens
                         : kDefaultSplitTokens;
    int split = tuning(PKV_TUNE_DECODE_SPLIT, base);
    split = (split + block_size - 1) / block_size * block_size;
    if (split <= 0) split = base;
    // Enough (sequence, head-group) units to fill the GPU many times over
    // without cutting the context: no split, no merge pass.
    if (units >= 16LL * sms) split = full;
    if (split > full) split = full;
    if (split / block_size > kMaxPagesPerSplit) split = kMaxPagesPerSplit * block_size;
    return split;
}

// The split merge's launch: 128 threads per CTA, allowed to start while the
// decode kernel before it on the stream still runs (the decode CTAs signal
// at their start, the merge waits for the decode grid's completion and
// memory before it reads a partial), which hides the kernel boundary.
// The PKV_TUNE_DECODE_PDL knob set to 0 launches it plainly after the decode kernel.
struct DependentLaunch {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    DependentLaunch(dim3 grid, cudaStream_t stream) {
        std::memset(&cfg, 0, sizeof(cfg));
        cfg.gridDim = grid;
        cfg.blockDim = dim3(128);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = tuning(PKV_TUNE_DECODE_PDL, 1) != 0 ? 1 : 0;
    }
};

// How decode CTAs find their work unit (DecodeParams::dense).  With 16 or
// more splits of the longest context, the dense list: where most contexts are
// shorter, most grid CTAs have no split, and placing them after the working
// ones pays (GB300, a 32K-token log-uniform GQA decode: 0.407 ms instead of
// 0.412 ms); where all are long, its head-group-fastest order reads the head
// slices of a block together (a 32K-token MHA decode: 1.231 instead of 1.269
// ms).  Fewer splits: grid order (the dense list's scan of the lengths in
// every CTA then costs more than it saves: 4K-token MHA 0.346 vs 0.341 ms).
// The PKV_TUNE_DECODE_ORDER knob (0, 1, or 2 = grid order with the head
// group fastest) forces one order.
int cta_order(int max_splits, int num_seqs) {
    const int forced = tuning(PKV_TUNE_DECODE_ORDER, -1);
    if (forced >= 0 && forced <= 2) return forced;
    return max_splits >= 16 && num_seqs <= kDenseMaxSeqs ? 1 : 0;
}

pkv_status make_config(int num_seqs, int n_heads, int n_kv_heads, int head_dim, int block_size,
                       int max_context_len, int split_tokens, int sm_count, DecodeConfig* c,
                       bool allow_stream = true, size_t smem_optin = 0, int smem_per_sm = 0) {
    const int stream_knob = tuning(PKV_TUNE_DECODE_STREAM, -1);
    // Many sequences: the streaming decode for any group size and context
    // length (on the tensor-core consumer), unless the knob says otherwise.
    const bool many = allow_stream && split_tokens == 0 && stream_knob != 0 &&
                      num_seqs >= kStreamManySeqs && num_seqs <= pkv::kStreamMaxSeqs;
    shape_config(n_heads, n_kv_heads, head_dim, block_size, c, many);
    // Too few (sequence, head-group) units to occupy the SMs: two kv heads per
    // CTA give more, shorter CTAs (measured on the tiny workload, 4 sequences
    // x 8 kv heads: 12.6 us per call instead of 14.8 us with 8 heads per CTA).
    if (!tuned(PKV_TUNE_DECODE_HPC) && c->hpc > 2 &&
        (long long)num_seqs * (n_kv_heads / c->hpc) < (sm_count > 0 ? sm_count : 1)) {
        DecodeConfig narrow;
        shape_config_hpc(n_heads, n_kv_heads, head_dim, block_size, 2, &narrow, many);
        *c = narrow;
    }
    // The whole longest context, in whole blocks.
    const long long full = ((long long)(max_context_len > 0 ? max_context_len : 1) +
                            block_size - 1) / block_size * block_size;
    // Streaming decode: the tensor-core consumer with the automatic split, at
    // most kStreamMaxSeqs sequences (their lengths live in shared memory),
    // 32-bit positions.  It cuts no context into splits (the work is cut at
    // the CTAs' shares instead), so the split length is the whole context.
    const long long all_pages = (long long)num_seqs * n_kv_heads * (full / block_size);
    c->stream = allow_stream && split_tokens == 0 && c->mma && c->wpt == 1 &&
                num_seqs <= pkv::kStreamMaxSeqs && all_pages <= 0x7fffffffLL &&
                full <= 0x7fffffffLL &&
                (stream_knob >= 0 ? stream_knob != 0
                                  : many || (num_seqs >= 2 && max_context_len <= kStreamMaxContext));
    c->stream_ctas = 0;
    if (c->stream) {
        // its shared memory must fit (the per-unit kernel runs otherwise)
        int stages = tuned(PKV_TUNE_DECODE_STAGES) ? c->stages : kStreamStages;
        const size_t limit = smem_optin > 0 ? smem_optin : (size_t)227 * 1024;
        const size_t per_sm_bytes = smem_per_sm > 0 ? (size_t)smem_per_sm : (size_t)228 * 1024;
        auto stream_smem = [&](int st) {
            return pkv::decode_stream_smem_bytes(head_dim, block_size, n_heads / n_kv_heads, 2,
                                                 c->hpc, st, num_seqs);
        };
        size_t smem = stream_smem(stages);
        // A third page in the ring where it costs no resident CTA (each CTA
        // also holds 1 KB of static shared memory and 1 KB the system
        // reserves): MHA and groups of 2 at
        // head_dim 128 with up to a few hundred sequences.  GB300, CUDA graphs
        // of flush + decode, MHA 32 heads, two pages / three: 256 Pareto
        // lengths 54.4 / 52.1 us, 384 Pareto 69.8 / 66.9 us, 320 of
        // U[512, 4096] 1828 / 1745 us, 256 of U[1, 1024] 336.4 / 318.9 us.
        if (!tuned(PKV_TUNE_DECODE_STAGES)) {
            const size_t smem3 = stream_smem(stages + 1);
            if (smem3 <= limit &&
                per_sm_bytes / (smem3 + 2048) == per_sm_bytes / (smem + 2048)) {
                stages += 1;
                smem = smem3;
            }
        }
        if (smem > limit) {
            c->stream = false;
        } else {
            c->stages = stages;
            // an upper bound of the resident CTAs (shared memory alone)
            int per_sm = (int)(per_sm_bytes / smem);
            per_sm = per_sm < 1 ? 1 : (per_sm > 32 ? 32 : per_sm);
            c->stream_ctas = (sm_count > 0 ? sm_count : 1) * per_sm;
        }
    }
    // The tensor-core consumer was taken for small groups only to stream.
    if (many && !c->stream && !tuned(PKV_TUNE_DECODE_MMA) && n_heads / n_kv_heads < 4)
        shape_config(n_heads, n_kv_heads, head_dim, block_size, c);
    if (split_tokens == 0) {
        split_tokens = c->stream ? (int)full
                                 : auto_split_tokens(num_seqs, n_kv_heads, c->hpc, block_size,
                                                     max_context_len, sm_count);
        if (split_tokens <= 0) split_tokens = block_size;
    } else if (split_tokens < 0 || split_tokens % block_size) {
        return invalid("split_tokens must be a positive multiple of block_size (or 0)");
    }
    if (!c->stream && split_tokens / block_size > kMaxPagesPerSplit)
        return invalid("split_tokens exceeds 4096 pages");
    c->split_tokens = split_tokens;
    const long long ms = ((long long)(max_context_len > 0 ? max_context_len : 0) + split_tokens - 1) /
                         split_tokens;
    c->max_splits = ms < 1 ? 1 : (int)ms;
    c->max_pages = split_tokens / block_size;
    // A grid that fits in one wave of resident CTAs: no CTA waits for a slot,
    // each waits only on its own chain of page loads and page work, so more
    // consumer warps and a deeper ring cost nothing.  Two warps take turns
    // on a kv head's pages, and the ring holds as many pages (8, 6 or 4) as
    // keep the grid in one wave.  GB300, CUDA graphs of L2 flush + decode:
    // the tiny workload 9.1 -> 7.0 us, 2 MHA sequences of 100-300 tokens
    // 11.9 -> 8.3 us, 4 of 1-2K tokens 31.0 -> 22.8 us, one of 8K tokens
    // 33.4 -> 27.9 us (256 CTAs, two per SM).
    if (!c->stream && !c->mma && !tuned(PKV_TUNE_DECODE_WPT) &&
        !tuned(PKV_TUNE_DECODE_STAGES) && c->wpt == 1 &&
        c->hpc * c->wpk * 2 <= pkv::kMaxConsumerWarps) {
        const long long ctas = (long long)num_seqs * (n_kv_heads / c->hpc) * c->max_splits;
        const size_t limit = smem_optin > 0 ? smem_optin : (size_t)227 * 1024;
        const size_t per_sm_bytes = smem_per_sm > 0 ? (size_t)smem_per_sm : (size_t)228 * 1024;
        for (int stages = 8; stages >= 4; stages -= 2) {
            const size_t smem = pkv::decode_smem_bytes(head_dim, block_size, c->qpw, 2, c->hpc,
                                                       c->wpk, 2, stages, c->max_pages);
            if (smem > limit) continue;
            const long long per_sm = (long long)(per_sm_bytes / (smem + 1024));
            if (ctas <= (long long)(sm_count > 0 ? sm_count : 1) * per_sm) {
                c->wpt = 2;
                c->stages = stages;
                c->threads = 32 * (1 + c->hpc * c->wpk * c->wpt);
                break;
            }
        }
    }
    if (c->stream)
        c->smem = pkv::decode_stream_smem_bytes(head_dim, block_size, n_heads / n_kv_heads, 2,
                                                c->hpc, c->stages, num_seqs);
    else
        c->smem = c->mma ? pkv::decode_mma_smem_bytes(head_dim, block_size, 2, c->hpc, c->stages,
                                                      c->max_pages)
                         : pkv::decode_smem_bytes(head_dim, block_size, c->qpw, 2, c->hpc,
                                                  c->wpk, c->wpt, c->stages, c->max_pages);
    return PKV_OK;
}

size_t workspace_bytes_for(int num_seqs, int n_heads, int head_dim, const DecodeConfig& c,
                           size_t* ml_offset, size_t* desc_offset = nullptr) {
    size_t units = 0;
    if (c.stream) {
        // a run of one page is never cut: no partial states
        if (c.max_pages > 1)
            units = pkv::decode_stream_partial_rows(c.stream_ctas, c.hpc, c.qpw);
    } else if (c.max_splits > 1) {
        units = (size_t)num_seqs * n_heads * c.max_splits;
    }
    if (units == 0) {
        if (ml_offset) *ml_offset = 0;
        return 0;
    }
    const size_t o_bytes = (units * head_dim * sizeof(float) + 255) / 256 * 256;
    if (ml_offset) *ml_offset = o_bytes;
    const size_t ml_bytes = units * 2 * sizeof(float);
    if (!c.stream) return o_bytes + ml_bytes;
    // then the boundary records (int4 per CTA), 16-byte aligned
    const size_t desc_at = (o_bytes + ml_bytes + 15) / 16 * 16;
    if (desc_offset) *desc_offset = desc_at;
    return desc_at + (size_t)c.stream_ctas * 16;
}

}  // namespace

namespace pkv {

// Lets other translation units of the library report a failure reason
// through pkv_last_error_detail().
void record_detail(const char* msg) { set_detail("%s", msg); }

// Address of the current device's error word (NULL if the device is unusable).
unsigned int* device_error_word() {
    DeviceInfo* d = nullptr;
    return device_info(&d) == cudaSuccess ? d->errors : nullptr;
}

cudaError_t ensure_smem_limit(const void* kernel, unsigned long long* done_mask, size_t bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (__atomic_load_n(done_mask, __ATOMIC_ACQUIRE) & bit) return cudaSuccess;
    int optin = 0;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)))
        return e;
    // The per-block limit covers the kernel's static shared memory too.
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, kernel))) return e;
    const size_t dyn_max = (size_t)optin > fa.sharedSizeBytes ? optin - fa.sharedSizeBytes : 0;
    if (bytes > dyn_max) return cudaErrorInvalidValue;
    if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)dyn_max)))
        return e;
    __atomic_fetch_or(done_mask, bit, __ATOMIC_RELEASE);
    return cudaSuccess;
}

}  // namespace pkv

// ================================================================== C ABI

extern "C" {

PKV_API const char* pkv_status_string(pkv_status status) {
    switch (status) {
        case PKV_OK: return "PKV_OK";
        case PKV_ERR_INVALID: return "PKV_ERR_INVALID";
        case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
        case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
        case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
        case PKV_ERR_NO_BLOCKS: return "PKV_ERR_NO_BLOCKS";
    }
    return "PKV_ERR_UNKNOWN";
}

PKV_API const char* pkv_last_error_detail(void) { return t_detail; }

PKV_API int pkv_version(void) { return 200; }

PKV_API pkv_status pkv_set_tuning(int knob, int value) {
    if (knob < 0 || knob >= PKV_TUNE_COUNT) return invalid("unknown tuning knob");
    tuning_init();
    g_tuning[knob].store(value, std::memory_order_relaxed);
    return PKV_OK;
}

PKV_API int pkv_get_tuning(int knob) {
    if (knob < 0 || knob >= PKV_TUNE_COUNT) return PKV_TUNE_AUTO;
    tuning_init();
    return g_tuning[knob].load(std::memory_order_relaxed);
}

PKV_API pkv_status pkv_device_errors(uint32_t* flags, int clear) {
    if (!flags) return invalid("flags is NULL");
    DeviceInfo* d = nullptr;
    cudaError_t e = device_info(&d);
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned int v = 0;
    if ((e = cudaMemcpy(&v, d->errors, sizeof(v), cudaMemcpyDeviceToHost))) return cuda_fail(e);
    *flags = v;
    if (clear) {
        if ((e = cudaMemset(d->errors, 0, sizeof(unsigned int)))) return cuda_fail(e);
        if ((e = cudaDeviceSynchronize())) return cuda_fail(e);
    }
    return PKV_OK;
}

PKV_API int pkv_decode_split_tokens(int num_seqs, int n_heads, int n_kv_heads, int head_dim,
                                    int block_size, int max_context_len) {
    if (!supported_shape(n_heads, n_kv_heads, head_dim, block_size) || num_seqs < 0) return 0;
    DeviceInfo* d = nullptr;
    const bool ok = device_info(&d) == cudaSuccess;
    DecodeConfig c;
    if (make_config(num_seqs, n_heads, n_kv_heads, head_dim, block_size, max_context_len, 0,
                    ok ? d->sm_count : 0, &c, true, ok ? (size_t)d->smem_optin : 0,
                    ok ? d->smem_per_sm : 0) != PKV_OK)
        return 0;
    return c.split_tokens;
}

PKV_API pkv_status pkv_decode_launch_shape(int num_seqs, int n_heads, int n_kv_heads,
                                           int head_dim, int block_size, int max_context_len,
                                           int split_tokens, int sm_count, int smem_optin,
                                           int smem_per_sm, pkv_decode_shape* shape) {
    if (!shape) return invalid("shape is required");
    if (num_seqs < 0 || max_context_len < 0 || sm_count < 1 || smem_optin < 1 ||
        smem_per_sm < 1)
        return invalid("negative sizes, or no SMs / shared memory");
    if (n_kv_heads <= 0 || n_heads <= 0 || n_heads % n_kv_heads)
        return invalid("n_heads must be a positive multiple of n_kv_heads");
    if (!supported_shape(n_heads, n_kv_heads, head_dim, block_size))
        return unsupported("head_dim, block_size or query-head group");
    DecodeConfig c;
    const pkv_status st = make_config(num_seqs, n_heads, n_kv_heads, head_dim, block_size,
                                      max_context_len, split_tokens, sm_count, &c, true,
                                      (size_t)smem_optin, smem_per_sm);
    if (st != PKV_OK) return st;
    if (c.smem > (size_t)smem_optin) return unsupported("shared memory of this configuration");
    shape->kernel = c.stream ? 2 : (c.mma ? 1 : 0);
    shape->split_tokens = c.split_tokens;
    shape->max_splits = c.max_splits;
    shape->heads_per_cta = c.hpc;
    shape->stages = c.stages;
    shape->warps_per_token = c.wpt;
    shape->threads = c.threads;
    shape->stream_ctas = c.stream ? c.stream_ctas : 0;
    shape->smem_bytes = c.smem;
    return PKV_OK;
}

PKV_API size_t pkv_decode_workspace_bytes(int num_seqs, int n_heads, int n_kv_heads,
                                          int head_dim, int block_size, int max_context_len,
                                          int split_tokens) {
    if (!supported_shape(n_heads, n_kv_heads, head_dim, block_size) || num_seqs < 0) return 0;
    DeviceInfo* d = nullptr;
    const bool ok = device_info(&d) == cudaSuccess;
    DecodeConfig c;
    if (make_config(num_seqs, n_heads, n_kv_heads, head_dim, block_size, max_context_len,
                    split_tokens, ok ? d->sm_count : 0, &c, true,
                    ok ? (size_t)d->smem_optin : 0, ok ? d->smem_per_sm : 0) != PKV_OK)
        return 0;
    return workspace_bytes_for(num_seqs, n_heads, head_dim, c, nullptr);
}

}  // extern "C"

namespace {

// paged_attn_decode, with the append of paged_attn_decode_append fused in
// when slot_mapping is not NULL.
pkv_status decode_impl(void* out, pkv_dtype out_dtype, const void* q, const void* k_pool,
                       const void* v_pool, pkv_dtype kv_dtype, const int32_t* block_tables,
                       int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                       int n_heads, int n_kv_heads, int head_dim, int block_size, int num_blocks,
                       float scale, int max_context_len, int split_tokens, void* workspace,
                       size_t workspace_bytes, const void* k_new, const void* v_new,
                       const int64_t* slot_mapping, void* stream) {
    // ---- host-side validation (nothing is launched on failure)
    if (num_seqs < 0) return invalid("num_seqs < 0");
    if (num_seqs > 65535) return unsupported("more than 65535 sequences per call");
    if (n_heads <= 0 || n_kv_heads <= 0 || n_heads % n_kv_heads)
        return invalid("n_heads must be a positive multiple of n_kv_heads");
    if (kv_dtype != PKV_BF16 && kv_dtype != PKV_F16) return unsupported("kv_dtype must be F16 or BF16");
    if (out_dtype != PKV_BF16 && out_dtype != PKV_F16 && out_dtype != PKV_F32)
        return invalid("out_dtype");
    if (!supported_shape(n_heads, n_kv_heads, head_dim, block_size))
        return unsupported("head_dim 64/128, block_size 16/32, group 1/2/4/8");
    if (num_blocks < 0) return invalid("num_blocks < 0");
    if (max_blocks_per_seq <= 0) return invalid("max_blocks_per_seq must be positive");
    if (!table_tokens_fit(max_blocks_per_seq, block_size))
        return unsupported("max_blocks_per_seq * block_size exceeds 2^31 - 1 tokens");
    if (max_context_len < 0) return invalid("max_context_len < 0");
    if (!std::isfinite(scale)) return invalid("scale is not finite");
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !block_tables || !context_lens)
        return invalid("a required pointer is NULL");
    if (num_blocks > 0 && (!k_pool || !v_pool)) return invalid("k_pool or v_pool is NULL");
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
        return invalid("out, q, k_pool and v_pool must be 16-byte aligned");
    if (!aligned16(block_tables) && ((uintptr_t)block_tables & 3)) return invalid("block_tables alignment");

    DeviceInfo* dev = nullptr;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return cuda_fail(e);

    DecodeConfig c;
    pkv_status st = make_config(num_seqs, n_heads, n_kv_heads, head_dim, block_size,
                                max_context_len, split_tokens, dev->sm_count, &c, true,
                                (size_t)dev->smem_optin, dev->smem_per_sm);
    if (st != PKV_OK) return st;
    if (c.smem > (size_t)dev->smem_optin) return unsupported("shared memory of this configuration");
    // The kernels clamp a context to min(table tokens, splits x split
    // length) in 32-bit arithmetic: both products must fit.
    if ((long long)c.max_splits * c.split_tokens > 0x7fffffffLL)
        return unsupported("max_context_len too close to 2^31 - 1 tokens for this split length");
    size_t ml_off = 0, desc_off = 0;
    const size_t need = workspace_bytes_for(num_seqs, n_heads, head_dim, c, &ml_off, &desc_off);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) {
            set_detail("%s", "workspace smaller than pkv_decode_workspace_bytes()");
            return PKV_ERR_WORKSPACE;
        }
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return invalid("workspace must be 256-byte aligned");
    }

    pkv::DecodeLaunch L;
    std::memset(&L, 0, sizeof(L));
    // An empty pool (every context empty) still needs well-formed maps; no
    // block id can pass the kernel's range check then, so nothing is loaded.
    const void* kmap_base = num_blocks > 0 ? k_pool : q;
    const void* vmap_base = num_blocks > 0 ? v_pool : q;
    const int map_blocks = num_blocks > 0 ? num_blocks : 1;
    if ((e = encode_pool_map(&L.tm_k, kmap_base, kv_dtype, map_blocks, block_size, n_kv_heads,
                             head_dim, c.hpc, c.mma)) != cudaSuccess)
        return cuda_fail(e);
    if ((e = encode_pool_map(&L.tm_v, vmap_base, kv_dtype, map_blocks, block_size, n_kv_heads,
                             head_dim, c.hpc, c.mma)) != cudaSuccess)
        return cuda_fail(e);
    // half-block boxes for a context's last block that it fills at most half
    if ((e = encode_pool_map(&L.tm_kh, kmap_base, kv_dtype, map_blocks, block_size, n_kv_heads,
                             head_dim, c.hpc, c.mma, block_size / 2)) != cudaSuccess ||
        (e = encode_pool_map(&L.tm_vh, vmap_base, kv_dtype, map_blocks, block_size, n_kv_heads,
                             head_dim, c.hpc, c.mma, block_size / 2)) != cudaSuccess)
        return cuda_fail(e);

    pkv::DecodeParams& p = L.p;
    p.out = out;
    p.out_dtype = out_dtype;
    p.q = q;
    p.block_tables = block_tables;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.context_lens = context_lens;
    p.num_seqs = num_seqs;
    p.n_heads = n_heads;
    p.n_kv_heads = n_kv_heads;
    p.group = n_heads / n_kv_heads;
    p.num_blocks = num_blocks;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.split_tokens = c.split_tokens;
    p.max_splits = c.max_splits;
    p.heads_per_cta = c.hpc;
    p.warps_per_kv = c.wpk;
    p.warps_per_tok = c.wpt;
    p.stages = c.stages;
    p.max_pages_per_split = c.max_pages;
    p.ws_o = need ? static_cast<float*>(workspace) : nullptr;
    p.ws_ml = need ? reinterpret_cast<float*>(static_cast<char*>(workspace) + ml_off) : nullptr;
    p.ws_desc = need && c.stream
                    ? reinterpret_cast<int4*>(static_cast<char*>(workspace) + desc_off)
                    : nullptr;
    p.errors = dev->errors;
    p.k_pool = const_cast<void*>(k_pool);
    p.v_pool = const_cast<void*>(v_pool);
    p.k_new = k_new;
    p.v_new = v_new;
    p.slot_mapping = slot_mapping;
    p.dense = cta_order(c.max_splits, num_seqs);

    L.grid = dim3((unsigned)c.max_splits, (unsigned)(n_kv_heads / c.hpc), (unsigned)num_seqs);
    L.block = dim3((unsigned)c.threads);
    L.smem_bytes = c.smem;
    L.stream = static_cast<cudaStream_t>(stream);
    L.sm_count = dev->sm_count;
    L.max_ctas = c.stream_ctas;
    if (c.max_splits > 65535 * 1024) return unsupported("context too long for the grid");

    int stream_ctas = 0;
    if (c.stream)
        e = kv_dtype == PKV_BF16
                ? pkv::launch_decode_stream_bf16(head_dim, block_size, L, &stream_ctas)
                : pkv::launch_decode_stream_f16(head_dim, block_size, L, &stream_ctas);
    else if (c.mma)
        e = kv_dtype == PKV_BF16 ? pkv::launch_decode_mma_bf16(head_dim, block_size, L)
                                 : pkv::launch_decode_mma_f16(head_dim, block_size, L);
    else
        e = kv_dtype == PKV_BF16 ? pkv::launch_decode_bf16(head_dim, block_size, c.qpw, L)
                                 : pkv::launch_decode_f16(head_dim, block_size, c.qpw, L);
    if (e != cudaSuccess) return cuda_fail(e);

    if (c.stream && need > 0) {
        // the runs cut by the stream decode's share boundaries
        const unsigned rows = (unsigned)(c.hpc * (n_heads / n_kv_heads));
        DependentLaunch dl(dim3((unsigned)stream_ctas, (rows + 3) / 4), L.stream);
        e = head_dim == 128
                ? cudaLaunchKernelEx(&dl.cfg, pkv::paged_decode_stream_merge_kernel<128>, p)
                : cudaLaunchKernelEx(&dl.cfg, pkv::paged_decode_stream_merge_kernel<64>, p);
        if (e != cudaSuccess) return cuda_fail(e);
    } else if (c.max_splits > 1) {
        pkv::ReduceParams r;
        r.out = out;
        r.out_dtype = out_dtype;
        r.context_lens = context_lens;
        r.num_seqs = num_seqs;
        r.n_heads = n_heads;
        r.split_tokens = c.split_tokens;
        r.max_splits = c.max_splits;
        r.cap_tokens = std::min((long long)max_blocks_per_seq * block_size,
                                (long long)c.max_splits * c.split_tokens) > 0x7fffffffLL
                           ? 0x7fffffff
                           : (int)std::min((long long)max_blocks_per_seq * block_size,
                                           (long long)c.max_splits * c.split_tokens);
        r.ws_o = p.ws_o;
        r.ws_ml = p.ws_ml;
        const unsigned units = (unsigned)num_seqs * (unsigned)n_heads;
        DependentLaunch dl(dim3((units + 3) / 4), L.stream);
        e = head_dim == 128 ? cudaLaunchKernelEx(&dl.cfg, pkv::paged_decode_reduce_kernel<128>, r)
                            : cudaLaunchKernelEx(&dl.cfg, pkv::paged_decode_reduce_kernel<64>, r);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return PKV_OK;
}

}  // namespace

extern "C" {

PKV_API pkv_status paged_attn_decode(void* out, pkv_dtype out_dtype, const void* q,
                                     const void* k_pool, const void* v_pool, pkv_dtype kv_dtype,
                                     const int32_t* block_tables, int max_blocks_per_seq,
                                     const int32_t* context_lens, int num_seqs, int n_heads,
                                     int n_kv_heads, int head_dim, int block_size, int num_blocks,
                                     float scale, int max_context_len, int split_tokens,
                                     void* workspace, size_t workspace_bytes, void* stream) {
    return decode_impl(out, out_dtype, q, k_pool, v_pool, kv_dtype, block_tables,
                       max_blocks_per_seq, context_lens, num_seqs, n_heads, n_kv_heads, head_dim,
                       block_size, num_blocks, scale, max_context_len, split_tokens, workspace,
                       workspace_bytes, nullptr, nullptr, nullptr, stream);
}

PKV_API pkv_status paged_attn_decode_append(
    void* out, pkv_dtype out_dtype, const void* q, void* k_pool, void* v_pool, pkv_dtype kv_dtype,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int num_seqs, int n_heads, int n_kv_heads, int head_dim, int block_size, int num_blocks,
    float scale, int max_context_len, int split_tokens, void* workspace, size_t workspace_bytes,
    const void* k_new, const void* v_new, const int64_t* slot_mapping, void* stream) {
    if (num_seqs > 0 && (!k_new || !v_new || !slot_mapping))
        return invalid("k_new, v_new and slot_mapping are required");
    if (!aligned16(k_new) || !aligned16(v_new) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return invalid("k_new and v_new must be 16-byte aligned, slot_mapping 8-byte aligned");
    return decode_impl(out, out_dtype, q, k_pool, v_pool, kv_dtype, block_tables,
                       max_blocks_per_seq, context_lens, num_seqs, n_heads, n_kv_heads, head_dim,
                       block_size, num_blocks, scale, max_context_len, split_tokens, workspace,
                       workspace_bytes, k_new, v_new, slot_mapping, stream);
}

PKV_API pkv_status paged_attn_decode_append_host(
    const pkv_copy* h2d, int n_h2d, void* out_host, size_t out_bytes, int synchronize,
    void* out, pkv_dtype out_dtype, const void* q, void* k_pool, void* v_pool, pkv_dtype kv_dtype,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int num_seqs, int n_heads, int n_kv_heads, int head_dim, int block_size, int num_blocks,
    float scale, int max_context_len, int split_tokens, void* workspace, size_t workspace_bytes,
    const void* k_new, const void* v_new, const int64_t* slot_mapping, void* stream) {
    if (n_h2d < 0 || (n_h2d > 0 && !h2d)) return invalid("h2d must list n_h2d copies");
    for (int i = 0; i < n_h2d; ++i)
        if (h2d[i].bytes > 0 && (!h2d[i].host || !h2d[i].device))
            return invalid("a host-to-device copy without a host or device address");
    if (out_bytes > 0) {
        if (!out_host || !out) return invalid("out_host and out are required when out_bytes > 0");
        const size_t es = out_dtype == PKV_F32 ? 4 : 2;
        if (num_seqs < 0 || n_heads < 0 || head_dim < 0 ||
            out_bytes > (size_t)num_seqs * n_heads * head_dim * es)
            return invalid("out_bytes exceeds the output");
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    for (int i = 0; i < n_h2d; ++i) {
        if (h2d[i].bytes == 0) continue;
        if ((e = cudaMemcpyAsync(h2d[i].device, h2d[i].host, h2d[i].bytes, cudaMemcpyHostToDevice,
                                 st)))
            return cuda_fail(e);
    }
    const pkv_status s = paged_attn_decode_append(
        out, out_dtype, q, k_pool, v_pool, kv_dtype, block_tables, max_blocks_per_seq,
        context_lens, num_seqs, n_heads, n_kv_heads, head_dim, block_size, num_blocks, scale,
        max_context_len, split_tokens, workspace, workspace_bytes, k_new, v_new, slot_mapping,
        stream);
    if (s != PKV_OK) return s;
    if (out_bytes > 0 &&
        (e = cudaMemcpyAsync(out_host, out, out_bytes, cudaMemcpyDeviceToHost, st)))
        return cuda_fail(e);
    if (synchronize && (e = cudaStreamSynchronize(st))) return cuda_fail(e);
    return PKV_OK;
}

}  // extern "C"

// ------------------------------------------------------------ batched decode

namespace {

constexpr uint32_t kPlanMagic = 0x504b5642u;

// What a plan remembers (inside the caller's pkv_decode_plan).
struct BatchPlan {
    uint32_t magic;
    int num_problems;
    int total_seqs;
    int n_heads;
    int head_dim;
    int block_size;
    int kv_dtype;
    int mma;
    int qpw;
    int groups;       // kv-head groups per sequence (n_kv_heads / heads per CTA)
    int max_splits;
    int threads;
    size_t smem;
    char* workspace;
    size_t seq_off;
};
static_assert(sizeof(BatchPlan) <= sizeof(pkv_decode_plan), "pkv_decode_plan is too small");

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Workspace of a batch: the problems' descriptors, the sequence offsets,
// then each problem's split partials (O, then (M, L)) when contexts split.
struct BatchLayout {
    size_t seq_off;
    size_t parts_off;
    size_t total;
};

BatchLayout batch_layout(const pkv_decode_problem* problems, int num_problems, int n_heads,
                         int head_dim, const DecodeConfig& c) {
    BatchLayout l;
    l.seq_off = align256((size_t)num_problems * sizeof(pkv::BatchedProblem));
    l.parts_off = l.seq_off + align256((size_t)(num_problems + 1) * sizeof(int));
    size_t t = l.parts_off;
    if (c.max_splits > 1)
        for (int i = 0; i < num_problems; ++i) {
            const size_t units =
                (size_t)std::max(problems[i].num_seqs, 0) * n_heads * c.max_splits;
            t += align256(units * head_dim * sizeof(float)) + align256(units * 2 * sizeof(float));
        }
    l.total = t;
    return l;
}

long long total_seqs_of(const pkv_decode_problem* problems, int num_problems) {
    long long t = 0;
    for (int i = 0; i < num_problems; ++i) t += std::max(problems[i].num_seqs, 0);
    return t;
}

}  // namespace

extern "C" {

PKV_API size_t pkv_decode_batched_workspace_bytes(const pkv_decode_problem* problems,
                                                  int num_problems, int n_heads, int n_kv_heads,
                                                  int head_dim, int block_size,
                                                  int max_context_len, int split_tokens) {
    if (num_problems < 0 || (num_problems > 0 && !problems) ||
        !supported_shape(n_heads, n_kv_heads, head_dim, block_size) || max_context_len < 0)
        return 0;
    DeviceInfo* dev = nullptr;
    if (device_info(&dev) != cudaSuccess) return 0;
    const long long total = total_seqs_of(problems, num_problems);
    DecodeConfig c;
    if (make_config((int)std::min(total, 65535LL), n_heads, n_kv_heads, head_dim, block_size,
                    max_context_len, split_tokens, dev->sm_count, &c, false) != PKV_OK)
        return 0;
    return batch_layout(problems, num_problems, n_heads, head_dim, c).total;
}

PKV_API pkv_status pkv_decode_batched_plan(pkv_decode_plan* plan,
                                           const pkv_decode_problem* problems, int num_problems,
                                           pkv_dtype out_dtype, pkv_dtype kv_dtype, int n_heads,
                                           int n_kv_heads, int head_dim, int block_size,
                                           float scale, int max_context_len, int split_tokens,
                                           void* workspace, size_t workspace_bytes, void* stream) {
    if (!plan) return invalid("plan is NULL");
    std::memset(plan, 0, sizeof(*plan));
    if (num_problems < 0 || (num_problems > 0 && !problems)) return invalid("problems");
    if (kv_dtype != PKV_BF16 && kv_dtype != PKV_F16) return unsupported("kv_dtype must be F16 or BF16");
    if (out_dtype != PKV_BF16 && out_dtype != PKV_F16 && out_dtype != PKV_F32)
        return invalid("out_dtype");
    if (!supported_shape(n_heads, n_kv_heads, head_dim, block_size))
        return unsupported("head_dim 64/128, block_size 16/32, group 1/2/4/8");
    if (max_context_len < 0) return invalid("max_context_len < 0");
    if (!std::isfinite(scale)) return invalid("scale is not finite");
    const long long total = total_seqs_of(problems, num_problems);
    if (total > 65535) return unsupported("more than 65535 sequences per batch");
    for (int i = 0; i < num_problems; ++i) {
        const pkv_decode_problem& q = problems[i];
        if (q.num_seqs < 0 || q.num_blocks < 0) return invalid("problem sizes");
        if (q.num_seqs == 0) continue;
        if (q.max_blocks_per_seq <= 0) return invalid("max_blocks_per_seq must be positive");
        if (!q.out || !q.q || !q.block_tables || !q.context_lens)
            return invalid("a problem's required pointer is NULL");
        if (q.num_blocks > 0 && (!q.k_pool || !q.v_pool)) return invalid("a problem's pool is NULL");
        if (!aligned16(q.out) || !aligned16(q.q) || !aligned16(q.k_pool) || !aligned16(q.v_pool))
            return invalid("out, q, k_pool and v_pool must be 16-byte aligned");
        if (q.slot_mapping &&
            (!q.k_new || !q.v_new || !aligned16(q.k_new) || !aligned16(q.v_new) ||
             (reinterpret_cast<uintptr_t>(q.slot_mapping) & 7u)))
            return invalid("a problem's append rows are NULL or misaligned");
    }
    DeviceInfo* dev = nullptr;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    DecodeConfig c;
    pkv_status st = make_config((int)std::max(total, 1LL), n_heads, n_kv_heads, head_dim,
                                block_size, max_context_len, split_tokens, dev->sm_count, &c,
                                false);
    if (st != PKV_OK) return st;
    if (c.smem > (size_t)dev->smem_optin) return unsupported("shared memory of this configuration");
    if (c.max_splits > 65535) return unsupported("more than 65535 splits per sequence");
    if ((long long)c.max_splits * c.split_tokens > 0x7fffffffLL)
        return unsupported("max_context_len too close to 2^31 - 1 tokens for this split length");
    for (int i = 0; i < num_problems; ++i)
        if (!table_tokens_fit(std::max(problems[i].max_blocks_per_seq, 1), block_size))
            return unsupported("max_blocks_per_seq * block_size exceeds 2^31 - 1 tokens");
    const BatchLayout lay = batch_layout(problems, num_problems, n_heads, head_dim, c);
    if (!workspace || workspace_bytes < lay.total) {
        set_detail("%s", "workspace smaller than pkv_decode_batched_workspace_bytes()");
        return PKV_ERR_WORKSPACE;
    }
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return invalid("workspace must be 256-byte aligned");

    char* ws = static_cast<char*>(workspace);
    std::vector<pkv::BatchedProblem> hp((size_t)num_problems);
    std::vector<int> seq_begin((size_t)num_problems + 1, 0);
    size_t part = lay.parts_off;
    const int cap_tokens =
        (int)std::min(0x7fffffffLL, (long long)c.max_splits * c.split_tokens);
    for (int i = 0; i < num_problems; ++i) {
        const pkv_decode_problem& q = problems[i];
        pkv::BatchedProblem& b = hp[(size_t)i];
        std::memset(&b, 0, sizeof(b));
        seq_begin[(size_t)i + 1] = seq_begin[(size_t)i] + std::max(q.num_seqs, 0);
        // an empty pool (or problem) still gets well-formed maps; no block id
        // passes the kernel's range check then, so nothing is loaded
        const void* kb = q.num_blocks > 0 ? q.k_pool : (q.q ? q.q : workspace);
        const void* vb = q.num_blocks > 0 ? q.v_pool : (q.q ? q.q : workspace);
        const int mb = q.num_blocks > 0 ? q.num_blocks : 1;
        if ((e = encode_pool_map(&b.tm_k, kb, kv_dtype, mb, block_size, n_kv_heads, head_dim,
                                 c.hpc, c.mma)) != cudaSuccess ||
            (e = encode_pool_map(&b.tm_v, vb, kv_dtype, mb, block_size, n_kv_heads, head_dim,
                                 c.hpc, c.mma)) != cudaSuccess ||
            (e = encode_pool_map(&b.tm_kh, kb, kv_dtype, mb, block_size, n_kv_heads, head_dim,
                                 c.hpc, c.mma, block_size / 2)) != cudaSuccess ||
            (e = encode_pool_map(&b.tm_vh, vb, kv_dtype, mb, block_size, n_kv_heads, head_dim,
                                 c.hpc, c.mma, block_size / 2)) != cudaSuccess)
            return cuda_fail(e);
        pkv::DecodeParams& p = b.p;
        p.out = q.out;
        p.out_dtype = out_dtype;
        p.q = q.q;
        p.block_tables = q.block_tables;
        p.max_blocks_per_seq = std::max(q.max_blocks_per_seq, 1);
        p.context_lens = q.context_lens;
        p.num_seqs = q.num_seqs;
        p.n_heads = n_heads;
        p.n_kv_heads = n_kv_heads;
        p.group = n_heads / n_kv_heads;
        p.num_blocks = q.num_blocks;
        p.scale_log2 = scale * 1.4426950408889634f;
        p.split_tokens = c.split_tokens;
        p.max_splits = c.max_splits;
        p.heads_per_cta = c.hpc;
        p.warps_per_kv = c.wpk;
        p.warps_per_tok = c.wpt;
        p.stages = c.stages;
        p.max_pages_per_split = c.max_pages;
        p.errors = dev->errors;
        p.k_pool = q.k_pool;
        p.v_pool = q.v_pool;
        p.k_new = q.k_new;
        p.v_new = q.v_new;
        p.slot_mapping = q.slot_mapping;
        p.dense = 0;  // the batched kernels map CTAs to problems by grid z
        if (c.max_splits > 1) {
            const size_t units = (size_t)std::max(q.num_seqs, 0) * n_heads * c.max_splits;
            p.ws_o = reinterpret_cast<float*>(ws + part);
            part += align256(units * head_dim * sizeof(float));
            p.ws_ml = reinterpret_cast<float*>(ws + part);
            part += align256(units * 2 * sizeof(float));
        }
        pkv::ReduceParams& r = b.r;
        r.out = q.out;
        r.out_dtype = out_dtype;
        r.context_lens = q.context_lens;
        r.num_seqs = q.num_seqs;
        r.n_heads = n_heads;
        r.split_tokens = c.split_tokens;
        r.max_splits = c.max_splits;
        r.cap_tokens = (int)std::min((long long)p.max_blocks_per_seq * block_size,
                                     (long long)cap_tokens);
        r.ws_o = p.ws_o;
        r.ws_ml = p.ws_ml;
    }
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (num_problems > 0) {
        if ((e = cudaMemcpyAsync(ws, hp.data(), hp.size() * sizeof(pkv::BatchedProblem),
                                 cudaMemcpyHostToDevice, cs)) != cudaSuccess ||
            (e = cudaMemcpyAsync(ws + lay.seq_off, seq_begin.data(),
                                 seq_begin.size() * sizeof(int), cudaMemcpyHostToDevice, cs)) !=
                cudaSuccess)
            return cuda_fail(e);
    }
    BatchPlan* bp = reinterpret_cast<BatchPlan*>(plan);
    bp->magic = kPlanMagic;
    bp->num_problems = num_problems;
    bp->total_seqs = (int)total;
    bp->n_heads = n_heads;
    bp->head_dim = head_dim;
    bp->block_size = block_size;
    bp->kv_dtype = kv_dtype;
    bp->mma = c.mma ? 1 : 0;
    bp->qpw = c.qpw;
    bp->groups = n_kv_heads / c.hpc;
    bp->max_splits = c.max_splits;
    bp->threads = c.threads;
    bp->smem = c.smem;
    bp->workspace = ws;
    bp->seq_off = lay.seq_off;
    return PKV_OK;
}

PKV_API pkv_status paged_attn_decode_batched(const pkv_decode_plan* plan, void* stream) {
    const BatchPlan* bp = reinterpret_cast<const BatchPlan*>(plan);
    if (!bp || bp->magic != kPlanMagic) return invalid("not a plan from pkv_decode_batched_plan");
    if (bp->total_seqs == 0) return PKV_OK;
    pkv::BatchedLaunch L;
    L.probs = reinterpret_cast<const pkv::BatchedProblem*>(bp->workspace);
    L.seq_begin = reinterpret_cast<const int*>(bp->workspace + bp->seq_off);
    L.num_problems = bp->num_problems;
    L.grid = dim3((unsigned)bp->max_splits, (unsigned)bp->groups, (unsigned)bp->total_seqs);
    L.block = dim3((unsigned)bp->threads);
    L.smem_bytes = bp->smem;
    L.stream = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (bp->mma)
        e = bp->kv_dtype == PKV_BF16
                ? pkv::launch_decode_mma_batched_bf16(bp->head_dim, bp->block_size, L)
                : pkv::launch_decode_mma_batched_f16(bp->head_dim, bp->block_size, L);
    else
        e = bp->kv_dtype == PKV_BF16
                ? pkv::launch_decode_batched_bf16(bp->head_dim, bp->block_size, bp->qpw, L)
                : pkv::launch_decode_batched_f16(bp->head_dim, bp->block_size, bp->qpw, L);
    if (e != cudaSuccess) return cuda_fail(e);
    if (bp->max_splits > 1) {
        const unsigned units = (unsigned)bp->total_seqs * (unsigned)bp->n_heads;
        DependentLaunch dl(dim3((units + 3) / 4), L.stream);
        const pkv::BatchedProblem* probs = L.probs;
        const int* seq_begin = L.seq_begin;
        e = bp->head_dim == 128
                ? cudaLaunchKernelEx(&dl.cfg, pkv::paged_decode_batched_reduce_kernel<128>, probs,
                                     seq_begin, L.num_problems, bp->n_heads)
                : cudaLaunchKernelEx(&dl.cfg, pkv::paged_decode_batched_reduce_kernel<64>, probs,
                                     seq_begin, L.num_problems, bp->n_heads);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return PKV_OK;
}

PKV_API pkv_status kv_append(void* k_pool, void* v_pool, const void* k_new, const void* v_new,
                             pkv_dtype dtype, const int64_t* slot_mapping, int num_seqs,
                             int n_kv_heads, int head_dim, int block_size, int num_blocks,
                             void* stream) {
    if (num_seqs < 0 || n_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks < 0)
        return invalid("sizes");
    int es = 0;
    switch (dtype) {
        case PKV_F16:
        case PKV_BF16: es = 2; break;
        case PKV_F32: es = 4; break;
        default: return invalid("dtype");
    }
    const long long row_bytes = (long long)n_kv_heads * head_dim * es;
    if (row_bytes % 16) return unsupported("n_kv_heads * head_dim * element size must be a multiple of 16 bytes");
    if (num_seqs == 0) return PKV_OK;
    if (!k_pool || !v_pool || !k_new || !v_new || !slot_mapping) return invalid("NULL pointer");
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_new) || !aligned16(v_new))
        return invalid("buffers must be 16-byte aligned");
    if (((uintptr_t)slot_mapping & 7) != 0) return invalid("slot_mapping must be 8-byte aligned");
    if (row_bytes / 16 > 0x7fffffffLL) return unsupported("row too large");
    DeviceInfo* dev = nullptr;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    const int row_vec = (int)(row_bytes / 16);
    const long long total = (long long)num_seqs * row_vec;
    long long blocks = (total + 255) / 256;
    const long long cap = 8LL * dev->sm_count;
    if (blocks > cap) blocks = cap;
    pkv::kv_append_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool),
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping,
        num_seqs, row_vec, (int64_t)num_blocks * block_size, dev->errors);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
    return PKV_OK;
}

}  // extern "C"

namespace {

// Whether a block copy takes the copy-engine path (cp.async.bulk through
// shared memory): only on request (the PKV_TUNE_SWAP_BULK knob), and only
// with device memory of the current device on both sides of every pool.
// By default the copy is the 16-byte load/store kernel, which measured
// ahead on GB300 (32 KB blocks, K and V, L2 cleared by a read before each
// call: 1024 pairs 23.2 us for both; 8192 pairs 0.974 of the copy peak
// against 0.939-0.950 for every bulk launch shape tried, and 0.88 against
// 0.82-0.83 back to back).  A source in pinned host memory (or on another
// device) always takes the load/store kernel, which reaches it through
// unified addressing.
bool use_bulk_copy(void* const* dst_pools, const void* const* src_pools, int n_pools) {
    if (tuning(PKV_TUNE_SWAP_BULK, 0) == 0) return false;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    for (int k = 0; k < n_pools; ++k) {
        for (const void* ptr : {static_cast<const void*>(dst_pools[k]), src_pools[k]}) {
            cudaPointerAttributes a;
            if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
                (void)cudaGetLastError();
                return false;
            }
            if (a.type != cudaMemoryTypeDevice || a.device != dev) return false;
        }
    }
    return true;
}

pkv_status launch_swap(void* const* dst_pools, const void* const* src_pools, int n_pools,
                       size_t block_bytes, const int64_t* pairs, int n_pairs,
                       int64_t num_src_blocks, int64_t num_dst_blocks, void* stream) {
    if (n_pairs < 0 || num_src_blocks < 0 || num_dst_blocks < 0) return invalid("sizes");
    if (block_bytes == 0 || block_bytes % 16)
        return invalid("block_bytes must be a positive multiple of 16");
    if (n_pairs == 0) return PKV_OK;
    if (!pairs) return invalid("NULL pointer");
    pkv::SwapPools pools;
    for (int k = 0; k < n_pools; ++k) {
        if (!dst_pools[k] || !src_pools[k]) return invalid("NULL pointer");
        if (!aligned16(dst_pools[k]) || !aligned16(src_pools[k]))
            return invalid("pools must be 16-byte aligned");
        pools.dst[k] = static_cast<uint4*>(dst_pools[k]);
        pools.src[k] = static_cast<const uint4*>(src_pools[k]);
    }
    if (((uintptr_t)pairs & 7) != 0) return invalid("pairs must be 8-byte aligned");
    DeviceInfo* dev = nullptr;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (use_bulk_copy(dst_pools, src_pools, n_pools)) {
        pkv::BulkSwapParams p;
        p.pools = pools;
        p.pairs = pairs;
        p.n_pairs = n_pairs;
        p.num_src = num_src_blocks;
        p.num_dst = num_dst_blocks;
        p.block_bytes = block_bytes;
        // One bulk copy moves a chunk of up to 32 KB (a whole block of the
        // 16-token, 8-head, d = 128 bf16 pools); three chunks in flight per
        // CTA and two CTAs per SM keep ~192 KB per SM moving.
        long long chunk = tuning(PKV_TUNE_SWAP_CHUNK, 32768);
        chunk = std::max(16LL, std::min(chunk, 65536LL)) / 16 * 16;
        if ((unsigned long long)chunk > block_bytes) chunk = (long long)block_bytes;
        int stages = std::max(2, std::min(tuning(PKV_TUNE_SWAP_STAGES, 3), pkv::kMaxBulkStages));
        while (stages > 2 && (size_t)stages * chunk > (size_t)dev->smem_optin - 4096) --stages;
        const int ctas = std::max(1, std::min(tuning(PKV_TUNE_SWAP_CTAS, 2), 32));
        p.chunk_bytes = (uint32_t)chunk;
        p.chunks = (int)((block_bytes + chunk - 1) / chunk);
        p.n_pools = n_pools;
        p.stages = stages;
        p.hint = tuning(PKV_TUNE_SWAP_HINT, 1) != 0 ? 1 : 0;
        p.errors = dev->errors;
        const size_t smem = (size_t)stages * chunk;
        static unsigned long long smem_done = 0;
        if ((e = pkv::ensure_smem_limit((const void*)pkv::swap_blocks_bulk_kernel, &smem_done,
                                        smem)) != cudaSuccess)
            return cuda_fail(e);
        const long long items = (long long)n_pairs * n_pools * p.chunks;
        const long long grid = std::min(items, (long long)dev->sm_count * ctas);
        pkv::swap_blocks_bulk_kernel<<<(unsigned)grid, 32, smem,
                                       static_cast<cudaStream_t>(stream)>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
        return PKV_OK;
    }
    const dim3 grid((unsigned)std::min<long long>(n_pairs, 1LL << 20), (unsigned)n_pools);
    pkv::swap_blocks_kernel<<<grid, pkv::kSwapThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        pools, (int64_t)(block_bytes / 16), pairs, n_pairs, num_src_blocks, num_dst_blocks,
        dev->errors);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
    return PKV_OK;
}

}  // namespace

extern "C" {

PKV_API pkv_status swap_blocks(void* dst_pool, const void* src_pool, size_t block_bytes,
                               const int64_t* pairs, int n_pairs, int64_t num_src_blocks,
                               int64_t num_dst_blocks, void* stream) {
    void* dst[1] = {dst_pool};
    const void* src[1] = {src_pool};
    return launch_swap(dst, src, 1, block_bytes, pairs, n_pairs, num_src_blocks, num_dst_blocks,
                       stream);
}

PKV_API pkv_status swap_blocks_kv(void* dst_k, void* dst_v, const void* src_k,
                                  const void* src_v, size_t block_bytes, const int64_t* pairs,
                                  int n_pairs, int64_t num_src_blocks, int64_t num_dst_blocks,
                                  void* stream) {
    void* dst[2] = {dst_k, dst_v};
    const void* src[2] = {src_k, src_v};
    return launch_swap(dst, src, 2, block_bytes, pairs, n_pairs, num_src_blocks, num_dst_blocks,
                       stream);
}

}  // extern "C"
