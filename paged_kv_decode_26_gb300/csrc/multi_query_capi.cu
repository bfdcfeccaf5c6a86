// multi_query_capi.cu -- paged_attn_multi_query of the C ABI: validation,
// the choice between the tcgen05 kernel (two query tiles of 128 rows per
// CTA) and the mma.sync kernel (16 rows per warp), tensor maps and launch.
// Declarations and contracts: pagedkv.h.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>

#include "capi_host.h"
#include "decode_launch.h"
#include "multi_query_tc_kernel.cuh"

using namespace pkv::host;

namespace {

// Every CTA of the tcgen05 kernel ranks the sequences by context length
// (S^2 / 352 comparisons per thread), so only up to this many.
constexpr int kLptMaxSeqs = 256;
constexpr int kLptMinContext = 8192;

// The queries [total_q, n_heads, D] as a 4-D tensor for the tcgen05
// multi-query kernel: dims (64, D/64, n_heads, total_q), box (64, 1, G, 128/G)
// with 128-byte swizzle, so one load per 64-element half brings the 128 rows
// (token, head of the group) of a query tile as [128][64], K-major.
cudaError_t encode_query_map(CUtensorMap* map, const void* q, pkv_dtype dt, int total_q,
                             int n_heads, int head_dim, int group) {
    auto encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t es = 2;
    cuuint64_t dims[4] = {64, (cuuint64_t)head_dim / 64, (cuuint64_t)n_heads, (cuuint64_t)total_q};
    cuuint64_t strides[3] = {64 * es, (cuuint64_t)head_dim * es,
                             (cuuint64_t)n_heads * head_dim * es};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)group, (cuuint32_t)(128 / group)};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = encode(map, dt == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        4, const_cast<void*>(q), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

extern "C" {

PKV_API pkv_status paged_attn_multi_query(void* out, pkv_dtype out_dtype, const void* q,
                                          const int32_t* q_start, int total_q, int max_q_len,
                                          const void* k_pool, const void* v_pool,
                                          pkv_dtype kv_dtype, const int32_t* block_tables,
                                          int max_blocks_per_seq, const int32_t* context_lens,
                                          int num_seqs, int n_heads, int n_kv_heads,
                                          int head_dim, int block_size, int num_blocks,
                                          float scale, int max_context_len, void* stream) {
    if (num_seqs < 0 || total_q < 0 || max_q_len < 0 || max_context_len < 0)
        return invalid("sizes");
    if (num_seqs > 65535) return unsupported("more than 65535 sequences per call");
    if (n_heads <= 0 || n_kv_heads <= 0 || n_heads % n_kv_heads)
        return invalid("n_heads must be a positive multiple of n_kv_heads");
    if (kv_dtype != PKV_BF16 && kv_dtype != PKV_F16) return unsupported("kv_dtype must be F16 or BF16");
    if (out_dtype != PKV_BF16 && out_dtype != PKV_F16 && out_dtype != PKV_F32)
        return invalid("out_dtype");
    if (!supported_shape(n_heads, n_kv_heads, head_dim, block_size))
        return unsupported("head_dim 64/128, block_size 16/32, group 1/2/4/8");
    if (num_blocks < 0 || max_blocks_per_seq <= 0) return invalid("pool / table sizes");
    if (!table_tokens_fit(max_blocks_per_seq, block_size))
        return unsupported("max_blocks_per_seq * block_size exceeds 2^31 - 1 tokens");
    if (!std::isfinite(scale)) return invalid("scale is not finite");
    if (num_seqs == 0 || total_q == 0 || max_q_len == 0) return PKV_OK;
    if (!out || !q || !q_start || !block_tables || !context_lens) return invalid("NULL pointer");
    if (num_blocks > 0 && (!k_pool || !v_pool)) return invalid("k_pool or v_pool is NULL");
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
        return invalid("out, q, k_pool and v_pool must be 16-byte aligned");
    const long long max_pages_ll = ((long long)max_context_len + block_size - 1) / block_size;
    if (max_pages_ll > max_blocks_per_seq || max_pages_ll > 16384)
        return invalid("max_context_len beyond the block table (or 16384 pages)");
    const int max_pages = (int)(max_pages_ll > 0 ? max_pages_ll : 1);
    DeviceInfo* dev = nullptr;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return cuda_fail(e);

    const int G = n_heads / n_kv_heads;
    const void* kmap_base = num_blocks > 0 ? k_pool : q;
    const void* vmap_base = num_blocks > 0 ? v_pool : q;
    const int map_blocks = num_blocks > 0 ? num_blocks : 1;

    // tcgen05 path: two query tiles of 128 rows (128/G tokens x G heads) per
    // CTA; the PKV_TUNE_MQ_TC knob forces it off/on where it applies.
    {
        const int tc_tokens = pkv::kTcRows / G;
        // Measured crossover (GB300): with groups of 4 the tcgen05 kernel wins
        // from 4-token chunks (16 rows); with groups of 1 the mma.sync kernel
        // wins up to 32 tokens and tcgen05 from 48.
        int want = tuning(PKV_TUNE_MQ_TC, -1);
        if (want < 0) {
            const long long rows = (long long)max_q_len * G;
            want = (G >= 4 ? rows >= 16 : rows >= 48) ? 1 : 0;
        }
        int stages = tuning(PKV_TUNE_MQ_TC_STAGES, head_dim == 64 ? 6 : 4);
        stages = stages < 2 ? 2 : (stages > 8 ? 8 : stages);
        // Longest context first (see longest_first) for batches small enough
        // to rank in every CTA, and only with contexts of 8K tokens or more:
        // the ranking adds ~1 us to each CTA's prologue (one CTA per SM, so
        // nothing hides it), which long CTAs absorb.  GB300, 256-token
        // chunks: log-uniform [128, 32768] contexts 3.409 -> 3.215 ms;
        // uniform [512, 4096] 0.729 -> 0.744 ms, hence the threshold.
        // The PKV_TUNE_MQ_LPT knob (0 / 1) forces index order / longest first.
        const int lpt_env = tuning(PKV_TUNE_MQ_LPT, -1);
        const bool lpt_on = lpt_env >= 0 ? lpt_env != 0 : max_context_len >= kLptMinContext;
        const int lpt = lpt_on && num_seqs <= kLptMaxSeqs ? num_seqs : 0;
        while (stages > 2 && pkv::multi_query_tc_smem_bytes(head_dim, stages, max_pages, lpt) >
                                 (size_t)dev->smem_optin)
            --stages;
        const size_t smem = pkv::multi_query_tc_smem_bytes(head_dim, stages, max_pages, lpt);
        if (want && total_q >= tc_tokens && smem <= (size_t)dev->smem_optin) {
            pkv::MultiQueryLaunch L;
            std::memset(&L, 0, sizeof(L));
            if ((e = encode_query_map(&L.tm_q, q, kv_dtype, total_q, n_heads, head_dim, G)) !=
                cudaSuccess)
                return cuda_fail(e);
            if ((e = encode_pool_map(&L.tm_k, kmap_base, kv_dtype, map_blocks, block_size,
                                     n_kv_heads, head_dim, 1, true)) != cudaSuccess)
                return cuda_fail(e);
            if ((e = encode_pool_map(&L.tm_v, vmap_base, kv_dtype, map_blocks, block_size,
                                     n_kv_heads, head_dim, 1, true)) != cudaSuccess)
                return cuda_fail(e);
            pkv::MultiQueryParams& p = L.p;
            p.out = out;
            p.out_dtype = out_dtype;
            p.q = q;
            p.q_start = q_start;
            p.total_q = total_q;
            p.max_q_len = max_q_len;
            p.block_tables = block_tables;
            p.max_blocks_per_seq = max_blocks_per_seq;
            p.context_lens = context_lens;
            p.num_seqs = num_seqs;
            p.n_heads = n_heads;
            p.n_kv_heads = n_kv_heads;
            p.group = G;
            p.num_blocks = num_blocks;
            p.scale_log2 = scale * 1.4426950408889634f;
            p.stages = stages;
            p.max_pages = max_pages;
            p.errors = dev->errors;
            p.lpt_seqs = lpt;
            const int cta_tokens = pkv::kTcQTiles * tc_tokens;
            L.grid = dim3((unsigned)((max_q_len + cta_tokens - 1) / cta_tokens),
                          (unsigned)n_kv_heads, (unsigned)num_seqs);
            L.block = dim3((unsigned)pkv::kTcThreads);
            L.smem_bytes = smem;
            L.stream = static_cast<cudaStream_t>(stream);
            e = kv_dtype == PKV_BF16 ? pkv::launch_multi_query_tc_bf16(head_dim, block_size, L)
                                     : pkv::launch_multi_query_tc_f16(head_dim, block_size, L);
            if (e != cudaSuccess) return cuda_fail(e);
            return PKV_OK;
        }
    }

    const int qt = 16 / G;  // query tokens per warp
    int warps = (max_q_len + qt - 1) / qt;
    warps = warps < 1 ? 1 : (warps > 4 ? 4 : warps);
    int stages = tuning(PKV_TUNE_MQ_STAGES, 4);
    stages = stages < 2 ? 2 : (stages > 8 ? 8 : stages);
    pkv::MultiQueryLaunch L;
    std::memset(&L, 0, sizeof(L));
    const size_t smem = pkv::multi_query_smem_bytes(head_dim, block_size, 2, stages, max_pages);
    if (smem > (size_t)dev->smem_optin) return unsupported("shared memory of this configuration");
    if ((e = encode_pool_map(&L.tm_k, kmap_base, kv_dtype, map_blocks, block_size, n_kv_heads,
                             head_dim, 1, true)) != cudaSuccess)
        return cuda_fail(e);
    if ((e = encode_pool_map(&L.tm_v, vmap_base, kv_dtype, map_blocks, block_size, n_kv_heads,
                             head_dim, 1, true)) != cudaSuccess)
        return cuda_fail(e);
    pkv::MultiQueryParams& p = L.p;
    p.out = out;
    p.out_dtype = out_dtype;
    p.q = q;
    p.q_start = q_start;
    p.total_q = total_q;
    p.max_q_len = max_q_len;
    p.block_tables = block_tables;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.context_lens = context_lens;
    p.num_seqs = num_seqs;
    p.n_heads = n_heads;
    p.n_kv_heads = n_kv_heads;
    p.group = G;
    p.num_blocks = num_blocks;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.stages = stages;
    p.max_pages = max_pages;
    p.errors = dev->errors;
    const int tile_tokens = warps * qt;
    L.grid = dim3((unsigned)((max_q_len + tile_tokens - 1) / tile_tokens), (unsigned)n_kv_heads,
                  (unsigned)num_seqs);
    L.block = dim3((unsigned)(32 * (1 + warps)));
    L.smem_bytes = smem;
    L.stream = static_cast<cudaStream_t>(stream);
    e = kv_dtype == PKV_BF16 ? pkv::launch_multi_query_bf16(head_dim, block_size, L)
                             : pkv::launch_multi_query_f16(head_dim, block_size, L);
    if (e != cudaSuccess) return cuda_fail(e);
    return PKV_OK;
}

}  // extern "C"
