// decode_launch.h -- host-side launch interface between the C ABI (capi.cu)
// and the translation units that instantiate the decode kernel templates.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "multi_query_kernel.cuh"

namespace pkv {

struct DecodeLaunch {
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    CUtensorMap tm_kh;   // boxes of half a block (a short last block)
    CUtensorMap tm_vh;
    DecodeParams p;
    dim3 grid;
    dim3 block;
    size_t smem_bytes;
    cudaStream_t stream;
    int sm_count;    // the stream kernel sizes its grid from it
    int max_ctas;    // stream kernel: at most this many CTAs (the workspace's bound)
};

// Launch paged_decode_kernel<D, BS, QPW, T> for T = __nv_bfloat16 / __half.
// Returns cudaErrorInvalidValue for a combination that is not compiled.
cudaError_t launch_decode_bf16(int D, int BS, int QPW, const DecodeLaunch& L);
cudaError_t launch_decode_f16(int D, int BS, int QPW, const DecodeLaunch& L);
// Launch paged_decode_mma_kernel<D, BS, T> (tensor-core path for query-head groups).
cudaError_t launch_decode_mma_bf16(int D, int BS, const DecodeLaunch& L);
cudaError_t launch_decode_mma_f16(int D, int BS, const DecodeLaunch& L);
// Launch paged_decode_mma_stream_kernel<D, BS, T> on every SM (as many CTAs
// as stay resident, at most L.max_ctas; L.grid is ignored).  *ctas receives
// the grid size, which the boundary merge launch must repeat.
cudaError_t launch_decode_stream_bf16(int D, int BS, const DecodeLaunch& L, int* ctas);
cudaError_t launch_decode_stream_f16(int D, int BS, const DecodeLaunch& L, int* ctas);

struct MultiQueryLaunch {
    CUtensorMap tm_q;   // tcgen05 kernel only
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    MultiQueryParams p;
    dim3 grid;
    dim3 block;
    size_t smem_bytes;
    cudaStream_t stream;
};

// Launch paged_multi_query_kernel<D, BS, T>.
cudaError_t launch_multi_query_bf16(int D, int BS, const MultiQueryLaunch& L);
cudaError_t launch_multi_query_f16(int D, int BS, const MultiQueryLaunch& L);
// Launch paged_multi_query_tc_kernel<D, BS, T> (tcgen05 tensor cores, 128 rows per CTA).
cudaError_t launch_multi_query_tc_bf16(int D, int BS, const MultiQueryLaunch& L);
cudaError_t launch_multi_query_tc_f16(int D, int BS, const MultiQueryLaunch& L);

struct BatchedProblem;

struct BatchedLaunch {
    const BatchedProblem* probs;   // device [num_problems]
    const int* seq_begin;          // device [num_problems + 1]
    int num_problems;
    dim3 grid;
    dim3 block;
    size_t smem_bytes;
    cudaStream_t stream;
};

// Launch paged_decode_batched_kernel<D, BS, QPW, T> / the tensor-core variant.
cudaError_t launch_decode_batched_bf16(int D, int BS, int QPW, const BatchedLaunch& L);
cudaError_t launch_decode_batched_f16(int D, int BS, int QPW, const BatchedLaunch& L);
cudaError_t launch_decode_mma_batched_bf16(int D, int BS, const BatchedLaunch& L);
cudaError_t launch_decode_mma_batched_f16(int D, int BS, const BatchedLaunch& L);

// Raise a kernel's dynamic shared-memory limit once per device.
cudaError_t ensure_smem_limit(const void* kernel, unsigned long long* done_mask, size_t bytes);

}  // namespace pkv
