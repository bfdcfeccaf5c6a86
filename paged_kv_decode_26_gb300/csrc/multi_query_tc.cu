// multi_query_tc.cu -- instances of the tcgen05 multi-query kernel for
// bf16 and f16 query / K / V, head dims 64 and 128, block sizes 16 and 32.
#include "decode_launch.h"
#include "multi_query_tc_kernel.cuh"

namespace pkv {
namespace {

template <int D, int BS, typename T>
cudaError_t launch_tc(const MultiQueryLaunch& L) {
    static unsigned long long done_mask = 0;
    const void* fn = reinterpret_cast<const void*>(&paged_multi_query_tc_kernel<D, BS, T>);
    cudaError_t e = ensure_smem_limit(fn, &done_mask, L.smem_bytes);
    if (e != cudaSuccess) return e;
    paged_multi_query_tc_kernel<D, BS, T>
        <<<L.grid, L.block, L.smem_bytes, L.stream>>>(L.tm_q, L.tm_k, L.tm_v, L.p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t by_shape(int D, int BS, const MultiQueryLaunch& L) {
    if (D == 64 && BS == 16) return launch_tc<64, 16, T>(L);
    if (D == 64 && BS == 32) return launch_tc<64, 32, T>(L);
    if (D == 128 && BS == 16) return launch_tc<128, 16, T>(L);
    if (D == 128 && BS == 32) return launch_tc<128, 32, T>(L);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_multi_query_tc_bf16(int D, int BS, const MultiQueryLaunch& L) {
    return by_shape<__nv_bfloat16>(D, BS, L);
}

cudaError_t launch_multi_query_tc_f16(int D, int BS, const MultiQueryLaunch& L) {
    return by_shape<__half>(D, BS, L);
}

}  // namespace pkv
