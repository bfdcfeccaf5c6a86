// decode_batched.cuh -- many independent decode problems in one launch.
//
// Each problem has its own K/V pools, block tables, lengths, queries and
// outputs (and optionally a fused append); all share head_dim, block size,
// head counts and dtypes, hence one kernel instance and one launch shape.
// A problem's TMA maps and parameters sit in device memory (written by the
// host once, when the batch is planned); CTA z of the grid serves global
// sequence z, i.e. sequence z - seq_begin[i] of problem i.  The CTA bodies
// are those of the single-problem kernels.
#pragma once

#include "decode_mma_kernel.cuh"

namespace pkv {

// One problem of a batched launch (aligned as CUtensorMap requires; arrays
// of it start on a 256-byte boundary).
struct BatchedProblem {
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    CUtensorMap tm_kh;   // boxes of half a block (a short last block)
    CUtensorMap tm_vh;
    DecodeParams p;
    ReduceParams r;
};

// The problem holding global sequence z: the last i with seq_begin[i] <= z
// (seq_begin non-decreasing, seq_begin[0] = 0).
__device__ __forceinline__ int problem_of(const int* __restrict__ seq_begin, int num_problems,
                                          int z) {
    int lo = 0, hi = num_problems - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (seq_begin[mid] <= z) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

template <int D, int BS, int QPW, typename T>
__global__ void __launch_bounds__(kMaxThreads, 1)
    paged_decode_batched_kernel(const BatchedProblem* __restrict__ probs,
                                const int* __restrict__ seq_begin, int num_problems) {
    launch_dependents();
    const int z = blockIdx.z;
    const int i = problem_of(seq_begin, num_problems, z);
    const BatchedProblem& b = probs[i];
    decode_cta<D, BS, QPW, T>(&b.tm_k, &b.tm_v, &b.tm_kh, &b.tm_vh, b.p, blockIdx.x, blockIdx.y,
                              z - seq_begin[i]);
}

template <int D, int BS, typename T>
__global__ void __launch_bounds__(kMmaMaxThreads, 1)
    paged_decode_mma_batched_kernel(const BatchedProblem* __restrict__ probs,
                                    const int* __restrict__ seq_begin, int num_problems) {
    launch_dependents();
    const int z = blockIdx.z;
    const int i = problem_of(seq_begin, num_problems, z);
    const BatchedProblem& b = probs[i];
    decode_mma_cta<D, BS, T>(&b.tm_k, &b.tm_v, &b.tm_kh, &b.tm_vh, b.p, blockIdx.x, blockIdx.y,
                             z - seq_begin[i]);
}

// Split merge over every problem: one warp per global (sequence, query head).
template <int D>
__global__ void __launch_bounds__(128)
    paged_decode_batched_reduce_kernel(const BatchedProblem* __restrict__ probs,
                                       const int* __restrict__ seq_begin, int num_problems,
                                       int n_heads) {
    dependency_wait();  // the decode kernel's partials (launched as its dependent)
    const int unit = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int z = unit / n_heads;
    if (z >= seq_begin[num_problems]) return;
    const int i = problem_of(seq_begin, num_problems, z);
    reduce_unit<D>(probs[i].r, unit - seq_begin[i] * n_heads, threadIdx.x & 31);
}

}  // namespace pkv
