// capi_host.h -- host helpers shared by the translation units of the C ABI
// (capi.cu, multi_query_capi.cu): failure reasons, per-device facts, TMA
// tensor maps of the K/V pools, shape support.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/pagedkv.h"

namespace pkv {
namespace host {

// Record a failure reason for pkv_last_error_detail() and return the status.
pkv_status invalid(const char* why);
pkv_status unsupported(const char* why);
pkv_status cuda_fail(cudaError_t e);

struct DeviceInfo {
    unsigned int* errors = nullptr;   // the device error word
    int sm_count = 0;
    int smem_optin = 0;               // dynamic shared memory a block may opt into
    int smem_per_sm = 0;
    bool ready = false;
};

// Facts of the current device, looked up once per device.
cudaError_t device_info(DeviceInfo** out);

bool aligned16(const void* p);

// Value of a launch-shape override (pkv_set_tuning), `fallback` while the
// knob holds PKV_TUNE_AUTO.
int tuning(pkv_tune_knob knob, int fallback);
// Whether the knob was set.
bool tuned(pkv_tune_knob knob);

// Tokens a block-table row can address (max_blocks_per_seq * block_size)
// fit the kernels' 32-bit token arithmetic.
bool table_tokens_fit(int max_blocks_per_seq, int block_size);

// head_dim 64/128, block_size 16/32, group 1/2/4/8.
bool supported_shape(int n_heads, int n_kv_heads, int head_dim, int block_size);

// The pool [num_blocks, B, Hk, D] as a 4-D tensor for TMA (see capi.cu).
// box_rows: token rows per box (0: the whole block).
cudaError_t encode_pool_map(CUtensorMap* map, const void* pool, pkv_dtype dt, int num_blocks,
                            int block_size, int n_kv_heads, int head_dim, int hpc, bool mma,
                            int box_rows = 0);

// The cuTensorMapEncodeTiled entry point of the driver (NULL if absent).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

}  // namespace host
}  // namespace pkv
