// decode_batched_bf16.cu -- batched decode kernel instances for bf16 query / K / V.
#define PKV_ELEM __nv_bfloat16
#define PKV_BATCHED_FN launch_decode_batched_bf16
#define PKV_BATCHED_MMA_FN launch_decode_mma_batched_bf16
#include "decode_batched_inst.inc"
