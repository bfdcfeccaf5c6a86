// decode_batched_f16.cu -- batched decode kernel instances for f16 query / K / V.
#define PKV_ELEM __half
#define PKV_BATCHED_FN launch_decode_batched_f16
#define PKV_BATCHED_MMA_FN launch_decode_mma_batched_f16
#include "decode_batched_inst.inc"
