// decode_bf16.cu -- decode kernel instances for bf16 query / K / V.
#define PKV_ELEM __nv_bfloat16
#define PKV_FN launch_decode_bf16
#define PKV_MMA_FN launch_decode_mma_bf16
#define PKV_MQ_FN launch_multi_query_bf16
#define PKV_STREAM_FN launch_decode_stream_bf16
#include "decode_inst.inc"
