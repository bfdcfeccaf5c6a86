// decode_f16.cu -- decode kernel instances for fp16 query / K / V.
#define PKV_ELEM __half
#define PKV_FN launch_decode_f16
#define PKV_MMA_FN launch_decode_mma_f16
#define PKV_MQ_FN launch_multi_query_f16
#define PKV_STREAM_FN launch_decode_stream_f16
#include "decode_inst.inc"
