// bwd_tc_d64.cu -- the tensor-core backward for head dim 64 (the kernel is bwd_tc_body.cuh).
#define RA_BWD_HD 64
#define RA_BWD_SUPPORTED tc_bwd_supported_d64
#define RA_BWD_LAUNCH launch_bwd_tc_d64
#include "bwd_tc_body.cuh"
