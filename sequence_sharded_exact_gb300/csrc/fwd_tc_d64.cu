// fwd_tc_d64.cu -- the tensor-core forward for head dim 64 (the kernel is fwd_tc_body.cuh).
#define RA_FWD_HD 64
#define RA_FWD_SUPPORTED tc_fwd_supported_d64
#define RA_FWD_LAUNCH launch_fwd_tc_d64
#include "fwd_tc_body.cuh"
