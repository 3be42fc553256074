// fwd_tc.cu -- the tensor-core forward for head dim 128 (the kernel is fwd_tc_body.cuh), and the
// dispatch of the forward over the head dims it is built for (128 here, 64 in fwd_tc_d64.cu).
#define RA_FWD_HD 128
#define RA_FWD_SUPPORTED tc_fwd_supported_d128
#define RA_FWD_LAUNCH launch_fwd_tc_d128
#include "fwd_tc_body.cuh"

namespace ra {

bool tc_fwd_supported_d64(const Problem& p);
cudaError_t launch_fwd_tc_d64(const Problem& p, const void* q, const void* k, const void* v, void* out, float* lse,
                              int mode, int step, unsigned int* status, cudaStream_t s,
                              unsigned long long* visits, const BlockView* blk);

bool tc_fwd_supported(const Problem& p)
{
    return p.d == 64 ? tc_fwd_supported_d64(p) : tc_fwd_supported_d128(p);
}

cudaError_t launch_fwd_tc(const Problem& p, const void* q, const void* k, const void* v, void* out, float* lse,
                          int mode, int step, unsigned int* status, cudaStream_t s, unsigned long long* visits,
                          const BlockView* blk)
{
    return p.d == 64 ? launch_fwd_tc_d64(p, q, k, v, out, lse, mode, step, status, s, visits, blk)
                     : launch_fwd_tc_d128(p, q, k, v, out, lse, mode, step, status, s, visits, blk);
}

}  // namespace ra
