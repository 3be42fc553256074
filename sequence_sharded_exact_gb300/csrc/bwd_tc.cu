// bwd_tc.cu -- the tensor-core backward for head dim 128 (the kernel is bwd_tc_body.cuh), and the
// dispatch of the backward over the head dims it is built for (128 here, 64 in bwd_tc_d64.cu).
#define RA_BWD_HD 128
#define RA_BWD_SUPPORTED tc_bwd_supported_d128
#define RA_BWD_LAUNCH launch_bwd_tc_d128
#include "bwd_tc_body.cuh"

namespace ra {

bool tc_bwd_supported_d64(const Problem& p);
cudaError_t launch_bwd_tc_d64(const Problem& p, const void* q, const void* k, const void* v, const void* dout,
                              const float* D, const float* lse, float* dq_acc, void* dk, void* dv, int grad_dtype,
                              unsigned int* status, cudaStream_t s, unsigned long long* visits,
                              const BlockView* blk);

bool tc_bwd_supported(const Problem& p)
{
    return p.d == 64 ? tc_bwd_supported_d64(p) : tc_bwd_supported_d128(p);
}

cudaError_t launch_bwd_tc(const Problem& p, const void* q, const void* k, const void* v, const void* dout,
                          const float* D, const float* lse, float* dq_acc, void* dk, void* dv, int grad_dtype,
                          unsigned int* status, cudaStream_t s, unsigned long long* visits, const BlockView* blk)
{
    return p.d == 64
               ? launch_bwd_tc_d64(p, q, k, v, dout, D, lse, dq_acc, dk, dv, grad_dtype, status, s, visits, blk)
               : launch_bwd_tc_d128(p, q, k, v, dout, D, lse, dq_acc, dk, dv, grad_dtype, status, s, visits, blk);
}

}  // namespace ra
