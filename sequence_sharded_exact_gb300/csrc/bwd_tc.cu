// bwd_tc.cu -- tensor-core backward (not yet enabled: every shape takes the SIMT backward).
#include "ra_internal.h"

namespace ra {

bool tc_bwd_supported(const Problem&) { return false; }

cudaError_t launch_bwd_tc(const Problem&, const void*, const void*, const void*, const void*,
                          const float*, const float*, float*, void*, void*, int, unsigned int*,
                          cudaStream_t)
{
    return cudaErrorNotSupported;
}

}  // namespace ra
