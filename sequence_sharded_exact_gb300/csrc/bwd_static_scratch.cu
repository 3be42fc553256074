// bwd_static_scratch.cu -- ring_attn_bwd_static_scratch: the backward for callers that cannot
// allocate device memory.
//
// ring_attn_bwd needs a caller-provided workspace (the row sums D and, for bf16 gradients, the
// float32 dQ accumulator).  Some callers cannot make one: a host framework that owns all device
// memory as one pre-sized pool and hands plugins nothing but their input and output buffers, or a
// latency-bound loop that is not allowed to call the allocator.  This entry point takes its scratch
// from a fixed array compiled into the library instead, so it allocates nothing.
//
// The array is kStaticScratchBytes (64 MiB) of device memory that every GPU which loads this
// library holds until the process exits.  Problems whose workspace would exceed it are rejected.
// The array is shared by every call on a device and keeps the last call's contents; everything the
// backward reads from it is rewritten (D) or cleared to zero (the dQ accumulator) by the call
// itself.  Calls whose work overlaps on the GPU (other streams, other threads) race on the array.
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "../../include/ringattn.h"
#include "ra_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;

__device__ __align__(256) unsigned char g_bwd_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices];

// Device address of the array on the current device, looked up once per device.
cudaError_t scratch_address(void** out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_bwd_static_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" {

size_t ring_attn_bwd_static_scratch_capacity(void) { return kStaticScratchBytes; }

ra_status ring_attn_bwd_static_scratch(const void* q, const void* k, const void* v,
                                       const void* out, const float* lse, const void* dout,
                                       void* dq, void* dk, void* dv, int grad_dtype, int B, int H,
                                       int Hkv, int L, int d, int n_shards, int causal,
                                       int layout, int dtype, void* stream)
{
    int path = 0;
    ra_status st = ring_attn_bwd_path(B, H, Hkv, L, d, n_shards, causal, layout, dtype, &path);
    if (st != RA_OK) return st;  // the problem itself is invalid (message already set)
    if (grad_dtype != RA_F32 && grad_dtype != RA_BF16)
        return ra::set_last_error(RA_ERR_INVALID_ARG, "unknown grad dtype");
    const size_t need = ring_attn_bwd_workspace_size(B, H, Hkv, L, d, grad_dtype);
    if (need > kStaticScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "ring_attn_bwd_static_scratch: this problem needs %zu bytes of scratch but the "
                 "library's static scratch holds %zu; use ring_attn_bwd with a workspace",
                 need, kStaticScratchBytes);
        return ra::set_last_error(RA_ERR_INVALID_ARG, msg);
    }
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
        cudaGetLastError();
        return ra::set_last_error(RA_ERR_NO_DEVICE, "no CUDA device available");
    }
    void* scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof(msg), "ring_attn_bwd_static_scratch: cudaGetSymbolAddress: %s",
                 cudaGetErrorString(e));
        return ra::set_last_error(RA_ERR_CUDA, msg);
    }
    return ring_attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, grad_dtype, scratch,
                         kStaticScratchBytes, B, H, Hkv, L, d, n_shards, causal, layout, dtype,
                         stream);
}

}  // extern "C"
