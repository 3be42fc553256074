// ra_internal.h -- declarations shared by the translation units of libringattn (not installed).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ra_geometry.h"

namespace ra {

// Arguments of one attention problem, validated by the entry points.
struct Problem {
    int B, H, Hkv, L, d, n, causal, layout, dtype;
    Geometry geo() const { return make_geometry(L, n, layout, causal); }
    long long q_rows() const { return (long long)B * H * L; }
    long long kv_rows() const { return (long long)B * Hkv * L; }
};

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// bits of the device status word (the ABI's RA_DEVICE_* values; api.cu checks they agree)
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned kStatusLayout = 2u;

// One device's block call (the per-device data path of the multi-device ring): the query rows are
// those of shard q_shard alone and the keys those of shard kv_shard alone, each in a local buffer
// of S = L / n rows per head holding rows [shard * S, (shard + 1) * S) of the whole-sequence
// layout.  Positions, masks and the ring step (q_shard - kv_shard) mod n come from the whole
// sequence's geometry; only the addressing of the buffers changes.
struct BlockView {
    int q_shard = 0, kv_shard = 0;
    int acc_kv = 0;  // backward: add dK, dV into the float32 outputs (1) or store them (0)
};

// Output mode of a forward kernel.
enum FwdMode {
    kFwdFused = 0,     // all ring steps, write out (dtype) + lse
    kFwdRingStep = 1,  // one ring step, write float32 partial + lse (-inf when nothing visible)
    kFwdRingStepAcc = 2,  // one ring step folded into a running float32 output + lse, in place
    kFwdFusedF32 = 3,  // all ring steps, write out as float32 (before any rounding to dtype) + lse
};

// Does the mode walk every ring step (the whole K/V sequence) rather than one?
__host__ __device__ inline bool fwd_all_steps(int mode) { return mode == kFwdFused || mode == kFwdFusedF32; }

// SIMT (CUDA-core) kernels: any shape, f32 or bf16 inputs.
// blk (optional): one device's block call; the forward then runs ring step
// (q_shard - kv_shard) mod n for shard q_shard only (mode kFwdRingStep or kFwdRingStepAcc), the
// backward adds dQ into a float32 dq and stores or adds dK, dV (float32) as blk->acc_kv says.
cudaError_t launch_fwd_simt(const Problem& p, const void* q, const void* k, const void* v,
                            void* out, float* lse, int mode, int step, cudaStream_t s,
                            const BlockView* blk = nullptr);
cudaError_t launch_bwd_simt(const Problem& p, const void* q, const void* k, const void* v,
                            const void* dout, const float* D, const float* lse, void* dq,
                            void* dk, void* dv, int grad_dtype, cudaStream_t s,
                            const BlockView* blk = nullptr);

// Tensor-core kernels (TMA + tcgen05 + TMEM), bf16, d = 128 or 64: forward with chunk length %
// 256 == 0, backward with chunk length % 128 == 0.
bool tc_fwd_supported(const Problem& p);
// visits (optional, n x n): +1 at [query shard][key shard] for every tile pair computed.
cudaError_t launch_fwd_tc(const Problem& p, const void* q, const void* k, const void* v,
                          void* out, float* lse, int mode, int step, unsigned int* status,
                          cudaStream_t s, unsigned long long* visits = nullptr,
                          const BlockView* blk = nullptr);
bool tc_bwd_supported(const Problem& p);
cudaError_t launch_bwd_tc(const Problem& p, const void* q, const void* k, const void* v,
                          const void* dout, const float* D, const float* lse, float* dq_acc,
                          void* dk, void* dv, int grad_dtype, unsigned int* status,
                          cudaStream_t s, unsigned long long* visits = nullptr,
                          const BlockView* blk = nullptr);

// HBM-bound helper kernels.
// Rotary position embedding by natural position, in place, of a [B][H][L][d] buffer (p.H heads),
// or (shard >= 0) of one device's [B][H][L/n][d] buffer holding shard `shard`'s rows.
cudaError_t launch_rope(const Problem& p, void* x, double base, int inverse, cudaStream_t s, int shard = -1);
// Ulysses all-to-all re-layout between the token split [n][B][S][H][row] and the head split
// [n][B][H/n][L][row] (direction 0 token -> head, 1 back); row_bytes a multiple of 4.
cudaError_t launch_ulysses_a2a(const Geometry& geo, int B, int H, int row_bytes, const void* src, void* dst,
                               int direction, cudaStream_t s);
cudaError_t launch_lse_merge(float* o_acc, float* lse_acc, const float* o_part,
                             const float* lse_part, long long rows, int d, cudaStream_t s);
cudaError_t launch_convert(const float* src, void* dst, int dst_dtype, long long count,
                           float scale, cudaStream_t s);
cudaError_t launch_bwd_preprocess(const void* out, const void* dout, int dtype, long long rows,
                                  int d, float* D, cudaStream_t s,
                                  int out_dtype = -1);
cudaError_t launch_zero(float* dst, long long count, cudaStream_t s);
// acc[i] += part[i] for count float32 values.
cudaError_t launch_add(float* acc, const float* part, long long count, cudaStream_t s);

// One thread waits on an mbarrier nothing completes (bounded wait of limit_ns); *returned = 1 when
// the wait gave up (and the timeout bit is set in *status), 2 if it completed.
cudaError_t launch_bounded_wait_selftest(unsigned int* status, unsigned long long limit_ns, unsigned int* returned,
                                         cudaStream_t s);

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Records `msg` as the calling thread's last error (ring_attn_last_error) and returns `status`.
int set_last_error(int status, const char* msg);

}  // namespace ra
