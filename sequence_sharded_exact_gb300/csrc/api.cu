// api.cu -- the C ABI of libringattn (declared in include/ringattn.h): argument checks, path
// selection, workspace carving, the device status word and the host-side shard scheduler queries.
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <new>
#include <string>

#include "../../include/ringattn.h"
#include "ra_internal.h"

static_assert(ra::kStatusTimeout == RA_DEVICE_TIMEOUT && ra::kStatusLayout == RA_DEVICE_LAYOUT,
              "device status bits agree with the ABI");

namespace ra {
namespace {

thread_local std::string g_last_error;

ra_status fail(ra_status st, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

ra_status cuda_fail(cudaError_t e, const char* what)
{
    return fail(RA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device status word: kernels set bits here when a bounded wait runs out.
__device__ unsigned int g_device_status;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int* g_status_ptr[kMaxDevices];
int g_sm_count[kMaxDevices];

int current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}

// Device address of the status word for the current device (looked up once per device).
unsigned int* status_word(cudaError_t* err)
{
    int dev = current_device();
    *err = cudaSuccess;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_device_status);
        if (*err != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<unsigned int*>(p);
    }
    return g_status_ptr[dev];
}

ra_status check_device()
{
    int n = 0;
    cudaError_t e = cudaGetDeviceCount(&n);
    if (e != cudaSuccess || n == 0) {
        cudaGetLastError();
        return fail(RA_ERR_NO_DEVICE, "no CUDA device available (%s)", cudaGetErrorName(e));
    }
    return RA_OK;
}

ra_status check_problem(const Problem& p)
{
    if (p.B < 1 || p.H < 1 || p.Hkv < 1 || p.L < 1 || p.n < 1)
        return fail(RA_ERR_INVALID_ARG, "B, H, Hkv, L, n_shards must be >= 1 (got %d %d %d %d %d)",
                    p.B, p.H, p.Hkv, p.L, p.n);
    if (p.H % p.Hkv != 0)
        return fail(RA_ERR_INVALID_ARG, "H (%d) must be a multiple of Hkv (%d)", p.H, p.Hkv);
    if (p.L % p.n != 0)
        return fail(RA_ERR_INVALID_ARG, "L (%d) must be a multiple of n_shards (%d)", p.L, p.n);
    if (p.layout != RA_LAYOUT_CONTIGUOUS && p.layout != RA_LAYOUT_ZIGZAG && p.layout != RA_LAYOUT_STRIPED)
        return fail(RA_ERR_INVALID_ARG, "unknown layout %d", p.layout);
    if (p.layout == RA_LAYOUT_ZIGZAG && p.L % (2 * p.n) != 0)
        return fail(RA_ERR_INVALID_ARG, "zigzag layout needs L (%d) to be a multiple of 2*n_shards",
                    p.L);
    if (p.causal != 0 && p.causal != 1)
        return fail(RA_ERR_INVALID_ARG, "causal must be 0 or 1 (got %d)", p.causal);
    if (p.dtype != RA_F32 && p.dtype != RA_BF16)
        return fail(RA_ERR_INVALID_ARG, "unknown dtype %d", p.dtype);
    if (p.d != 64 && p.d != 128)
        return fail(RA_ERR_UNSUPPORTED, "head dim %d not supported (64 or 128)", p.d);
    if ((long long)p.B * p.H * p.L * p.d >= (1LL << 40))
        return fail(RA_ERR_UNSUPPORTED, "problem too large");
    return RA_OK;
}

ra_status check_ptrs(std::initializer_list<const void*> ptrs)
{
    int i = 0;
    for (const void* x : ptrs) {
        if (!x) return fail(RA_ERR_INVALID_ARG, "pointer argument %d is NULL", i);
        if (!aligned16(x)) return fail(RA_ERR_INVALID_ARG, "pointer argument %d is not 16-byte aligned", i);
        ++i;
    }
    return RA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

int set_last_error(int status, const char* msg)
{
    g_last_error = msg ? msg : "";
    return status;
}

int device_sm_count()
{
    int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return 148;
    if (g_sm_count[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1) v = 148;
        g_sm_count[dev] = v;
    }
    return g_sm_count[dev];
}

}  // namespace ra

using namespace ra;

extern "C" {

int ring_attn_abi_version(void) { return 1; }

const char* ring_attn_last_error(void) { return g_last_error.c_str(); }

ra_status ring_attn_fwd_path(int B, int H, int Hkv, int L, int d, int n_shards, int causal,
                             int layout, int dtype, int* path)
{
    Problem p{B, H, Hkv, L, d, n_shards, causal, layout, dtype};
    ra_status st = check_problem(p);
    if (st != RA_OK) return st;
    if (!path) return fail(RA_ERR_INVALID_ARG, "path is NULL");
    *path = tc_fwd_supported(p) ? RA_PATH_TCGEN05 : RA_PATH_SIMT;
    return RA_OK;
}

ra_status ring_attn_bwd_path(int B, int H, int Hkv, int L, int d, int n_shards, int causal,
                             int layout, int dtype, int* path)
{
    Problem p{B, H, Hkv, L, d, n_shards, causal, layout, dtype};
    ra_status st = check_problem(p);
    if (st != RA_OK) return st;
    if (!path) return fail(RA_ERR_INVALID_ARG, "path is NULL");
    *path = tc_bwd_supported(p) ? RA_PATH_TCGEN05 : RA_PATH_SIMT;
    return RA_OK;
}

namespace {

ra_status fwd_impl(const void* q, const void* k, const void* v, void* out, float* lse, const Problem& p,
                   unsigned long long* visits, void* stream, int mode = kFwdFused)
{
    ra_status st = check_problem(p);
    if (st != RA_OK) return st;
    if ((st = check_ptrs({q, k, v, out, lse})) != RA_OK) return st;
    const bool tc = tc_fwd_supported(p);
    if (visits) {
        if ((st = check_ptrs({visits})) != RA_OK) return st;
        if (!tc) return fail(RA_ERR_UNSUPPORTED, "tile visits are counted on the tensor-core path only");
    }
    if ((st = check_device()) != RA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (tc) {
        unsigned int* sw = status_word(&e);
        if (!sw) return cuda_fail(e, "status word");
        e = launch_fwd_tc(p, q, k, v, out, lse, mode, 0, sw, s, visits);
    } else {
        e = launch_fwd_simt(p, q, k, v, out, lse, mode, 0, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "ring_attn_fwd launch");
    return RA_OK;
}

}  // namespace

ra_status ring_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                        int H, int Hkv, int L, int d, int n_shards, int causal, int layout,
                        int dtype, void* stream)
{
    return fwd_impl(q, k, v, out, lse, Problem{B, H, Hkv, L, d, n_shards, causal, layout, dtype},
                    nullptr, stream);
}

ra_status ring_attn_fwd_f32out(const void* q, const void* k, const void* v, float* out, float* lse, int B,
                               int H, int Hkv, int L, int d, int n_shards, int causal, int layout,
                               int dtype, void* stream)
{
    return fwd_impl(q, k, v, out, lse, Problem{B, H, Hkv, L, d, n_shards, causal, layout, dtype},
                    nullptr, stream, kFwdFusedF32);
}

ra_status ring_attn_fwd_tile_visits(const void* q, const void* k, const void* v, void* out,
                                    float* lse, int B, int H, int Hkv, int L, int d, int n_shards,
                                    int causal, int layout, int dtype,
                                    unsigned long long* visits, void* stream)
{
    if (!visits) return fail(RA_ERR_INVALID_ARG, "visits is NULL");
    return fwd_impl(q, k, v, out, lse, Problem{B, H, Hkv, L, d, n_shards, causal, layout, dtype},
                    visits, stream);
}

ra_status ring_attn_ring_step_fwd(const void* q, const void* k, const void* v, float* o_part,
                                  float* lse_part, int B, int H, int Hkv, int L, int d,
                                  int n_shards, int step, int causal, int layout, int dtype,
                                  void* stream)
{
    Problem p{B, H, Hkv, L, d, n_shards, causal, layout, dtype};
    ra_status st = check_problem(p);
    if (st != RA_OK) return st;
    if (step < 0 || step >= n_shards)
        return fail(RA_ERR_INVALID_ARG, "step %d outside [0, n_shards)", step);
    if ((st = check_ptrs({q, k, v, o_part, lse_part})) != RA_OK) return st;
    if ((st = check_device()) != RA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (tc_fwd_supported(p)) {
        unsigned int* sw = status_word(&e);
        if (!sw) return cuda_fail(e, "status word");
        e = launch_fwd_tc(p, q, k, v, o_part, lse_part, kFwdRingStep, step, sw, s);
    } else {
        e = launch_fwd_simt(p, q, k, v, o_part, lse_part, kFwdRingStep, step, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "ring_attn_ring_step_fwd launch");
    return RA_OK;
}

ra_status ring_attn_ring_step_fwd_accumulate(const void* q, const void* k, const void* v, float* o_acc,
                                             float* lse_acc, int B, int H, int Hkv, int L, int d, int n_shards,
                                             int step, int causal, int layout, int dtype, void* stream)
{
    Problem p{B, H, Hkv, L, d, n_shards, causal, layout, dtype};
    ra_status st = check_problem(p);
    if (st != RA_OK) return st;
    if (step < 0 || step >= n_shards)
        return fail(RA_ERR_INVALID_ARG, "step %d outside [0, n_shards)", step);
    if ((st = check_ptrs({q, k, v, o_acc, lse_acc})) != RA_OK) return st;
    if ((st = check_device()) != RA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (tc_fwd_supported(p)) {
        unsigned int* sw = status_word(&e);
        if (!sw) return cuda_fail(e, "status word");
        e = launch_fwd_tc(p, q, k, v, o_acc, lse_acc, kFwdRingStepAcc, step, sw, s);
    } else {
        e = launch_fwd_simt(p, q, k, v, o_acc, lse_acc, kFwdRingStepAcc, step, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "ring_attn_ring_step_fwd_accumulate launch");
    return RA_OK;
}

ra_status ring_attn_lse_merge(float* o_acc, float* lse_acc, const float* o_part,
                              const float* lse_part, long long rows, int d, void* stream)
{
    if (rows < 0 || d < 1) return fail(RA_ERR_INVALID_ARG, "rows must be >= 0 and d >= 1");
    if (rows == 0) return RA_OK;
    ra_status st = check_ptrs({o_acc, lse_acc, o_part, lse_part});
    if (st != RA_OK) return st;
    if ((st = check_device()) != RA_OK) return st;
    cudaError_t e = launch_lse_merge(o_acc, lse_acc, o_part, lse_part, rows, d,
                                     static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ring_attn_lse_merge launch");
    return RA_OK;
}

size_t ring_attn_fwd_stepwise_workspace_size(int B, int H, int L, int d)
{
    if (B < 1 || H < 1 || L < 1 || d < 1) return 0;
    const size_t rows = (size_t)B * H * L;
    return align256(rows * d * sizeof(float));  // the float32 running output
}

ra_status ring_attn_fwd_stepwise(const void* q, const void* k, const void* v, void* out,
                                 float* lse, int B, int H, int Hkv, int L, int d, int n_shards,
                                 int causal, int layout, int dtype, void* workspace,
                                 size_t workspace_bytes, void* stream)
{
    Problem p{B, H, Hkv, L, d, n_shards, causal, layout, dtype};
    ra_status st = check_problem(p);
    if (st != RA_OK) return st;
    if ((st = check_ptrs({q, k, v, out, lse, workspace})) != RA_OK) return st;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(RA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    const size_t need = ring_attn_fwd_stepwise_workspace_size(B, H, L, d);
    if (workspace_bytes < need)
        return fail(RA_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
    if ((st = check_device()) != RA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long rows = p.q_rows();
    float* o_acc = static_cast<float*>(workspace);
    const bool tc = tc_fwd_supported(p);
    cudaError_t e = cudaSuccess;
    unsigned int* sw = nullptr;
    if (tc && !(sw = status_word(&e))) return cuda_fail(e, "status word");
    // step 0 writes the running (o, lse); every later step folds its block into it in its epilogue
    for (int step = 0; step < n_shards && e == cudaSuccess; ++step) {
        const int mode = step == 0 ? kFwdRingStep : kFwdRingStepAcc;
        e = tc ? launch_fwd_tc(p, q, k, v, o_acc, lse, mode, step, sw, s)
               : launch_fwd_simt(p, q, k, v, o_acc, lse, mode, step, s);
    }
    if (e == cudaSuccess) e = launch_convert(o_acc, out, dtype, rows * d, 1.0f, s);
    if (e != cudaSuccess) return cuda_fail(e, "ring_attn_fwd_stepwise launch");
    return RA_OK;
}

size_t ring_attn_bwd_workspace_size(int B, int H, int Hkv, int L, int d, int grad_dtype)
{
    (void)Hkv;
    if (B < 1 || H < 1 || L < 1 || d < 1) return 0;
    const size_t rows = (size_t)B * H * L;
    size_t bytes = align256(rows * sizeof(float));                   // D
    if (grad_dtype != RA_F32) bytes += align256(rows * d * sizeof(float));  // dQ accumulator
    return bytes;
}

namespace {

ra_status bwd_impl(const void* q, const void* k, const void* v, const void* out, const float* lse,
                   const void* dout, void* dq, void* dk, void* dv, int grad_dtype, void* workspace,
                   size_t workspace_bytes, const Problem& p, unsigned long long* visits, void* stream,
                   int out_dtype = -1)
{
    const int B = p.B, H = p.H, Hkv = p.Hkv, L = p.L, d = p.d, dtype = p.dtype;
    ra_status st = check_problem(p);
    if (st != RA_OK) return st;
    if (grad_dtype != RA_F32 && grad_dtype != RA_BF16)
        return fail(RA_ERR_INVALID_ARG, "unknown grad dtype %d", grad_dtype);
    if ((st = check_ptrs({q, k, v, out, lse, dout, dq, dk, dv, workspace})) != RA_OK) return st;
    const bool tc = tc_bwd_supported(p);
    if (visits) {
        if ((st = check_ptrs({visits})) != RA_OK) return st;
        if (!tc) return fail(RA_ERR_UNSUPPORTED, "tile visits are counted on the tensor-core path only");
    }
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(RA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    const size_t need = ring_attn_bwd_workspace_size(B, H, Hkv, L, d, grad_dtype);
    if (workspace_bytes < need)
        return fail(RA_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
    if ((st = check_device()) != RA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long rows = p.q_rows();
    char* ws = static_cast<char*>(workspace);
    float* D = reinterpret_cast<float*>(ws);
    cudaError_t e = launch_bwd_preprocess(out, dout, dtype, rows, d, D, s, out_dtype);
    if (e != cudaSuccess) return cuda_fail(e, "ring_attn_bwd preprocess launch");
    if (tc) {
        unsigned int* sw = status_word(&e);
        if (!sw) return cuda_fail(e, "status word");
        float* dq_acc = grad_dtype == RA_F32
                            ? static_cast<float*>(dq)
                            : reinterpret_cast<float*>(ws + align256((size_t)rows * sizeof(float)));
        e = launch_zero(dq_acc, rows * d, s);
        if (e == cudaSuccess)
            e = launch_bwd_tc(p, q, k, v, dout, D, lse, dq_acc, dk, dv, grad_dtype, sw, s, visits);
        if (e == cudaSuccess && grad_dtype != RA_F32)
            e = launch_convert(dq_acc, dq, grad_dtype, rows * d, 1.0f, s);
    } else {
        e = launch_bwd_simt(p, q, k, v, dout, D, lse, dq, dk, dv, grad_dtype, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "ring_attn_bwd launch");
    return RA_OK;
}

}  // namespace

ra_status ring_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                        const float* lse, const void* dout, void* dq, void* dk, void* dv,
                        int grad_dtype, void* workspace, size_t workspace_bytes, int B, int H,
                        int Hkv, int L, int d, int n_shards, int causal, int layout, int dtype,
                        void* stream)
{
    return bwd_impl(q, k, v, out, lse, dout, dq, dk, dv, grad_dtype, workspace, workspace_bytes,
                    Problem{B, H, Hkv, L, d, n_shards, causal, layout, dtype}, nullptr, stream);
}

ra_status ring_attn_bwd_f32out(const void* q, const void* k, const void* v, const float* out,
                               const float* lse, const void* dout, void* dq, void* dk, void* dv,
                               int grad_dtype, void* workspace, size_t workspace_bytes, int B, int H,
                               int Hkv, int L, int d, int n_shards, int causal, int layout, int dtype,
                               void* stream)
{
    return bwd_impl(q, k, v, out, lse, dout, dq, dk, dv, grad_dtype, workspace, workspace_bytes,
                    Problem{B, H, Hkv, L, d, n_shards, causal, layout, dtype}, nullptr, stream, RA_F32);
}

ra_status ring_attn_bwd_tile_visits(const void* q, const void* k, const void* v, const void* out,
                                    const float* lse, const void* dout, void* dq, void* dk,
                                    void* dv, int grad_dtype, void* workspace,
                                    size_t workspace_bytes, int B, int H, int Hkv, int L, int d,
                                    int n_shards, int causal, int layout, int dtype,
                                    unsigned long long* visits, void* stream)
{
    if (!visits) return fail(RA_ERR_INVALID_ARG, "visits is NULL");
    return bwd_impl(q, k, v, out, lse, dout, dq, dk, dv, grad_dtype, workspace, workspace_bytes,
                    Problem{B, H, Hkv, L, d, n_shards, causal, layout, dtype}, visits, stream);
}

// ---------------------------------------------------------------------------------------------
// One device's data path of the multi-device ring (block calls and their helpers)
// ---------------------------------------------------------------------------------------------
namespace {

ra_status check_block(const Problem& p, int shard_q, int shard_kv, int flag, const char* flag_name)
{
    ra_status st = check_problem(p);
    if (st != RA_OK) return st;
    if (shard_q < 0 || shard_q >= p.n || shard_kv < 0 || shard_kv >= p.n)
        return fail(RA_ERR_INVALID_ARG, "shard indices (%d, %d) outside [0, n_shards = %d)", shard_q, shard_kv, p.n);
    if (flag != 0 && flag != 1) return fail(RA_ERR_INVALID_ARG, "%s must be 0 or 1 (got %d)", flag_name, flag);
    return RA_OK;
}

ra_status check_count(long long count)
{
    if (count < 0) return fail(RA_ERR_INVALID_ARG, "count must be >= 0 (got %lld)", count);
    return RA_OK;
}

}  // namespace

ra_status ring_attn_block_fwd(const void* q, const void* k, const void* v, float* o_acc, float* lse_acc, int B,
                              int H, int Hkv, int L, int d, int n_shards, int shard_q, int shard_kv, int accumulate,
                              int causal, int layout, int dtype, void* stream)
{
    Problem p{B, H, Hkv, L, d, n_shards, causal, layout, dtype};
    ra_status st = check_block(p, shard_q, shard_kv, accumulate, "accumulate");
    if (st != RA_OK) return st;
    if ((st = check_ptrs({q, k, v, o_acc, lse_acc})) != RA_OK) return st;
    if ((st = check_device()) != RA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const BlockView blk{shard_q, shard_kv, 0};
    const int step = (shard_q - shard_kv + n_shards) % n_shards;
    const int mode = accumulate ? kFwdRingStepAcc : kFwdRingStep;
    cudaError_t e;
    if (tc_fwd_supported(p)) {
        unsigned int* sw = status_word(&e);
        if (!sw) return cuda_fail(e, "status word");
        e = launch_fwd_tc(p, q, k, v, o_acc, lse_acc, mode, step, sw, s, nullptr, &blk);
    } else {
        e = launch_fwd_simt(p, q, k, v, o_acc, lse_acc, mode, step, s, &blk);
    }
    if (e != cudaSuccess) return cuda_fail(e, "ring_attn_block_fwd launch");
    return RA_OK;
}

ra_status ring_attn_block_bwd(const void* q, const void* k, const void* v, const void* dout, const float* lse,
                              const float* D, float* dq_acc, float* dk, float* dv, int B, int H, int Hkv, int L,
                              int d, int n_shards, int shard_q, int shard_kv, int accumulate_kv, int causal,
                              int layout, int dtype, void* stream)
{
    Problem p{B, H, Hkv, L, d, n_shards, causal, layout, dtype};
    ra_status st = check_block(p, shard_q, shard_kv, accumulate_kv, "accumulate_kv");
    if (st != RA_OK) return st;
    if ((st = check_ptrs({q, k, v, dout, lse, D, dq_acc, dk, dv})) != RA_OK) return st;
    if ((st = check_device()) != RA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const BlockView blk{shard_q, shard_kv, accumulate_kv};
    cudaError_t e;
    if (tc_bwd_supported(p)) {
        unsigned int* sw = status_word(&e);
        if (!sw) return cuda_fail(e, "status word");
        e = launch_bwd_tc(p, q, k, v, dout, D, lse, dq_acc, dk, dv, RA_F32, sw, s, nullptr, &blk);
    } else {
        e = launch_bwd_simt(p, q, k, v, dout, D, lse, dq_acc, dk, dv, RA_F32, s, &blk);
    }
    if (e != cudaSuccess) return cuda_fail(e, "ring_attn_block_bwd launch");
    return RA_OK;
}

ra_status ring_attn_bwd_preprocess(const void* out, const void* dout, float* D, long long rows, int d, int dtype,
                                   void* stream)
{
    ra_status st = check_count(rows);
    if (st != RA_OK) return st;
    if (d < 1) return fail(RA_ERR_INVALID_ARG, "d must be >= 1");
    if (dtype != RA_F32 && dtype != RA_BF16) return fail(RA_ERR_INVALID_ARG, "unknown dtype %d", dtype);
    if (rows == 0) return RA_OK;
    if ((st = check_ptrs({out, dout, D})) != RA_OK) return st;
    if ((st = check_device()) != RA_OK) return st;
    cudaError_t e = launch_bwd_preprocess(out, dout, dtype, rows, d, D, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ring_attn_bwd_preprocess launch");
    return RA_OK;
}

ra_status ring_attn_bwd_preprocess_f32out(const float* out, const void* dout, float* D, long long rows, int d,
                                          int dtype, void* stream)
{
    ra_status st = check_count(rows);
    if (st != RA_OK) return st;
    if (d < 1) return fail(RA_ERR_INVALID_ARG, "d must be >= 1");
    if (dtype != RA_F32 && dtype != RA_BF16) return fail(RA_ERR_INVALID_ARG, "unknown dtype %d", dtype);
    if (rows == 0) return RA_OK;
    if ((st = check_ptrs({out, dout, D})) != RA_OK) return st;
    if ((st = check_device()) != RA_OK) return st;
    cudaError_t e = launch_bwd_preprocess(out, dout, dtype, rows, d, D, static_cast<cudaStream_t>(stream), RA_F32);
    if (e != cudaSuccess) return cuda_fail(e, "ring_attn_bwd_preprocess_f32out launch");
    return RA_OK;
}

ra_status ring_attn_f32_zero(float* x, long long count, void* stream)
{
    ra_status st = check_count(count);
    if (st != RA_OK || count == 0) return st;
    if ((st = check_ptrs({x})) != RA_OK) return st;
    if ((st = check_device()) != RA_OK) return st;
    cudaError_t e = launch_zero(x, count, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ring_attn_f32_zero launch");
    return RA_OK;
}

ra_status ring_attn_f32_add(float* acc, const float* part, long long count, void* stream)
{
    ra_status st = check_count(count);
    if (st != RA_OK || count == 0) return st;
    if ((st = check_ptrs({acc, part})) != RA_OK) return st;
    if ((st = check_device()) != RA_OK) return st;
    cudaError_t e = launch_add(acc, part, count, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ring_attn_f32_add launch");
    return RA_OK;
}

ra_status ring_attn_f32_convert(const float* src, void* dst, long long count, int dtype, void* stream)
{
    ra_status st = check_count(count);
    if (st != RA_OK) return st;
    if (dtype != RA_F32 && dtype != RA_BF16) return fail(RA_ERR_INVALID_ARG, "unknown dtype %d", dtype);
    if (count == 0) return RA_OK;
    if ((st = check_ptrs({src, dst})) != RA_OK) return st;
    if ((st = check_device()) != RA_OK) return st;
    cudaError_t e = launch_convert(src, dst, dtype, count, 1.0f, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ring_attn_f32_convert launch");
    return RA_OK;
}

ra_status ring_attn_rope(void* x, int B, int H, int L, int d, int n_shards, int layout, int dtype,
                         double base, int inverse, void* stream)
{
    Problem p{B, H, H, L, d, n_shards, 0, layout, dtype};
    ra_status st = check_problem(p);
    if (st != RA_OK) return st;
    if (!(base > 0.0) || !isfinite(base)) return fail(RA_ERR_INVALID_ARG, "base must be positive and finite");
    if ((st = check_ptrs({x})) != RA_OK) return st;
    if ((st = check_device()) != RA_OK) return st;
    cudaError_t e = launch_rope(p, x, base, inverse, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ring_attn_rope launch");
    return RA_OK;
}

ra_status ring_attn_block_rope(void* x, int B, int H, int L, int d, int n_shards, int shard, int layout, int dtype,
                               double base, int inverse, void* stream)
{
    Problem p{B, H, H, L, d, n_shards, 0, layout, dtype};
    ra_status st = check_block(p, shard, shard, 0, "-");
    if (st != RA_OK) return st;
    if (!(base > 0.0) || !isfinite(base)) return fail(RA_ERR_INVALID_ARG, "base must be positive and finite");
    if ((st = check_ptrs({x})) != RA_OK) return st;
    if ((st = check_device()) != RA_OK) return st;
    cudaError_t e = launch_rope(p, x, base, inverse, static_cast<cudaStream_t>(stream), shard);
    if (e != cudaSuccess) return cuda_fail(e, "ring_attn_block_rope launch");
    return RA_OK;
}

namespace {

ra_status check_ulysses_heads(const Problem& p)
{
    if (p.H % p.n != 0 || p.Hkv % p.n != 0)
        return fail(RA_ERR_INVALID_ARG,
                    "Ulysses splits heads across the shards: H (%d) and Hkv (%d) must be multiples of n_shards (%d)",
                    p.H, p.Hkv, p.n);
    return RA_OK;
}

size_t elem_size(int dtype) { return dtype == RA_F32 ? 4 : 2; }

}  // namespace

ra_status ring_attn_ulysses_a2a(const void* src, void* dst, int B, int H, int L, int d, int n_shards, int layout,
                                int dtype, int direction, void* stream)
{
    Problem p{B, H, H, L, 64, n_shards, 0, layout, dtype};  // d checked below: any row length
    ra_status st = check_problem(p);
    if (st != RA_OK) return st;
    if (d < 1 || (long long)d * elem_size(dtype) % 4 != 0)
        return fail(RA_ERR_INVALID_ARG, "row of %d elements is not a whole number of 4-byte words", d);
    if ((long long)B * H * L * d * (long long)elem_size(dtype) / 4 >= (1LL << 32))
        return fail(RA_ERR_UNSUPPORTED, "tensor of 2^34 bytes or more");
    if (direction != 0 && direction != 1) return fail(RA_ERR_INVALID_ARG, "direction must be 0 or 1");
    if ((st = check_ulysses_heads(p)) != RA_OK) return st;
    if ((st = check_ptrs({src, dst})) != RA_OK) return st;
    if (src == dst) return fail(RA_ERR_INVALID_ARG, "src and dst must not be the same buffer");
    if ((st = check_device()) != RA_OK) return st;
    cudaError_t e = launch_ulysses_a2a(p.geo(), B, H, (int)(d * elem_size(dtype)), src, dst, direction,
                                       static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ring_attn_ulysses_a2a launch");
    return RA_OK;
}

size_t ring_attn_ulysses_workspace_size(int B, int H, int Hkv, int L, int d, int dtype)
{
    if (B < 1 || H < 1 || Hkv < 1 || L < 1 || d < 1) return 0;
    const size_t e = elem_size(dtype);
    const size_t qrows = (size_t)B * H * L, kvrows = (size_t)B * Hkv * L;
    // head-split q, k, v, out, lse
    return 2 * align256(qrows * d * e) + 2 * align256(kvrows * d * e) + align256(qrows * sizeof(float));
}

ra_status ring_attn_ulysses_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int H,
                                int Hkv, int L, int d, int n_shards, int causal, int layout, int dtype,
                                void* workspace, size_t workspace_bytes, void* stream)
{
    Problem p{B, H, Hkv, L, d, n_shards, causal, layout, dtype};
    ra_status st = check_problem(p);
    if (st != RA_OK) return st;
    if ((st = check_ulysses_heads(p)) != RA_OK) return st;
    if ((long long)B * H * L * d * (long long)elem_size(dtype) / 4 >= (1LL << 32))
        return fail(RA_ERR_UNSUPPORTED, "tensor of 2^34 bytes or more");
    if ((st = check_ptrs({q, k, v, out, lse, workspace})) != RA_OK) return st;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(RA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    const size_t need = ring_attn_ulysses_workspace_size(B, H, Hkv, L, d, dtype);
    if (workspace_bytes < need)
        return fail(RA_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
    if ((st = check_device()) != RA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t e = elem_size(dtype);
    const size_t qrows = (size_t)B * H * L, kvrows = (size_t)B * Hkv * L;
    char* ws = static_cast<char*>(workspace);
    void* qh = ws;
    void* kh = ws + align256(qrows * d * e);
    void* vh = static_cast<char*>(kh) + align256(kvrows * d * e);
    void* oh = static_cast<char*>(vh) + align256(kvrows * d * e);
    float* lh = reinterpret_cast<float*>(static_cast<char*>(oh) + align256(qrows * d * e));
    const Geometry geo = p.geo();
    const int row = (int)(d * e);
    // first all-to-all: token split -> head split
    cudaError_t err = launch_ulysses_a2a(geo, B, H, row, q, qh, 0, s);
    if (err == cudaSuccess) err = launch_ulysses_a2a(geo, B, Hkv, row, k, kh, 0, s);
    if (err == cudaSuccess) err = launch_ulysses_a2a(geo, B, Hkv, row, v, vh, 0, s);
    // each rank: ordinary attention over the whole sequence (natural order) for its H / n heads, all
    // ranks in one launch as a batch of n * B problems
    if (err == cudaSuccess) {
        const Problem pr{n_shards * B, H / n_shards, Hkv / n_shards, L, d, 1, causal, RA_LAYOUT_CONTIGUOUS, dtype};
        if (tc_fwd_supported(pr)) {
            unsigned int* sw = status_word(&err);
            if (sw) err = launch_fwd_tc(pr, qh, kh, vh, oh, lh, kFwdFused, 0, sw, s);
        } else {
            err = launch_fwd_simt(pr, qh, kh, vh, oh, lh, kFwdFused, 0, s);
        }
    }
    // second all-to-all: head split -> token split, for out and lse
    if (err == cudaSuccess) err = launch_ulysses_a2a(geo, B, H, row, oh, out, 1, s);
    if (err == cudaSuccess) err = launch_ulysses_a2a(geo, B, H, 4, lh, lse, 1, s);
    if (err != cudaSuccess) return cuda_fail(err, "ring_attn_ulysses_fwd launch");
    return RA_OK;
}

size_t ring_attn_ulysses_bwd_workspace_size(int B, int H, int Hkv, int L, int d, int n_shards, int dtype,
                                            int grad_dtype)
{
    if (B < 1 || H < 1 || Hkv < 1 || L < 1 || d < 1 || n_shards < 1 || H % n_shards || Hkv % n_shards) return 0;
    const size_t e = elem_size(dtype), ge = elem_size(grad_dtype);
    const size_t qrows = (size_t)B * H * L, kvrows = (size_t)B * Hkv * L;
    // head-split q, out, dout, k, v, lse, dq, dk, dv, then the per-shard backward's own workspace
    return 3 * align256(qrows * d * e) + 2 * align256(kvrows * d * e) + align256(qrows * sizeof(float)) +
           align256(qrows * d * ge) + 2 * align256(kvrows * d * ge) +
           align256(ring_attn_bwd_workspace_size(n_shards * B, H / n_shards, Hkv / n_shards, L, d, grad_dtype));
}

ra_status ring_attn_ulysses_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                                const void* dout, void* dq, void* dk, void* dv, int grad_dtype, void* workspace,
                                size_t workspace_bytes, int B, int H, int Hkv, int L, int d, int n_shards,
                                int causal, int layout, int dtype, void* stream)
{
    Problem p{B, H, Hkv, L, d, n_shards, causal, layout, dtype};
    ra_status st = check_problem(p);
    if (st != RA_OK) return st;
    if ((st = check_ulysses_heads(p)) != RA_OK) return st;
    if (grad_dtype != RA_F32 && grad_dtype != RA_BF16)
        return fail(RA_ERR_INVALID_ARG, "unknown grad dtype %d", grad_dtype);
    if ((long long)B * H * L * d >= (1LL << 32))  // the float32 dq all-to-all indexes 4-byte words in 32 bits
        return fail(RA_ERR_UNSUPPORTED, "tensor of 2^32 elements or more");
    if ((st = check_ptrs({q, k, v, out, lse, dout, dq, dk, dv, workspace})) != RA_OK) return st;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(RA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    const size_t need = ring_attn_ulysses_bwd_workspace_size(B, H, Hkv, L, d, n_shards, dtype, grad_dtype);
    if (workspace_bytes < need)
        return fail(RA_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
    if ((st = check_device()) != RA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t e = elem_size(dtype), ge = elem_size(grad_dtype);
    const size_t qrows = (size_t)B * H * L, kvrows = (size_t)B * Hkv * L;
    char* w = static_cast<char*>(workspace);
    auto take = [&](size_t bytes) { char* x = w; w += align256(bytes); return x; };
    void* qh = take(qrows * d * e);
    void* oh = take(qrows * d * e);
    void* doh = take(qrows * d * e);
    void* kh = take(kvrows * d * e);
    void* vh = take(kvrows * d * e);
    float* lh = reinterpret_cast<float*>(take(qrows * sizeof(float)));
    void* dqh = take(qrows * d * ge);
    void* dkh = take(kvrows * d * ge);
    void* dvh = take(kvrows * d * ge);
    const int pn = n_shards;
    const size_t inner = ring_attn_bwd_workspace_size(pn * B, H / pn, Hkv / pn, L, d, grad_dtype);
    void* iw = take(inner);
    const Geometry geo = p.geo();
    const int row = (int)(d * e), grow = (int)(d * ge);
    cudaError_t err = launch_ulysses_a2a(geo, B, H, row, q, qh, 0, s);
    if (err == cudaSuccess) err = launch_ulysses_a2a(geo, B, H, row, out, oh, 0, s);
    if (err == cudaSuccess) err = launch_ulysses_a2a(geo, B, H, row, dout, doh, 0, s);
    if (err == cudaSuccess) err = launch_ulysses_a2a(geo, B, Hkv, row, k, kh, 0, s);
    if (err == cudaSuccess) err = launch_ulysses_a2a(geo, B, Hkv, row, v, vh, 0, s);
    if (err == cudaSuccess) err = launch_ulysses_a2a(geo, B, H, 4, lse, lh, 0, s);
    if (err != cudaSuccess) return cuda_fail(err, "ring_attn_ulysses_bwd launch");
    // every shard: the ordinary backward over the whole sequence for its heads (one call, n * B problems)
    st = bwd_impl(qh, kh, vh, oh, lh, doh, dqh, dkh, dvh, grad_dtype, iw, inner,
                  Problem{pn * B, H / pn, Hkv / pn, L, d, 1, causal, RA_LAYOUT_CONTIGUOUS, dtype}, nullptr, stream);
    if (st != RA_OK) return st;
    err = launch_ulysses_a2a(geo, B, H, grow, dqh, dq, 1, s);
    if (err == cudaSuccess) err = launch_ulysses_a2a(geo, B, Hkv, grow, dkh, dk, 1, s);
    if (err == cudaSuccess) err = launch_ulysses_a2a(geo, B, Hkv, grow, dvh, dv, 1, s);
    if (err != cudaSuccess) return cuda_fail(err, "ring_attn_ulysses_bwd launch");
    return RA_OK;
}

namespace {

// Copy streams and events of the host-buffer forward, created once per device.
struct HostPipe {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaStream_t comp[2] = {};  // the groups' kernels alternate between two streams (see below)
    cudaEvent_t entry = nullptr, in_done[2] = {}, compute_done[2] = {}, out_done[2] = {};
    std::mutex mu;  // one host-buffer forward enqueues at a time per device (the events are shared)
};
HostPipe g_pipe[kMaxDevices];

cudaError_t host_pipe_init(HostPipe& hp)
{
    if (hp.ready) return cudaSuccess;
    cudaError_t e = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking);
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaStreamCreateWithFlags(&hp.comp[i], cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.entry, cudaEventDisableTiming);
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
        e = cudaEventCreateWithFlags(&hp.in_done[i], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.compute_done[i], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.out_done[i], cudaEventDisableTiming);
    }
    if (e == cudaSuccess) hp.ready = true;
    return e;
}

}  // namespace

size_t ring_attn_fwd_host_workspace_size(int H, int Hkv, int L, int d, int dtype)
{
    if (H < 1 || Hkv < 1 || L < 1 || d < 1 || H % Hkv) return 0;
    const size_t e = elem_size(dtype), G = (size_t)(H / Hkv), rows = (size_t)L;
    // per slot: q and out of one kv group's query heads, its k and v, its lse; two slots
    const size_t slot = 2 * align256(G * rows * d * e) + 2 * align256(rows * d * e) + align256(G * rows * 4);
    return 2 * slot;
}

ra_status ring_attn_fwd_host(const void* q, const void* k, const void* v, void* out, float* lse, int B, int H,
                             int Hkv, int L, int d, int n_shards, int causal, int layout, int dtype, void* workspace,
                             size_t workspace_bytes, void* stream)
{
    Problem p{B, H, Hkv, L, d, n_shards, causal, layout, dtype};
    ra_status st = check_problem(p);
    if (st != RA_OK) return st;
    if (!q || !k || !v || !out || !lse) return fail(RA_ERR_INVALID_ARG, "a host buffer is NULL");
    if ((st = check_ptrs({workspace})) != RA_OK) return st;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(RA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    const size_t need = ring_attn_fwd_host_workspace_size(H, Hkv, L, d, dtype);
    if (workspace_bytes < need)
        return fail(RA_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
    if ((st = check_device()) != RA_OK) return st;
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return fail(RA_ERR_NO_DEVICE, "device index out of range");
    HostPipe& hp = g_pipe[dev];
    std::lock_guard<std::mutex> lock(hp.mu);
    cudaError_t e = host_pipe_init(hp);
    if (e != cudaSuccess) return cuda_fail(e, "ring_attn_fwd_host streams");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int* sw = nullptr;
    const Problem pg{1, H / Hkv, 1, L, d, n_shards, causal, layout, dtype};  // one kv group
    const bool tc = tc_fwd_supported(pg);
    if (tc && !(sw = status_word(&e))) return cuda_fail(e, "status word");
    const size_t es = elem_size(dtype), G = (size_t)(H / Hkv);
    const size_t qbytes = G * L * d * es, kbytes = (size_t)L * d * es, lbytes = G * L * 4;
    char* base = static_cast<char*>(workspace);
    const size_t slot_bytes = 2 * align256(qbytes) + 2 * align256(kbytes) + align256(lbytes);
    // earlier work on the caller's stream (a previous call using this workspace) comes first
    e = cudaEventRecord(hp.entry, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp.h2d, hp.entry, 0);
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(hp.comp[i], hp.entry, 0);
    const int groups = B * Hkv;
    for (int gi = 0; gi < groups && e == cudaSuccess; ++gi) {
        const int sl = gi & 1;
        char* w = base + sl * slot_bytes;
        char* dq = w;
        char* dout = dq + align256(qbytes);
        char* dk = dout + align256(qbytes);
        char* dv = dk + align256(kbytes);
        float* dl = reinterpret_cast<float*>(dv + align256(kbytes));
        // the slot is free once the group two back has been copied out
        if (gi >= 2) e = cudaStreamWaitEvent(hp.h2d, hp.out_done[sl], 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(dq, static_cast<const char*>(q) + (size_t)gi * qbytes, qbytes,
                                                  cudaMemcpyHostToDevice, hp.h2d);
        if (e == cudaSuccess) e = cudaMemcpyAsync(dk, static_cast<const char*>(k) + (size_t)gi * kbytes, kbytes,
                                                  cudaMemcpyHostToDevice, hp.h2d);
        if (e == cudaSuccess) e = cudaMemcpyAsync(dv, static_cast<const char*>(v) + (size_t)gi * kbytes, kbytes,
                                                  cudaMemcpyHostToDevice, hp.h2d);
        if (e == cudaSuccess) e = cudaEventRecord(hp.in_done[sl], hp.h2d);
        // the group's attention, on the compute stream of its slot: consecutive groups' kernels sit
        // on different streams, so the next one's CTAs take the SMs that the previous one's last
        // CTAs leave (one persistent CTA per SM cannot keep every SM busy to the end)
        cudaStream_t cs = hp.comp[sl];
        if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, hp.in_done[sl], 0);
        if (e == cudaSuccess)
            e = tc ? launch_fwd_tc(pg, dq, dk, dv, dout, dl, kFwdFused, 0, sw, cs)
                   : launch_fwd_simt(pg, dq, dk, dv, dout, dl, kFwdFused, 0, cs);
        if (e == cudaSuccess) e = cudaEventRecord(hp.compute_done[sl], cs);
        // and its results back
        if (e == cudaSuccess) e = cudaStreamWaitEvent(hp.d2h, hp.compute_done[sl], 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(static_cast<char*>(out) + (size_t)gi * qbytes, dout, qbytes,
                                                  cudaMemcpyDeviceToHost, hp.d2h);
        if (e == cudaSuccess) e = cudaMemcpyAsync(reinterpret_cast<char*>(lse) + (size_t)gi * lbytes, dl, lbytes,
                                                  cudaMemcpyDeviceToHost, hp.d2h);
        if (e == cudaSuccess) e = cudaEventRecord(hp.out_done[sl], hp.d2h);
    }
    // the caller's stream completes only after the last results are on the host
    for (int sl = 0; sl < 2 && sl < groups && e == cudaSuccess; ++sl) e = cudaStreamWaitEvent(s, hp.out_done[sl], 0);
    if (e != cudaSuccess) return cuda_fail(e, "ring_attn_fwd_host");
    return RA_OK;
}

ra_status ring_attn_selftest_bounded_wait(unsigned long long limit_ns, unsigned int* returned, void* stream)
{
    if (limit_ns < 1000ull || limit_ns > 100000000ull)
        return fail(RA_ERR_INVALID_ARG, "limit_ns must be in [1e3, 1e8] (1 us to 100 ms)");
    ra_status st = check_ptrs({returned});
    if (st != RA_OK) return st;
    if ((st = check_device()) != RA_OK) return st;
    cudaError_t e;
    unsigned int* sw = status_word(&e);
    if (!sw) return cuda_fail(e, "status word");
    e = launch_bounded_wait_selftest(sw, limit_ns, static_cast<unsigned int*>(returned),
                                     static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ring_attn_selftest_bounded_wait launch");
    return RA_OK;
}

ra_status ring_attn_device_status(unsigned int* status, void* stream)
{
    if (!status) return fail(RA_ERR_INVALID_ARG, "status is NULL");
    ra_status st = check_device();
    if (st != RA_OK) return st;
    cudaError_t e;
    unsigned int* sw = status_word(&e);
    if (!sw) return cuda_fail(e, "status word");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int host = 0;
    e = cudaMemcpyAsync(&host, sw, sizeof(host), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(sw, 0, sizeof(unsigned int), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "ring_attn_device_status");
    *status = host;
    return RA_OK;
}

ra_status ring_attn_device_check(void* stream)
{
    unsigned int st = 0;
    ra_status r = ring_attn_device_status(&st, stream);
    if (r != RA_OK) return r;
    if (st & RA_DEVICE_TIMEOUT)
        return fail(RA_ERR_TIMEOUT,
                    "a bounded wait inside a kernel ran out: that kernel stopped early and its results are "
                    "incomplete (status word 0x%x)", st);
    if (st & RA_DEVICE_LAYOUT)
        return fail(RA_ERR_CUDA, "a kernel found its shared memory misaligned and did nothing (status word 0x%x)", st);
    return RA_OK;
}

// Host-side shard scheduler query.  Tiles are `tile` consecutive buffer rows from each shard's
// first row; a (query tile, key tile) pair counts when the smallest natural key position of the
// key tile does not exceed the largest natural query position of the query tile.  The per-tile
// extremes come from the chunk geometry, and the count uses the sorted key minima.
ra_status ring_attn_shard_tiles(int L, int n_shards, int causal, int layout, int tile,
                                long long* tiles_per_shard)
{
    if (!tiles_per_shard) return fail(RA_ERR_INVALID_ARG, "tiles_per_shard is NULL");
    if (tile < 1) return fail(RA_ERR_INVALID_ARG, "tile must be >= 1");
    Problem p{1, 1, 1, L, 64, n_shards, causal, layout, RA_F32};
    ra_status st = check_problem(p);
    if (st != RA_OK) return st;
    const Geometry g = p.geo();
    const long long tps = (g.S + tile - 1) / tile;
    const long long nt = tps * g.n;
    long long* kmin = new (std::nothrow) long long[nt];
    long long* qmax = new (std::nothrow) long long[nt];
    if (!kmin || !qmax) {
        delete[] kmin;
        delete[] qmax;
        return fail(RA_ERR_INVALID_ARG, "out of host memory");
    }
    for (long long x = 0; x < nt; ++x) {
        const int shard = (int)(x / tps);
        const int r0 = shard * g.S + (int)(x % tps) * tile;
        const int r1 = r0 + tile < (shard + 1) * g.S ? r0 + tile : (shard + 1) * g.S;
        long long lo = (long long)1 << 62, hi = -1;
        // the tile's rows split into runs of consecutive natural positions, one per chunk
        for (int r = r0; r < r1;) {
            const int c = r / g.Lc;
            const int run_end = (c + 1) * g.Lc < r1 ? (c + 1) * g.Lc : r1;
            const long long a = natural_position(g, r), b = natural_position(g, run_end - 1);
            lo = a < lo ? a : lo;
            hi = b > hi ? b : hi;
            r = run_end;
        }
        kmin[x] = lo;
        qmax[x] = hi;
    }
    // sort key minima (insertion into a counting array over natural positions)
    long long* hist = new (std::nothrow) long long[(size_t)L + 1];
    if (!hist) {
        delete[] kmin;
        delete[] qmax;
        return fail(RA_ERR_INVALID_ARG, "out of host memory");
    }
    memset(hist, 0, sizeof(long long) * ((size_t)L + 1));
    for (long long x = 0; x < nt; ++x) hist[kmin[x]] += 1;
    for (int pos = 1; pos <= L; ++pos) hist[pos] += hist[pos - 1];  // hist[p] = #tiles with min <= p
    for (int i = 0; i < g.n; ++i) {
        long long cnt = 0;
        for (long long a = 0; a < tps; ++a) {
            const long long x = (long long)i * tps + a;
            cnt += causal ? hist[qmax[x]] : nt;
        }
        tiles_per_shard[i] = cnt;
    }
    delete[] hist;
    delete[] kmin;
    delete[] qmax;
    return RA_OK;
}

}  // extern "C"
