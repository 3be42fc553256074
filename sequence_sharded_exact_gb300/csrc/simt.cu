// simt.cu -- CUDA-core kernels of libringattn for every shape the tensor-core path does not take
// (float32 inputs, head dim 64, chunks that are not a multiple of 256 rows, ...).
//
// Forward: one warp per query row.  The row walks the ring schedule (step r uses the K/V of shard
// (i - r) mod n; LLM-101-CN "distributed hands-on code" section 6.2) in groups of 32 keys: each lane
// scores one key, warp shuffles give the group's maximum and sum, and the running state
// (max M, sum L, output O) is rescaled by exp(M - M_new) as in block_attention.  Causal keys past
// the row's natural position are never visited (airsota M4-051 section 3).
// Backward: one warp per query row for dQ and one warp per key row for dK/dV, recomputing
// P = exp(s - lse) from the saved lse.
// Block calls (one device of the multi-device ring): the rows are those of one query shard and the
// keys those of one K/V shard, in local buffers of qL = S rows per head; a whole-sequence buffer
// row r is local row r - q_off (queries) or r - kv_off (keys).  Whole-sequence calls have zero
// offsets and qL = L.
#include <cuda_bf16.h>
#include <math.h>

#include "ra_internal.h"

namespace ra {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarps = 8;  // warps per block

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_max(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    return x;
}

template <typename T, int D>
__device__ __forceinline__ float dot_row(const float* __restrict__ a_smem, const T* __restrict__ b)
{
    float acc = 0.f;
#pragma unroll 16
    for (int c = 0; c < D; ++c) acc = fmaf(a_smem[c], to_f(b[c]), acc);
    return acc;
}

// ---------------------------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32)
fwd_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                void* __restrict__ out, float* __restrict__ lse, Geometry geo, int B, int H,
                int Hkv, int mode, int step, float scale_log2, int q_off, int kv_off, int qL)
{
    constexpr int EPL = D / 32;
    __shared__ float qs[kWarps][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kWarps + warp;
    if (row >= (long long)B * H * qL) return;
    const int r = (int)(row % qL) + q_off;  // whole-sequence buffer row
    const int h = (int)((row / qL) % H);
    const int b = (int)(row / ((long long)qL * H));
    const int g = h / (H / Hkv);
    for (int c = lane; c < D; c += 32) qs[warp][c] = to_f(q[row * D + c]);
    __syncwarp();
    const T* kh = k + ((long long)b * Hkv + g) * qL * D;  // key row t (whole sequence) is local row t - kv_off
    const T* vh = v + ((long long)b * Hkv + g) * qL * D;
    const int i = r / geo.S;
    const int p = natural_position(geo, r);

    float m = -INFINITY, l = 0.f, o[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] = 0.f;
    const int s0 = fwd_all_steps(mode) ? 0 : step;
    const int s1 = fwd_all_steps(mode) ? geo.n : step + 1;
    for (int st = s0; st < s1; ++st) {
        for (int c = 0; c < geo.cps; ++c) {
            const KvRange kr = kv_range(geo, i, st, c, p);
            for (int base = 0; base < kr.count; base += 32) {
                const int t = base + lane;
                float s = -INFINITY;
                if (t < kr.count) s = dot_row<T, D>(qs[warp], kh + (long long)(kr.row0 - kv_off + t) * D) * scale_log2;
                const float m_new = fmaxf(m, warp_max(s));
                const float ref = m_new == -INFINITY ? 0.f : m_new;
                const float alpha = exp2f(m - ref);
                const float pr = exp2f(s - ref);
                l = l * alpha + warp_sum(pr);
#pragma unroll
                for (int e = 0; e < EPL; ++e) o[e] *= alpha;
                const int nvalid = min(32, kr.count - base);
                for (int tt = 0; tt < nvalid; ++tt) {
                    const float pt = __shfl_sync(kFull, pr, tt);
                    const T* vrow = vh + (long long)(kr.row0 - kv_off + base + tt) * D;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) o[e] = fmaf(pt, to_f(vrow[lane + 32 * e]), o[e]);
                }
                m = m_new;
            }
        }
    }
    if (mode == kFwdFused) {
        const float inv = 1.f / l;
        T* orow = static_cast<T*>(out) + row * D;
#pragma unroll
        for (int e = 0; e < EPL; ++e) orow[lane + 32 * e] = from_f<T>(o[e] * inv);
        if (lane == 0) lse[row] = (m + log2f(l)) * kLn2;
    } else if (mode == kFwdRingStepAcc) {
        // fold this step into the running (out, lse); an empty step leaves the row as it is
        if (!(l > 0.f)) return;
        const float b = (m + log2f(l)) * kLn2;
        const float acc = lse[row];
        __syncwarp();  // every lane has read lse before lane 0 overwrites it
        const float mx = fmaxf(acc, b);
        const float nl = mx + log1pf(expf(-fabsf(acc - b)));
        const float wa = acc == -INFINITY ? 0.f : expf(acc - nl);
        const float wb = expf(b - nl) / l;
        float* orow = static_cast<float*>(out) + row * D;
        // a running row with lse = -inf holds nothing yet: its o_acc is not read
#pragma unroll
        for (int e = 0; e < EPL; ++e) orow[lane + 32 * e] = (wa != 0.f ? wa * orow[lane + 32 * e] : 0.f) + wb * o[e];
        if (lane == 0) lse[row] = nl;
    } else {
        float* orow = static_cast<float*>(out) + row * D;
        const bool any = l > 0.f;
        const float inv = any ? 1.f / l : 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) orow[lane + 32 * e] = any ? o[e] * inv : 0.f;
        if (lane == 0) lse[row] = any ? (m + log2f(l)) * kLn2 : -INFINITY;
    }
}

// ---------------------------------------------------------------------------------------------
// backward
// ---------------------------------------------------------------------------------------------
template <typename T, typename G, int D>
__global__ void __launch_bounds__(kWarps * 32)
bwd_dq_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                   const T* __restrict__ dout, const float* __restrict__ Dv,
                   const float* __restrict__ lse, G* __restrict__ dq, Geometry geo, int B, int H,
                   int Hkv, float scale, float scale_log2, int s0, int s1, int q_off, int kv_off, int qL,
                   int acc_dq)
{
    constexpr int EPL = D / 32;
    __shared__ float qs[kWarps][D];
    __shared__ float ds[kWarps][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kWarps + warp;
    if (row >= (long long)B * H * qL) return;
    const int r = (int)(row % qL) + q_off;  // whole-sequence buffer row
    const int h = (int)((row / qL) % H);
    const int b = (int)(row / ((long long)qL * H));
    const int g = h / (H / Hkv);
    for (int c = lane; c < D; c += 32) {
        qs[warp][c] = to_f(q[row * D + c]);
        ds[warp][c] = to_f(dout[row * D + c]);
    }
    __syncwarp();
    const T* kh = k + ((long long)b * Hkv + g) * qL * D;  // key row t (whole sequence) is local row t - kv_off
    const T* vh = v + ((long long)b * Hkv + g) * qL * D;
    const int i = r / geo.S;
    const int p = natural_position(geo, r);
    const float lse2 = lse[row] * kLog2e;
    const float Drow = Dv[row];
    float acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    for (int st = s0; st < s1; ++st) {
        for (int c = 0; c < geo.cps; ++c) {
            const KvRange kr = kv_range(geo, i, st, c, p);
            for (int base = 0; base < kr.count; base += 32) {
                const int t = base + lane;
                float dS = 0.f;
                if (t < kr.count) {
                    const long long kv = (long long)(kr.row0 - kv_off + t) * D;
                    const float s = dot_row<T, D>(qs[warp], kh + kv) * scale_log2;
                    const float dP = dot_row<T, D>(ds[warp], vh + kv);
                    dS = exp2f(s - lse2) * (dP - Drow);
                }
                const int nvalid = min(32, kr.count - base);
                for (int tt = 0; tt < nvalid; ++tt) {
                    const float w = __shfl_sync(kFull, dS, tt);
                    const T* krow = kh + (long long)(kr.row0 - kv_off + base + tt) * D;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) acc[e] = fmaf(w, to_f(krow[lane + 32 * e]), acc[e]);
                }
            }
        }
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        const long long x = row * D + lane + 32 * e;
        dq[x] = from_f<G>(acc_dq ? to_f(dq[x]) + acc[e] * scale : acc[e] * scale);
    }
}

// One warp per key row t of kv head (b, g): the query rows that see it are visited shard by shard
// in the order the K/V block of shard j meets them on the ring (shard (j + step) mod n at step).
template <typename T, typename G, int D>
__global__ void __launch_bounds__(kWarps * 32)
bwd_dkv_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                    const T* __restrict__ dout, const float* __restrict__ Dv,
                    const float* __restrict__ lse, G* __restrict__ dk, G* __restrict__ dv,
                    Geometry geo, int B, int H, int Hkv, float scale, float scale_log2, int s0, int s1,
                    int q_off, int kv_off, int qL, int acc_kv)
{
    constexpr int EPL = D / 32;
    __shared__ float ks[kWarps][D];
    __shared__ float vs[kWarps][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long krow = (long long)blockIdx.x * kWarps + warp;
    if (krow >= (long long)B * Hkv * qL) return;
    const int t = (int)(krow % qL) + kv_off;  // whole-sequence buffer row
    const int g = (int)((krow / qL) % Hkv);
    const int b = (int)(krow / ((long long)qL * Hkv));
    const int G_ = H / Hkv;
    for (int c = lane; c < D; c += 32) {
        ks[warp][c] = to_f(k[krow * D + c]);
        vs[warp][c] = to_f(v[krow * D + c]);
    }
    __syncwarp();
    const int j = t / geo.S;
    const int pt = natural_position(geo, t);
    float ak[EPL], av[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) ak[e] = av[e] = 0.f;
    for (int hh = 0; hh < G_; ++hh) {
        // local query row = whole-sequence row - q_off
        const long long hb = ((long long)b * H + (long long)g * G_ + hh) * qL - q_off;
        for (int st = s0; st < s1; ++st) {
            for (int c = 0; c < geo.cps; ++c) {
                const KvRange qr = q_range(geo, j, st, c, pt);
                for (int base = 0; base < qr.count; base += 32) {
                    const int x = base + lane;
                    float P = 0.f, dS = 0.f;
                    if (x < qr.count) {
                        const long long prow = hb + qr.row0 + x;
                        const float s = dot_row<T, D>(ks[warp], q + prow * D) * scale_log2;
                        const float dP = dot_row<T, D>(vs[warp], dout + prow * D);
                        P = exp2f(s - lse[prow] * kLog2e);
                        dS = P * (dP - Dv[prow]);
                    }
                    const int nvalid = min(32, qr.count - base);
                    for (int tt = 0; tt < nvalid; ++tt) {
                        const float wp = __shfl_sync(kFull, P, tt);
                        const float ws = __shfl_sync(kFull, dS, tt);
                        const long long prow = (hb + qr.row0 + base + tt) * D;
#pragma unroll
                        for (int e = 0; e < EPL; ++e) {
                            av[e] = fmaf(wp, to_f(dout[prow + lane + 32 * e]), av[e]);
                            ak[e] = fmaf(ws, to_f(q[prow + lane + 32 * e]), ak[e]);
                        }
                    }
                }
            }
        }
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        const long long x = krow * D + lane + 32 * e;
        dk[x] = from_f<G>(acc_kv ? to_f(dk[x]) + ak[e] * scale : ak[e] * scale);
        dv[x] = from_f<G>(acc_kv ? to_f(dv[x]) + av[e] : av[e]);
    }
}

// Row addressing of a call: whole-sequence buffers, or one device's block call (local shard buffers).
struct Rows {
    int q_off, kv_off, qL;
};

Rows rows_of(const Problem& p, const BlockView* blk)
{
    const int S = p.L / p.n;
    return blk ? Rows{blk->q_shard * S, blk->kv_shard * S, S} : Rows{0, 0, p.L};
}

template <typename T, int D>
cudaError_t fwd_simt_typed(const Problem& p, const void* q, const void* k, const void* v,
                           void* out, float* lse, int mode, int step, cudaStream_t s, const BlockView* blk)
{
    const Rows rw = rows_of(p, blk);
    const long long rows = (long long)p.B * p.H * rw.qL;
    const unsigned grid = (unsigned)((rows + kWarps - 1) / kWarps);
    const float scale_log2 = kLog2e / sqrtf((float)D);
    fwd_simt_kernel<T, D><<<grid, kWarps * 32, 0, s>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), out, lse,
        p.geo(), p.B, p.H, p.Hkv, mode, step, scale_log2, rw.q_off, rw.kv_off, rw.qL);
    return cudaGetLastError();
}

template <typename T, typename G, int D>
cudaError_t bwd_simt_typed(const Problem& p, const void* q, const void* k, const void* v,
                           const void* dout, const float* Dv, const float* lse, void* dq,
                           void* dk, void* dv, cudaStream_t s, const BlockView* blk)
{
    const float scale = 1.f / sqrtf((float)D);
    const float scale_log2 = kLog2e * scale;
    const Rows rw = rows_of(p, blk);
    // a block call walks its one ring step and adds dQ (and, if asked, dK, dV) into float32 outputs
    const int s0 = blk ? (blk->q_shard - blk->kv_shard + p.n) % p.n : 0;
    const int s1 = blk ? s0 + 1 : p.n;
    const unsigned gq = (unsigned)(((long long)p.B * p.H * rw.qL + kWarps - 1) / kWarps);
    bwd_dq_simt_kernel<T, G, D><<<gq, kWarps * 32, 0, s>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v),
        static_cast<const T*>(dout), Dv, lse, static_cast<G*>(dq), p.geo(), p.B, p.H, p.Hkv, scale,
        scale_log2, s0, s1, rw.q_off, rw.kv_off, rw.qL, blk ? 1 : 0);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const unsigned gk = (unsigned)(((long long)p.B * p.Hkv * rw.qL + kWarps - 1) / kWarps);
    bwd_dkv_simt_kernel<T, G, D><<<gk, kWarps * 32, 0, s>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v),
        static_cast<const T*>(dout), Dv, lse, static_cast<G*>(dk), static_cast<G*>(dv), p.geo(),
        p.B, p.H, p.Hkv, scale, scale_log2, s0, s1, rw.q_off, rw.kv_off, rw.qL, blk ? blk->acc_kv : 0);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t bwd_simt_grad(const Problem& p, const void* q, const void* k, const void* v,
                          const void* dout, const float* Dv, const float* lse, void* dq, void* dk,
                          void* dv, int grad_dtype, cudaStream_t s, const BlockView* blk)
{
    if (grad_dtype == 0 || blk)  // a block call's gradients are float32
        return bwd_simt_typed<T, float, D>(p, q, k, v, dout, Dv, lse, dq, dk, dv, s, blk);
    return bwd_simt_typed<T, __nv_bfloat16, D>(p, q, k, v, dout, Dv, lse, dq, dk, dv, s, blk);
}

}  // namespace

cudaError_t launch_fwd_simt(const Problem& p, const void* q, const void* k, const void* v,
                            void* out, float* lse, int mode, int step, cudaStream_t s, const BlockView* blk)
{
    if (p.dtype == 0)
        return p.d == 64 ? fwd_simt_typed<float, 64>(p, q, k, v, out, lse, mode, step, s, blk)
                         : fwd_simt_typed<float, 128>(p, q, k, v, out, lse, mode, step, s, blk);
    return p.d == 64 ? fwd_simt_typed<__nv_bfloat16, 64>(p, q, k, v, out, lse, mode, step, s, blk)
                     : fwd_simt_typed<__nv_bfloat16, 128>(p, q, k, v, out, lse, mode, step, s, blk);
}

cudaError_t launch_bwd_simt(const Problem& p, const void* q, const void* k, const void* v,
                            const void* dout, const float* Dv, const float* lse, void* dq,
                            void* dk, void* dv, int grad_dtype, cudaStream_t s, const BlockView* blk)
{
    if (p.dtype == 0)
        return p.d == 64
                   ? bwd_simt_grad<float, 64>(p, q, k, v, dout, Dv, lse, dq, dk, dv, grad_dtype, s, blk)
                   : bwd_simt_grad<float, 128>(p, q, k, v, dout, Dv, lse, dq, dk, dv, grad_dtype, s, blk);
    return p.d == 64 ? bwd_simt_grad<__nv_bfloat16, 64>(p, q, k, v, dout, Dv, lse, dq, dk, dv,
                                                        grad_dtype, s, blk)
                     : bwd_simt_grad<__nv_bfloat16, 128>(p, q, k, v, dout, Dv, lse, dq, dk, dv,
                                                         grad_dtype, s, blk);
}

}  // namespace ra
