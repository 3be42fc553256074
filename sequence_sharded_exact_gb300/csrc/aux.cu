// aux.cu -- HBM-bound kernels of libringattn: the log-sum-exp merge of ring-step partials, the
// backward preprocess D = rowsum(dO * O), float32 -> output conversion, and zero fill.
// All are grid-stride loops sized to a multiple of the SM count, with 16-byte accesses where the
// row length allows.
#include <cuda_bf16.h>
#include <math.h>

#include "ra_internal.h"

namespace ra {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// Merge of two normalised partial results of the same rows (online softmax across ring steps,
// LLM-101-CN "distributed hands-on code" section 6.2, rewritten for normalised partials):
//   lse = max(a, b) + log(1 + exp(-|a - b|)),  o = exp(a - lse) o_a + exp(b - lse) o_b.
// One warp per row.  For d = 128 (one float4 per lane) a warp takes four rows at a time and issues
// every load of them before it needs any, so that enough bytes are in flight to keep
// HBM busy; every lane reads both lse values before lane 0 overwrites lse_acc.
__device__ __forceinline__ void merge_weights(float a, float b, float& wa, float& wb, float& lse)
{
    const float mx = fmaxf(a, b);
    lse = mx + log1pf(expf(-fabsf(a - b)));
    wa = expf(a - lse);
    wb = expf(b - lse);
}

__global__ void __launch_bounds__(256)
lse_merge_kernel(float* __restrict__ o_acc, float* __restrict__ lse_acc,
                 const float* __restrict__ o_part, const float* __restrict__ lse_part,
                 long long rows, int d)
{
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    const long long w0 = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (d == 128) {
        constexpr int R = 4;  // rows per warp per iteration, all loaded before any is used
        for (long long r0 = R * w0; r0 < rows; r0 += R * warps) {
            float a[R], b[R];
            float4 x[R], y[R];
#pragma unroll
            for (int k = 0; k < R; ++k) {
                const long long r = r0 + k < rows ? r0 + k : r0;
                a[k] = lse_acc[r];
                b[k] = lse_part[r];
                x[k] = reinterpret_cast<const float4*>(o_acc + r * 128)[lane];
                y[k] = reinterpret_cast<const float4*>(o_part + r * 128)[lane];
            }
            __syncwarp();
#pragma unroll
            for (int k = 0; k < R; ++k) {
                const long long r = r0 + k;
                if (r >= rows || b[k] == -INFINITY) continue;  // an empty partial leaves the row unchanged
                float wa, wb, lse;
                merge_weights(a[k], b[k], wa, wb, lse);
                reinterpret_cast<float4*>(o_acc + r * 128)[lane] =
                    make_float4(wa * x[k].x + wb * y[k].x, wa * x[k].y + wb * y[k].y, wa * x[k].z + wb * y[k].z,
                                wa * x[k].w + wb * y[k].w);
                if (lane == 0) lse_acc[r] = lse;
            }
        }
        return;
    }
    for (long long row = w0; row < rows; row += warps) {
        const float a = lse_acc[row];
        const float b = lse_part[row];
        __syncwarp();
        if (b == -INFINITY) continue;
        float wa, wb, lse;
        merge_weights(a, b, wa, wb, lse);
        float* oa = o_acc + row * d;
        const float* ob = o_part + row * d;
        if ((d & 3) == 0) {
            for (int c = lane * 4; c < d; c += 128) {
                float4 x = *reinterpret_cast<const float4*>(oa + c);
                const float4 y = *reinterpret_cast<const float4*>(ob + c);
                x.x = wa * x.x + wb * y.x;
                x.y = wa * x.y + wb * y.y;
                x.z = wa * x.z + wb * y.z;
                x.w = wa * x.w + wb * y.w;
                *reinterpret_cast<float4*>(oa + c) = x;
            }
        } else {
            for (int c = lane; c < d; c += 32) oa[c] = wa * oa[c] + wb * ob[c];
        }
        if (lane == 0) lse_acc[row] = lse;
    }
}

template <typename T>
__device__ __forceinline__ float ldf(const T* p, long long i);
template <>
__device__ __forceinline__ float ldf<float>(const float* p, long long i) { return p[i]; }
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p, long long i)
{
    return __bfloat162float(p[i]);
}

// D[row] = sum_c out[row][c] * dout[row][c]; one warp per row.
template <typename T>
__global__ void __launch_bounds__(256)
bwd_preprocess_kernel(const T* __restrict__ out, const T* __restrict__ dout, long long rows, int d,
                      float* __restrict__ D)
{
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
         row += warps) {
        float acc = 0.f;
        const long long base = row * d;
        if (sizeof(T) == 2 && (d & 7) == 0) {
            for (int c = lane * 8; c < d; c += 256) {
                const uint4 xo = *reinterpret_cast<const uint4*>(out + base + c);
                const uint4 xd = *reinterpret_cast<const uint4*>(dout + base + c);
                const __nv_bfloat162* po = reinterpret_cast<const __nv_bfloat162*>(&xo);
                const __nv_bfloat162* pd = reinterpret_cast<const __nv_bfloat162*>(&xd);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 fo = __bfloat1622float2(po[e]);
                    const float2 fd = __bfloat1622float2(pd[e]);
                    acc = fmaf(fo.x, fd.x, acc);
                    acc = fmaf(fo.y, fd.y, acc);
                }
            }
        } else {
            for (int c = lane; c < d; c += 32) acc = fmaf(ldf(out, base + c), ldf(dout, base + c), acc);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
        if (lane == 0) D[row] = acc;
    }
}

// The same for bf16 rows of kD = 64 or 128 elements: kD / 8 lanes per row, 16 bytes each, so a warp
// covers 256 / kD rows per load and the whole warp is busy; four such row groups per iteration with
// all their loads issued before any is used (one row per warp, half the lanes idle at kD = 128 and one
// row's loads in flight, reached 0.74 of the copy bandwidth).
template <int kD>
__global__ void __launch_bounds__(256)
bwd_preprocess_bf16_kernel(const __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ dout,
                           long long rows, float* __restrict__ D)
{
    constexpr int kLanesPerRow = kD / 8;
    constexpr int kRowsPerLoad = 32 / kLanesPerRow;
    constexpr int kGroups = 4;
    constexpr int kRowsPerIter = kRowsPerLoad * kGroups;
    const int lane = threadIdx.x & 31;
    const int sub = lane / kLanesPerRow;
    const int c = (lane % kLanesPerRow) * 8;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    const long long w0 = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    for (long long r0 = w0 * kRowsPerIter; r0 < rows; r0 += warps * kRowsPerIter) {
        uint4 xo[kGroups], xd[kGroups];
#pragma unroll
        for (int k = 0; k < kGroups; ++k) {
            const long long row = r0 + k * kRowsPerLoad + sub;
            if (row < rows) {
                xo[k] = *reinterpret_cast<const uint4*>(out + row * kD + c);
                xd[k] = *reinterpret_cast<const uint4*>(dout + row * kD + c);
            } else {
                xo[k] = make_uint4(0u, 0u, 0u, 0u);
                xd[k] = xo[k];
            }
        }
#pragma unroll
        for (int k = 0; k < kGroups; ++k) {
            const __nv_bfloat162* po = reinterpret_cast<const __nv_bfloat162*>(&xo[k]);
            const __nv_bfloat162* pd = reinterpret_cast<const __nv_bfloat162*>(&xd[k]);
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 fo = __bfloat1622float2(po[e]);
                const float2 fd = __bfloat1622float2(pd[e]);
                acc = fmaf(fo.x, fd.x, acc);
                acc = fmaf(fo.y, fd.y, acc);
            }
#pragma unroll
            for (int o = kLanesPerRow / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
            const long long row = r0 + k * kRowsPerLoad + sub;
            if (lane % kLanesPerRow == 0 && row < rows) D[row] = acc;
        }
    }
}

// D from a float32 output and a bf16 dout (the forward's output kept before rounding): one warp per
// row, lanes over the row's elements.
__global__ void __launch_bounds__(256)
bwd_preprocess_f32out_kernel(const float* __restrict__ out, const __nv_bfloat16* __restrict__ dout, long long rows,
                             int d, float* __restrict__ D)
{
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
         row += warps) {
        const long long base = row * d;
        float acc = 0.f;
        for (int c = lane; c < d; c += 32) acc = fmaf(out[base + c], __bfloat162float(dout[base + c]), acc);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
        if (lane == 0) D[row] = acc;
    }
}

// The same for kD = 64 or 128: kD / 4 lanes per row, each 16 bytes of out and 8 of dout, four row
// groups per warp iteration with all their loads issued before any is used.
template <int kD>
__global__ void __launch_bounds__(256)
bwd_preprocess_f32out_vec_kernel(const float* __restrict__ out, const __nv_bfloat16* __restrict__ dout,
                                 long long rows, float* __restrict__ D)
{
    constexpr int kLanesPerRow = kD / 4;
    constexpr int kRowsPerLoad = 32 / kLanesPerRow;
    constexpr int kGroups = 4;
    constexpr int kRowsPerIter = kRowsPerLoad * kGroups;
    const int lane = threadIdx.x & 31;
    const int sub = lane / kLanesPerRow;
    const int c = (lane % kLanesPerRow) * 4;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    const long long w0 = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    for (long long r0 = w0 * kRowsPerIter; r0 < rows; r0 += warps * kRowsPerIter) {
        float4 xo[kGroups];
        uint2 xd[kGroups];
#pragma unroll
        for (int k = 0; k < kGroups; ++k) {
            const long long row = r0 + k * kRowsPerLoad + sub;
            if (row < rows) {
                xo[k] = *reinterpret_cast<const float4*>(out + row * kD + c);
                xd[k] = *reinterpret_cast<const uint2*>(dout + row * kD + c);
            } else {
                xo[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                xd[k] = make_uint2(0u, 0u);
            }
        }
#pragma unroll
        for (int k = 0; k < kGroups; ++k) {
            const __nv_bfloat162* pd = reinterpret_cast<const __nv_bfloat162*>(&xd[k]);
            const float2 d0 = __bfloat1622float2(pd[0]);
            const float2 d1 = __bfloat1622float2(pd[1]);
            float acc = fmaf(xo[k].x, d0.x, 0.f);
            acc = fmaf(xo[k].y, d0.y, acc);
            acc = fmaf(xo[k].z, d1.x, acc);
            acc = fmaf(xo[k].w, d1.y, acc);
#pragma unroll
            for (int o = kLanesPerRow / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
            const long long row = r0 + k * kRowsPerLoad + sub;
            if (lane % kLanesPerRow == 0 && row < rows) D[row] = acc;
        }
    }
}

__global__ void __launch_bounds__(256)
convert_kernel(const float* __restrict__ src, void* __restrict__ dst, int dst_dtype,
               long long count, float scale)
{
    const long long stride = (long long)gridDim.x * blockDim.x;
    const long long n4 = count >> 2;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
        float4 x = reinterpret_cast<const float4*>(src)[i];
        x.x *= scale;
        x.y *= scale;
        x.z *= scale;
        x.w *= scale;
        if (dst_dtype == 0) {
            reinterpret_cast<float4*>(dst)[i] = x;
        } else {
            __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(x.z, x.w);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&lo);
            pk.y = *reinterpret_cast<uint32_t*>(&hi);
            reinterpret_cast<uint2*>(dst)[i] = pk;
        }
    }
    for (long long i = (n4 << 2) + (long long)blockIdx.x * blockDim.x + threadIdx.x; i < count;
         i += stride) {
        const float x = src[i] * scale;
        if (dst_dtype == 0)
            static_cast<float*>(dst)[i] = x;
        else
            static_cast<__nv_bfloat16*>(dst)[i] = __float2bfloat16_rn(x);
    }
}

__global__ void __launch_bounds__(256) zero_kernel(float* __restrict__ dst, long long count)
{
    const long long stride = (long long)gridDim.x * blockDim.x;
    const long long n4 = count >> 2;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride)
        reinterpret_cast<float4*>(dst)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long i = (n4 << 2) + (long long)blockIdx.x * blockDim.x + threadIdx.x; i < count;
         i += stride)
        dst[i] = 0.f;
}

__global__ void __launch_bounds__(256)
add_kernel(float* __restrict__ acc, const float* __restrict__ part, long long count)
{
    const long long stride = (long long)gridDim.x * blockDim.x;
    const long long n4 = count >> 2;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
        const float4 a = reinterpret_cast<const float4*>(acc)[i];
        const float4 b = reinterpret_cast<const float4*>(part)[i];
        reinterpret_cast<float4*>(acc)[i] = make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
    }
    for (long long i = (n4 << 2) + (long long)blockIdx.x * blockDim.x + threadIdx.x; i < count;
         i += stride)
        acc[i] += part[i];
}

unsigned grid_for(long long work_items, int per_block)
{
    const long long want = (work_items + per_block - 1) / per_block;
    const long long cap = (long long)device_sm_count() * 8;  // 8 resident blocks of 256 per SM
    long long g = want < cap ? want : cap;
    return (unsigned)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_lse_merge(float* o_acc, float* lse_acc, const float* o_part,
                             const float* lse_part, long long rows, int d, cudaStream_t s)
{
    if (rows == 0) return cudaSuccess;
    lse_merge_kernel<<<grid_for(rows, 8), 256, 0, s>>>(o_acc, lse_acc, o_part, lse_part, rows, d);
    return cudaGetLastError();
}

cudaError_t launch_bwd_preprocess(const void* out, const void* dout, int dtype, long long rows,
                                  int d, float* D, cudaStream_t s, int out_dtype)
{
    if (rows == 0) return cudaSuccess;
    if (out_dtype == 0 && dtype == 1 && d == 128)
        bwd_preprocess_f32out_vec_kernel<128><<<grid_for((rows + 3) / 4, 8), 256, 0, s>>>(
            static_cast<const float*>(out), static_cast<const __nv_bfloat16*>(dout), rows, D);
    else if (out_dtype == 0 && dtype == 1 && d == 64)
        bwd_preprocess_f32out_vec_kernel<64><<<grid_for((rows + 7) / 8, 8), 256, 0, s>>>(
            static_cast<const float*>(out), static_cast<const __nv_bfloat16*>(dout), rows, D);
    else if (out_dtype == 0 && dtype == 1)
        bwd_preprocess_f32out_kernel<<<grid_for(rows, 8), 256, 0, s>>>(
            static_cast<const float*>(out), static_cast<const __nv_bfloat16*>(dout), rows, d, D);
    else if (dtype == 0)
        bwd_preprocess_kernel<float><<<grid_for(rows, 8), 256, 0, s>>>(
            static_cast<const float*>(out), static_cast<const float*>(dout), rows, d, D);
    else if (d == 128)
        bwd_preprocess_bf16_kernel<128><<<grid_for((rows + 7) / 8, 8), 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout), rows, D);
    else if (d == 64)
        bwd_preprocess_bf16_kernel<64><<<grid_for((rows + 15) / 16, 8), 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout), rows, D);
    else
        bwd_preprocess_kernel<__nv_bfloat16><<<grid_for(rows, 8), 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout), rows,
            d, D);
    return cudaGetLastError();
}

cudaError_t launch_convert(const float* src, void* dst, int dst_dtype, long long count,
                           float scale, cudaStream_t s)
{
    if (count == 0) return cudaSuccess;
    convert_kernel<<<grid_for((count + 3) / 4, 256), 256, 0, s>>>(src, dst, dst_dtype, count,
                                                                   scale);
    return cudaGetLastError();
}

cudaError_t launch_zero(float* dst, long long count, cudaStream_t s)
{
    if (count == 0) return cudaSuccess;
    zero_kernel<<<grid_for((count + 3) / 4, 256), 256, 0, s>>>(dst, count);
    return cudaGetLastError();
}

cudaError_t launch_add(float* acc, const float* part, long long count, cudaStream_t s)
{
    if (count == 0) return cudaSuccess;
    add_kernel<<<grid_for((count + 3) / 4, 256), 256, 0, s>>>(acc, part, count);
    return cudaGetLastError();
}

}  // namespace ra
