// rope.cu -- rotary position embedding by natural position, in place (HBM-bound).
//
// LLM-101-CN "distributed hands-on code" (section 6, the questions after the 6.2 implementation)
// asks how position information must be handled once K/V blocks travel round the ring.  Here every
// row turns by the angle of its natural position p -- its place in the whole sequence, which the
// layout fixes -- and never by its buffer row or its index inside a shard, so a K/V block carries
// its positions with it wherever the ring takes it.  The rotation is the RoFormer one: for i in [0, d/2) with
// theta_i = base^(-2i/d) the pair (x[2i], x[2i+1]) turns by p * theta_i (by -p * theta_i for the
// inverse, which maps gradients with respect to rotated rows back to the unrotated ones).
//
// Angle reduction: theta_i / (2 pi) is held as a 64-bit fixed-point fraction of a turn, so that
// p * theta_i modulo one turn is an exact integer product (mod 2^64); its top 32 bits give the
// fraction of a turn for sincospif.  The error stays below 1e-6 rad at any position the int index
// reaches, where float32 arithmetic on p * theta_i would lose ~1e-2 rad at p = 131072.
//
// One thread owns a 16-byte chunk of one (batch, position) row and computes its angles once, then
// rotates that chunk in every head (the heads of a position share its angles).
// A buffer holds `rows` rows per head: the whole sequence (rows = L, row_off = 0), or one device's
// shard (rows = S = L / n, row_off = shard * S: local row r is whole-sequence row r + row_off).
#include <cuda_bf16.h>
#include <math.h>

#include "ra_internal.h"

namespace ra {
namespace {

struct RopeArgs {
    Geometry geo;
    int B, H;
    int rows, row_off;  // rows per head in the buffer; whole-sequence row of local row 0
    int inverse;
    unsigned long long turn[64];  // theta_i / (2 pi) in units of 2^-64 turn
};

__device__ __forceinline__ void rotate(float& x0, float& x1, float c, float s)
{
    const float y0 = x0 * c - x1 * s;
    const float y1 = x0 * s + x1 * c;
    x0 = y0;
    x1 = y1;
}

template <int D>
__global__ void __launch_bounds__(256) rope_bf16_kernel(__nv_bfloat16* __restrict__ x, const RopeArgs a)
{
    constexpr int kChunks = D / 8;  // 8 bf16 = 4 pairs per chunk
    const long long L = a.rows;
    const long long total = (long long)a.B * L * kChunks;
    const long long step = (long long)gridDim.x * blockDim.x;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += step) {
        const int ch = (int)(idx % kChunks);
        const long long br = idx / kChunks;
        const int r = (int)(br % L);
        const int b = (int)(br / L);
        const unsigned long long p = (unsigned long long)natural_position(a.geo, r + a.row_off);
        float c[4], s[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const unsigned long long u = p * a.turn[ch * 4 + j];
            const float t = (float)(unsigned)(u >> 32) * 2.3283064365386963e-10f;  // 2^-32
            sincospif(2.0f * t, &s[j], &c[j]);
            if (a.inverse) s[j] = -s[j];
        }
        uint4* ptr = reinterpret_cast<uint4*>(x + ((long long)b * a.H * L + r) * D) + ch;
        const long long hstride = L * D / 8;
        for (int h = 0; h < a.H; ++h, ptr += hstride) {
            uint4 v = *ptr;
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                __nv_bfloat162 pr = *reinterpret_cast<__nv_bfloat162*>(&w[j]);
                float x0 = __low2float(pr), x1 = __high2float(pr);
                rotate(x0, x1, c[j], s[j]);
                pr = __floats2bfloat162_rn(x0, x1);
                w[j] = *reinterpret_cast<uint32_t*>(&pr);
            }
            *ptr = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

template <int D>
__global__ void __launch_bounds__(256) rope_f32_kernel(float* __restrict__ x, const RopeArgs a)
{
    constexpr int kChunks = D / 4;  // 4 floats = 2 pairs per chunk
    const long long L = a.rows;
    const long long total = (long long)a.B * L * kChunks;
    const long long step = (long long)gridDim.x * blockDim.x;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += step) {
        const int ch = (int)(idx % kChunks);
        const long long br = idx / kChunks;
        const int r = (int)(br % L);
        const int b = (int)(br / L);
        const unsigned long long p = (unsigned long long)natural_position(a.geo, r + a.row_off);
        float c[2], s[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const unsigned long long u = p * a.turn[ch * 2 + j];
            const float t = (float)(unsigned)(u >> 32) * 2.3283064365386963e-10f;  // 2^-32
            sincospif(2.0f * t, &s[j], &c[j]);
            if (a.inverse) s[j] = -s[j];
        }
        float4* ptr = reinterpret_cast<float4*>(x + ((long long)b * a.H * L + r) * D) + ch;
        const long long hstride = L * D / 4;
        for (int h = 0; h < a.H; ++h, ptr += hstride) {
            float4 v = *ptr;
            rotate(v.x, v.y, c[0], s[0]);
            rotate(v.z, v.w, c[1], s[1]);
            *ptr = v;
        }
    }
}

unsigned rope_grid(long long items)
{
    const long long want = (items + 255) / 256;
    const long long cap = (long long)device_sm_count() * 8;
    const long long g = want < cap ? want : cap;
    return (unsigned)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_rope(const Problem& p, void* x, double base, int inverse, cudaStream_t s, int shard)
{
    RopeArgs a;
    a.geo = p.geo();
    a.B = p.B;
    a.H = p.H;
    a.rows = shard < 0 ? p.L : p.L / p.n;
    a.row_off = shard < 0 ? 0 : shard * (p.L / p.n);
    a.inverse = inverse ? 1 : 0;
    const double two_pi = 6.283185307179586476925;
    for (int i = 0; i < 64; ++i) {
        a.turn[i] = 0;
        if (i < p.d / 2) {
            double frac = pow(base, -2.0 * i / p.d) / two_pi;  // turns per position
            frac -= floor(frac);                                 // only the fraction of a turn matters
            a.turn[i] = (unsigned long long)ldexp(frac, 64);
        }
    }
    const long long rows = (long long)p.B * a.rows;
    if (p.dtype == 1) {
        const long long items = rows * (p.d / 8);
        if (p.d == 128)
            rope_bf16_kernel<128><<<rope_grid(items), 256, 0, s>>>(static_cast<__nv_bfloat16*>(x), a);
        else
            rope_bf16_kernel<64><<<rope_grid(items), 256, 0, s>>>(static_cast<__nv_bfloat16*>(x), a);
    } else {
        const long long items = rows * (p.d / 4);
        if (p.d == 128)
            rope_f32_kernel<128><<<rope_grid(items), 256, 0, s>>>(static_cast<float*>(x), a);
        else
            rope_f32_kernel<64><<<rope_grid(items), 256, 0, s>>>(static_cast<float*>(x), a);
    }
    return cudaGetLastError();
}

}  // namespace ra
