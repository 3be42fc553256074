// ulysses.cu -- the all-to-all re-layout of the Ulysses variant of sequence parallelism (HBM-bound).
//
// "Lecture 30: TP/PP/SP/CP", section 3.3 (DeepSpeed-Ulysses; section 3.4 compares it with the ring)
// describes the other context-parallel design: every one of n devices holds all heads of its
// S = L / n tokens, [B, S, H, d]; an all-to-all turns that into H / n heads of the whole sequence,
// [B, L, H / n, d];
// each device then runs ordinary attention over the full sequence for its heads, and a second
// all-to-all brings the output back to the token split.  The heads must therefore divide by n.
//
// On one GPU the n devices are n slices of one allocation and the all-to-all is a permutation of
// rows.  A row is the d contiguous elements of one (token, head); it is contiguous in both forms,
// so the permutation moves whole rows with 16-byte accesses:
//   token split  [n][B][S][H][d]: rank i, local token s (the layout fixes which natural token that
//                 is: contiguous, zigzag or striped, as for the ring), head h;
//   head split   [n][B][H/n][L][d]: rank h / (H/n), head h % (H/n), natural position p -- the
//                 head-major form the attention kernels read, one full-sequence problem per rank.
// direction 0 maps the token split to the head split, direction 1 the reverse.  Rows of 4 bytes
// (the float32 lse) use 4-byte words.
#include <cuda_bf16.h>
#include <stdint.h>

#include "ra_internal.h"

namespace ra {
namespace {

struct A2AArgs {
    Geometry geo;      // L, n, layout of the token split
    int B, H;          // heads of the tensor (all ranks)
    int words;         // words of Word type per row
    int direction;     // 0: token split -> head split, 1: head split -> token split
};

// One thread per word; WORDS words per row (0: a.words at run time).  Index arithmetic in 32 bits
// (the caller guarantees rows * words < 2^32): the row decomposition is most of the work.
template <typename Word, int WORDS>
__global__ void __launch_bounds__(256) a2a_kernel(const Word* __restrict__ src, Word* __restrict__ dst, const A2AArgs a)
{
    const unsigned words = WORDS > 0 ? (unsigned)WORDS : (unsigned)a.words;
    const unsigned S = (unsigned)a.geo.S, L = (unsigned)a.geo.L, H = (unsigned)a.H, B = (unsigned)a.B;
    const unsigned Hn = H / (unsigned)a.geo.n;
    const unsigned total = (unsigned)a.geo.L * B * H * words;
    const unsigned step = gridDim.x * blockDim.x;
    for (unsigned idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += step) {
        const unsigned wi = idx % words;
        const unsigned t = idx / words;  // token-split row: ((i * B + b) * S + s) * H + h
        const unsigned h = t % H;
        unsigned rest = t / H;
        const unsigned s = rest % S;
        rest /= S;
        const unsigned b = rest % B;
        const unsigned i = rest / B;
        const unsigned p = (unsigned)natural_position(a.geo, (int)(i * S + s));
        const unsigned long long hrow = ((unsigned long long)((h / Hn) * B + b) * Hn + (h % Hn)) * L + p;
        if (a.direction == 0)
            dst[hrow * words + wi] = src[(unsigned long long)t * words + wi];
        else
            dst[(unsigned long long)t * words + wi] = src[hrow * words + wi];
    }
}

unsigned a2a_grid(long long items)
{
    const long long want = (items + 255) / 256;
    const long long cap = (long long)device_sm_count() * 8;
    const long long g = want < cap ? want : cap;
    return (unsigned)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_ulysses_a2a(const Geometry& geo, int B, int H, int row_bytes, const void* src, void* dst,
                               int direction, cudaStream_t s)
{
    A2AArgs a;
    a.geo = geo;
    a.B = B;
    a.H = H;
    a.direction = direction;
    const long long rows = (long long)geo.L * B * H;
    a.words = row_bytes % 16 == 0 ? row_bytes / 16 : row_bytes / 4;
    const long long items = rows * a.words;
    if (items >= (1LL << 32)) return cudaErrorInvalidValue;  // the kernels index in 32 bits
    const unsigned grid = a2a_grid(items);
    if (row_bytes % 16 == 0) {
        const uint4* in = static_cast<const uint4*>(src);
        uint4* out = static_cast<uint4*>(dst);
        if (a.words == 16)
            a2a_kernel<uint4, 16><<<grid, 256, 0, s>>>(in, out, a);  // bf16, d = 128
        else if (a.words == 8)
            a2a_kernel<uint4, 8><<<grid, 256, 0, s>>>(in, out, a);
        else if (a.words == 32)
            a2a_kernel<uint4, 32><<<grid, 256, 0, s>>>(in, out, a);
        else
            a2a_kernel<uint4, 0><<<grid, 256, 0, s>>>(in, out, a);
    } else if (a.words == 1) {
        a2a_kernel<uint32_t, 1><<<grid, 256, 0, s>>>(static_cast<const uint32_t*>(src), static_cast<uint32_t*>(dst), a);
    } else {
        a2a_kernel<uint32_t, 0><<<grid, 256, 0, s>>>(static_cast<const uint32_t*>(src), static_cast<uint32_t*>(dst), a);
    }
    return cudaGetLastError();
}

}  // namespace ra
