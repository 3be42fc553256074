// fwd_tc_body.cuh -- tensor-core forward of Ring Attention for sm_103a: bf16 inputs, head dim
// RA_FWD_HD (128 or 64), shard (contiguous, striped) or chunk (zigzag) length a multiple of 256.
// Compiled once per head dim (fwd_tc.cu: 128, fwd_tc_d64.cu: 64); the including file names the
// two host entry points through RA_FWD_SUPPORTED and RA_FWD_LAUNCH.
//
// Method (web pages on Ring Attention, cited by title and section):
//   block attention with a running max / running sum / running output (LLM-101-CN "distributed
//   hands-on code", section 6.2, block_attention), visited in ring order: the rows of shard i see
//   the K/V of shard (i - r) mod n at step r (same page, forward; "Lecture 30: TP/PP/SP/CP",
//   section 3.2); causal blocks entirely in the future are skipped and the diagonal is masked
//   (airsota "M4-051 Ring Attention and sequence parallelism", section 3); zigzag layout
//   (M4-051 section 4 item 2).  On one GPU the shards are row ranges of one buffer: the ring is the
//   order in which this kernel walks K/V tiles.
//
// Design (one CTA per SM, persistent):
//   * a work unit is one head and 256 consecutive query rows inside one chunk (two 128-row Q
//     tiles that share every K/V tile); units come in mirrored pairs (natural block u and U-1-u)
//     so that every CTA gets the same causal work; pairs are ordered kv head by kv head so that
//     concurrently running CTAs read the same K/V from L2.
//   * warp 8 (one thread) issues TMA loads: Q tiles, and K/V tiles through a 2-stage ring;
//     warps 10-11 only complete the third warpgroup, whose registers go to the softmax warps.
//   * warp 9 (one thread) issues tcgen05.mma: S_w = Q_w K^T into TMEM (w = 0, 1), then
//     O_w += P_w V with P_w read from TMEM; the S MMA of the next tile is issued between the two
//     P V products so that the tensor core works while the softmax warps do.
//   * warps 0-3 and 4-7 are the softmax warpgroups of Q tile 0 and 1: thread = row.  They read S
//     from TMEM (the whole row is in one thread, so row max and row sum need no shuffles), apply
//     the causal mask on diagonal tiles, compute P = 2^(S*scale*log2e - m) with ex2, write P as
//     bf16 over the S columns, keep the running sum, and rescale O in TMEM only when the running
//     max grows by more than 2^8 (the final O / l is exact whatever reference max is used, as
//     long as l and O share it).  They also write the epilogue: O / l in bf16, and lse.
//   * TMEM: S0 cols [0,128), S1 [128,256), O0 from 256, O1 from 384 (head-dim columns each).
//   * every wait is bounded; a wait that runs out sets the device status word and the CTA stops.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "ra_internal.h"
#include "ra_ptx.cuh"

namespace ra {
namespace {

constexpr int kTile = 128;                        // rows of a Q tile (MMA M) and of a K/V tile
constexpr int kHd = RA_FWD_HD;                    // head dim: 128 or 64
constexpr int kHalves = kHd / 64;                 // 128-byte-swizzle boxes (64 columns) per row
static_assert(kHd == 128 || kHd == 64, "head dim");
constexpr int kBlock = 2 * kTile;                 // query rows per work unit
constexpr int kStages = 2;                        // K/V pipeline depth
constexpr int kThreads = 384;                     // 12 warps (warps 10-11 idle)
constexpr uint32_t kHalfBytes = kTile * 64 * 2;   // 128 rows x 64 bf16 (one 128-byte-swizzle box)
constexpr uint32_t kTileBytes = kHalves * kHalfBytes;  // 128 rows x kHd bf16

constexpr uint32_t kSmemQ = 0;
constexpr uint32_t kSmemK = kSmemQ + 2 * kTileBytes;
constexpr uint32_t kSmemV = kSmemK + kStages * kTileBytes;
constexpr uint32_t kSmemBar = kSmemV + kStages * kTileBytes;

enum : int {
    BAR_Q_FULL = 0,
    BAR_Q_EMPTY = 1,
    BAR_K_FULL = 2,
    BAR_V_FULL = BAR_K_FULL + kStages,
    BAR_K_EMPTY = BAR_V_FULL + kStages,   // K tile read by both S MMAs of its K/V tile
    BAR_V_EMPTY = BAR_K_EMPTY + kStages,  // V tile read by both P V MMAs
    BAR_S_FULL = BAR_V_EMPTY + kStages,
    BAR_P_FULL = BAR_S_FULL + 2,
    BAR_O_DONE = BAR_P_FULL + 2,
    BAR_DRAIN = BAR_O_DONE + 2,
    BAR_COUNT = BAR_DRAIN + 1
};

constexpr uint32_t kSmemTmemSlot = kSmemBar + BAR_COUNT * 8;
constexpr uint32_t kSmemAbort = kSmemTmemSlot + 8;
constexpr uint32_t kSmemUsed = kSmemAbort + 8;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // slack for 1024-byte alignment of the base

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColO0 = 256;

constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s

struct FwdArgs {
    Geometry geo;
    int B, H, Hkv, G;
    int mode, step;
    int U;           // 256-row blocks per head (striped, block call: per shard)
    int pairs;       // mirrored block pairs per head (striped, block call: per shard)
    long long items; // B * H * pairs (striped: B * H * n * pairs)
    // One device's block call: only the rows of query shard q_shard, against one K/V block, with
    // q / out / lse and k / v in local buffers of qL = S rows per head.  A whole-sequence buffer row
    // r is local row r - q_off (queries) or r - kv_off (keys).  Otherwise blk = 0, the offsets are 0
    // and qL = L.
    int blk, q_shard, q_off, kv_off, qL;
    void* out;
    float* lse;
    unsigned int* status;
    unsigned long long* visits;  // optional [n][n] tile-pair counter
    float scale_log2;
};

struct Unit {
    int b, h, g;
    int r0;      // buffer row of the unit's first query row
    int p0;      // its natural position
    int p_hi;    // largest natural position among its rows
    int shard;   // query shard
    int ntiles;  // K/V tiles walked
};

// K/V tiles of a unit in ring order.
struct KvWalk {
    Geometry geo;
    int shard, p_hi, st, st_end, c, t, nt;
    KvRange kr;

    __device__ __forceinline__ void settle()
    {
        while (st < st_end) {
            kr = kv_range(geo, shard, st, c, p_hi);
            nt = (kr.count + kTile - 1) / kTile;  // a partial last tile is masked element-wise
            if (nt > 0) return;
            if (++c == geo.cps) {
                c = 0;
                ++st;
            }
        }
        nt = 0;
    }
    __device__ __forceinline__ void begin(const FwdArgs& a, const Unit& u)
    {
        geo = a.geo;
        shard = u.shard;
        p_hi = u.p_hi;
        st = fwd_all_steps(a.mode) ? 0 : a.step;
        st_end = fwd_all_steps(a.mode) ? a.geo.n : a.step + 1;
        c = 0;
        t = 0;
        settle();
    }
    __device__ __forceinline__ void next(int& row, int& nat)
    {
        row = kr.row0 + t * kTile;
        nat = kr.nat0 + t * kTile;
        if (++t == nt) {
            t = 0;
            if (++c == geo.cps) {
                c = 0;
                ++st;
            }
            settle();
        }
    }
};

__device__ __forceinline__ bool unit_of(const FwdArgs& a, long long item, int member, Unit& u)
{
    const int pair = (int)(item % a.pairs);
    long long rest = item / a.pairs;
    // striped and block calls: blocks of consecutive rows inside one shard
    const bool rowwise = a.geo.layout == 2 || a.blk;
    int shard = a.blk ? a.q_shard : 0;
    if (a.geo.layout == 2 && !a.blk) {
        shard = (int)(rest % a.geo.n);
        rest /= a.geo.n;
    }
    const int hg = (int)(rest % a.G);
    rest /= a.G;
    u.g = (int)(rest % a.Hkv);
    u.b = (int)(rest / a.Hkv);
    u.h = u.g * a.G + hg;
    const int blk = member == 0 ? pair : a.U - 1 - pair;
    if (member == 1 && blk == pair) return false;
    if (rowwise) {
        u.r0 = shard * a.geo.S + blk * kBlock;
        u.p0 = natural_position(a.geo, u.r0);
    } else {
        u.p0 = blk * kBlock;
        u.r0 = buffer_row(a.geo, u.p0);
    }
    u.p_hi = natural_position(a.geo, u.r0 + kBlock - 1);
    u.shard = u.r0 / a.geo.S;
    int nt = 0;
    const int s0 = fwd_all_steps(a.mode) ? 0 : a.step;
    const int s1 = fwd_all_steps(a.mode) ? a.geo.n : a.step + 1;
    for (int st = s0; st < s1; ++st)
        for (int c = 0; c < a.geo.cps; ++c) nt += (kv_range(a.geo, u.shard, st, c, u.p_hi).count + kTile - 1) / kTile;
    u.ntiles = nt;
    return true;
}

// Wait without the abort shortcut, for draining copies and MMAs already in flight.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > 1000000000ull) return;
    }
}

// ------------------------------------------------------------------------------------------------
// softmax warpgroups
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void softmax_role(const FwdArgs& a, uint32_t sbase, uint32_t tmem,
                                             const WaitCtl& ctl)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int w = warp >> 2;               // Q tile of this warpgroup
    const int rw = (warp & 3) * 32 + lane; // row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + kColS0 + (uint32_t)w * 128;
    const uint32_t tO = tmem + lane_off + kColO0 + (uint32_t)w * 128;
    const uint32_t bar_s = sbase + kSmemBar + 8 * (BAR_S_FULL + w);
    const uint32_t bar_p = sbase + kSmemBar + 8 * (BAR_P_FULL + w);
    const uint32_t bar_o = sbase + kSmemBar + 8 * (BAR_O_DONE + w);
    const float sl2 = a.scale_log2;
    uint32_t tcount = 0;

    for (long long item = blockIdx.x; item < a.items; item += gridDim.x) {
        for (int member = 0; member < 2; ++member) {
            Unit u;
            if (!unit_of(a, item, member, u)) continue;
            const long long row_g = ((long long)u.b * a.H + u.h) * a.qL + (u.r0 - a.q_off) + w * kTile + rw;
            if (u.ntiles == 0) {  // ring-step modes only: nothing visible from this block
                if (a.mode == kFwdRingStepAcc) continue;  // the running result stays as it is
                float* orow = static_cast<float*>(a.out) + row_g * kHd;
#pragma unroll
                for (int c = 0; c < kHd; c += 4)
                    *reinterpret_cast<float4*>(orow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
                a.lse[row_g] = -INFINITY;
                continue;
            }
            const int pq = u.p0 + w * kTile;  // natural position of this Q tile's first row (not striped)
            // l_run: running sum of the weights; c_run: running sum of (bf16(P_max) - P_max) over the
            // tiles (see below).  O is normalised by l_run + c_run, lse is m_run + log2(l_run).
            float m_run = -INFINITY, l_run = 0.f, c_run = 0.f;
            KvWalk walk;
            walk.begin(a, u);
            for (int jj = 0; jj < u.ntiles; ++jj, ++tcount) {
                int kv_row, kv_nat;
                walk.next(kv_row, kv_nat);
                // 0 all visible, 1 / 3 diagonal (key c visible to row r iff c <= r / c < r), 2 none;
                // the natural positions of tile starts decide it unless the layout is striped
                const int mask = a.geo.layout == 2 ? tile_mask(a.geo, u.r0 + w * kTile, kv_row)
                                 : (!a.geo.causal ? 0 : (kv_nat < pq ? 0 : (kv_nat == pq ? 1 : 2)));
                // keys c > lim of this row are masked
                const int lim = mask == 2 ? -1 : (mask == 3 ? rw - 1 : rw);
                if (!mbar_wait(bar_s, tcount & 1, ctl)) return;
                tc_fence_after_sync();
                __syncwarp();
                uint32_t r[4][32];
                // First half of the row, then the second half's loads overlap the first half's max.
                tmem_ld_32x32b_x32(tS + 0, r[0]);
                tmem_ld_32x32b_x32(tS + 32, r[1]);
                tmem_ld_wait(r[0]);
                tmem_ld_wait(r[1]);
                tmem_ld_32x32b_x32(tS + 64, r[2]);
                tmem_ld_32x32b_x32(tS + 96, r[3]);
                float m8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) m8[i] = -INFINITY;
                if (mask != 0) {
#pragma unroll
                    for (int c4 = 0; c4 < 2; ++c4)
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if ((c4 * 32 + e) > lim) r[c4][e] = __float_as_uint(-INFINITY);
                }
#pragma unroll
                for (int c4 = 0; c4 < 2; ++c4)
#pragma unroll
                    for (int e = 0; e < 32; e += 2)
                        m8[(e >> 1) & 7] = max3f(m8[(e >> 1) & 7], __uint_as_float(r[c4][e]), __uint_as_float(r[c4][e + 1]));
                tmem_ld_wait(r[2]);
                tmem_ld_wait(r[3]);
                if (mask != 0) {
#pragma unroll
                    for (int c4 = 2; c4 < 4; ++c4)
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if ((c4 * 32 + e) > lim) r[c4][e] = __float_as_uint(-INFINITY);
                }
#pragma unroll
                for (int c4 = 2; c4 < 4; ++c4)
#pragma unroll
                    for (int e = 0; e < 32; e += 2)
                        m8[(e >> 1) & 7] = max3f(m8[(e >> 1) & 7], __uint_as_float(r[c4][e]), __uint_as_float(r[c4][e + 1]));
                const float mx = max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
                const float m_tile = mx * sl2;
                float m_new = m_run;
                if (m_tile > m_run + 8.0f) m_new = m_tile;
                const float alpha = (m_new == m_run) ? 1.0f : ex2_approx(m_run - m_new);
                const float ref = m_new == -INFINITY ? 0.f : m_new;
                const float2 scale2 = make_float2(sl2, sl2), nref2 = make_float2(-ref, -ref);
                float2 s4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) s4[i] = make_float2(0.f, 0.f);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t pk[32];
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const int c4 = half * 2 + cc;
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float2 x2 = fma2(make_float2(__uint_as_float(r[c4][e]), __uint_as_float(r[c4][e + 1])),
                                                   scale2, nref2);
                            const float2 p2 = make_float2(ex2_approx(x2.x), ex2_approx(x2.y));
                            s4[(e >> 1) & 3] = add2(s4[(e >> 1) & 3], p2);
                            pk[cc * 16 + e / 2] = pack_bf16x2(p2.x, p2.y);
                        }
                    }
                    tmem_st_32x32b_x32(tS + half * 32, pk);
                }
                const float2 s2 = add2(add2(s4[0], s4[1]), add2(s4[2], s4[3]));
                // P V multiplies V by the weights rounded to bf16, while the sum above adds them
                // unrounded.  For the tile's largest weight the difference is kept, so that the output
                // of a row dominated by one key is normalised by exactly the weight its V row received
                // (the same fma and ex2 as that element: the same value bit for bit); lse keeps the
                // unrounded sum.
                const float p_max = ex2_approx(fmaf(mx, sl2, -ref));
                const float p_max_bf16 = __uint_as_float(pack_bf16x2(p_max, 0.f) << 16);
                const float rsum = s2.x + s2.y;
                l_run = l_run * alpha + rsum;
                c_run = c_run * alpha + (p_max_bf16 - p_max);
                tmem_st_wait();
                const bool need = jj > 0 && alpha != 1.0f;
                if (__any_sync(0xffffffffu, need)) {
                    // O of the previous tile must be complete before it is rescaled.
                    if (!mbar_wait(bar_o, (tcount - 1) & 1, ctl)) return;
                    tc_fence_after_sync();
#pragma unroll 1
                    for (int c4 = 0; c4 < kHd / 32; ++c4) {
                        uint32_t o[32];
                        tmem_ld_32x32b_x32(tO + c4 * 32, o);
                        tmem_ld_wait(o);
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float2 v = mul2(make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])),
                                                  make_float2(alpha, alpha));
                            o[e] = __float_as_uint(v.x);
                            o[e + 1] = __float_as_uint(v.y);
                        }
                        tmem_st_32x32b_x32(tO + c4 * 32, o);
                    }
                    tmem_st_wait();
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_p);
                m_run = m_new;
            }
            // epilogue: wait for the last P V product of this tile
            if (!mbar_wait(bar_o, (tcount - 1) & 1, ctl)) return;
            tc_fence_after_sync();
            __syncwarp();
            const bool any = l_run > 0.f;
            const float inv = any ? 1.0f / (l_run + c_run) : 0.f;
            if (a.mode == kFwdFused) {
                __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) + row_g * kHd;
#pragma unroll 1
                for (int c4 = 0; c4 < kHd / 32; ++c4) {
                    uint32_t o[32];
                    tmem_ld_32x32b_x32(tO + c4 * 32, o);
                    tmem_ld_wait(o);
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
                    uint4* dst = reinterpret_cast<uint4*>(orow + c4 * 32);
#pragma unroll
                    for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                }
            } else if (a.mode == kFwdRingStepAcc) {
                // fold this step into the running (out, lse): the online-softmax update across ring
                // steps, on normalised results.  A row that saw no key in this step stays as it is;
                // the TMEM loads stay warp-uniform, only the global update is per row.
                const float acc = a.lse[row_g];
                float wa = 1.f, wb = 0.f, lse = acc;
                if (any) {
                    const float b = (m_run + log2f(l_run)) * kLn2;
                    const float mx = fmaxf(acc, b);
                    lse = mx + log1pf(expf(-fabsf(acc - b)));
                    wa = acc == -INFINITY ? 0.f : expf(acc - lse);
                    wb = expf(b - lse) * inv;
                }
                float* orow = static_cast<float*>(a.out) + row_g * kHd;
#pragma unroll 1
                for (int c4 = 0; c4 < kHd / 32; ++c4) {
                    uint32_t o[32];
                    tmem_ld_32x32b_x32(tO + c4 * 32, o);
                    tmem_ld_wait(o);
                    if (!any) continue;
                    float4* dst = reinterpret_cast<float4*>(orow + c4 * 32);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        // a running row with lse = -inf holds nothing yet: its o_acc is not read
                        const float4 x = wa != 0.f ? dst[e] : make_float4(0.f, 0.f, 0.f, 0.f);
                        dst[e] = make_float4(wa * x.x + wb * __uint_as_float(o[4 * e]), wa * x.y + wb * __uint_as_float(o[4 * e + 1]),
                                             wa * x.z + wb * __uint_as_float(o[4 * e + 2]),
                                             wa * x.w + wb * __uint_as_float(o[4 * e + 3]));
                    }
                }
                a.lse[row_g] = lse;
                continue;
            } else {
                float* orow = static_cast<float*>(a.out) + row_g * kHd;
#pragma unroll 1
                for (int c4 = 0; c4 < kHd / 32; ++c4) {
                    uint32_t o[32];
                    tmem_ld_32x32b_x32(tO + c4 * 32, o);
                    tmem_ld_wait(o);
                    float4* dst = reinterpret_cast<float4*>(orow + c4 * 32);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        dst[e] = make_float4(__uint_as_float(o[4 * e]) * inv, __uint_as_float(o[4 * e + 1]) * inv,
                                             __uint_as_float(o[4 * e + 2]) * inv, __uint_as_float(o[4 * e + 3]) * inv);
                }
            }
            a.lse[row_g] = any ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
        }
    }
}

// ------------------------------------------------------------------------------------------------
// TMA producer (one thread)
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void producer_role(const FwdArgs& a, uint32_t sbase, const CUtensorMap* tmQ,
                                              const CUtensorMap* tmK, const CUtensorMap* tmV,
                                              const WaitCtl& ctl)
{
    auto bar = [&](int i) { return sbase + kSmemBar + 8u * (uint32_t)i; };
    tma_prefetch_desc(tmQ);
    tma_prefetch_desc(tmK);
    tma_prefetch_desc(tmV);
    // Each Q tile is read once; K/V tiles are read again by every unit of the kv head.  Q's lines go
    // first when L2 needs room (L = 131072, one A/B on one box: DRAM reads per launch 4.3 -> 3.6 GB,
    // time unchanged; across boxes the reads vary by as much; the same hint on K/V as evict_last,
    // or on the output stores, raised the reads instead).
    const uint64_t pol_q = l2_policy_evict_first();
    uint32_t kc = 0, qc = 0;
    bool ok = true;
    for (long long item = blockIdx.x; ok && item < a.items; item += gridDim.x) {
        for (int member = 0; ok && member < 2; ++member) {
            Unit u;
            if (!unit_of(a, item, member, u) || u.ntiles == 0) continue;
            if (qc > 0 && !mbar_wait(bar(BAR_Q_EMPTY), (qc - 1) & 1, ctl)) { ok = false; break; }
            mbar_arrive_expect_tx(bar(BAR_Q_FULL), 2 * kTileBytes);
            const int zq = u.b * a.H + u.h;
#pragma unroll
            for (int w = 0; w < 2; ++w)
#pragma unroll
                for (int half = 0; half < kHalves; ++half)
                    tma_load_3d_hint(sbase + kSmemQ + (uint32_t)(w * kHalves + half) * kHalfBytes, tmQ,
                                     bar(BAR_Q_FULL), half * 64, u.r0 - a.q_off + w * kTile, zq, pol_q);
            ++qc;
            const int zkv = u.b * a.Hkv + u.g;
            KvWalk walk;
            walk.begin(a, u);
            for (int jj = 0; jj < u.ntiles; ++jj, ++kc) {
                int kv_row, kv_nat;
                walk.next(kv_row, kv_nat);
                if (a.visits) atomicAdd(a.visits + (long long)u.shard * a.geo.n + kv_row / a.geo.S, 1ull);
                const int stage = (int)(kc % kStages);
                const uint32_t use = kc / kStages;
                // K and V stages are released separately: K once both S MMAs of its tile are done,
                // about a K/V-tile period before V, so the next K loads that much earlier.
                if (use > 0 && !mbar_wait(bar(BAR_K_EMPTY + stage), (use - 1) & 1, ctl)) { ok = false; break; }
                mbar_arrive_expect_tx(bar(BAR_K_FULL + stage), kTileBytes);
#pragma unroll
                for (int half = 0; half < kHalves; ++half)
                    tma_load_3d(sbase + kSmemK + (uint32_t)stage * kTileBytes + (uint32_t)half * kHalfBytes, tmK,
                                bar(BAR_K_FULL + stage), half * 64, kv_row - a.kv_off, zkv);
                if (use > 0 && !mbar_wait(bar(BAR_V_EMPTY + stage), (use - 1) & 1, ctl)) { ok = false; break; }
                mbar_arrive_expect_tx(bar(BAR_V_FULL + stage), kTileBytes);
#pragma unroll
                for (int half = 0; half < kHalves; ++half)
                    tma_load_3d(sbase + kSmemV + (uint32_t)stage * kTileBytes + (uint32_t)half * kHalfBytes, tmV,
                                bar(BAR_V_FULL + stage), half * 64, kv_row - a.kv_off, zkv);
            }
        }
    }
    // Copies still in flight must land before the CTA's shared memory goes away.
    if (qc > 0) drain_wait(bar(BAR_Q_FULL), (qc - 1) & 1);
    for (uint32_t s = 0; s < kStages && s < kc; ++s) {
        const uint32_t last_use = (kc - 1 - s) / kStages;  // stage (kc-1-s) % kStages
        const int stage = (int)((kc - 1 - s) % kStages);
        drain_wait(bar(BAR_K_FULL + stage), last_use & 1);
        drain_wait(bar(BAR_V_FULL + stage), last_use & 1);
    }
}

// ------------------------------------------------------------------------------------------------
// MMA issuer (one thread)
// ------------------------------------------------------------------------------------------------
struct UnitCursor {
    long long item;
    int member;
    Unit u;
    __device__ __forceinline__ bool advance(const FwdArgs& a)
    {
        while (true) {
            if (++member == 2) {
                member = 0;
                item += gridDim.x;
            }
            if (item >= a.items) return false;
            if (unit_of(a, item, member, u) && u.ntiles > 0) return true;
        }
    }
};

// Operand descriptors of the issue loops: low words of the Q, K and V tiles' descriptors (K and V
// at stage 0), built once; a k-step or a stage is a constant added to them.
struct FwdDesc {
    uint32_t q, k, v;
};
constexpr uint32_t kDescHi = sdesc_sw128_hi(1024);

__device__ __forceinline__ void issue_qk(const FwdDesc& dsc, uint32_t tmem, int w, int stage)
{
    constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, false);
    const uint32_t kb = dsc.k + (uint32_t)stage * (kTileBytes >> 4);
#pragma unroll
    for (int kk = 0; kk < kHd / 16; ++kk) {
        const uint32_t half = (uint32_t)(kk >> 2), koff = (uint32_t)(kk & 3) * 32u;
        const uint64_t ad = sdesc_at(dsc.q, ((uint32_t)w * kHalves + half) * kHalfBytes + koff, kDescHi);
        const uint64_t bd = sdesc_at(kb, half * kHalfBytes + koff, kDescHi);
        mma_ss(tmem + kColS0 + (uint32_t)w * 128, ad, bd, idesc, kk > 0 ? 1u : 0u);
    }
}

__device__ __forceinline__ void issue_pv(const FwdDesc& dsc, uint32_t tmem, int w, int stage, bool accumulate)
{
    constexpr uint32_t idesc = idesc_bf16_f32(128, kHd, false, true);
    const uint32_t vb = dsc.v + (uint32_t)stage * (kTileBytes >> 4);
    const uint32_t acc0 = accumulate ? 1u : 0u;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint64_t bd = sdesc_at(vb, (uint32_t)kk * 2048u, kDescHi);
        mma_ts(tmem + kColO0 + (uint32_t)w * 128, tmem + kColS0 + (uint32_t)w * 128 + (uint32_t)kk * 8, bd, idesc,
               kk > 0 ? 1u : acc0);
    }
}

__device__ __forceinline__ void mma_role(const FwdArgs& a, uint32_t sbase, uint32_t tmem, const WaitCtl& ctl)
{
    auto bar = [&](int i) { return sbase + kSmemBar + 8u * (uint32_t)i; };
    UnitCursor cur;
    cur.item = blockIdx.x;
    cur.member = -1;
    bool issued = false;
    FwdDesc dsc;
    dsc.q = sdesc_sw128_lo(sbase + kSmemQ, 16);
    dsc.k = sdesc_sw128_lo(sbase + kSmemK, 16);
    dsc.v = sdesc_sw128_lo(sbase + kSmemV, kHalfBytes);
    if (cur.advance(a)) {
        issued = true;
        uint32_t kc = 0, tc = 0, qc = 0;
        int jj = 0;
        // prologue: S of the first tile
        if (!mbar_wait(bar(BAR_Q_FULL), qc & 1, ctl)) goto drain;
        if (!mbar_wait(bar(BAR_K_FULL + 0), 0, ctl)) goto drain;
        tc_fence_after_sync();
        issue_qk(dsc, tmem, 0, 0);
        tc_commit(bar(BAR_S_FULL + 0));
        issue_qk(dsc, tmem, 1, 0);
        tc_commit(bar(BAR_S_FULL + 1));
        tc_commit(bar(BAR_K_EMPTY + 0));
        if (cur.u.ntiles == 1) tc_commit(bar(BAR_Q_EMPTY));
        while (true) {
            const int stage = (int)(kc % kStages);
            const uint32_t use = kc / kStages;
            // next tile
            UnitCursor nxt = cur;
            int jn = jj + 1;
            bool has_next = true;
            if (jn == cur.u.ntiles) {
                jn = 0;
                has_next = nxt.advance(a);
            }
            const uint32_t nkc = kc + 1;
            const int nstage = (int)(nkc % kStages);
            const uint32_t nuse = nkc / kStages;

            if (!mbar_wait(bar(BAR_V_FULL + stage), use & 1, ctl)) goto drain;
            if (!mbar_wait(bar(BAR_P_FULL + 0), tc & 1, ctl)) goto drain;
            tc_fence_after_sync();
            issue_pv(dsc, tmem, 0, stage, jj > 0);
            tc_commit(bar(BAR_O_DONE + 0));
            if (has_next) {
                if (jn == 0) {
                    ++qc;
                    if (!mbar_wait(bar(BAR_Q_FULL), qc & 1, ctl)) goto drain;
                }
                if (!mbar_wait(bar(BAR_K_FULL + nstage), nuse & 1, ctl)) goto drain;
                tc_fence_after_sync();
                issue_qk(dsc, tmem, 0, nstage);
                tc_commit(bar(BAR_S_FULL + 0));
            }
            if (!mbar_wait(bar(BAR_P_FULL + 1), tc & 1, ctl)) goto drain;
            tc_fence_after_sync();
            issue_pv(dsc, tmem, 1, stage, jj > 0);
            tc_commit(bar(BAR_O_DONE + 1));
            tc_commit(bar(BAR_V_EMPTY + stage));
            if (!has_next) break;
            issue_qk(dsc, tmem, 1, nstage);
            tc_commit(bar(BAR_S_FULL + 1));
            tc_commit(bar(BAR_K_EMPTY + nstage));
            if (jn == nxt.u.ntiles - 1) tc_commit(bar(BAR_Q_EMPTY));
            cur = nxt;
            jj = jn;
            kc = nkc;
            ++tc;
        }
    }
drain:
    if (issued) {
        // every MMA issued by this thread has completed once this barrier flips
        tc_commit(bar(BAR_DRAIN));
        drain_wait(bar(BAR_DRAIN), 0);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const FwdArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemAbort);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmemTmemSlot);

    if (threadIdx.x == 0) {
        for (int i = 0; i < BAR_COUNT; ++i) {
            const uint32_t cnt = (i == BAR_P_FULL || i == BAR_P_FULL + 1) ? 4u : 1u;
            mbar_init(sbase + kSmemBar + 8u * (uint32_t)i, cnt);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl ctl{abort_flag, a.status, kWaitLimitNs};

    // Register split: launched with 384 x 168 = 64512 registers; softmax warpgroups 2 x 128 x 192
    // plus the TMA/MMA warpgroup 128 x 120 = 64512 (per SM sub-partition 192 + 192 + 120 = 504).
    if (warp < 8)
        asm volatile("setmaxnreg.inc.sync.aligned.u32 192;" ::: "memory");
    else
        asm volatile("setmaxnreg.dec.sync.aligned.u32 120;" ::: "memory");

    if (warp < 8) {
        softmax_role(a, sbase, tmem, ctl);
    } else if (warp == 8) {
        if ((threadIdx.x & 31) == 0) producer_role(a, sbase, &tmQ, &tmK, &tmV, ctl);
    } else if (warp == 9) {
        if ((threadIdx.x & 31) == 0) mma_role(a, sbase, tmem, ctl);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 3-D map over a [heads][L][kHd] bf16 tensor, box = 64 columns x 128 rows x 1 head, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int L, long long heads)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kHd, (cuuint64_t)L, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)kHd * 2, (cuuint64_t)L * kHd * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kTile, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

bool RA_FWD_SUPPORTED(const Problem& p)
{
    if (p.dtype != 1 || p.d != kHd) return false;
    const Geometry g = p.geo();
    return g.Lc % kBlock == 0;
}

cudaError_t RA_FWD_LAUNCH(const Problem& p, const void* q, const void* k, const void* v, void* out,
                          float* lse, int mode, int step, unsigned int* status, cudaStream_t s,
                          unsigned long long* visits, const BlockView* blk)
{
    FwdArgs a;
    a.geo = p.geo();
    a.blk = blk ? 1 : 0;
    a.q_shard = blk ? blk->q_shard : 0;
    a.q_off = blk ? blk->q_shard * a.geo.S : 0;
    a.kv_off = blk ? blk->kv_shard * a.geo.S : 0;
    a.qL = blk ? a.geo.S : p.L;  // rows per head of every buffer (local shard buffers in a block call)
    CUtensorMap tq, tk, tv;
    if (!make_map(&tq, q, a.qL, (long long)p.B * p.H) || !make_map(&tk, k, a.qL, (long long)p.B * p.Hkv) ||
        !make_map(&tv, v, a.qL, (long long)p.B * p.Hkv))
        return cudaErrorInvalidValue;
    a.B = p.B;
    a.H = p.H;
    a.Hkv = p.Hkv;
    a.G = p.H / p.Hkv;
    a.mode = mode;
    a.step = step;
    a.U = (p.layout == 2 || blk ? p.L / p.n : p.L) / kBlock;
    a.pairs = (a.U + 1) / 2;
    a.items = (long long)p.B * p.H * a.pairs * (p.layout == 2 && !blk ? p.n : 1);
    a.out = out;
    a.lse = lse;
    a.status = status;
    a.visits = visits;
    a.scale_log2 = kLog2e / sqrtf((float)kHd);

    // The shared-memory opt-in is set once per device; the lock makes concurrent first launches from
    // several host threads safe.
    static std::mutex attr_mu;
    static bool attr_done[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lk(attr_mu);
        if (!attr_done[dev]) {
            e = cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
            if (e != cudaSuccess) return e;
            attr_done[dev] = true;
        }
    }
    const long long sms = device_sm_count();
    const unsigned grid = (unsigned)(a.items < sms ? a.items : sms);
    fwd_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(tq, tk, tv, a);
    return cudaGetLastError();
}

}  // namespace ra
