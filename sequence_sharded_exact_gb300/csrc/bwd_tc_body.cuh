// bwd_tc_body.cuh -- tensor-core backward of Ring Attention for sm_103a: bf16 inputs, head dim
// RA_BWD_HD (128 or 64), shard (contiguous, striped) or chunk (zigzag) length a multiple of 128.
// Compiled once per head dim (bwd_tc.cu: 128, bwd_tc_d64.cu: 64); the including file names the
// two host entry points through RA_BWD_SUPPORTED and RA_BWD_LAUNCH.
//
// The pages describe the forward only; the backward is the derivative of the same definition,
// with the attention weights recomputed from the saved log-sum-exp (never stored):
//   P = exp(s - lse),  dS = P (dO . v - D),  D = rowsum(dO * O),
//   dV = P^T dO,  dK = scale dS^T Q,  dQ = scale dS K,
// dK and dV summed over the query heads that share a kv head.  Causal blocks that are entirely
// masked are skipped and the diagonal tiles are masked element by element.
// Ring order: the K/V block of shard j meets the queries of shard (j + r) mod n at step r (the K/V
// travels to the next device at every step, LLM-101-CN "distributed hands-on code" section 6.2),
// so a K/V tile walks the query shards in that order.
//
// Design (one CTA per SM, persistent; a work unit is one 128-row K/V tile of one kv head, units in
// mirrored pairs so that causal work is equal across CTAs, the leftover pairs of the last round
// split into single tiles; the unit walks 128-row query tiles, so
// that every product is a 128 x 128 x 128 one -- an N = 64 instruction costs nearly as long as an
// N = 128 one on this tensor core):
//   * warp 12: TMA loads of the unit's K and V tiles and, through 2 stages, of each query tile's Q
//     (with its lse) and dO (with its D); the vectors come by bulk copy into shared memory.
//   * warp 13: tcgen05.mma issue, per query tile t, in this order:
//       dV += P^T_t dO_t (P^T from TMEM), S^T_{t+1} = K Q_{t+1}^T, dQ^T_t = K^T dS^T_t,
//       dK += dS^T_t Q_t (dS^T from shared memory for both), dP^T_{t+1} = V dO_{t+1}^T.
//     S^T of the next tile runs while the math warps compute dS^T of this one; dQ^T goes before
//     dK so that its read-out (which frees the columns of the next dP^T) overlaps dK.
//   * warps 0-7 (two warpgroups, each owning 64 of the 128 query columns; thread = key row), per
//     query tile t:
//       phase A: P^T_t = 2^(S^T c - lse2) -> registers and, as bf16, TMEM (A operand of dV);
//       phase B: dS^T_t = P^T_t (dP^T_t - D) / sqrt(d) -> shared memory (operand of dK and dQ^T);
//     at the end of a unit, the dK, dV write-out.
//   * warps 8-11 (thread = head-dim index): read dQ^T_t out of TMEM, free its columns and add it
//     into the float32 accumulator in global memory with coalesced reductions (one warp
//     instruction covers 32 consecutive head-dim entries of one query row), paced so that they do
//     not crowd the other warps' shared-memory traffic out of the memory-instruction queue.
//   * TMEM columns (head dim 128): X = [0,128) S^T then P^T; Y = [128,256) dP^T, then dQ^T once
//     phase B has read dP^T; dK [256,384), dV [384,512).
//   * head dim 64: K, V, Q and dO tiles are one 128-byte-swizzle box wide instead of two, and
//     dK, dV use 64 columns.  dQ^T = K^T dS^T keeps M = 128 (the tensor core's 128-lane layout,
//     the one the dQ warps read) with K loaded twice, so that its rows 64-127 repeat rows 0-63:
//     warps 8-9 add query columns 0-63, warps 10-11 columns 64-127.  dQ^T has TMEM columns of its
//     own there (X 0, Y 128, dQ^T 256, dK 384, dV 448), so the next dP^T does not wait for the
//     dQ read-out.
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

constexpr int kKT = 128;       // K/V tile rows
constexpr int kQT = 128;       // query tile rows
constexpr int kHd = RA_BWD_HD;  // head dim: 128 or 64
static_assert(kHd == 128 || kHd == 64, "head dim");
constexpr int kHalves = kHd / 64;  // 128-byte-swizzle boxes (64 bf16 head-dim columns) per row
constexpr int kStages = 2;     // query-tile stages (Q + lse, dO + D)
constexpr int kThreads = 512;  // 16 warps: 0-7 math, 8-11 dQ, 12 TMA loads, 13 MMA, 14-15 idle
constexpr uint32_t kHalf = 128 * 128;            // 16 KB: 128 rows x 64 bf16 columns
constexpr uint32_t kTileBytes = kHalves * kHalf; // a 128-row K, V, Q or dO tile (32 KB at d = 128)
constexpr uint32_t kDsBytes = 2 * kHalf;         // dS^T: 128 keys x 128 queries (bf16)
constexpr uint32_t kVecBytes = kQT * 4;          // lse or D of one query tile (float32)

// Head dim 64 has TMEM and shared memory to spare: dQ^T gets columns of its own (so the next dP^T
// need not wait for the dQ read-out), and K is loaded twice, back to back, so that the M = 128
// product dQ^T = K^T dS^T computes its rows 0-63 twice and all four dQ warps can reduce (rows
// 0-63 give the query columns 0-63, rows 64-127 the columns 64-127).
constexpr bool kD64 = kHd == 64;
constexpr uint32_t kSmemK = 0;                                   // d = 64: K, then K again
constexpr uint32_t kSmemV = kSmemK + (kD64 ? 2 : 1) * kTileBytes;
constexpr uint32_t kSmemQ = kSmemV + kTileBytes;                 // kStages x 32 KB
constexpr uint32_t kSmemDO = kSmemQ + kStages * kTileBytes;      // kStages x 32 KB
constexpr uint32_t kSmemDS = kSmemDO + kStages * kTileBytes;     // dS^T: 2 query blocks x 128 keys x 128 B
constexpr uint32_t kSmemLse = kSmemDS + kDsBytes;                // kStages x 512 B
constexpr uint32_t kSmemD = kSmemLse + kStages * kVecBytes;      // kStages x 512 B
constexpr uint32_t kSmemBar = kSmemD + kStages * kVecBytes;

enum : int {
    BAR_KV_FULL = 0,
    BAR_KV_EMPTY,
    BAR_Q_FULL,                           // kStages: Q tile and its lse landed
    BAR_DO_FULL = BAR_Q_FULL + kStages,   // kStages: dO tile and its D landed
    BAR_Q_EMPTY = BAR_DO_FULL + kStages,  // kStages: S^T and dK have read the Q tile
    BAR_DO_EMPTY = BAR_Q_EMPTY + kStages, // kStages: dP^T and dV have read the dO tile
    BAR_ST_FULL = BAR_DO_EMPTY + kStages,
    BAR_DPT_FULL,
    BAR_P_READY,   // 8 math warps
    BAR_DS_READY,  // 8 math warps
    BAR_DQ_FULL,
    BAR_DQ_FREE,   // 4 dQ warps
    BAR_ACC_FULL,
    BAR_ACC_FREE,  // 8 math warps
    BAR_DRAIN,
    BAR_COUNT
};

constexpr uint32_t kSmemTmemSlot = kSmemBar + BAR_COUNT * 8;
constexpr uint32_t kSmemAbort = kSmemTmemSlot + 8;
constexpr uint32_t kSmemBytes = kSmemAbort + 8;
// The base of dynamic shared memory sits right after the 1 KB the system reserves, so it is
// 1024-byte aligned (the 128-byte swizzle atoms need that); the kernel checks it and stops with
// RA_DEVICE_LAYOUT if not, instead of reserving 1 KB of slack that this layout does not have.
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kColX = 0, kColY = 128;
constexpr uint32_t kColDQ = kD64 ? 256 : kColY;  // d = 128: dQ^T reuses Y once phase B has read dP^T
constexpr uint32_t kColDK = kD64 ? 384 : 256, kColDV = kD64 ? 448 : 384;
constexpr uint64_t kWaitLimitNs = 4000000000ull;

struct BwdArgs {
    Geometry geo;
    int B, H, Hkv, G;
    int T;            // 128-row K/V tiles per head (striped, block call: per shard)
    int pairs;        // mirrored tile pairs per kv head (striped, block call: per shard)
    long long items;  // B * Hkv * pairs (striped: B * Hkv * n * pairs)
    // One device's block call: only the K/V tiles of shard kv_shard, met by the queries of shard
    // (kv_shard + step) mod n at ring step `step` alone, with q / dout / lse / D / dq in local
    // buffers of qL = S rows per head and k / v / dk / dv in local buffers of S rows: a
    // whole-sequence row r is local row r - q_off (queries) or r - kv_off (keys).  dK and dV are then
    // float32 and added to (acc_kv = 1) or stored (acc_kv = 0; a tile that meets no query gets zeros).
    // Otherwise blk = 0, every step is walked, the offsets are 0 and qL = L.
    int blk, kv_shard, step, q_off, kv_off, qL, acc_kv;
    const float* lse;
    const float* Dv;
    float* dq_acc;
    void* dk;
    void* dv;
    int grad_bf16;
    unsigned int* status;
    unsigned long long* visits;  // optional [n][n] tile-pair counter
    float scale, scale_log2;
};

struct KvUnit {
    int b, g;
    int rk;        // buffer row of the K/V tile
    int pk;        // natural position of its first row
    int shard;     // kv shard
    int per_head;  // query tiles per head
    int ntiles;    // query tiles over all heads of the group
    int rev;       // walk the heads of the group last to first (the second tile of a mirrored pair)
};

// The query rows of chunk c of the shard the K/V tile meets at step st that can see it, widened
// down to a query-tile boundary (striped: the first visible row may sit inside a tile).
__device__ __forceinline__ KvRange q_tile_range(const Geometry& g, int shard, int st, int c, int pk)
{
    KvRange qr = q_range(g, shard, st, c, pk);
    if (qr.count == 0) return qr;
    int i = shard + st;
    if (i >= g.n) i -= g.n;
    const int cs = (i * g.cps + c) * g.Lc;  // first row of that chunk
    const int off = (qr.row0 - cs) / kQT * kQT;
    qr.nat0 -= (qr.row0 - cs - off) * g.stride;
    qr.row0 = cs + off;
    qr.count = g.Lc - off;
    return qr;
}

__device__ __forceinline__ int q_tiles_per_head(const BwdArgs& a, int shard, int pk)
{
    int nt = 0;
    const int s0 = a.blk ? a.step : 0, s1 = a.blk ? a.step + 1 : a.geo.n;
    for (int st = s0; st < s1; ++st)
        for (int c = 0; c < a.geo.cps; ++c) nt += q_tile_range(a.geo, shard, st, c, pk).count / kQT;
    return nt;
}

__device__ __forceinline__ bool unit_of(const BwdArgs& a, long long item, int member, KvUnit& u)
{
    // striped and block calls: tiles of consecutive rows inside one shard
    const bool rowwise = a.geo.layout == 2 || a.blk;
    int shard = a.blk ? a.kv_shard : 0;
    int pair;
    long long rest;
    if (a.geo.layout == 2 && !a.blk) {
        // Striped: the shard index varies fastest, so that the CTAs running at the same time hold the
        // same few local tiles of every shard -- tiles whose query walks are equally long.  With the
        // pair index fastest they held every local tile of a few shards, walked the query heads at
        // rates up to 1.9x apart, and spread their Q, dO and dQ over all heads of the group at once
        // (L2 read misses 30%, 206 GB of DRAM traffic per 64K launch).
        shard = (int)(item % a.geo.n);
        rest = item / a.geo.n;
        pair = (int)(rest % a.pairs);
        rest /= a.pairs;
    } else {
        pair = (int)(item % a.pairs);
        rest = item / a.pairs;
    }
    u.g = (int)(rest % a.Hkv);
    u.b = (int)(rest / a.Hkv);
    const int tile = member == 0 ? pair : a.T - 1 - pair;
    if (member == 1 && tile == pair) return false;
    if (rowwise) {
        u.rk = shard * a.geo.S + tile * kKT;
        u.pk = natural_position(a.geo, u.rk);
    } else {
        u.pk = tile * kKT;
        u.rk = buffer_row(a.geo, u.pk);
    }
    u.shard = u.rk / a.geo.S;
    u.per_head = q_tiles_per_head(a, u.shard, u.pk);
    u.rev = member & 1;
    u.ntiles = u.per_head * a.G;
    return true;
}

// The CTA's sequence of units: mirrored pairs, items c, c + G, ... (G = gridDim.x, c = blockIdx.x).
// When the pairs left for the last round fill at most half the CTAs, they are split into their two
// tiles instead, one tile per CTA: the last round then costs about half a pair instead of a whole
// one on some CTAs while the others idle (64K training: 2048 pairs = 13 rounds of 152 + 72).
// Slot 2r + m is member m of round r's pair; the one slot after them holds a split tile.
__device__ __forceinline__ bool split_last_round(const BwdArgs& a)
{
    const long long G = gridDim.x, rem = a.items % G;
    return rem > 0 && 2 * rem <= G;
}

__device__ __forceinline__ int unit_slots(const BwdArgs& a)
{
    const long long G = gridDim.x;
    const long long pair_rounds = split_last_round(a) ? a.items / G : (a.items + G - 1) / G;
    return (int)(2 * pair_rounds + (split_last_round(a) ? 1 : 0));
}

__device__ __forceinline__ bool unit_in_slot(const BwdArgs& a, int s, KvUnit& u)
{
    const long long G = gridDim.x, c = blockIdx.x, R = a.items / G;
    const bool split = split_last_round(a);
    if (!split || s < 2 * R) {
        const long long item = (long long)(s >> 1) * G + c;
        return item < a.items && unit_of(a, item, s & 1, u);
    }
    const long long tu = c;  // tile index among the leftover pairs (one slot: 2 rem <= G)
    if (tu >= 2 * (a.items - R * G)) return false;
    return unit_of(a, R * G + (tu >> 1), (int)(tu & 1), u);
}

// Query tiles of a unit: heads of the group in turn, each walking the query shards in ring order.
// The second tile of a mirrored pair walks the heads last to first, so that a CTA goes on with the
// head it has just finished and the CTAs running together keep to the same heads (their Q, dO and
// dQ stay in L2).  Striped layout (whole sequence): the query shards are walked in one order for
// every unit (shard 0, 1, ...), so that the CTAs running together -- the same local tile of every
// shard, which see the same query tiles -- walk them in step (in ring order they started at 16
// different shards and each query tile was read at widely spread times).  The order of the sum
// over query tiles changes only the rounding of dK, dV and dQ.
struct QWalk {
    Geometry geo;
    int shard, pk, st, st0, st1, c, t, nt, hh, G, rev, global;
    // ring step at which this unit meets walk position st
    __device__ __forceinline__ int step_of(int s) const { return global ? (s - shard + geo.n) % geo.n : s; }
    KvRange qr;
    __device__ __forceinline__ void settle()
    {
        while (true) {
            while (st < st1) {
                qr = q_tile_range(geo, shard, step_of(st), c, pk);
                nt = qr.count / kQT;
                if (nt > 0) return;
                if (++c == geo.cps) {
                    c = 0;
                    ++st;
                }
            }
            ++hh;
            st = st0;
            c = 0;
            if (hh > 1 << 20) return;  // callers never walk past the unit's tile count
        }
    }
    __device__ __forceinline__ void begin(const BwdArgs& a, const KvUnit& u)
    {
        geo = a.geo;
        shard = u.shard;
        pk = u.pk;
        G = a.G;
        rev = u.rev;
        global = a.geo.layout == 2 && !a.blk;
        st0 = a.blk ? a.step : 0;  // a block call walks its one ring step
        st1 = a.blk ? a.step + 1 : a.geo.n;
        st = st0;
        c = 0;
        t = 0;
        hh = 0;
        settle();
    }
    // head within the group, buffer row and natural position of the next query tile
    __device__ __forceinline__ void next(int& head, int& row, int& nat)
    {
        head = rev ? G - 1 - hh : hh;
        row = qr.row0 + t * kQT;
        nat = qr.nat0 + t * kQT * geo.stride;
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

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > 1000000000ull) return;
    }
}

// 128-byte-swizzled address of 16-byte chunk `ch` of row `r` in a region of 128-byte rows.
__device__ __forceinline__ uint32_t sw128(uint32_t region, int r, int ch)
{
    return region + (uint32_t)r * 128u + ((uint32_t)(ch ^ (r & 7)) << 4);
}

// 16 bytes of shared memory (every lane of a warp reads the same words: one broadcast)
__device__ __forceinline__ float4 lds_f4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint32_t stage_of(uint32_t x) { return x % kStages; }
__device__ __forceinline__ uint32_t phase_of(uint32_t x) { return (x / kStages) & 1u; }

// ------------------------------------------------------------------------------------------------
// math warpgroups
// ------------------------------------------------------------------------------------------------
// Phase A: P^T = 2^(S^T c - lse2) for the warpgroup's query columns [64w, 64w+64), kept in p[] for
// phase B and written to TMEM as bf16 pairs (columns [64w, 64w+32) of X) for dV += P^T dO.
// Query columns c < lim of this key row are masked.
__device__ __forceinline__ void phase_a(const BwdArgs& a, uint32_t tmem, uint32_t lane_off, int w, int lim,
                                        uint32_t s_lse, float (&p)[64])
{
    const uint32_t tx = tmem + lane_off + kColX + (uint32_t)w * 64;
    uint32_t sv[64];
    tmem_ld_32x32b_x64(tx, sv);
    tmem_ld_wait(sv);
    uint32_t pk[32];
    const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
    const float2 nl2e = make_float2(-kLog2e, -kLog2e);
#pragma unroll
    for (int e4 = 0; e4 < 16; ++e4) {
        const float4 l4 = lds_f4(s_lse + (uint32_t)(w * 64 + e4 * 4) * 4u);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int col = e4 * 4 + h * 2;
            const uint32_t x0 = sv[col];
            const uint32_t x1 = sv[col + 1];
            const float2 lq = h == 0 ? make_float2(l4.x, l4.y) : make_float2(l4.z, l4.w);
            const float2 xv = fma2(make_float2(__uint_as_float(x0), __uint_as_float(x1)), sc2, mul2(lq, nl2e));
            float p0 = ex2_approx(xv.x), p1 = ex2_approx(xv.y);
            if (col < lim) p0 = 0.f;
            if (col + 1 < lim) p1 = 0.f;
            p[col] = p0;
            p[col + 1] = p1;
            pk[e4 * 2 + h] = pack_bf16x2(p0, p1);
        }
    }
    tmem_st_32x32b_x32(tx, pk);
    tmem_st_wait();
}

// Phase B: dS^T = P^T (dP^T - D) / sqrt(d) for the warpgroup's query columns, in two halves of 32,
// -> 128-byte-swizzled shared memory (query block w: key row r, its 128-byte row), where it is
// both the A operand of dK (K-major: key rows, query columns contiguous) and the B operand of
// dQ^T (N-major).
__device__ __forceinline__ void phase_b(const BwdArgs& a, uint32_t sbase, uint32_t tmem, uint32_t lane_off, int w,
                                        int r, uint32_t s_d, const float (&p)[64])
{
    const uint32_t ty = tmem + lane_off + kColY + (uint32_t)w * 64;
    const float2 sc = make_float2(a.scale, a.scale), neg1 = make_float2(-1.f, -1.f);
    const uint32_t region = sbase + kSmemDS + (uint32_t)w * kHalf;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        uint32_t dp[32];
        tmem_ld_32x32b_x32(ty + (uint32_t)hf * 32, dp);
        tmem_ld_wait(dp);
        uint32_t dsp[16];
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
            const float4 dq = lds_f4(s_d + (uint32_t)(w * 64 + hf * 32 + e4 * 4) * 4u);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int col = e4 * 4 + h * 2;
                const int pc = hf * 32 + col;
                const float2 d2 = h == 0 ? make_float2(dq.x, dq.y) : make_float2(dq.z, dq.w);
                // dS = (dP - D) * P * scale
                const float2 t = fma2(d2, neg1, make_float2(__uint_as_float(dp[col]), __uint_as_float(dp[col + 1])));
                const float2 ds = mul2(t, mul2(make_float2(p[pc], p[pc + 1]), sc));
                dsp[e4 * 2 + h] = pack_bf16x2(ds.x, ds.y);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sw128(region, r, hf * 4 + j)),
                         "r"(dsp[4 * j]), "r"(dsp[4 * j + 1]), "r"(dsp[4 * j + 2]), "r"(dsp[4 * j + 3])
                         : "memory");
    }
}

// Per query tile t the warpgroups run phase A then phase B; dQ^T is the dQ warps' business.
__device__ __forceinline__ void math_role(const BwdArgs& a, uint32_t sbase, uint32_t tmem, const WaitCtl& ctl)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int w = warp >> 2;                    // query-column half owned by this warpgroup
    const int r = (warp & 3) * 32 + lane;       // TMEM lane = key row
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    auto bar = [&](int i) { return sbase + kSmemBar + 8u * (uint32_t)i; };
    uint32_t gt = 0, uc = 0;
    const int slots = unit_slots(a);
    for (int slot = 0; slot < slots; ++slot) {
        {
            KvUnit u;
            if (!unit_in_slot(a, slot, u)) continue;
            if (u.ntiles == 0) {
                // a block call's tile that meets no query in this block: stored gradients are zero
                if (a.blk && !a.acc_kv) {
                    const long long krow = ((long long)u.b * a.Hkv + u.g) * a.qL + (u.rk - a.kv_off) + r;
#pragma unroll 1
                    for (int which = 0; which < 2; ++which) {
                        float4* d = reinterpret_cast<float4*>(static_cast<float*>(which == 0 ? a.dk : a.dv) +
                                                              krow * kHd + w * (kHd / 2));
#pragma unroll
                        for (int e = 0; e < kHd / 8; ++e) d[e] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                continue;
            }
            QWalk walk;
            walk.begin(a, u);
            for (int t = 0; t < u.ntiles; ++t, ++gt) {
                int hh, qrow, qnat;
                walk.next(hh, qrow, qnat);
                (void)hh;
                // Causal mask: query column c (of this warpgroup's 64) is masked for key row r iff
                // c < lim.  Natural positions: key pk + r vs query qnat + 64w + c.  Striped: local
                // rows t0 + r (shard j) vs u0 + 64w + c (shard i) and a key equal in local row is
                // visible only when j <= i.
                int lim = -(1 << 30);
                if (a.geo.causal) {
                    int delta;
                    if (a.geo.layout == 2) {
                        const int i = qrow / a.geo.S;
                        delta = (u.rk - u.shard * a.geo.S) - (qrow - i * a.geo.S) + (u.shard > i ? 1 : 0);
                    } else {
                        delta = u.pk - qnat;
                    }
                    lim = r + delta - 64 * w;
                }
                const uint32_t st = stage_of(gt), sp = phase_of(gt);
                float p[64];
                if (!mbar_wait(bar(BAR_ST_FULL), gt & 1, ctl)) goto done;
                if (!mbar_wait(bar(BAR_Q_FULL + (int)st), sp, ctl)) goto done;
                tc_fence_after_sync();
                __syncwarp();
                phase_a(a, tmem, lane_off, w, lim, sbase + kSmemLse + st * kVecBytes, p);
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(BAR_P_READY));
                if (!mbar_wait(bar(BAR_DPT_FULL), gt & 1, ctl)) goto done;
                if (!mbar_wait(bar(BAR_DO_FULL + (int)st), sp, ctl)) goto done;
                tc_fence_after_sync();
                __syncwarp();
                phase_b(a, sbase, tmem, lane_off, w, r, sbase + kSmemD + st * kVecBytes, p);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(BAR_DS_READY));
            }
            // epilogue: dK, dV of key row r, columns [w d/2, (w+1) d/2)
            if (!mbar_wait(bar(BAR_ACC_FULL), uc & 1, ctl)) goto done;
            tc_fence_after_sync();
            __syncwarp();
            const long long krow = ((long long)u.b * a.Hkv + u.g) * a.qL + (u.rk - a.kv_off) + r;
#pragma unroll 1
            for (int which = 0; which < 2; ++which) {
                const uint32_t col = (which == 0 ? kColDK : kColDV) + (uint32_t)w * (kHd / 2);
                void* base = which == 0 ? a.dk : a.dv;
#pragma unroll 1
                for (int c = 0; c < kHd / 64; ++c) {
                    uint32_t x[32];
                    tmem_ld_32x32b_x32(tmem + lane_off + col + c * 32, x);
                    tmem_ld_wait(x);
                    const long long off = krow * kHd + w * (kHd / 2) + c * 32;
                    if (a.acc_kv) {  // block call: add into the float32 gradients that travel with the block
                        float4* d = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float4 y = d[e];
                            d[e] = make_float4(y.x + __uint_as_float(x[4 * e]), y.y + __uint_as_float(x[4 * e + 1]),
                                               y.z + __uint_as_float(x[4 * e + 2]), y.w + __uint_as_float(x[4 * e + 3]));
                        }
                    } else if (a.grad_bf16) {
                        uint4* d = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + off);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            d[e] = make_uint4(pack_bf16x2(__uint_as_float(x[8 * e]), __uint_as_float(x[8 * e + 1])),
                                              pack_bf16x2(__uint_as_float(x[8 * e + 2]), __uint_as_float(x[8 * e + 3])),
                                              pack_bf16x2(__uint_as_float(x[8 * e + 4]), __uint_as_float(x[8 * e + 5])),
                                              pack_bf16x2(__uint_as_float(x[8 * e + 6]), __uint_as_float(x[8 * e + 7])));
                    } else {
                        float4* d = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            d[e] = make_float4(__uint_as_float(x[4 * e]), __uint_as_float(x[4 * e + 1]),
                                               __uint_as_float(x[4 * e + 2]), __uint_as_float(x[4 * e + 3]));
                    }
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(BAR_ACC_FREE));
            ++uc;
        }
    }
done:
    return;
}

// ------------------------------------------------------------------------------------------------
// dQ warpgroup (warps 8-11, thread = head-dim index): dQ^T of each query tile out of TMEM, then
// added into the float32 accumulator [heads][L][d] (at d = 64 by warps 8-9 only).  Its columns are freed as soon as they are
// in registers, so the next dP^T does not wait for the reductions.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void red_add_f32(float* addr, float v)
{
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

// The reductions go out in 16 groups of 8 per thread with an 80 ns pause between groups: issued at
// once they fill the SM's memory-instruction queue, and every other warp's shared-memory and
// barrier traffic then waits behind them (64K training backward: ~78 ms unpaced, ~71 paced).
// Pauses of 80-115 ns per group all give the same time; from ~130 ns on, the reductions fall
// behind the tiles (90 ms and worse), so 80 ns keeps a wide margin on boxes that run the tiles
// faster.  A tile whose successor is already waiting goes out without pauses.
__device__ __forceinline__ void red_group(float* dst, const uint32_t (&x)[64], int c0, uint32_t gap_ns)
{
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        if (gap_ns) __nanosleep(gap_ns);
#pragma unroll
        for (int c = 0; c < 8; ++c) red_add_f32(dst + (long long)(c0 + 8 * g + c) * kHd, __uint_as_float(x[8 * g + c]));
    }
}

__device__ __forceinline__ void dq_role(const BwdArgs& a, uint32_t sbase, uint32_t tmem, const WaitCtl& ctl)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int dcol = (warp & 3) * 32 + lane;  // TMEM lane = head-dim index
    const uint32_t ty = tmem + ((uint32_t)((warp & 3) * 32) << 16) + kColDQ;
    const uint32_t dq_c0 = kD64 && (warp & 3) >= 2 ? 64u : 0u;  // d = 64: this warp's query columns
    auto bar = [&](int i) { return sbase + kSmemBar + 8u * (uint32_t)i; };
    uint32_t gt = 0;
    const int slots = unit_slots(a);
    for (int slot = 0; slot < slots; ++slot) {
        {
            KvUnit u;
            if (!unit_in_slot(a, slot, u) || u.ntiles == 0) continue;
            QWalk walk;
            walk.begin(a, u);
            for (int t = 0; t < u.ntiles; ++t, ++gt) {
                int hh, qrow, qnat;
                walk.next(hh, qrow, qnat);
                (void)qnat;
                const bool behind = __shfl_sync(0xffffffffu, mbar_test_wait(bar(BAR_DQ_FULL), gt & 1), 0) != 0;
                const uint32_t gap_ns = behind ? 0u : 80u;
                if (!mbar_wait(bar(BAR_DQ_FULL), gt & 1, ctl)) return;
                tc_fence_after_sync();
                __syncwarp();
                if constexpr (kD64) {
                    // rows 0-63 (warps 8-9): query columns 0-63; rows 64-127 (warps 10-11, the same
                    // values from the second copy of K): query columns 64-127
                    uint32_t xa[64], xb[64];
                    tmem_ld_32x32b_x64(ty, xa);
                    tmem_ld_32x32b_x64(ty + 64, xb);
                    tmem_ld_wait(xa);
                    tmem_ld_wait(xb);
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(BAR_DQ_FREE));
                    const int zq = u.b * a.H + u.g * a.G + hh;
                    float* dst = a.dq_acc + ((long long)zq * a.qL + qrow - a.q_off) * kHd + (dcol & 63);
                    if (dq_c0 == 0)
                        red_group(dst, xa, 0, gap_ns);
                    else
                        red_group(dst, xb, 64, gap_ns);
                } else {
                    uint32_t xa[64], xb[64];
                    tmem_ld_32x32b_x64(ty, xa);
                    tmem_ld_32x32b_x64(ty + 64, xb);
                    tmem_ld_wait(xa);
                    tmem_ld_wait(xb);
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(BAR_DQ_FREE));
                    const int zq = u.b * a.H + u.g * a.G + hh;
                    float* dst = a.dq_acc + ((long long)zq * a.qL + qrow - a.q_off) * kHd + dcol;
                    red_group(dst, xa, 0, gap_ns);
                    red_group(dst, xb, 64, gap_ns);
                }
            }
        }
    }
}

// ------------------------------------------------------------------------------------------------
// TMA producer (one thread)
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void producer_role(const BwdArgs& a, uint32_t sbase, const CUtensorMap* tmQ,
                                              const CUtensorMap* tmK, const CUtensorMap* tmV,
                                              const CUtensorMap* tmDO, const WaitCtl& ctl)
{
    auto bar = [&](int i) { return sbase + kSmemBar + 8u * (uint32_t)i; };
    tma_prefetch_desc(tmQ);
    tma_prefetch_desc(tmK);
    tma_prefetch_desc(tmV);
    tma_prefetch_desc(tmDO);
    uint32_t uc = 0, qc = 0;
    bool ok = true;
    const int slots = unit_slots(a);
    for (int slot = 0; ok && slot < slots; ++slot) {
        {
            KvUnit u;
            if (!unit_in_slot(a, slot, u) || u.ntiles == 0) continue;
            if (uc > 0 && !mbar_wait(bar(BAR_KV_EMPTY), (uc - 1) & 1, ctl)) { ok = false; break; }
            const int zkv = u.b * a.Hkv + u.g;
            mbar_arrive_expect_tx(bar(BAR_KV_FULL), (kD64 ? 3 : 2) * kTileBytes);
#pragma unroll
            for (int half = 0; half < kHalves; ++half) {
                tma_load_3d(sbase + kSmemK + (uint32_t)half * kHalf, tmK, bar(BAR_KV_FULL), half * 64, u.rk - a.kv_off, zkv);
                tma_load_3d(sbase + kSmemV + (uint32_t)half * kHalf, tmV, bar(BAR_KV_FULL), half * 64, u.rk - a.kv_off, zkv);
            }
            if constexpr (kD64)
                tma_load_3d(sbase + kSmemK + kTileBytes, tmK, bar(BAR_KV_FULL), 0, u.rk - a.kv_off, zkv);
            ++uc;
            QWalk walk;
            walk.begin(a, u);
            for (int t = 0; t < u.ntiles; ++t, ++qc) {
                int hh, qrow, qnat;
                walk.next(hh, qrow, qnat);
                if (a.visits) atomicAdd(a.visits + (long long)(qrow / a.geo.S) * a.geo.n + u.shard, 1ull);
                const uint32_t st = stage_of(qc), use = qc / kStages;
                const int zq = u.b * a.H + u.g * a.G + hh;
                const long long qbase = (long long)zq * a.qL + qrow - a.q_off;  // first row's index in lse / D
                // Q with its lse first: S^T and phase A need them; dO and D follow
                if (use > 0 && !mbar_wait(bar(BAR_Q_EMPTY + (int)st), (use - 1) & 1, ctl)) { ok = false; break; }
                mbar_arrive_expect_tx(bar(BAR_Q_FULL + (int)st), kTileBytes + kVecBytes);
#pragma unroll
                for (int half = 0; half < kHalves; ++half)
                    tma_load_3d(sbase + kSmemQ + st * kTileBytes + (uint32_t)half * kHalf, tmQ,
                                bar(BAR_Q_FULL + (int)st), half * 64, qrow - a.q_off, zq);
                bulk_load_1d(sbase + kSmemLse + st * kVecBytes, a.lse + qbase, kVecBytes, bar(BAR_Q_FULL + (int)st));
                if (use > 0 && !mbar_wait(bar(BAR_DO_EMPTY + (int)st), (use - 1) & 1, ctl)) { ok = false; break; }
                mbar_arrive_expect_tx(bar(BAR_DO_FULL + (int)st), kTileBytes + kVecBytes);
#pragma unroll
                for (int half = 0; half < kHalves; ++half)
                    tma_load_3d(sbase + kSmemDO + st * kTileBytes + (uint32_t)half * kHalf, tmDO,
                                bar(BAR_DO_FULL + (int)st), half * 64, qrow - a.q_off, zq);
                bulk_load_1d(sbase + kSmemD + st * kVecBytes, a.Dv + qbase, kVecBytes, bar(BAR_DO_FULL + (int)st));
            }
        }
    }
    // Copies still in flight must land before the CTA's shared memory goes away.
    if (uc > 0) drain_wait(bar(BAR_KV_FULL), (uc - 1) & 1);
    for (uint32_t s = 0; s < (uint32_t)kStages && s < qc; ++s) {
        const uint32_t x = qc - 1 - s;
        drain_wait(bar(BAR_Q_FULL + (int)stage_of(x)), phase_of(x));
        drain_wait(bar(BAR_DO_FULL + (int)stage_of(x)), phase_of(x));
    }
}

// ------------------------------------------------------------------------------------------------
// MMA issuer (one thread)
// ------------------------------------------------------------------------------------------------
// Operand descriptors, as the low words of their shared-memory descriptors (query-tile operands
// at stage 0): K-major views have LBO 16, N- or M-major views LBO = the distance between their
// 64-element column blocks (16 KB everywhere here).  A stage or a k-step is a constant added.
// At d = 64 the M-major K view's second block (rows 64-127 of dQ^T) is the V tile, which follows
// K in shared memory: those rows are computed and never read.
struct BwdDesc {
    uint32_t k_k, v_k;    // K and V tiles, K-major (A of S^T and dP^T)
    uint32_t k_m;         // K tile, M-major (A of dQ^T = K^T dS^T)
    uint32_t q_k, do_k;   // Q and dO tiles, K-major (B of S^T and dP^T)
    uint32_t q_n, do_n;   // Q and dO tiles, N-major (B of dK and dV)
    uint32_t ds_n;        // dS^T, N-major (B of dQ^T)
    uint32_t ds_k;        // dS^T, K-major (A of dK)
};
constexpr uint32_t kDescHi = sdesc_sw128_hi(1024);
constexpr uint32_t kId = idesc_bf16_f32(128, 128, false, false);     // S^T, dP^T: both K-major
constexpr uint32_t kIdTs = idesc_bf16_f32(128, kHd, false, true);    // dV (A TMEM), dK (A K-major): B N-major
constexpr uint32_t kIdDQ = idesc_bf16_f32(128, 128, true, true);     // dQ^T: A M-major, B N-major

__device__ __forceinline__ BwdDesc make_desc(uint32_t sbase)
{
    BwdDesc d;
    d.k_k = sdesc_sw128_lo(sbase + kSmemK, 16);
    d.v_k = sdesc_sw128_lo(sbase + kSmemV, 16);
    d.k_m = sdesc_sw128_lo(sbase + kSmemK, kHalf);
    d.q_k = sdesc_sw128_lo(sbase + kSmemQ, 16);
    d.do_k = sdesc_sw128_lo(sbase + kSmemDO, 16);
    d.q_n = sdesc_sw128_lo(sbase + kSmemQ, kHalf);
    d.do_n = sdesc_sw128_lo(sbase + kSmemDO, kHalf);
    d.ds_n = sdesc_sw128_lo(sbase + kSmemDS, kHalf);
    d.ds_k = sdesc_sw128_lo(sbase + kSmemDS, 16);
    return d;
}

// TMEM column of the A operand for k-step kk of a product over the 128 query columns: the bf16
// pairs of warpgroup w's columns [64w, 64w+64) sit at [64w, 64w+32) of the region.
__device__ __forceinline__ uint32_t a_col(int kk) { return (uint32_t)(kk >> 2) * 64u + (uint32_t)(kk & 3) * 8u; }

// The issue helpers take their descriptor words through this, so that the compiler rebuilds the
// eight k-step descriptors at each call (eight 32-bit adds) instead of keeping every product's
// descriptors live across the tile loop, which would not fit the issuing warp's registers.
__device__ __forceinline__ uint32_t opaque(uint32_t x)
{
    asm volatile("" : "+r"(x));
    return x;
}

// D (tmem) = A B over the head dimension, both K-major in shared memory (S^T = K Q^T, dP^T = V dO^T)
__device__ __forceinline__ void issue_kmajor(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo)
{
    a_lo = opaque(a_lo);
    b_lo = opaque(b_lo);
#pragma unroll
    for (int kk = 0; kk < kHd / 16; ++kk) {
        const uint32_t off = (uint32_t)(kk >> 2) * kHalf + (uint32_t)(kk & 3) * 32u;
        mma_ss(d_tmem, sdesc_at(a_lo, off, kDescHi), sdesc_at(b_lo, off, kDescHi), kId, kk > 0);
    }
}

// acc (tmem) += A (tmem, bf16 pairs) B over the 128 query rows, B N-major in shared memory
// (dV += P^T dO)
__device__ __forceinline__ void issue_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, bool accumulate)
{
    const uint32_t acc0 = accumulate ? 1u : 0u;
    b_lo = opaque(b_lo);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        mma_ts(d_tmem, a_tmem + a_col(kk), sdesc_at(b_lo, (uint32_t)kk * 2048u, kDescHi), kIdTs, kk > 0 ? 1u : acc0);
}

// dK += dS^T Q over the 128 query rows: A = dS^T K-major (query block kk / 4, 16 queries = 32 bytes
// of each 128-byte key row), B = Q N-major
__device__ __forceinline__ void issue_dk(uint32_t tmem, const BwdDesc& dsc, uint32_t q_lo, bool accumulate)
{
    const uint32_t a_lo = opaque(dsc.ds_k), b_lo = opaque(q_lo);
    const uint32_t acc0 = accumulate ? 1u : 0u;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        mma_ss(tmem + kColDK, sdesc_at(a_lo, (uint32_t)(kk >> 2) * kHalf + (uint32_t)(kk & 3) * 32u, kDescHi),
               sdesc_at(b_lo, (uint32_t)kk * 2048u, kDescHi), kIdTs, kk > 0 ? 1u : acc0);
}

// dQ^T = K^T dS^T over the 128 key rows
__device__ __forceinline__ void issue_dq(uint32_t tmem, const BwdDesc& dsc)
{
    const uint32_t a_lo = opaque(dsc.k_m), b_lo = opaque(dsc.ds_n);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        mma_ss(tmem + kColDQ, sdesc_at(a_lo, (uint32_t)kk * 2048u, kDescHi), sdesc_at(b_lo, (uint32_t)kk * 2048u, kDescHi),
               kIdDQ, kk > 0);
}

__device__ __forceinline__ void mma_role(const BwdArgs& a, uint32_t sbase, uint32_t tmem, const WaitCtl& ctl)
{
    auto bar = [&](int i) { return sbase + kSmemBar + 8u * (uint32_t)i; };
    constexpr uint32_t kStageLo = kTileBytes >> 4;  // one query-tile stage, in descriptor units
    uint32_t gt = 0, uc = 0;
    bool issued = false;
    const BwdDesc dsc = make_desc(sbase);
    const int slots = unit_slots(a);
    for (int slot = 0; slot < slots; ++slot) {
        {
            KvUnit u;
            if (!unit_in_slot(a, slot, u) || u.ntiles == 0) continue;
            if (!mbar_wait(bar(BAR_KV_FULL), uc & 1, ctl)) goto drain;
            issued = true;
            tc_fence_after_sync();
            // the unit's first S^T and dP^T; later ones are issued one tile ahead (below)
            {
                const uint32_t st = stage_of(gt), sp = phase_of(gt);
                if (!mbar_wait(bar(BAR_Q_FULL + (int)st), sp, ctl)) goto drain;
                tc_fence_after_sync();
                issue_kmajor(tmem + kColX, dsc.k_k, dsc.q_k + st * kStageLo);
                tc_commit(bar(BAR_ST_FULL));
                // Y: the previous tile's dQ^T must have been read out (d = 128, where it shares Y)
                if (!kD64 && gt > 0 && !mbar_wait(bar(BAR_DQ_FREE), (gt - 1) & 1, ctl)) goto drain;
                if (!mbar_wait(bar(BAR_DO_FULL + (int)st), sp, ctl)) goto drain;
                tc_fence_after_sync();
                issue_kmajor(tmem + kColY, dsc.v_k, dsc.do_k + st * kStageLo);
                tc_commit(bar(BAR_DPT_FULL));
            }
            for (int t = 0; t < u.ntiles; ++t, ++gt) {
                const uint32_t st = stage_of(gt);
                // dV += P^T dO (P^T in X); the accumulators must have been written out at a unit's start
                if (!mbar_wait(bar(BAR_P_READY), gt & 1, ctl)) goto drain;
                if (t == 0 && uc > 0 && !mbar_wait(bar(BAR_ACC_FREE), (uc - 1) & 1, ctl)) goto drain;
                tc_fence_after_sync();
                issue_ts(tmem + kColDV, tmem + kColX, dsc.do_n + st * kStageLo, t > 0);
                tc_commit(bar(BAR_DO_EMPTY + (int)st));
                const bool more = t + 1 < u.ntiles;
                const uint32_t nst = stage_of(gt + 1), nsp = phase_of(gt + 1);
                // next S^T into X, which dV above has read; it runs while phase B computes dS^T
                if (more) {
                    if (!mbar_wait(bar(BAR_Q_FULL + (int)nst), nsp, ctl)) goto drain;
                    tc_fence_after_sync();
                    issue_kmajor(tmem + kColX, dsc.k_k, dsc.q_k + nst * kStageLo);
                    tc_commit(bar(BAR_ST_FULL));
                }
                // dQ^T = K^T dS^T (d = 128: into Y, whose dP^T phase B has read; d = 64: into its own
                // columns, once the previous tile's dQ^T is out), then dK += dS^T Q
                if (!mbar_wait(bar(BAR_DS_READY), gt & 1, ctl)) goto drain;
                if (kD64 && gt > 0 && !mbar_wait(bar(BAR_DQ_FREE), (gt - 1) & 1, ctl)) goto drain;
                tc_fence_after_sync();
                issue_dq(tmem, dsc);
                tc_commit(bar(BAR_DQ_FULL));
                issue_dk(tmem, dsc, dsc.q_n + st * kStageLo, t > 0);
                tc_commit(bar(BAR_Q_EMPTY + (int)st));
                // next dP^T into Y (d = 128: once dQ^T has been read out of it)
                if (more) {
                    if (!kD64 && !mbar_wait(bar(BAR_DQ_FREE), gt & 1, ctl)) goto drain;
                    if (!mbar_wait(bar(BAR_DO_FULL + (int)nst), nsp, ctl)) goto drain;
                    tc_fence_after_sync();
                    issue_kmajor(tmem + kColY, dsc.v_k, dsc.do_k + nst * kStageLo);
                    tc_commit(bar(BAR_DPT_FULL));
                }
            }
            tc_commit(bar(BAR_KV_EMPTY));
            tc_commit(bar(BAR_ACC_FULL));
            ++uc;
        }
    }
drain:
    if (issued) {
        tc_commit(bar(BAR_DRAIN));
        drain_wait(bar(BAR_DRAIN), 0);
    }
}

// ------------------------------------------------------------------------------------------------
// kernel
// ------------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO, const BwdArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    if (sbase & 1023u) {  // see kSmemBytes; uniform across the CTA, before any barrier or TMEM use
        if (threadIdx.x == 0) atomicOr(a.status, kStatusLayout);
        return;
    }
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemAbort);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmemTmemSlot);
    if (threadIdx.x == 0) {
        for (int i = 0; i < BAR_COUNT; ++i) {
            const bool by_math = i == BAR_P_READY || i == BAR_DS_READY || i == BAR_ACC_FREE;
            mbar_init(sbase + kSmemBar + 8u * (uint32_t)i, by_math ? 8u : (i == BAR_DQ_FREE ? 4u : 1u));
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 13) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl ctl{abort_flag, a.status, kWaitLimitNs};
    // Register split: launched with 512 x 128 = 65536 registers; math warpgroups 2 x 128 x 144, the
    // dQ warpgroup 128 x 152 and the TMA/MMA warpgroup 128 x 72 = 65536 (per SM sub-partition
    // 144 + 144 + 152 + 72 = 512).
    if (warp < 8)
        asm volatile("setmaxnreg.inc.sync.aligned.u32 144;" ::: "memory");
    else if (warp < 12)
        asm volatile("setmaxnreg.inc.sync.aligned.u32 152;" ::: "memory");
    else
        asm volatile("setmaxnreg.dec.sync.aligned.u32 72;" ::: "memory");
    if (warp < 8) {
        math_role(a, sbase, tmem, ctl);
    } else if (warp < 12) {
        dq_role(a, sbase, tmem, ctl);
    } else if (warp == 12) {
        if ((threadIdx.x & 31) == 0) producer_role(a, sbase, &tmQ, &tmK, &tmV, &tmDO, ctl);
    } else if (warp == 13) {
        if ((threadIdx.x & 31) == 0) mma_role(a, sbase, tmem, ctl);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 13) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

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

// 3-D map over a bf16 [heads][L][d] tensor: box 64 columns x `rows` rows x 1 head, 128-byte
// swizzle.
bool make_map(CUtensorMap* map, const void* base, int L, long long heads, int rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kHd, (cuuint64_t)L, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)kHd * 2, (cuuint64_t)L * kHd * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool RA_BWD_SUPPORTED(const Problem& p)
{
    if (p.dtype != 1 || p.d != kHd) return false;
    return p.geo().Lc % kKT == 0 && p.geo().Lc % kQT == 0;
}

cudaError_t RA_BWD_LAUNCH(const Problem& p, const void* q, const void* k, const void* v, const void* dout,
                          const float* D, const float* lse, float* dq_acc, void* dk, void* dv, int grad_dtype,
                          unsigned int* status, cudaStream_t s, unsigned long long* visits, const BlockView* blk)
{
    BwdArgs a;
    a.geo = p.geo();
    a.blk = blk ? 1 : 0;
    a.kv_shard = blk ? blk->kv_shard : 0;
    a.step = blk ? (blk->q_shard - blk->kv_shard + p.n) % p.n : 0;
    a.q_off = blk ? blk->q_shard * a.geo.S : 0;
    a.kv_off = blk ? blk->kv_shard * a.geo.S : 0;
    a.qL = blk ? a.geo.S : p.L;  // rows per head of every buffer (local shard buffers in a block call)
    a.acc_kv = blk ? blk->acc_kv : 0;
    CUtensorMap tq, tk, tv, tdo;
    if (!make_map(&tq, q, a.qL, (long long)p.B * p.H, kQT) || !make_map(&tk, k, a.qL, (long long)p.B * p.Hkv, kKT) ||
        !make_map(&tv, v, a.qL, (long long)p.B * p.Hkv, kKT) || !make_map(&tdo, dout, a.qL, (long long)p.B * p.H, kQT))
        return cudaErrorInvalidValue;
    a.B = p.B;
    a.H = p.H;
    a.Hkv = p.Hkv;
    a.G = p.H / p.Hkv;
    a.T = (p.layout == 2 || blk ? p.L / p.n : p.L) / kKT;
    a.pairs = (a.T + 1) / 2;
    a.items = (long long)p.B * p.Hkv * a.pairs * (p.layout == 2 && !blk ? p.n : 1);
    a.lse = lse;
    a.Dv = D;
    a.dq_acc = dq_acc;
    a.dk = dk;
    a.dv = dv;
    a.grad_bf16 = !blk && grad_dtype == 1;  // a block call's gradients are float32
    a.status = status;
    a.visits = visits;
    a.scale = 1.0f / sqrtf((float)kHd);
    a.scale_log2 = a.scale * kLog2e;
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
            e = cudaFuncSetAttribute(bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
            if (e != cudaSuccess) return e;
            attr_done[dev] = true;
        }
    }
    const long long sms = device_sm_count();
    const unsigned grid = (unsigned)(a.items < sms ? a.items : sms);
    bwd_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(tq, tk, tv, tdo, a);
    return cudaGetLastError();
}

}  // namespace ra
