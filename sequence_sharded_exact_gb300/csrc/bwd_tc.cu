// bwd_tc.cu -- tensor-core backward of Ring Attention for sm_103a: bf16 inputs, head dim 128,
// shard (contiguous, striped) or chunk (zigzag) length a multiple of 128.
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
// mirrored pairs so that causal work is equal across CTAs; the unit walks 64-row query tiles):
//   * warp 8: TMA loads of the unit's K and V tiles and, through 3 stages, of each query tile's Q
//     (with its lse) and dO (with its D); the vectors come by bulk copy into shared memory.
//   * warp 9: tcgen05.mma issue, per query tile t:
//       dK += dS^T_{t-1} Q_{t-1} (dS^T from TMEM), then dQ^T_{t-1} = K^T dS^T_{t-1} (dS^T from
//       shared memory, N-major) interleaved step by step with dP^T_t = V dO_t^T, then
//       dV += P^T_t dO_t (P^T from TMEM) and S^T_{t+1} = K Q_{t+1}^T (K from TMEM).
//     Products whose A operand sits in TMEM run at about twice the rate of those reading both
//     operands from shared memory, so every operand that can stay in TMEM does.
//   * warps 0-7 (two warpgroups, each owning 32 of the 64 query columns), per query tile t:
//       phase A: P^T_t from S^T_t and lse (thread = key row) -> registers and TMEM;
//       phase C of t - 1: dQ^T_{t-1} out of TMEM (thread = head-dim index), into the dQ staging
//         buffer -- its products ran on the tensor cores during phase A;
//       phase B: dS^T_t = P^T_t (dP^T_t - D) -> shared memory;
//     at the end of a unit, phase C of the last tile and the dK, dV write-out.
//   * warp 10: adds each staged dQ tile into the float32 accumulator in HBM with TMA bulk
//     reductions and frees the staging buffer once the reductions have read it.  The staging
//     buffer is nothing else's, so the reductions (bound by the L2's rate for them) never hold up
//     the loads of later query tiles.
//   * TMEM columns: S^T/P^T [0,64), dP^T [64,128), dQ^T [128,192), the unit's K tile [192,256)
//     (copied in from shared memory once per unit: S^T reads its A operand there, which leaves
//     shared-memory bandwidth, the scarce resource here, to the other products), dK [256,384),
//     dV [384,512).
//   * every wait is bounded; a wait that runs out sets the device status word and the CTA stops.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "ra_internal.h"
#include "ra_ptx.cuh"

namespace ra {
namespace {

constexpr int kKT = 128;       // K/V tile rows
constexpr int kQT = 64;        // query tile rows
constexpr int kHd = 128;
constexpr int kStages = 3;     // query-tile stages (Q, dO, lse, D)
constexpr int kThreads = 384;  // 12 warps: 0-7 math, 8 TMA loads, 9 MMA, 10 dQ reductions, 11 idle
constexpr uint32_t kKHalf = kKT * 128;           // 16 KB: 128 rows x 64 head-dim columns (bf16)
constexpr uint32_t kKBytes = 2 * kKHalf;         // 32 KB
constexpr uint32_t kQHalf = kQT * 128;           // 8 KB
constexpr uint32_t kQBytes = 2 * kQHalf;         // 16 KB
constexpr uint32_t kVecBytes = kQT * 4;          // lse or D of one query tile (float32)

constexpr uint32_t kSmemK = 0;
constexpr uint32_t kSmemV = kSmemK + kKBytes;
constexpr uint32_t kSmemQ = kSmemV + kKBytes;                // kStages x 16 KB
constexpr uint32_t kSmemDO = kSmemQ + kStages * kQBytes;     // kStages x 16 KB
constexpr uint32_t kSmemDS = kSmemDO + kStages * kQBytes;    // dS^T: 128 key rows x 64 queries (bf16)
constexpr uint32_t kSmemDQ = kSmemDS + kKT * 128;            // dQ staging: 64 queries x 128 (float32)
constexpr uint32_t kSmemLse = kSmemDQ + kQT * kHd * 4;       // kStages x 256 B
constexpr uint32_t kSmemD = kSmemLse + kStages * kVecBytes;  // kStages x 256 B
constexpr uint32_t kSmemBar = kSmemD + kStages * kVecBytes;

enum : int {
    BAR_KV_FULL = 0,
    BAR_KV_EMPTY,
    BAR_Q_FULL,                           // kStages: Q tile and its lse landed
    BAR_DO_FULL = BAR_Q_FULL + kStages,   // kStages: dO tile and its D landed
    BAR_Q_EMPTY = BAR_DO_FULL + kStages,  // kStages: dK has read the Q tile
    BAR_DO_EMPTY = BAR_Q_EMPTY + kStages, // kStages: dP^T and dV have read the dO tile
    BAR_ST_FULL = BAR_DO_EMPTY + kStages,
    BAR_DPT_FULL,
    BAR_P_READY,
    BAR_DS_READY,
    BAR_DQ_FULL,
    BAR_DQ_FREE,
    BAR_DQ_STAGED,
    BAR_STG_FREE,
    BAR_ACC_FULL,
    BAR_ACC_FREE,
    BAR_DRAIN,
    BAR_COUNT
};

constexpr uint32_t kSmemTmemSlot = kSmemBar + BAR_COUNT * 8;
constexpr uint32_t kSmemAbort = kSmemTmemSlot + 8;
constexpr uint32_t kSmemUsed = kSmemAbort + 8;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // slack for 1024-byte alignment of the base
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kColST = 0, kColDPT = 64, kColDQ = 128, kColK = 192, kColDK = 256, kColDV = 384;
constexpr uint64_t kWaitLimitNs = 4000000000ull;

struct BwdArgs {
    Geometry geo;
    int B, H, Hkv, G;
    int T;            // 128-row K/V tiles per head (striped: per shard)
    int pairs;        // mirrored tile pairs per kv head (striped: per shard)
    long long items;  // B * Hkv * pairs (striped: B * Hkv * n * pairs)
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
    for (int st = 0; st < a.geo.n; ++st)
        for (int c = 0; c < a.geo.cps; ++c) nt += q_tile_range(a.geo, shard, st, c, pk).count / kQT;
    return nt;
}

__device__ __forceinline__ bool unit_of(const BwdArgs& a, long long item, int member, KvUnit& u)
{
    const int pair = (int)(item % a.pairs);
    long long rest = item / a.pairs;
    int shard = 0;
    if (a.geo.layout == 2) {  // striped: tiles of consecutive rows inside one shard
        shard = (int)(rest % a.geo.n);
        rest /= a.geo.n;
    }
    u.g = (int)(rest % a.Hkv);
    u.b = (int)(rest / a.Hkv);
    const int tile = member == 0 ? pair : a.T - 1 - pair;
    if (member == 1 && tile == pair) return false;
    if (a.geo.layout == 2) {
        u.rk = shard * a.geo.S + tile * kKT;
        u.pk = natural_position(a.geo, u.rk);
    } else {
        u.pk = tile * kKT;
        u.rk = buffer_row(a.geo, u.pk);
    }
    u.shard = u.rk / a.geo.S;
    u.per_head = q_tiles_per_head(a, u.shard, u.pk);
    u.ntiles = u.per_head * a.G;
    return true;
}

// Query tiles of a unit: heads of the group in turn, each walking the query shards in ring order.
struct QWalk {
    Geometry geo;
    int shard, pk, st, c, t, nt, hh;
    KvRange qr;
    __device__ __forceinline__ void settle()
    {
        while (true) {
            while (st < geo.n) {
                qr = q_tile_range(geo, shard, st, c, pk);
                nt = qr.count / kQT;
                if (nt > 0) return;
                if (++c == geo.cps) {
                    c = 0;
                    ++st;
                }
            }
            ++hh;
            st = 0;
            c = 0;
            if (hh > 1 << 20) return;  // callers never walk past the unit's tile count
        }
    }
    __device__ __forceinline__ void begin(const BwdArgs& a, const KvUnit& u)
    {
        geo = a.geo;
        shard = u.shard;
        pk = u.pk;
        st = 0;
        c = 0;
        t = 0;
        hh = 0;
        settle();
    }
    // head within the group, buffer row and natural position of the next query tile
    __device__ __forceinline__ void next(int& head, int& row, int& nat)
    {
        head = hh;
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

// TMA: global tile at {x, y, z} += the box in shared memory at `src` (float32 add, bulk group).
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z)
{
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
        ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until the shared memory of every bulk copy this thread committed has been read.
__device__ __forceinline__ void bulk_wait_read_all()
{
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Waits until every bulk copy this thread committed has completed.
__device__ __forceinline__ void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
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
// elementwise + dQ + epilogue warpgroups
// ------------------------------------------------------------------------------------------------
// Phase A: P^T = 2^(S^T c - lse2) for the warpgroup's query columns [32w, 32w+32), kept in p[] for
// phase B and written to TMEM as bf16 (columns [32w, 32w+16)) for dV += P^T dO.  Query columns
// c < lim of this key row are masked.
__device__ __forceinline__ void phase_a(const BwdArgs& a, uint32_t tmem, uint32_t lane_off, int w, int lim,
                                        uint32_t s_lse, float (&p)[32])
{
    uint32_t s[32];
    tmem_ld_32x32b_x32(tmem + lane_off + kColST + (uint32_t)w * 32, s);
    tmem_ld_wait(s);
    uint32_t pk[16];
    const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
    const float2 nl2e = make_float2(-kLog2e, -kLog2e);
#pragma unroll
    for (int e4 = 0; e4 < 8; ++e4) {
        const float4 l4 = lds_f4(s_lse + (uint32_t)(w * 32 + e4 * 4) * 4u);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int col = e4 * 4 + h * 2;
            const float2 lq = h == 0 ? make_float2(l4.x, l4.y) : make_float2(l4.z, l4.w);
            const float2 xv = fma2(make_float2(__uint_as_float(s[col]), __uint_as_float(s[col + 1])), sc2,
                                   mul2(lq, nl2e));
            float p0 = ex2_approx(xv.x), p1 = ex2_approx(xv.y);
            if (col < lim) p0 = 0.f;
            if (col + 1 < lim) p1 = 0.f;
            p[col] = p0;
            p[col + 1] = p1;
            pk[e4 * 2 + h] = pack_bf16x2(p0, p1);
        }
    }
    tmem_st_32x32b_x16(tmem + lane_off + kColST + (uint32_t)w * 32, pk);
    tmem_st_wait();
}

// Phase B: dS^T = P^T (dP^T - D) / sqrt(d) for the warpgroup's query columns -> 128-byte-swizzled
// shared memory (key row r, bytes [64w, 64w+64) of its 128-byte row; the B operand of dQ^T) and,
// as bf16 pairs, TMEM columns [64 + 32w, 64 + 32w + 16) (the A operand of dK).
__device__ __forceinline__ void phase_b(const BwdArgs& a, uint32_t sbase, uint32_t tmem, uint32_t lane_off, int w,
                                        int r, uint32_t s_d, const float (&p)[32])
{
    uint32_t dp[32];
    tmem_ld_32x32b_x32(tmem + lane_off + kColDPT + (uint32_t)w * 32, dp);
    tmem_ld_wait(dp);
    uint32_t dsp[16];
    const float2 sc = make_float2(a.scale, a.scale), neg1 = make_float2(-1.f, -1.f);
#pragma unroll
    for (int e4 = 0; e4 < 8; ++e4) {
        const float4 dq = lds_f4(s_d + (uint32_t)(w * 32 + e4 * 4) * 4u);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int col = e4 * 4 + h * 2;
            const float2 d2 = h == 0 ? make_float2(dq.x, dq.y) : make_float2(dq.z, dq.w);
            // dS = (dP - D) * P * scale
            const float2 t = fma2(d2, neg1, make_float2(__uint_as_float(dp[col]), __uint_as_float(dp[col + 1])));
            const float2 ds = mul2(t, mul2(make_float2(p[col], p[col + 1]), sc));
            dsp[e4 * 2 + h] = pack_bf16x2(ds.x, ds.y);
        }
    }
    const uint32_t region = sbase + kSmemDS;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sw128(region, r, 4 * w + j)), "r"(dsp[4 * j]),
                     "r"(dsp[4 * j + 1]), "r"(dsp[4 * j + 2]), "r"(dsp[4 * j + 3])
                     : "memory");
    // and into this warpgroup's dP^T columns, just read: the A operand of dK += dS^T Q
    tmem_st_32x32b_x16(tmem + lane_off + kColDPT + (uint32_t)w * 32, dsp);
    tmem_st_wait();
}

// Phase C of query tile gx: read dQ^T (thread = head-dim index r, the warpgroup's 32 query
// columns) out of TMEM, release its columns at once and stage it in the dQ buffer as the TMA
// reduction boxes want it: box (query block w, head-dim block r / 32) of 32 x 32 float32, rows =
// queries, 128-byte swizzled.  The reducer warp adds the boxes into the float32 accumulator.
__device__ __forceinline__ bool phase_c(uint32_t sbase, uint32_t tmem, uint32_t lane_off, int warp, int w, int lane,
                                        uint32_t gx, const WaitCtl& ctl)
{
    auto bar = [&](int i) { return sbase + kSmemBar + 8u * (uint32_t)i; };
    if (!mbar_wait(bar(BAR_DQ_FULL), gx & 1, ctl)) return false;
    tc_fence_after_sync();
    __syncwarp();
    uint32_t x[32];
    tmem_ld_32x32b_x32(tmem + lane_off + kColDQ + (uint32_t)w * 32, x);
    tmem_ld_wait(x);
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(BAR_DQ_FREE));
    // the reductions of the previous tile must have read the buffer
    if (gx > 0 && !mbar_wait(bar(BAR_STG_FREE), (gx - 1) & 1, ctl)) return false;
    const uint32_t box = sbase + kSmemDQ + (uint32_t)(w * 4 + (warp & 3)) * 4096u;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const uint32_t addr = box + (uint32_t)j * 128u + ((uint32_t)((lane >> 2) ^ (j & 7)) << 4) + (uint32_t)(lane & 3) * 4u;
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(x[j]) : "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(BAR_DQ_STAGED));
    return true;
}

// Per query tile t the warpgroups run phase A of t, phase C of t - 1 (whose dK and dQ products
// ran during phase A), then phase B of t.
__device__ __forceinline__ void math_role(const BwdArgs& a, uint32_t sbase, uint32_t tmem, const WaitCtl& ctl)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int w = warp >> 2;                    // query-column half owned by this warpgroup
    const int r = (warp & 3) * 32 + lane;       // TMEM lane = key row (S^T, dP^T) or head-dim index (dQ^T)
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    auto bar = [&](int i) { return sbase + kSmemBar + 8u * (uint32_t)i; };
    uint32_t gt = 0, uc = 0;
    for (long long item = blockIdx.x; item < a.items; item += gridDim.x) {
        for (int member = 0; member < 2; ++member) {
            KvUnit u;
            if (!unit_of(a, item, member, u) || u.ntiles == 0) continue;
            QWalk walk;
            walk.begin(a, u);
            for (int t = 0; t < u.ntiles; ++t, ++gt) {
                int hh, qrow, qnat;
                walk.next(hh, qrow, qnat);
                (void)hh;
                // Causal mask: query column c (of this warpgroup's 32) is masked for key row r iff
                // c < lim.  Natural positions: key pk + r vs query qnat + 32w + c.  Striped: local
                // rows t0 + r (shard j) vs u0 + 32w + c (shard i) and a key equal in local row is
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
                    lim = r + delta - 32 * w;
                }
                const uint32_t st = stage_of(gt), sp = phase_of(gt);
                float p[32];
                if (!mbar_wait(bar(BAR_ST_FULL), gt & 1, ctl)) goto done;
                if (!mbar_wait(bar(BAR_Q_FULL + (int)st), sp, ctl)) goto done;
                tc_fence_after_sync();
                __syncwarp();
                phase_a(a, tmem, lane_off, w, lim, sbase + kSmemLse + st * kVecBytes, p);
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(BAR_P_READY));
                if (t > 0 && !phase_c(sbase, tmem, lane_off, warp, w, lane, gt - 1, ctl)) goto done;
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
            if (!phase_c(sbase, tmem, lane_off, warp, w, lane, gt - 1, ctl)) goto done;
            // epilogue: dK, dV of key row r, columns [64w, 64w+64)
            if (!mbar_wait(bar(BAR_ACC_FULL), uc & 1, ctl)) goto done;
            tc_fence_after_sync();
            __syncwarp();
            const long long krow = ((long long)u.b * a.Hkv + u.g) * a.geo.L + u.rk + r;
#pragma unroll 1
            for (int which = 0; which < 2; ++which) {
                const uint32_t col = (which == 0 ? kColDK : kColDV) + (uint32_t)w * 64;
                void* base = which == 0 ? a.dk : a.dv;
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                    uint32_t x[32];
                    tmem_ld_32x32b_x32(tmem + lane_off + col + c * 32, x);
                    tmem_ld_wait(x);
                    const long long off = krow * kHd + w * 64 + c * 32;
                    if (a.grad_bf16) {
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
// dQ reducer (one thread): adds each staged dQ tile into the float32 accumulator with TMA bulk
// reductions, then frees the staging buffer.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void reducer_role(const BwdArgs& a, uint32_t sbase, const CUtensorMap* tmDQ,
                                             const WaitCtl& ctl)
{
    auto bar = [&](int i) { return sbase + kSmemBar + 8u * (uint32_t)i; };
    tma_prefetch_desc(tmDQ);
    uint32_t gt = 0;
    for (long long item = blockIdx.x; item < a.items; item += gridDim.x) {
        for (int member = 0; member < 2; ++member) {
            KvUnit u;
            if (!unit_of(a, item, member, u) || u.ntiles == 0) continue;
            QWalk walk;
            walk.begin(a, u);
            for (int t = 0; t < u.ntiles; ++t, ++gt) {
                int hh, qrow, qnat;
                walk.next(hh, qrow, qnat);
                if (!mbar_wait(bar(BAR_DQ_STAGED), gt & 1, ctl)) goto done;
                const int zq = u.b * a.H + u.g * a.G + hh;
#pragma unroll 1
                for (int bx = 0; bx < 8; ++bx)  // box (query block bx / 4, head-dim block bx % 4)
                    tma_reduce_add_3d(tmDQ, sbase + kSmemDQ + (uint32_t)bx * 4096u, (bx & 3) * 32, qrow + (bx >> 2) * 32,
                                      zq);
                bulk_commit();
                bulk_wait_read_all();
                mbar_arrive(bar(BAR_STG_FREE));
            }
        }
    }
done:
    bulk_wait_all();  // every reduction has been applied before the CTA exits
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
    for (long long item = blockIdx.x; ok && item < a.items; item += gridDim.x) {
        for (int member = 0; ok && member < 2; ++member) {
            KvUnit u;
            if (!unit_of(a, item, member, u) || u.ntiles == 0) continue;
            if (uc > 0 && !mbar_wait(bar(BAR_KV_EMPTY), (uc - 1) & 1, ctl)) { ok = false; break; }
            const int zkv = u.b * a.Hkv + u.g;
            mbar_arrive_expect_tx(bar(BAR_KV_FULL), 2 * kKBytes);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                tma_load_3d(sbase + kSmemK + (uint32_t)half * kKHalf, tmK, bar(BAR_KV_FULL), half * 64, u.rk, zkv);
                tma_load_3d(sbase + kSmemV + (uint32_t)half * kKHalf, tmV, bar(BAR_KV_FULL), half * 64, u.rk, zkv);
            }
            ++uc;
            QWalk walk;
            walk.begin(a, u);
            for (int t = 0; t < u.ntiles; ++t, ++qc) {
                int hh, qrow, qnat;
                walk.next(hh, qrow, qnat);
                if (a.visits) atomicAdd(a.visits + (long long)(qrow / a.geo.S) * a.geo.n + u.shard, 1ull);
                const uint32_t st = stage_of(qc), use = qc / kStages;
                const int zq = u.b * a.H + u.g * a.G + hh;
                const long long qbase = (long long)zq * a.geo.L + qrow;  // first row's index in lse / D
                // Q with its lse first: S^T and phase A need them; dO and D follow
                if (use > 0 && !mbar_wait(bar(BAR_Q_EMPTY + (int)st), (use - 1) & 1, ctl)) { ok = false; break; }
                mbar_arrive_expect_tx(bar(BAR_Q_FULL + (int)st), kQBytes + kVecBytes);
#pragma unroll
                for (int half = 0; half < 2; ++half)
                    tma_load_3d(sbase + kSmemQ + st * kQBytes + (uint32_t)half * kQHalf, tmQ, bar(BAR_Q_FULL + (int)st),
                                half * 64, qrow, zq);
                bulk_load_1d(sbase + kSmemLse + st * kVecBytes, a.lse + qbase, kVecBytes, bar(BAR_Q_FULL + (int)st));
                if (use > 0 && !mbar_wait(bar(BAR_DO_EMPTY + (int)st), (use - 1) & 1, ctl)) { ok = false; break; }
                mbar_arrive_expect_tx(bar(BAR_DO_FULL + (int)st), kQBytes + kVecBytes);
#pragma unroll
                for (int half = 0; half < 2; ++half)
                    tma_load_3d(sbase + kSmemDO + st * kQBytes + (uint32_t)half * kQHalf, tmDO,
                                bar(BAR_DO_FULL + (int)st), half * 64, qrow, zq);
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
// Operand descriptors of the issue loops, as the low words of their shared-memory descriptors
// (query-tile operands at stage 0): K-major views have LBO 16, N- or M-major views LBO = the
// distance between their 64-element column blocks.  A stage or a k-step is a constant added to them.
struct BwdDesc {
    uint32_t q_k, q_n;    // Q tile, K-major (S^T) and N-major (dK)
    uint32_t do_k, do_n;  // dO tile, K-major (dP^T) and N-major (dV)
    uint32_t v_k;         // V tile, K-major (dP^T)
    uint32_t k_m, ds_n;   // K tile M-major and dS^T N-major (dQ^T)
};
constexpr uint32_t kDescHi = sdesc_sw128_hi(1024);

__device__ __forceinline__ BwdDesc make_desc(uint32_t sbase)
{
    BwdDesc d;
    d.q_k = sdesc_sw128_lo(sbase + kSmemQ, 16);
    d.q_n = sdesc_sw128_lo(sbase + kSmemQ, kQHalf);
    d.do_k = sdesc_sw128_lo(sbase + kSmemDO, 16);
    d.do_n = sdesc_sw128_lo(sbase + kSmemDO, kQHalf);
    d.v_k = sdesc_sw128_lo(sbase + kSmemV, 16);
    d.k_m = sdesc_sw128_lo(sbase + kSmemK, kKHalf);
    d.ds_n = sdesc_sw128_lo(sbase + kSmemDS, kKHalf);
    return d;
}

// S^T = K Q^T into TMEM columns [0, 64): A = K from TMEM (lane = key row, 8 columns per 16 head-dim
// elements), B = Q K-major from shared memory (stage st).
__device__ __forceinline__ void issue_st(uint32_t tmem, const BwdDesc& dsc, uint32_t st)
{
    constexpr uint32_t id = idesc_bf16_f32(128, 64, false, false);
    const uint32_t qb = dsc.q_k + st * (kQBytes >> 4);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        mma_ts(tmem + kColST, tmem + kColK + (uint32_t)kk * 8u,
               sdesc_at(qb, (uint32_t)(kk >> 2) * kQHalf + (uint32_t)(kk & 3) * 32u, kDescHi), id, kk > 0);
}

constexpr uint32_t kIdDK = idesc_bf16_f32(128, 128, false, true);  // dK: A dS^T (TMEM), B Q N-major
constexpr uint32_t kIdDQ = idesc_bf16_f32(128, 64, true, true);    // dQ^T: A K^T M-major, B dS^T N-major
constexpr uint32_t kIdDP = idesc_bf16_f32(128, 64, false, false);  // dP^T: both K-major

// TMEM column of the A operand (bf16 pairs written by the two warpgroups) for k-step kk of a
// product over the 64 query columns: columns [0,32) at [0,16), [32,64) at [32,48) of the region.
__device__ __forceinline__ uint32_t a_col(int kk) { return kk < 2 ? (uint32_t)kk * 8u : 32u + (uint32_t)(kk - 2) * 8u; }

// dK += dS^T Q for query tile gx (tile t of its unit), once phase B has finished, then wait until
// the previous dQ^T has been read out; the dQ^T product itself is issued by the caller.
__device__ __forceinline__ bool issue_dk(uint32_t sbase, uint32_t tmem, const BwdDesc& dsc, uint32_t gx, int t,
                                         const WaitCtl& ctl)
{
    auto bar = [&](int i) { return sbase + kSmemBar + 8u * (uint32_t)i; };
    const uint32_t qb = dsc.q_n + stage_of(gx) * (kQBytes >> 4);
    const uint32_t acc0 = t > 0 ? 1u : 0u;
    if (!mbar_wait(bar(BAR_DS_READY), gx & 1, ctl)) return false;
    tc_fence_after_sync();
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_ts(tmem + kColDK, tmem + kColDPT + a_col(kk), sdesc_at(qb, (uint32_t)kk * 2048u, kDescHi), kIdDK,
               kk > 0 ? 1u : acc0);
    tc_commit(bar(BAR_Q_EMPTY + (int)stage_of(gx)));
    // dQ^T's columns: the previous tile's dQ^T must have been read out
    if (gx > 0 && !mbar_wait(bar(BAR_DQ_FREE), (gx - 1) & 1, ctl)) return false;
    tc_fence_after_sync();
    return true;
}

// k-step kk of dQ^T = K^T dS^T.
__device__ __forceinline__ void issue_dq_step(uint32_t tmem, const BwdDesc& dsc, int kk)
{
    mma_ss(tmem + kColDQ, sdesc_at(dsc.k_m, (uint32_t)kk * 2048u, kDescHi),
           sdesc_at(dsc.ds_n, (uint32_t)kk * 2048u, kDescHi), kIdDQ, kk > 0);
}

__device__ __forceinline__ void mma_role(const BwdArgs& a, uint32_t sbase, uint32_t tmem, const WaitCtl& ctl)
{
    auto bar = [&](int i) { return sbase + kSmemBar + 8u * (uint32_t)i; };
    constexpr uint32_t id_dv = idesc_bf16_f32(128, 128, false, true);  // dV: A P^T (TMEM), B dO N-major
    uint32_t gt = 0, uc = 0;
    bool issued = false;
    const BwdDesc dsc = make_desc(sbase);
    for (long long item = blockIdx.x; item < a.items; item += gridDim.x) {
        for (int member = 0; member < 2; ++member) {
            KvUnit u;
            if (!unit_of(a, item, member, u) || u.ntiles == 0) continue;
            if (!mbar_wait(bar(BAR_KV_FULL), uc & 1, ctl)) goto drain;
            issued = true;
            tc_fence_after_sync();
            // the unit's K tile into TMEM (after every S^T of the previous unit, in issue order)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tmem_cp_128x256b(tmem + kColK + (uint32_t)kk * 8u,
                                 sdesc_sw128(sbase + kSmemK + (uint32_t)(kk >> 2) * kKHalf + (uint32_t)(kk & 3) * 32u, 16,
                                             1024));
            // the unit's first S^T; later ones are issued one tile ahead (below)
            if (!mbar_wait(bar(BAR_Q_FULL + (int)stage_of(gt)), phase_of(gt), ctl)) goto drain;
            tc_fence_after_sync();
            issue_st(tmem, dsc, stage_of(gt));
            tc_commit(bar(BAR_ST_FULL));
            for (int t = 0; t < u.ntiles; ++t, ++gt) {
                const uint32_t st = stage_of(gt), sp = phase_of(gt);
                const uint32_t dok = dsc.do_k + st * (kQBytes >> 4), don = dsc.do_n + st * (kQBytes >> 4);
                // dK of the previous tile (its dS^T is ready when phase B ends; dK reads it from the
                // dP^T columns, so it goes before the new dP^T)
                if (t > 0 && !issue_dk(sbase, tmem, dsc, gt - 1, t - 1, ctl)) goto drain;
                // dP^T = V dO^T, its k-steps interleaved with those of the previous tile's dQ^T: two
                // independent accumulators keep the tensor pipe busier than one chain at a time
                if (!mbar_wait(bar(BAR_DO_FULL + (int)st), sp, ctl)) goto drain;
                tc_fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    if (t > 0) issue_dq_step(tmem, dsc, kk);
                    mma_ss(tmem + kColDPT,
                           sdesc_at(dsc.v_k, (uint32_t)(kk >> 2) * kKHalf + (uint32_t)(kk & 3) * 32u, kDescHi),
                           sdesc_at(dok, (uint32_t)(kk >> 2) * kQHalf + (uint32_t)(kk & 3) * 32u, kDescHi), kIdDP,
                           kk > 0);
                }
                if (t > 0) tc_commit(bar(BAR_DQ_FULL));
                tc_commit(bar(BAR_DPT_FULL));
                // dV += P^T dO   (P^T in TMEM: query columns [0,32) at cols [0,16), [32,64) at [32,48))
                if (!mbar_wait(bar(BAR_P_READY), gt & 1, ctl)) goto drain;
                if (t == 0 && uc > 0 && !mbar_wait(bar(BAR_ACC_FREE), (uc - 1) & 1, ctl)) goto drain;
                tc_fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ts(tmem + kColDV, tmem + kColST + a_col(kk), sdesc_at(don, (uint32_t)kk * 2048u, kDescHi),
                           id_dv, (t > 0 || kk > 0) ? 1u : 0u);
                tc_commit(bar(BAR_DO_EMPTY + (int)st));
                // next S^T, into the columns P^T leaves once the dV product above has read it
                if (t + 1 < u.ntiles) {
                    const uint32_t nst = stage_of(gt + 1);
                    if (!mbar_wait(bar(BAR_Q_FULL + (int)nst), phase_of(gt + 1), ctl)) goto drain;
                    tc_fence_after_sync();
                    issue_st(tmem, dsc, nst);
                    tc_commit(bar(BAR_ST_FULL));
                }
            }
            if (!issue_dk(sbase, tmem, dsc, gt - 1, u.ntiles - 1, ctl)) goto drain;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) issue_dq_step(tmem, dsc, kk);
            tc_commit(bar(BAR_DQ_FULL));
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

__global__ void __launch_bounds__(kThreads, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
              const __grid_constant__ CUtensorMap tmDQ, const BwdArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemAbort);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmemTmemSlot);
    if (threadIdx.x == 0) {
        for (int i = 0; i < BAR_COUNT; ++i) {
            const bool by_warps = i == BAR_P_READY || i == BAR_DS_READY || i == BAR_DQ_FREE || i == BAR_ACC_FREE ||
                                  i == BAR_DQ_STAGED;
            mbar_init(sbase + kSmemBar + 8u * (uint32_t)i, by_warps ? 8u : 1u);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl ctl{abort_flag, a.status, kWaitLimitNs};
    // Register split: launched with 384 x 168 = 64512 registers; math warpgroups 2 x 128 x 192 plus
    // the TMA/MMA warpgroup 128 x 120 = 64512 (per SM sub-partition 192 + 192 + 120 = 504).
    if (warp < 8)
        asm volatile("setmaxnreg.inc.sync.aligned.u32 192;" ::: "memory");
    else
        asm volatile("setmaxnreg.dec.sync.aligned.u32 120;" ::: "memory");
    if (warp < 8) {
        math_role(a, sbase, tmem, ctl);
    } else if (warp == 8) {
        if ((threadIdx.x & 31) == 0) producer_role(a, sbase, &tmQ, &tmK, &tmV, &tmDO, ctl);
    } else if (warp == 9) {
        if ((threadIdx.x & 31) == 0) mma_role(a, sbase, tmem, ctl);
    } else if (warp == 10) {
        if ((threadIdx.x & 31) == 0) reducer_role(a, sbase, &tmDQ, ctl);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        tried = true;
    }
    return fn;
}

// 3-D map over a bf16 [heads][L][128] tensor: box 64 columns x `rows` rows x 1 head, 128-byte
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

// 3-D map over the float32 dQ accumulator [heads][L][128]: box 32 columns x 32 rows x 1 head,
// 128-byte swizzle (the layout the math warps stage it in).
bool make_dq_map(CUtensorMap* map, float* base, int L, long long heads)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kHd, (cuuint64_t)L, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)kHd * 4, (cuuint64_t)L * kHd * 4};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

}  // namespace

bool tc_bwd_supported(const Problem& p)
{
    if (p.dtype != 1 || p.d != kHd) return false;
    return p.geo().Lc % kKT == 0;
}

cudaError_t launch_bwd_tc(const Problem& p, const void* q, const void* k, const void* v, const void* dout,
                          const float* D, const float* lse, float* dq_acc, void* dk, void* dv, int grad_dtype,
                          unsigned int* status, cudaStream_t s, unsigned long long* visits)
{
    CUtensorMap tq, tk, tv, tdo, tdq;
    if (!make_map(&tq, q, p.L, (long long)p.B * p.H, kQT) || !make_map(&tk, k, p.L, (long long)p.B * p.Hkv, kKT) ||
        !make_map(&tv, v, p.L, (long long)p.B * p.Hkv, kKT) || !make_map(&tdo, dout, p.L, (long long)p.B * p.H, kQT) ||
        !make_dq_map(&tdq, dq_acc, p.L, (long long)p.B * p.H))
        return cudaErrorInvalidValue;
    BwdArgs a;
    a.geo = p.geo();
    a.B = p.B;
    a.H = p.H;
    a.Hkv = p.Hkv;
    a.G = p.H / p.Hkv;
    a.T = (p.layout == 2 ? p.L / p.n : p.L) / kKT;
    a.pairs = (a.T + 1) / 2;
    a.items = (long long)p.B * p.Hkv * a.pairs * (p.layout == 2 ? p.n : 1);
    a.lse = lse;
    a.Dv = D;
    a.dq_acc = dq_acc;
    a.dk = dk;
    a.dv = dv;
    a.grad_bf16 = grad_dtype == 1;
    a.status = status;
    a.visits = visits;
    a.scale = 1.0f / sqrtf((float)kHd);
    a.scale_log2 = a.scale * kLog2e;
    static bool attr_done[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_done[dev]) {
        e = cudaFuncSetAttribute(bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    const long long sms = device_sm_count();
    const unsigned grid = (unsigned)(a.items < sms ? a.items : sms);
    bwd_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(tq, tk, tv, tdo, tdq, a);
    return cudaGetLastError();
}

}  // namespace ra
