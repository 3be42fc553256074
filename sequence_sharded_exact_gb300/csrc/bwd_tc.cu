// bwd_tc.cu -- tensor-core backward of Ring Attention for sm_103a: bf16 inputs, head dim 128,
// shard (contiguous) or chunk (zigzag) length a multiple of 128.
//
// The pages describe the forward only; the backward is the derivative of the same definition,
// with the attention weights recomputed from the saved log-sum-exp (never stored):
//   P = exp(s - lse),  dS = P (dO . v - D),  D = rowsum(dO * O),
//   dV = P^T dO,  dK = scale dS^T Q,  dQ = scale dS K,
// dK and dV summed over the query heads that share a kv head.  Causal blocks that are entirely
// masked are skipped and the diagonal tile is masked element by element.
// Ring order: the K/V block of shard j meets the queries of shard (j + r) mod n at step r (the K/V
// travels to the next device at every step, LLM-101-CN "distributed hands-on code" section 6.2),
// so a K/V tile walks the query shards in that order.
//
// Design (one CTA per SM, persistent; a work unit is one 128-row K/V tile of one kv head, units in
// mirrored pairs so that causal work is equal across CTAs):
//   * warp 8: TMA loads of the unit's K and V tiles and of the (Q, dO) tiles through 2 stages.
//   * warp 9: tcgen05.mma issue, per query tile t:
//       S^T = K Q^T, dP^T = V dO^T (TMEM), then dV += P^T dO (P^T read from TMEM),
//       dK += dS^T Q and dQ_t = dS K (dS^T read from shared memory, as a K-major operand for dK
//       and as an M-major operand for dQ).
//   * warps 0-7 (two warpgroups, each owning half of the 128 columns): read S^T and dP^T
//     (thread = key row), form P^T and dS^T, write P^T to TMEM and dS^T to shared memory; then read
//     dQ_t from TMEM (thread = query row) and stage it in shared memory; at the end of a unit write
//     dK and dV.
//   * warp 10: adds each staged dQ tile into the float32 accumulator in HBM with TMA bulk
//     reductions and hands the staging buffer back to the producer.
//   * TMEM columns: S^T/P^T [0,128), dP^T/dQ [128,256), dK [256,384), dV [384,512).
//   * every wait is bounded; a wait that runs out sets the device status word and the CTA stops.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "ra_internal.h"
#include "ra_ptx.cuh"

namespace ra {
namespace {

constexpr int kTile = 128;
constexpr int kHd = 128;
constexpr int kThreads = 384;  // 12 warps: 0-7 math, 8 TMA loads, 9 MMA, 10 dQ reductions, 11 idle
constexpr uint32_t kHalfBytes = kTile * 64 * 2;  // 16 KB
constexpr uint32_t kTileBytes = 2 * kHalfBytes;  // 32 KB

constexpr uint32_t kSmemK = 0;
constexpr uint32_t kSmemV = kSmemK + kTileBytes;
constexpr uint32_t kSmemQ = kSmemV + kTileBytes;      // 2 stages x (Q, dO)
constexpr uint32_t kSmemDO = kSmemQ + kTileBytes;     // stage s at + s * 2 * kTileBytes
constexpr uint32_t kStageBytes = 2 * kTileBytes;
constexpr uint32_t kSmemDS = kSmemQ + 2 * kStageBytes;
constexpr uint32_t kSmemBar = kSmemDS + kTileBytes;

enum : int {
    BAR_KV_FULL = 0,
    BAR_KV_EMPTY,
    BAR_QD_FULL,              // 2 stages
    BAR_QD_EMPTY = BAR_QD_FULL + 2,
    BAR_ST_FULL = BAR_QD_EMPTY + 2,
    BAR_DPT_FULL,
    BAR_P_READY,
    BAR_DS_READY,
    BAR_DQ_FULL,
    BAR_DQ_FREE,
    BAR_ACC_FULL,
    BAR_ACC_FREE,
    BAR_DQ_STAGED,            // 2 stages
    BAR_DRAIN = BAR_DQ_STAGED + 2,
    BAR_COUNT
};

constexpr uint32_t kSmemTmemSlot = kSmemBar + BAR_COUNT * 8;
constexpr uint32_t kSmemAbort = kSmemTmemSlot + 8;
constexpr uint32_t kSmemUsed = kSmemAbort + 8;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kColST = 0, kColDPT = 128, kColDK = 256, kColDV = 384;
constexpr uint64_t kWaitLimitNs = 4000000000ull;

struct BwdArgs {
    Geometry geo;
    int B, H, Hkv, G;
    int T;            // 128-row tiles per head (striped: per shard)
    int pairs;        // mirrored tile pairs per kv head
    long long items;  // B * Hkv * pairs
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
    int rk;      // buffer row of the K/V tile
    int pk;      // natural position of its first row
    int shard;   // kv shard
    int per_head;  // query tiles per head
    int ntiles;  // query tiles over all heads of the group
};

// The query rows of chunk c of the shard the K/V tile meets at step st that can see it, widened
// down to a tile boundary (striped: the first visible row may sit inside the diagonal tile).
__device__ __forceinline__ KvRange q_tile_range(const Geometry& g, int shard, int st, int c, int pk)
{
    KvRange qr = q_range(g, shard, st, c, pk);
    if (qr.count == 0) return qr;
    int i = shard + st;
    if (i >= g.n) i -= g.n;
    const int cs = (i * g.cps + c) * g.Lc;  // first row of that chunk
    const int off = (qr.row0 - cs) / kTile * kTile;
    qr.row0 = cs + off;
    qr.count = g.Lc - off;
    return qr;
}

__device__ __forceinline__ int q_tiles_per_head(const BwdArgs& a, int shard, int pk)
{
    int nt = 0;
    for (int st = 0; st < a.geo.n; ++st)
        for (int c = 0; c < a.geo.cps; ++c) nt += q_tile_range(a.geo, shard, st, c, pk).count / kTile;
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
        u.rk = shard * a.geo.S + tile * kTile;
        u.pk = natural_position(a.geo, u.rk);
    } else {
        u.pk = tile * kTile;
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
                nt = qr.count / kTile;
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
        row = qr.row0 + t * kTile;
        nat = qr.nat0 + t * kTile;
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

// ------------------------------------------------------------------------------------------------
// elementwise + dQ + epilogue warpgroups
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void math_role(const BwdArgs& a, uint32_t sbase, uint32_t tmem, const WaitCtl& ctl)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int w = warp >> 2;                    // column half owned by this warpgroup
    const int r = (warp & 3) * 32 + lane;       // TMEM lane = key row (S^T) or query row (dQ)
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    auto bar = [&](int i) { return sbase + kSmemBar + 8u * (uint32_t)i; };
    uint32_t gt = 0, uc = 0;
    for (long long item = blockIdx.x; item < a.items; item += gridDim.x) {
        for (int member = 0; member < 2; ++member) {
            KvUnit u;
            if (!unit_of(a, item, member, u) || u.ntiles == 0) continue;
            QWalk walk;
            walk.begin(a, u);
            float4 lv[16];  // lse of this step's query columns, loaded one step ahead
            for (int t = 0; t < u.ntiles; ++t, ++gt) {
                int hh, qrow, qnat;
                walk.next(hh, qrow, qnat);
                // 0 all visible, 1 / 3 diagonal (key row r visible to query column q iff r <= q /
                // r < q), 2 none; outside the striped layout only the diagonal tile is masked
                const int mk = a.geo.layout == 2 ? tile_mask(a.geo, qrow, u.rk) : (a.geo.causal && qnat == u.pk ? 1 : 0);
                // this key row's query columns 64w + c with c < lim are masked
                const int lim = (mk == 0 ? 0 : (mk == 1 ? r : (mk == 3 ? r + 1 : 1 << 20))) - w * 64;
                const long long qbase = ((long long)u.b * a.H + u.g * a.G + hh) * a.geo.L + qrow;
                if (t == 0) {
                    const float4* l4 = reinterpret_cast<const float4*>(a.lse + qbase + w * 64);
#pragma unroll
                    for (int e4 = 0; e4 < 16; ++e4) lv[e4] = __ldg(l4 + e4);
                }
                if (!mbar_wait(bar(BAR_ST_FULL), gt & 1, ctl)) goto done;
                tc_fence_after_sync();
                __syncwarp();
                // phase A: P^T = 2^(S^T c - lse2) for query columns [64w, 64w+64), kept in registers
                // for phase B and written to TMEM as bf16 for dV += P^T dO.
                float p[64];
                {
                    uint32_t s0[32], s1[32];
                    tmem_ld_32x32b_x32(tmem + lane_off + kColST + (uint32_t)w * 64, s0);
                    tmem_ld_32x32b_x32(tmem + lane_off + kColST + (uint32_t)w * 64 + 32, s1);
                    tmem_ld_wait(s0);
                    tmem_ld_wait(s1);
                    uint32_t pk[32];
                    const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
                    const float2 nl2e = make_float2(-kLog2e, -kLog2e);
#pragma unroll
                    for (int e4 = 0; e4 < 16; ++e4) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int col = e4 * 4 + h * 2;
                            const float2 lq = h == 0 ? make_float2(lv[e4].x, lv[e4].y) : make_float2(lv[e4].z, lv[e4].w);
                            const uint32_t sa = col < 32 ? s0[col] : s1[col - 32];
                            const uint32_t sb = col < 32 ? s0[col + 1] : s1[col - 31];
                            const float2 xv = fma2(make_float2(__uint_as_float(sa), __uint_as_float(sb)), sc2, mul2(lq, nl2e));
                            float p0 = ex2_approx(xv.x), p1 = ex2_approx(xv.y);
                            if (col < lim) p0 = 0.f;
                            if (col + 1 < lim) p1 = 0.f;
                            p[col] = p0;
                            p[col + 1] = p1;
                            pk[e4 * 2 + h] = pack_bf16x2(p0, p1);
                        }
                    }
                    // P^T of query columns [64w, 64w+64) -> TMEM columns [64w, 64w+32)
                    tmem_st_32x32b_x32(tmem + lane_off + kColST + (uint32_t)w * 64, pk);
                    tmem_st_wait();
                }
                // D of these columns for phase B, in flight while dP^T is computed
                float4 dv4[16];
                {
                    const float4* d4 = reinterpret_cast<const float4*>(a.Dv + qbase + w * 64);
#pragma unroll
                    for (int e4 = 0; e4 < 16; ++e4) dv4[e4] = __ldg(d4 + e4);
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(BAR_P_READY));
                // phase B: dS^T = P^T (dP^T - D) / sqrt(d) -> 128-byte-swizzled shared memory
                if (!mbar_wait(bar(BAR_DPT_FULL), gt & 1, ctl)) goto done;
                tc_fence_after_sync();
                __syncwarp();
                {
                    const uint32_t region = sbase + kSmemDS + (uint32_t)w * kHalfBytes;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t dp[32];
                        tmem_ld_32x32b_x32(tmem + lane_off + kColDPT + (uint32_t)(w * 64 + c * 32), dp);
                        tmem_ld_wait(dp);
                        uint32_t dsp[16];
                        const float2 sc = make_float2(a.scale, a.scale), neg1 = make_float2(-1.f, -1.f);
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {
                            const float4 dq = dv4[c * 8 + e4];
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int col = e4 * 4 + h * 2;
                                const float2 d2 = h == 0 ? make_float2(dq.x, dq.y) : make_float2(dq.z, dq.w);
                                // dS = (dP - D) * P * scale
                                const float2 t = fma2(d2, neg1, make_float2(__uint_as_float(dp[col]), __uint_as_float(dp[col + 1])));
                                const float2 ds = mul2(t, mul2(make_float2(p[c * 32 + col], p[c * 32 + col + 1]), sc));
                                dsp[e4 * 2 + h] = pack_bf16x2(ds.x, ds.y);
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int ch = (c * 32 + j * 8) >> 3;  // 16-byte chunk within the 128-byte row
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sw128(region, r, ch)),
                                         "r"(dsp[4 * j]), "r"(dsp[4 * j + 1]), "r"(dsp[4 * j + 2]), "r"(dsp[4 * j + 3])
                                         : "memory");
                        }
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(BAR_DS_READY));
                {  // next step's lse, in flight during the dQ readout (the last step reloads its own)
                    long long qbase2 = qbase;
                    if (t + 1 < u.ntiles) {
                        QWalk peek = walk;
                        int hh2, qrow2, qnat2;
                        peek.next(hh2, qrow2, qnat2);
                        qbase2 = ((long long)u.b * a.H + u.g * a.G + hh2) * a.geo.L + qrow2;
                    }
                    const float4* l4 = reinterpret_cast<const float4*>(a.lse + qbase2 + w * 64);
#pragma unroll
                    for (int e4 = 0; e4 < 16; ++e4) lv[e4] = __ldg(l4 + e4);
                }
                // dQ_t (thread = query row) added into the float32 accumulator
                if (!mbar_wait(bar(BAR_DQ_FULL), gt & 1, ctl)) goto done;
                tc_fence_after_sync();
                __syncwarp();
                // Read dQ out of TMEM and release its columns at once; stage it in this warp's 8 KB
                // slice of the step's (Q, dO) buffer, which no MMA reads any more.  The reducer warp
                // adds it into the float32 accumulator with TMA and hands the buffer back.
                {
                    uint32_t x0[32], x1[32];
                    tmem_ld_32x32b_x32(tmem + lane_off + kColDPT + (uint32_t)(w * 64), x0);
                    tmem_ld_32x32b_x32(tmem + lane_off + kColDPT + (uint32_t)(w * 64 + 32), x1);
                    tmem_ld_wait(x0);
                    tmem_ld_wait(x1);
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(BAR_DQ_FREE));
                    const uint32_t slice = sbase + kSmemQ + (uint32_t)(gt & 1) * kStageBytes + (uint32_t)warp * 8192u;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sw128(slice, lane, j)),
                                     "r"(x0[4 * j]), "r"(x0[4 * j + 1]), "r"(x0[4 * j + 2]), "r"(x0[4 * j + 3])
                                     : "memory");
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sw128(slice + 4096u, lane, j)),
                                     "r"(x1[4 * j]), "r"(x1[4 * j + 1]), "r"(x1[4 * j + 2]), "r"(x1[4 * j + 3])
                                     : "memory");
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(BAR_DQ_STAGED + (int)(gt & 1)));
                }
            }
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
// dQ reducer (one thread): adds each step's staged dQ tile into the float32 accumulator with TMA
// bulk reductions, then returns the step's (Q, dO) buffer to the producer.
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
                const int stage = (int)(gt & 1);
                if (!mbar_wait(bar(BAR_DQ_STAGED + stage), (gt >> 1) & 1, ctl)) goto done;
                const int zq = u.b * a.H + u.g * a.G + hh;
                const uint32_t buf = sbase + kSmemQ + (uint32_t)stage * kStageBytes;
#pragma unroll 1
                for (int wi = 0; wi < 8; ++wi) {
                    const uint32_t slice = buf + (uint32_t)wi * 8192u;
                    const int y = qrow + (wi & 3) * 32;
                    tma_reduce_add_3d(tmDQ, slice, (wi >> 2) * 64, y, zq);
                    tma_reduce_add_3d(tmDQ, slice + 4096u, (wi >> 2) * 64 + 32, y, zq);
                }
                bulk_commit();
                bulk_wait_read_all();
                mbar_arrive(bar(BAR_QD_EMPTY + stage));
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
            mbar_arrive_expect_tx(bar(BAR_KV_FULL), 2 * kTileBytes);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                tma_load_3d(sbase + kSmemK + (uint32_t)half * kHalfBytes, tmK, bar(BAR_KV_FULL), half * 64, u.rk, zkv);
                tma_load_3d(sbase + kSmemV + (uint32_t)half * kHalfBytes, tmV, bar(BAR_KV_FULL), half * 64, u.rk, zkv);
            }
            ++uc;
            QWalk walk;
            walk.begin(a, u);
            for (int t = 0; t < u.ntiles; ++t, ++qc) {
                int hh, qrow, qnat;
                walk.next(hh, qrow, qnat);
                if (a.visits) atomicAdd(a.visits + (long long)(qrow / a.geo.S) * a.geo.n + u.shard, 1ull);
                const int stage = (int)(qc & 1);
                const uint32_t use = qc >> 1;
                if (use > 0 && !mbar_wait(bar(BAR_QD_EMPTY + stage), (use - 1) & 1, ctl)) { ok = false; break; }
                const int zq = u.b * a.H + u.g * a.G + hh;
                const uint32_t sq = sbase + kSmemQ + (uint32_t)stage * kStageBytes;
                const uint32_t sd = sbase + kSmemDO + (uint32_t)stage * kStageBytes;
                mbar_arrive_expect_tx(bar(BAR_QD_FULL + stage), 2 * kTileBytes);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    tma_load_3d(sq + (uint32_t)half * kHalfBytes, tmQ, bar(BAR_QD_FULL + stage), half * 64, qrow, zq);
                    tma_load_3d(sd + (uint32_t)half * kHalfBytes, tmDO, bar(BAR_QD_FULL + stage), half * 64, qrow, zq);
                }
            }
        }
    }
    if (uc > 0) drain_wait(bar(BAR_KV_FULL), (uc - 1) & 1);
    for (uint32_t s = 0; s < 2 && s < qc; ++s) {
        const uint32_t x = qc - 1 - s;
        drain_wait(bar(BAR_QD_FULL + (int)(x & 1)), (x >> 1) & 1);
    }
}

// ------------------------------------------------------------------------------------------------
// MMA issuer (one thread)
// ------------------------------------------------------------------------------------------------
// S^T = K Q^T into TMEM columns [0, 128) (both operands K-major).
__device__ __forceinline__ void issue_st(uint32_t sbase, uint32_t tmem, uint32_t sq)
{
    constexpr uint32_t id_kk = idesc_bf16_f32(128, 128, false, false);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (uint32_t)(kk >> 2) * kHalfBytes + (uint32_t)(kk & 3) * 32u;
        mma_ss(tmem + kColST, sdesc_sw128(sbase + kSmemK + off, 16, 1024), sdesc_sw128(sq + off, 16, 1024), id_kk,
               kk > 0);
    }
}

__device__ __forceinline__ void mma_role(const BwdArgs& a, uint32_t sbase, uint32_t tmem, const WaitCtl& ctl)
{
    auto bar = [&](int i) { return sbase + kSmemBar + 8u * (uint32_t)i; };
    constexpr uint32_t id_kk = idesc_bf16_f32(128, 128, false, false);  // both operands K-major
    constexpr uint32_t id_kn = idesc_bf16_f32(128, 128, false, true);   // B N-major
    constexpr uint32_t id_mn = idesc_bf16_f32(128, 128, true, true);    // A M-major, B N-major
    uint32_t gt = 0, uc = 0;
    bool issued = false;
    for (long long item = blockIdx.x; item < a.items; item += gridDim.x) {
        for (int member = 0; member < 2; ++member) {
            KvUnit u;
            if (!unit_of(a, item, member, u) || u.ntiles == 0) continue;
            if (!mbar_wait(bar(BAR_KV_FULL), uc & 1, ctl)) goto drain;
            issued = true;
            for (int t = 0; t < u.ntiles; ++t, ++gt) {
                const int stage = (int)(gt & 1);
                const uint32_t use = gt >> 1;
                const uint32_t sq = sbase + kSmemQ + (uint32_t)stage * kStageBytes;
                const uint32_t sd = sbase + kSmemDO + (uint32_t)stage * kStageBytes;
                if (t == 0) {
                    // the first S^T of a unit; later ones are issued one step ahead (below)
                    if (!mbar_wait(bar(BAR_QD_FULL + stage), use & 1, ctl)) goto drain;
                    tc_fence_after_sync();
                    issue_st(sbase, tmem, sq);
                    tc_commit(bar(BAR_ST_FULL));
                }
                // dP^T = V dO^T (its columns also hold the previous dQ: wait until that was read)
                if (gt > 0 && !mbar_wait(bar(BAR_DQ_FREE), (gt - 1) & 1, ctl)) goto drain;
                tc_fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 2) * kHalfBytes + (uint32_t)(kk & 3) * 32u;
                    mma_ss(tmem + kColDPT, sdesc_sw128(sbase + kSmemV + off, 16, 1024), sdesc_sw128(sd + off, 16, 1024),
                           id_kk, kk > 0);
                }
                tc_commit(bar(BAR_DPT_FULL));
                // dV += P^T dO   (P^T in TMEM: query columns [0,64) at cols [0,32), [64,128) at [64,96))
                if (!mbar_wait(bar(BAR_P_READY), gt & 1, ctl)) goto drain;
                if (t == 0 && uc > 0 && !mbar_wait(bar(BAR_ACC_FREE), (uc - 1) & 1, ctl)) goto drain;
                tc_fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t acol = kColST + (kk < 4 ? (uint32_t)kk * 8u : 64u + (uint32_t)(kk - 4) * 8u);
                    mma_ts(tmem + kColDV, tmem + acol, sdesc_sw128(sd + (uint32_t)kk * 2048u, kHalfBytes, 1024), id_kn,
                           (t > 0 || kk > 0) ? 1u : 0u);
                }
                // next S^T, into the columns P^T leaves once the dV product above has read it
                if (t + 1 < u.ntiles) {
                    const int nstage = (int)((gt + 1) & 1);
                    if (!mbar_wait(bar(BAR_QD_FULL + nstage), ((gt + 1) >> 1) & 1, ctl)) goto drain;
                    tc_fence_after_sync();
                    issue_st(sbase, tmem, sbase + kSmemQ + (uint32_t)nstage * kStageBytes);
                    tc_commit(bar(BAR_ST_FULL));
                }
                // dK += dS^T Q ; dQ_t = dS K
                if (!mbar_wait(bar(BAR_DS_READY), gt & 1, ctl)) goto drain;
                tc_fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 2) * kHalfBytes + (uint32_t)(kk & 3) * 32u;
                    mma_ss(tmem + kColDK, sdesc_sw128(sbase + kSmemDS + off, 16, 1024),
                           sdesc_sw128(sq + (uint32_t)kk * 2048u, kHalfBytes, 1024), id_kn, (t > 0 || kk > 0) ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    mma_ss(tmem + kColDPT, sdesc_sw128(sbase + kSmemDS + (uint32_t)kk * 2048u, kHalfBytes, 1024),
                           sdesc_sw128(sbase + kSmemK + (uint32_t)kk * 2048u, kHalfBytes, 1024), id_mn, kk > 0);
                }
                tc_commit(bar(BAR_DQ_FULL));
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
                                  i == BAR_DQ_STAGED || i == BAR_DQ_STAGED + 1;
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

bool make_map(CUtensorMap* map, const void* base, int L, long long heads)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kHd, (cuuint64_t)L, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)kHd * 2, (cuuint64_t)L * kHd * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kTile, 1};
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
    return p.geo().Lc % kTile == 0;
}

cudaError_t launch_bwd_tc(const Problem& p, const void* q, const void* k, const void* v, const void* dout,
                          const float* D, const float* lse, float* dq_acc, void* dk, void* dv, int grad_dtype,
                          unsigned int* status, cudaStream_t s, unsigned long long* visits)
{
    CUtensorMap tq, tk, tv, tdo, tdq;
    if (!make_map(&tq, q, p.L, (long long)p.B * p.H) || !make_map(&tk, k, p.L, (long long)p.B * p.Hkv) ||
        !make_map(&tv, v, p.L, (long long)p.B * p.Hkv) || !make_map(&tdo, dout, p.L, (long long)p.B * p.H) ||
        !make_dq_map(&tdq, dq_acc, p.L, (long long)p.B * p.H))
        return cudaErrorInvalidValue;
    BwdArgs a;
    a.geo = p.geo();
    a.B = p.B;
    a.H = p.H;
    a.Hkv = p.Hkv;
    a.G = p.H / p.Hkv;
    a.T = (p.layout == 2 ? p.L / p.n : p.L) / kTile;
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
