// ra_geometry.h -- sequence layout and ring schedule of Ring Attention, shared by the host
// scheduler and the device kernels of libringattn.
//
// The sequence (length L) is cut into n shards of S = L/n rows (airsota "M4-051 Ring Attention and
// sequence parallelism", section 3).  Buffers store the sequence axis as the concatenation of the
// shards' local buffers.  Each shard is made of "chunks" whose rows are consecutive natural
// positions:
//   contiguous layout: 1 chunk per shard, natural range [i*S, (i+1)*S);
//   zigzag layout:     2 chunks per shard of C = L/(2n) rows: natural chunk i, then natural chunk
//                      2n-1-i (M4-051 section 4 item 2; "Lecture 30: TP/PP/SP/CP" section 3.2);
//   striped layout:    1 chunk per shard holding natural positions i, i + n, i + 2n, ... (the
//                      round-robin token split of "Lecture 30" section 3.2): consecutive rows of a
//                      chunk are `stride` = n positions apart (1 in the other layouts).
// Ring schedule (LLM-101-CN "distributed hands-on code", section 6.2; Lecture 30 section 3.2): at
// step r the rows of shard i use the K/V of shard (i - r) mod n.  Within a shard the chunks are
// walked in buffer order and, causally, only keys whose natural position does not exceed the
// largest natural position of the query rows are visited (blocks entirely in the future are
// skipped, M4-051 section 3).
#pragma once

#ifdef __CUDACC__
#define RA_HD __host__ __device__ __forceinline__
#else
#define RA_HD inline
#endif

namespace ra {

struct Geometry {
    int L;       // sequence length
    int n;       // shards
    int layout;  // 0 contiguous, 1 zigzag, 2 striped
    int causal;  // 0 / 1
    int S;       // rows per shard
    int Lc;      // rows per chunk
    int cps;     // chunks per shard (1 or 2)
    int stride;  // natural-position step between consecutive rows of a chunk (n if striped, else 1)
};

RA_HD Geometry make_geometry(int L, int n, int layout, int causal)
{
    Geometry g;
    g.L = L;
    g.n = n;
    g.layout = layout;
    g.causal = causal;
    g.S = L / n;
    g.cps = layout == 1 ? 2 : 1;
    g.Lc = g.S / g.cps;
    g.stride = layout == 2 ? n : 1;
    return g;
}

// Natural position of the first row of buffer chunk c.
RA_HD int chunk_natural_start(const Geometry& g, int c)
{
    if (g.layout == 2) return c;
    if (g.cps == 1) return c * g.Lc;
    int shard = c >> 1;
    int nat_chunk = (c & 1) ? (2 * g.n - 1 - shard) : shard;
    return nat_chunk * g.Lc;
}

// Natural position of buffer row r.
RA_HD int natural_position(const Geometry& g, int r)
{
    int c = r / g.Lc;
    return chunk_natural_start(g, c) + (r - c * g.Lc) * g.stride;
}

// Buffer row holding natural position p.
RA_HD int buffer_row(const Geometry& g, int p)
{
    if (g.layout == 2) return (p % g.n) * g.S + p / g.n;
    if (g.cps == 1) return p;
    int nc = p / g.Lc;
    int off = p - nc * g.Lc;
    int shard = nc < g.n ? nc : 2 * g.n - 1 - nc;
    return shard * g.S + (nc < g.n ? 0 : g.Lc) + off;
}

// One run of key rows of a ring step: buffer rows [row0, row0 + count) hold natural positions
// nat0, nat0 + stride, ..., in increasing order.
struct KvRange {
    int row0;
    int nat0;
    int count;
};

// Keys of chunk `c` (0..cps-1) of the shard visited by query shard `i` at ring step `step`, limited
// (causal) to natural positions <= p_hi.
RA_HD KvRange kv_range(const Geometry& g, int i, int step, int c, int p_hi)
{
    int j = i - step;
    if (j < 0) j += g.n;
    int ck = j * g.cps + c;
    KvRange kr;
    kr.row0 = ck * g.Lc;
    kr.nat0 = chunk_natural_start(g, ck);
    int cnt = g.Lc;
    if (g.causal) {
        // rows at positions <= p_hi
        cnt = p_hi < kr.nat0 ? 0 : (g.stride == 1 ? p_hi - kr.nat0 : (p_hi - kr.nat0) / g.stride) + 1;
        if (cnt > g.Lc) cnt = g.Lc;
    }
    kr.count = cnt;
    return kr;
}

// Query rows of chunk `c` of the shard that holds kv shard `j`'s block at backward step `step`
// (the K/V block of shard j meets the queries of shard (j + step) mod n), limited (causal) to
// natural positions >= p_lo.
RA_HD KvRange q_range(const Geometry& g, int j, int step, int c, int p_lo)
{
    int i = j + step;
    if (i >= g.n) i -= g.n;
    int cq = i * g.cps + c;
    KvRange qr;
    qr.row0 = cq * g.Lc;
    qr.nat0 = chunk_natural_start(g, cq);
    int first = 0;
    if (g.causal) {
        // rows at positions >= p_lo
        first = p_lo <= qr.nat0 ? 0
                : (g.stride == 1 ? p_lo - qr.nat0 : (p_lo - qr.nat0 + g.stride - 1) / g.stride);
        if (first > g.Lc) first = g.Lc;
    }
    qr.row0 += first;
    qr.nat0 += first * g.stride;
    qr.count = g.Lc - first;
    return qr;
}

// Causal relation of a query tile and a key tile of `tile` rows each, both starting at multiples
// of `tile` inside their chunks (chunk lengths multiples of `tile`), given by their first buffer
// rows.  0: every key visible to every query; 1: diagonal, key c visible to query r iff c <= r;
// 3: diagonal, iff c < r (striped, key shard after the query shard); 2: no key visible.
RA_HD int tile_mask(const Geometry& g, int q_row0, int kv_row0)
{
    if (!g.causal) return 0;
    if (g.layout == 2) {
        const int i = q_row0 / g.S, u0 = q_row0 - i * g.S;
        const int j = kv_row0 / g.S, t0 = kv_row0 - j * g.S;
        if (t0 < u0) return 0;
        if (t0 > u0) return 2;
        return j <= i ? 1 : 3;
    }
    const int pq = natural_position(g, q_row0), pk = natural_position(g, kv_row0);
    return pk < pq ? 0 : (pk == pq ? 1 : 2);
}

}  // namespace ra
