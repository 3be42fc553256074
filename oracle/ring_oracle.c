/*
 * ring_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, float64 CPU statement of what Ring Attention computes: exact softmax attention
 * softmax(Q K^T / sqrt(d)) V over a sequence that has been cut into n shards, causal or not,
 * contiguous or zigzag layout, with grouped K/V heads.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this file's library.  The CUDA product path never
 * includes, links or calls anything here, and nothing here is shared with it.
 *
 * Sources (web pages on Ring Attention; cited by page title and section):
 *  [LLM101]  LLM-101-CN, "distributed hands-on code", section 6 "Ring Attention / sequence
 *            parallelism": 6.1 (each rank keeps its Q block; K/V blocks go round the ring) and 6.2
 *            (block_attention: S = Q K^T / sqrt(head_dim), running max M, running sum L, running
 *            output O, rescale by exp(M - M_new); final O / L).
 *  [M4-051]  airsota "M4-051 Ring Attention and sequence parallelism", section 3 (device i holds
 *            Q_i, K_i, V_i of length L/n; at step r it uses the K/V block it currently holds; after
 *            n steps the result equals full attention; causal: device i only needs blocks before
 *            it) and section 4 item 2 (zigzag layout balances causal work).
 *  [CP-30]   "Lecture 30: TP/PP/SP/CP", section 3.2 (the 4-GPU ring walk: step 0 uses the local
 *            K/V, each later step the block received from the previous GPU).
 *
 * Readings where the pages are silent or garbled (each also listed in the design notes):
 *  - zigzag: the sequence is cut into 2n chunks of C = L/(2n); shard i holds chunk i followed by
 *    chunk 2n-1-i (the page's "segments i and n-1-i" cannot hold for n segments).
 *  - striped (the round-robin token split of "Lecture 30" section 3.2): shard i holds the natural
 *    positions i, i + n, i + 2n, ... in increasing order.
 *  - every buffer (q, k, v, out, lse, dout, grads) stores the sequence axis in the layout's order,
 *    i.e. as the concatenation of the shards' local buffers; masking uses natural positions.
 *  - causal mask: key t is visible to query p iff pos(t) <= pos(p) (the query sees itself).
 *  - scale is 1/sqrt(d); GQA query head h uses kv head h / (H/Hkv).
 *  - lse is the natural-log log-sum-exp of the scaled scores.
 *  - ring direction: at step r shard i uses the K/V of shard (i - r) mod n (the page's code sends
 *    to rank+1 and receives from rank-1).
 *  - running max starts at -infinity (the page's -1e4 fails when all scores are below -1e4); a
 *    block in which a row sees no key leaves that row's state unchanged.
 *  - rotary positions (oracle_rope): natural positions, RoFormer pair rotation (see there).
 *  - backward (absent from the pages): the plain derivative of the forward definition,
 *    P = exp(s - lse), D = <dO, O>, dS = P (dO.v - D), dQ = scale dS K, dK = scale dS^T Q,
 *    dV = P^T dO, with dK and dV summed over the query heads of a group.
 *
 * Tensor layouts: q, out, dout, dq are [B][H][L][d]; k, v, dk, dv are [B][Hkv][L][d]; lse is
 * [B][H][L].  Inputs are float (exact copies of the values the GPU reads); results are double.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARGS 1
#define ORACLE_NO_MEMORY 2

/* Natural sequence position of buffer row r ([M4-051] section 4 item 2 and [CP-30] section 3.2;
 * zigzag and striped readings above).  layout 0 contiguous, 1 zigzag, 2 striped. */
long oracle_natural_position(long r, long L, int n, int layout)
{
    if (layout == 0) return r;
    if (layout == 2) {
        long S = L / n;
        return (r % S) * n + r / S;
    }
    long C = L / (2L * n);
    long shard = r / (2 * C);
    long off = r % (2 * C);
    if (off < C) return shard * C + off;
    return (2L * n - 1 - shard) * C + (off - C);
}

static int check_args(int B, int H, int Hkv, long L, int d, int n, int layout)
{
    if (B < 1 || H < 1 || Hkv < 1 || L < 1 || d < 1 || n < 1) return 0;
    if (H % Hkv != 0) return 0;
    if (L % n != 0) return 0;
    if (layout != 0 && layout != 1 && layout != 2) return 0;
    if (layout == 1 && L % (2L * n) != 0) return 0;
    return 1;
}

/* One query row by definition: two passes (max first, then the sums), float64 throughout.
 * Writes o[d] and returns lse.  scores is caller-provided scratch of length L. */
static double attention_row(const float* q, const float* k, const float* v, int H, int Hkv, long L,
                            int d, int n, int causal, int layout, int b, int h, long r,
                            double* o, double* scores)
{
    const int g = h / (H / Hkv);
    const double scale = 1.0 / sqrt((double)d);
    const float* qrow = q + (((long)b * H + h) * L + r) * d;
    const float* kh = k + ((long)b * Hkv + g) * L * d;
    const float* vh = v + ((long)b * Hkv + g) * L * d;
    const long p = oracle_natural_position(r, L, n, layout);

    double mx = -INFINITY;
    for (long t = 0; t < L; ++t) {
        int visible = !causal || oracle_natural_position(t, L, n, layout) <= p;
        if (!visible) { scores[t] = -INFINITY; continue; }
        double s = 0.0;
        for (int c = 0; c < d; ++c) s += (double)qrow[c] * (double)kh[t * d + c];
        s *= scale;
        scores[t] = s;
        if (s > mx) mx = s;
    }
    double sum = 0.0;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (long t = 0; t < L; ++t) {
        if (scores[t] == -INFINITY) continue;
        double e = exp(scores[t] - mx);
        sum += e;
        for (int c = 0; c < d; ++c) o[c] += e * (double)vh[t * d + c];
    }
    for (int c = 0; c < d; ++c) o[c] /= sum;
    return mx + log(sum);
}

/* Forward for a list of query rows.  rows[i] is the flat index (b*H + h)*L + r.
 * out is [nrows][d], lse is [nrows]. */
int oracle_attn_fwd_rows(const float* q, const float* k, const float* v, int B, int H, int Hkv,
                         long L, int d, int n, int causal, int layout, long nrows, const long* rows,
                         double* out, double* lse)
{
    if (!check_args(B, H, Hkv, L, d, n, layout)) return ORACLE_BAD_ARGS;
    int status = ORACLE_OK;
#pragma omp parallel
    {
        double* scores = (double*)malloc(sizeof(double) * L);
        if (!scores) {
#pragma omp atomic write
            status = ORACLE_NO_MEMORY;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long i = 0; i < nrows; ++i) {
                long idx = rows[i];
                long r = idx % L;
                int h = (int)((idx / L) % H);
                int b = (int)(idx / ((long)H * L));
                lse[i] = attention_row(q, k, v, H, Hkv, L, d, n, causal, layout, b, h, r,
                                       out + i * d, scores);
            }
            free(scores);
        }
    }
    return status;
}

/* Forward for every row: out [B][H][L][d], lse [B][H][L]. */
int oracle_attn_fwd(const float* q, const float* k, const float* v, int B, int H, int Hkv, long L,
                    int d, int n, int causal, int layout, double* out, double* lse)
{
    if (!check_args(B, H, Hkv, L, d, n, layout)) return ORACLE_BAD_ARGS;
    long nrows = (long)B * H * L;
    long* rows = (long*)malloc(sizeof(long) * nrows);
    if (!rows) return ORACLE_NO_MEMORY;
    for (long i = 0; i < nrows; ++i) rows[i] = i;
    int st = oracle_attn_fwd_rows(q, k, v, B, H, Hkv, L, d, n, causal, layout, nrows, rows, out, lse);
    free(rows);
    return st;
}

/* The ring walk itself ([LLM101] 6.2, [CP-30] 3.2): for every shard i and step r = 0..n-1 the rows
 * of shard i take the keys of shard j = (i - r) mod n and fold them into a running (M, L, O) state
 * with the page's update
 *     M_new = max(M, rowmax S);  L = L e^{M - M_new} + sum e^{S - M_new};
 *     O = O e^{M - M_new} + e^{S - M_new} V,
 * and finish with O / L, lse = M + ln L.  pairs[i*n + j] counts the (query, key) pairs with a
 * visible key that step (i, j) touched, summed over batch and heads; it may be NULL. */
int oracle_ring_fwd(const float* q, const float* k, const float* v, int B, int H, int Hkv, long L,
                    int d, int n, int causal, int layout, double* out, double* lse, long* pairs)
{
    if (!check_args(B, H, Hkv, L, d, n, layout)) return ORACLE_BAD_ARGS;
    const long S = L / n;
    const double scale = 1.0 / sqrt((double)d);
    if (pairs) memset(pairs, 0, sizeof(long) * n * n);
    int status = ORACLE_OK;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * S);
        long* my_pairs = (long*)calloc((size_t)n * n, sizeof(long));
        if (!s || !my_pairs) {
#pragma omp atomic write
            status = ORACLE_NO_MEMORY;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long idx = 0; idx < (long)B * H * L; ++idx) {
                long r = idx % L;
                int h = (int)((idx / L) % H);
                int b = (int)(idx / ((long)H * L));
                int g = h / (H / Hkv);
                int i = (int)(r / S);
                long pq = oracle_natural_position(r, L, n, layout);
                const float* qrow = q + idx * d;
                const float* kh = k + ((long)b * Hkv + g) * L * d;
                const float* vh = v + ((long)b * Hkv + g) * L * d;
                double M = -INFINITY, Lsum = 0.0;
                double* O = out + idx * d;
                for (int c = 0; c < d; ++c) O[c] = 0.0;
                for (int step = 0; step < n; ++step) {
                    int j = ((i - step) % n + n) % n;
                    double mloc = -INFINITY;
                    long seen = 0;
                    for (long tt = 0; tt < S; ++tt) {
                        long t = (long)j * S + tt;
                        if (causal && oracle_natural_position(t, L, n, layout) > pq) {
                            s[tt] = -INFINITY;
                            continue;
                        }
                        double acc = 0.0;
                        for (int c = 0; c < d; ++c) acc += (double)qrow[c] * (double)kh[t * d + c];
                        s[tt] = acc * scale;
                        if (s[tt] > mloc) mloc = s[tt];
                        ++seen;
                    }
                    my_pairs[i * n + j] += seen;
                    if (seen == 0) continue; /* the row sees nothing in this block */
                    double Mnew = M > mloc ? M : mloc;
                    double alpha = exp(M - Mnew); /* M = -inf gives 0 */
                    double lloc = 0.0;
                    for (int c = 0; c < d; ++c) O[c] *= alpha;
                    for (long tt = 0; tt < S; ++tt) {
                        if (s[tt] == -INFINITY) continue;
                        double e = exp(s[tt] - Mnew);
                        lloc += e;
                        const float* vrow = vh + ((long)j * S + tt) * d;
                        for (int c = 0; c < d; ++c) O[c] += e * (double)vrow[c];
                    }
                    Lsum = Lsum * alpha + lloc;
                    M = Mnew;
                }
                for (int c = 0; c < d; ++c) O[c] /= Lsum;
                lse[idx] = M + log(Lsum);
            }
            if (pairs) {
#pragma omp critical
                for (long x = 0; x < (long)n * n; ++x) pairs[x] += my_pairs[x];
            }
        }
        free(s);
        free(my_pairs);
    }
    return status;
}

/* Tiles of T x T (query tile, key tile) that contain at least one visible pair, per query shard.
 * Tiles are T consecutive buffer rows starting at each shard's first row (the last one of a shard
 * may be shorter).  A tile pair holds a visible pair iff the smallest natural key position in the
 * key tile is <= the largest natural query position in the query tile.  Brute force over tile pairs. */
int oracle_shard_tiles(long L, int n, int causal, int layout, int T, long* tiles_per_shard)
{
    if (L < 1 || n < 1 || T < 1 || L % n != 0) return ORACLE_BAD_ARGS;
    if (layout != 0 && layout != 1 && layout != 2) return ORACLE_BAD_ARGS;
    if (layout == 1 && L % (2L * n) != 0) return ORACLE_BAD_ARGS;
    const long S = L / n;
    const long tps = (S + T - 1) / T; /* tiles per shard */
    const long nt = tps * n;
    long* tmin = (long*)malloc(sizeof(long) * nt);
    long* tmax = (long*)malloc(sizeof(long) * nt);
    if (!tmin || !tmax) { free(tmin); free(tmax); return ORACLE_NO_MEMORY; }
    for (long x = 0; x < nt; ++x) {
        long shard = x / tps, a = x % tps;
        long r0 = shard * S + a * T, r1 = r0 + T < (shard + 1) * S ? r0 + T : (shard + 1) * S;
        long lo = L, hi = -1;
        for (long r = r0; r < r1; ++r) {
            long p = oracle_natural_position(r, L, n, layout);
            if (p < lo) lo = p;
            if (p > hi) hi = p;
        }
        tmin[x] = lo;
        tmax[x] = hi;
    }
    for (int i = 0; i < n; ++i) {
        long cnt = 0;
        for (long a = 0; a < tps; ++a) {
            long xq = (long)i * tps + a;
            for (long xk = 0; xk < nt; ++xk)
                if (!causal || tmin[xk] <= tmax[xq]) ++cnt;
        }
        tiles_per_shard[i] = cnt;
    }
    free(tmin);
    free(tmax);
    return ORACLE_OK;
}

/* ---------------------------------------------------------------------------------------------
 * Backward (not on the pages; the derivative of the forward definition, reading above).
 * ------------------------------------------------------------------------------------------- */

/* lse and D = <dO, O> of one query row.  lse is the forward definition's; O is the forward
 * definition's output row, or, when out_given is not NULL, that row of out_given: the output a
 * backward receives as its input (a stored, rounded forward result), read like the rounded q, k, v. */
static void row_stats(const float* q, const float* k, const float* v, const float* dout,
                      const float* out_given, int H, int Hkv, long L, int d, int n, int causal,
                      int layout, long idx, double* lse_out, double* D_out, double* o, double* scores)
{
    long r = idx % L;
    int h = (int)((idx / L) % H);
    int b = (int)(idx / ((long)H * L));
    *lse_out = attention_row(q, k, v, H, Hkv, L, d, n, causal, layout, b, h, r, o, scores);
    double D = 0.0;
    for (int c = 0; c < d; ++c)
        D += (double)dout[idx * d + c] * (out_given ? (double)out_given[idx * d + c] : o[c]);
    *D_out = D;
}

/* dQ for a list of query rows (flat (b*H+h)*L + r); dq is [nrows][d].  out: NULL, or the output
 * [B][H][L][d] whose rows give D (see row_stats). */
int oracle_attn_bwd_dq_rows(const float* q, const float* k, const float* v, const float* dout,
                            const float* out, int B, int H, int Hkv, long L, int d, int n, int causal,
                            int layout, long nrows, const long* rows, double* dq)
{
    if (!check_args(B, H, Hkv, L, d, n, layout)) return ORACLE_BAD_ARGS;
    const double scale = 1.0 / sqrt((double)d);
    int status = ORACLE_OK;
#pragma omp parallel
    {
        double* scores = (double*)malloc(sizeof(double) * L);
        double* o = (double*)malloc(sizeof(double) * d);
        if (!scores || !o) {
#pragma omp atomic write
            status = ORACLE_NO_MEMORY;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long i = 0; i < nrows; ++i) {
                long idx = rows[i];
                int h = (int)((idx / L) % H);
                int b = (int)(idx / ((long)H * L));
                int g = h / (H / Hkv);
                double lse, D;
                row_stats(q, k, v, dout, out, H, Hkv, L, d, n, causal, layout, idx, &lse, &D, o, scores);
                /* attention_row left the scaled scores (or -inf) in scores[] */
                const float* kh = k + ((long)b * Hkv + g) * L * d;
                const float* vh = v + ((long)b * Hkv + g) * L * d;
                const float* dorow = dout + idx * d;
                double* dqx = dq + i * d;
                for (int c = 0; c < d; ++c) dqx[c] = 0.0;
                for (long t = 0; t < L; ++t) {
                    if (scores[t] == -INFINITY) continue;
                    double P = exp(scores[t] - lse);
                    double dP = 0.0;
                    for (int c = 0; c < d; ++c) dP += (double)dorow[c] * (double)vh[t * d + c];
                    double dS = P * (dP - D);
                    for (int c = 0; c < d; ++c) dqx[c] += scale * dS * (double)kh[t * d + c];
                }
            }
        }
        free(scores);
        free(o);
    }
    return status;
}

/* dK and dV for a list of key rows (flat (b*Hkv+g)*L + t); dk, dv are [nkeys][d].  out: NULL, or
 * the output whose rows give D (see row_stats).
 * Phase 1 marks the query rows that see any listed key, phase 2 evaluates their lse and D by the
 * forward definition, phase 3 sums the contributions. */
int oracle_attn_bwd_dkv_rows(const float* q, const float* k, const float* v, const float* dout,
                             const float* out, int B, int H, int Hkv, long L, int d, int n, int causal,
                             int layout, long nkeys, const long* keys, double* dk, double* dv)
{
    if (!check_args(B, H, Hkv, L, d, n, layout)) return ORACLE_BAD_ARGS;
    const int G = H / Hkv;
    const double scale = 1.0 / sqrt((double)d);
    const long nq = (long)B * H * L;
    char* need = (char*)calloc(nq, 1);
    double* lse = (double*)malloc(sizeof(double) * nq);
    double* Dv = (double*)malloc(sizeof(double) * nq);
    if (!need || !lse || !Dv) { free(need); free(lse); free(Dv); return ORACLE_NO_MEMORY; }

    /* phase 1: for each listed key, the query rows of its group that can see it */
    for (long x = 0; x < nkeys; ++x) {
        long t = keys[x] % L;
        int g = (int)((keys[x] / L) % Hkv);
        int b = (int)(keys[x] / ((long)Hkv * L));
        long pt = oracle_natural_position(t, L, n, layout);
        for (int hh = 0; hh < G; ++hh) {
            int h = g * G + hh;
            for (long r = 0; r < L; ++r)
                if (!causal || oracle_natural_position(r, L, n, layout) >= pt)
                    need[((long)b * H + h) * L + r] = 1;
        }
    }
    int status = ORACLE_OK;
    /* phase 2 */
#pragma omp parallel
    {
        double* scores = (double*)malloc(sizeof(double) * L);
        double* o = (double*)malloc(sizeof(double) * d);
        if (!scores || !o) {
#pragma omp atomic write
            status = ORACLE_NO_MEMORY;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (long idx = 0; idx < nq; ++idx)
                if (need[idx])
                    row_stats(q, k, v, dout, out, H, Hkv, L, d, n, causal, layout, idx, &lse[idx],
                              &Dv[idx], o, scores);
        }
        free(scores);
        free(o);
    }
    if (status != ORACLE_OK) { free(need); free(lse); free(Dv); return status; }
    /* phase 3 */
#pragma omp parallel for schedule(dynamic, 1)
    for (long x = 0; x < nkeys; ++x) {
        long t = keys[x] % L;
        int g = (int)((keys[x] / L) % Hkv);
        int b = (int)(keys[x] / ((long)Hkv * L));
        long pt = oracle_natural_position(t, L, n, layout);
        const float* krow = k + (((long)b * Hkv + g) * L + t) * d;
        const float* vrow = v + (((long)b * Hkv + g) * L + t) * d;
        double* dkx = dk + x * d;
        double* dvx = dv + x * d;
        for (int c = 0; c < d; ++c) { dkx[c] = 0.0; dvx[c] = 0.0; }
        for (int hh = 0; hh < G; ++hh) {
            int h = g * G + hh;
            for (long r = 0; r < L; ++r) {
                if (causal && oracle_natural_position(r, L, n, layout) < pt) continue;
                long idx = ((long)b * H + h) * L + r;
                const float* qrow = q + idx * d;
                const float* dorow = dout + idx * d;
                double s = 0.0, dP = 0.0;
                for (int c = 0; c < d; ++c) {
                    s += (double)qrow[c] * (double)krow[c];
                    dP += (double)dorow[c] * (double)vrow[c];
                }
                double P = exp(s * scale - lse[idx]);
                double dS = P * (dP - Dv[idx]);
                for (int c = 0; c < d; ++c) {
                    dvx[c] += P * (double)dorow[c];
                    dkx[c] += scale * dS * (double)qrow[c];
                }
            }
        }
    }
    free(need);
    free(lse);
    free(Dv);
    return ORACLE_OK;
}

/* Full backward: dq [B][H][L][d], dk and dv [B][Hkv][L][d]. */
int oracle_attn_bwd(const float* q, const float* k, const float* v, const float* dout, int B, int H,
                    int Hkv, long L, int d, int n, int causal, int layout, double* dq, double* dk,
                    double* dv)
{
    if (!check_args(B, H, Hkv, L, d, n, layout)) return ORACLE_BAD_ARGS;
    long nq = (long)B * H * L, nk = (long)B * Hkv * L;
    long* rows = (long*)malloc(sizeof(long) * (nq > nk ? nq : nk));
    if (!rows) return ORACLE_NO_MEMORY;
    for (long i = 0; i < nq; ++i) rows[i] = i;
    int st = oracle_attn_bwd_dq_rows(q, k, v, dout, NULL, B, H, Hkv, L, d, n, causal, layout, nq, rows, dq);
    if (st == ORACLE_OK) {
        for (long i = 0; i < nk; ++i) rows[i] = i;
        st = oracle_attn_bwd_dkv_rows(q, k, v, dout, NULL, B, H, Hkv, L, d, n, causal, layout, nk, rows,
                                      dk, dv);
    }
    free(rows);
    return st;
}

/* ---------------------------------------------------------------------------------------------
 * One device of the multi-device ring ([LLM101] 6.2 block_attention; [M4-051] section 3): device i
 * holds only shard i's rows; at ring step r it meets the K/V block of shard j = (i - r) mod n.
 * Local buffers hold S = L/n rows per head: q_i, dout_i [B][H][S][d] and k_j, v_j [B][Hkv][S][d]
 * are rows [i*S, (i+1)*S) (resp. [j*S, (j+1)*S)) of the whole-sequence buffers.  Positions and the
 * causal mask come from the whole sequence (L, n, layout).
 * ------------------------------------------------------------------------------------------- */

/* The block attention by definition: for every local row of shard i, attention restricted to the
 * keys of shard j it may see (two passes, float64).  o_part [B][H][S][d] is normalised by the
 * block's own sum, lse_part [B][H][S] is the log-sum-exp over those keys; a row that sees no key
 * of the block gets o_part = 0 and lse_part = -inf.  The n blocks of a row together are the row's
 * full key set, so their (o_part, lse_part) recombine into full attention. */
int oracle_block_fwd(const float* q_i, const float* k_j, const float* v_j, int B, int H, int Hkv, long L, int d,
                     int n, int causal, int layout, int i, int j, double* o_part, double* lse_part)
{
    if (!check_args(B, H, Hkv, L, d, n, layout) || i < 0 || i >= n || j < 0 || j >= n) return ORACLE_BAD_ARGS;
    const long S = L / n;
    const double scale = 1.0 / sqrt((double)d);
    int status = ORACLE_OK;
#pragma omp parallel
    {
        double* sc = (double*)malloc(sizeof(double) * S);
        if (!sc) {
#pragma omp atomic write
            status = ORACLE_NO_MEMORY;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long idx = 0; idx < (long)B * H * S; ++idx) {
                const long u = idx % S; /* local row */
                const int h = (int)((idx / S) % H);
                const int b = (int)(idx / ((long)H * S));
                const int g = h / (H / Hkv);
                const long p = oracle_natural_position((long)i * S + u, L, n, layout);
                const float* qrow = q_i + idx * d;
                const float* kh = k_j + ((long)b * Hkv + g) * S * d;
                const float* vh = v_j + ((long)b * Hkv + g) * S * d;
                double mx = -INFINITY;
                for (long t = 0; t < S; ++t) {
                    if (causal && oracle_natural_position((long)j * S + t, L, n, layout) > p) {
                        sc[t] = -INFINITY;
                        continue;
                    }
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c) acc += (double)qrow[c] * (double)kh[t * d + c];
                    sc[t] = acc * scale;
                    if (sc[t] > mx) mx = sc[t];
                }
                double* o = o_part + idx * d;
                for (int c = 0; c < d; ++c) o[c] = 0.0;
                if (mx == -INFINITY) { /* nothing of this block is visible */
                    lse_part[idx] = -INFINITY;
                    continue;
                }
                double sum = 0.0;
                for (long t = 0; t < S; ++t) {
                    if (sc[t] == -INFINITY) continue;
                    const double e = exp(sc[t] - mx);
                    sum += e;
                    for (int c = 0; c < d; ++c) o[c] += e * (double)vh[t * d + c];
                }
                for (int c = 0; c < d; ++c) o[c] /= sum;
                lse_part[idx] = mx + log(sum);
            }
        }
        free(sc);
    }
    return status;
}

/* The backward contributions of one block by definition: only the pairs (query p of shard i, key t
 * of shard j) with t visible to p, with P = exp(s - lse_p) from the query row's FULL log-sum-exp and
 * D_p = <dO_p, O_p> of the full output (both given, [B][H][S], float64):
 *   dq_part_p = scale sum_t dS_pt k_t,  dk_part_t = scale sum_{p, h in group} dS_pt q_p,
 *   dv_part_t = sum_{p, h in group} P_pt dO_p,   dS_pt = P_pt (<dO_p, v_t> - D_p).
 * dq_part [B][H][S][d], dk_part and dv_part [B][Hkv][S][d].  Summed over the n blocks these are
 * the full gradients (oracle_attn_bwd). */
int oracle_block_bwd(const float* q_i, const float* k_j, const float* v_j, const float* dout_i, const double* lse_i,
                     const double* D_i, int B, int H, int Hkv, long L, int d, int n, int causal, int layout, int i,
                     int j, double* dq_part, double* dk_part, double* dv_part)
{
    if (!check_args(B, H, Hkv, L, d, n, layout) || i < 0 || i >= n || j < 0 || j >= n) return ORACLE_BAD_ARGS;
    const long S = L / n;
    const int G = H / Hkv;
    const double scale = 1.0 / sqrt((double)d);
    /* dQ: one query row at a time */
#pragma omp parallel for schedule(dynamic, 4)
    for (long idx = 0; idx < (long)B * H * S; ++idx) {
        const long u = idx % S;
        const int h = (int)((idx / S) % H);
        const int b = (int)(idx / ((long)H * S));
        const int g = h / G;
        const long p = oracle_natural_position((long)i * S + u, L, n, layout);
        const float* qrow = q_i + idx * d;
        const float* dorow = dout_i + idx * d;
        const float* kh = k_j + ((long)b * Hkv + g) * S * d;
        const float* vh = v_j + ((long)b * Hkv + g) * S * d;
        double* out = dq_part + idx * d;
        for (int c = 0; c < d; ++c) out[c] = 0.0;
        for (long t = 0; t < S; ++t) {
            if (causal && oracle_natural_position((long)j * S + t, L, n, layout) > p) continue;
            double s = 0.0, dP = 0.0;
            for (int c = 0; c < d; ++c) {
                s += (double)qrow[c] * (double)kh[t * d + c];
                dP += (double)dorow[c] * (double)vh[t * d + c];
            }
            const double P = exp(s * scale - lse_i[idx]);
            const double dS = P * (dP - D_i[idx]);
            for (int c = 0; c < d; ++c) out[c] += scale * dS * (double)kh[t * d + c];
        }
    }
    /* dK, dV: one key row at a time, summed over the query heads of its group */
#pragma omp parallel for schedule(dynamic, 4)
    for (long kidx = 0; kidx < (long)B * Hkv * S; ++kidx) {
        const long t = kidx % S;
        const int g = (int)((kidx / S) % Hkv);
        const int b = (int)(kidx / ((long)Hkv * S));
        const long pt = oracle_natural_position((long)j * S + t, L, n, layout);
        const float* krow = k_j + kidx * d;
        const float* vrow = v_j + kidx * d;
        double* dkx = dk_part + kidx * d;
        double* dvx = dv_part + kidx * d;
        for (int c = 0; c < d; ++c) { dkx[c] = 0.0; dvx[c] = 0.0; }
        for (int hh = 0; hh < G; ++hh) {
            const long hbase = ((long)b * H + (long)g * G + hh) * S;
            for (long u = 0; u < S; ++u) {
                if (causal && oracle_natural_position((long)i * S + u, L, n, layout) < pt) continue;
                const long idx = hbase + u;
                const float* qrow = q_i + idx * d;
                const float* dorow = dout_i + idx * d;
                double s = 0.0, dP = 0.0;
                for (int c = 0; c < d; ++c) {
                    s += (double)qrow[c] * (double)krow[c];
                    dP += (double)dorow[c] * (double)vrow[c];
                }
                const double P = exp(s * scale - lse_i[idx]);
                const double dS = P * (dP - D_i[idx]);
                for (int c = 0; c < d; ++c) {
                    dvx[c] += P * (double)dorow[c];
                    dkx[c] += scale * dS * (double)qrow[c];
                }
            }
        }
    }
    return ORACLE_OK;
}

/* Rotary position embedding with natural positions.  [LLM101] section 6 (the questions after 6.2)
 * asks how position information must be treated once K/V blocks travel round the ring; reading C17: every row is rotated by the angle of
 * its NATURAL position p (its place in the whole sequence, from the layout), never by its buffer
 * row or its index inside a shard, so a K/V block carries its positions with it.  The rotation is
 * the RoFormer one (not given by the pages, reading C18): for i in [0, d/2) with
 * theta_i = base^(-2i/d), the pair (x[2i], x[2i+1]) turns by the angle p * theta_i:
 *   y[2i]   = x[2i] cos(p theta_i) - x[2i+1] sin(p theta_i)
 *   y[2i+1] = x[2i] sin(p theta_i) + x[2i+1] cos(p theta_i).
 * inverse != 0 turns by -p * theta_i instead (the transposed rotation: what maps the gradient with
 * respect to the rotated rows back to the unrotated ones).
 * x and y are [nheads][L][d] (nheads = B * H); d even. */
int oracle_rope(const float* x, long nheads, long L, int d, int n, int layout, double base, int inverse,
                double* y)
{
    if (nheads < 1 || L < 1 || d < 2 || d % 2 != 0 || n < 1 || L % n != 0 || base <= 0.0)
        return ORACLE_BAD_ARGS;
    if (layout != 0 && layout != 1 && layout != 2) return ORACLE_BAD_ARGS;
    if (layout == 1 && L % (2L * n) != 0) return ORACLE_BAD_ARGS;
    const double sign = inverse ? -1.0 : 1.0;
#pragma omp parallel for schedule(static)
    for (long hr = 0; hr < nheads * L; ++hr) {
        const long r = hr % L;
        const double p = (double)oracle_natural_position(r, L, n, layout);
        const float* xr = x + hr * d;
        double* yr = y + hr * d;
        for (int i = 0; i < d / 2; ++i) {
            const double theta = pow(base, -2.0 * i / d);
            const double ang = sign * p * theta;
            const double c = cos(ang), sn = sin(ang);
            const double x0 = xr[2 * i], x1 = xr[2 * i + 1];
            yr[2 * i] = x0 * c - x1 * sn;
            yr[2 * i + 1] = x0 * sn + x1 * c;
        }
    }
    return ORACLE_OK;
}

/* Number of OpenMP threads the oracle runs on (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
