/*
 * ringattn.h -- C ABI of libringattn.so: Ring Attention's blockwise exact attention on one GB300.
 *
 * What is computed (sources are web pages on Ring Attention, cited by title and section):
 *   The sequence of length L is cut into n shards; shard i holds Q_i, K_i, V_i
 *   (airsota "M4-051 Ring Attention and sequence parallelism", section 3).  At ring step
 *   r = 0..n-1 shard i takes the K/V block of shard (i - r) mod n, computes the block attention
 *   S = Q K^T / sqrt(d) and folds it into a running max / running sum / running output
 *   (LLM-101-CN "distributed hands-on code", section 6.2, block_attention and forward; "Lecture 30:
 *   TP/PP/SP/CP", section 3.2).  After n steps the output O / L equals full softmax attention.
 *   Causal: a key is visible to a query iff its natural position is <= the query's; blocks that
 *   are entirely masked are skipped (M4-051 sections 3 and 5).  Zigzag layout: the sequence is cut
 *   into 2n chunks and shard i holds chunks i and 2n-1-i, which equalises causal work
 *   (M4-051 section 4 item 2; Lecture 30 section 3.2, "Zigzag / Striped").
 *   On one GPU the n shards are virtual: they are row ranges of the same buffers, and the ring
 *   schedule is the order in which the kernels walk K/V tiles.  No data moves between shards.
 *
 * Conventions shared by every entry point:
 *   - Layout of the sequence axis: every buffer stores it in the layout's order, i.e. as the
 *     concatenation of the shards' local buffers (shard i occupies rows [i*L/n, (i+1)*L/n)).
 *     With RA_LAYOUT_ZIGZAG, rows [i*S, i*S + C) of shard i are natural positions [i*C, (i+1)*C)
 *     and rows [i*S + C, (i+1)*S) are natural positions [(2n-1-i)*C, (2n-i)*C), with S = L/n and
 *     C = L/(2n).  With RA_LAYOUT_STRIPED, row i*S + t of shard i is natural position t*n + i
 *     (shard i holds tokens i, i + n, i + 2n, ...: the round-robin split of "Lecture 30:
 *     TP/PP/SP/CP", section 3.2).  Outputs come back in the same order as the inputs.
 *   - Shapes (row-major, d contiguous): q, out, dout, dq: [B][H][L][d]; k, v, dk, dv:
 *     [B][Hkv][L][d]; lse: [B][H][L] float32, natural logarithm of sum_t exp(s_t).
 *     Query head h reads kv head h / (H / Hkv) (grouped-query attention).  Scale is 1/sqrt(d).
 *   - dtype: RA_F32 (float) or RA_BF16 (bfloat16) for q, k, v, out, dout.  Accumulation is float32.
 *   - Pointers are DEVICE pointers unless stated otherwise, allocated and owned by the caller,
 *     16-byte aligned.  The library never allocates or frees device memory and keeps no pointer
 *     after a call returns.
 *   - stream is a cudaStream_t passed as void* (NULL = legacy default stream).  Work is enqueued on
 *     it; no call synchronises the host unless stated.  The device calls enqueue kernel launches
 *     only: after one call on a device has run outside stream capture (it sets the kernels'
 *     launch attributes and looks up the status word), they may be recorded into a CUDA graph
 *     (not ring_attn_fwd_host, whose copies and kernels run on streams of the library).
 *   - Errors: arguments are checked before anything is enqueued; a rejected call returns
 *     RA_ERR_INVALID_ARG or RA_ERR_UNSUPPORTED and enqueues nothing.  A failed launch returns
 *     RA_ERR_CUDA.  ring_attn_last_error() gives a message for the calling thread's last failure.
 *     Kernels never trap: every wait inside a kernel is bounded, and a wait that runs out sets a
 *     device status word and the kernel returns; ring_attn_device_status reads the word,
 *     ring_attn_device_check turns it into RA_ERR_TIMEOUT.  Nothing throws across this interface.
 */
#ifndef RINGATTN_H
#define RINGATTN_H

#include <stddef.h>

#if defined(__GNUC__)
#define RA_API __attribute__((visibility("default")))
#else
#define RA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef int ra_status;
#define RA_OK 0
#define RA_ERR_INVALID_ARG 1
#define RA_ERR_UNSUPPORTED 2
#define RA_ERR_CUDA 3
#define RA_ERR_NO_DEVICE 4
#define RA_ERR_TIMEOUT 5   /* returned by ring_attn_device_check: a bounded wait in a kernel ran out */

#define RA_LAYOUT_CONTIGUOUS 0
#define RA_LAYOUT_ZIGZAG 1
#define RA_LAYOUT_STRIPED 2

#define RA_F32 0
#define RA_BF16 1

/* Kernel paths reported by ring_attn_fwd_path / ring_attn_bwd_path. */
#define RA_PATH_SIMT 1      /* CUDA-core kernels: any shape, f32 or bf16 */
#define RA_PATH_TCGEN05 2   /* tensor-core kernels (TMA + tcgen05 + TMEM): bf16, d = 128 or 64,
                               shard (contiguous, striped) or chunk (zigzag) length a multiple of
                               256 (forward) or 128 (backward) */

/* Device status bits (ring_attn_device_status). */
#define RA_DEVICE_TIMEOUT 1u  /* a bounded wait inside a kernel ran out; the kernel stopped */
#define RA_DEVICE_LAYOUT 2u   /* a kernel found its shared memory misaligned and did nothing */

/*
 * ring_attn_fwd -- the whole ring forward in one launch.
 * For every shard i and ring step r = 0..n_shards-1, the rows of shard i attend to the K/V of
 * shard (i - r) mod n_shards, with the running-max / running-sum rescale of LLM-101-CN section 6.2,
 * fully masked causal blocks skipped (M4-051 section 3).  Writes out (dtype) and lse.
 *   q, k, v   inputs as above (dtype);   out [B][H][L][d] (dtype);   lse [B][H][L] float32.
 *   L % n_shards == 0; zigzag also needs L % (2 n_shards) == 0; H % Hkv == 0; d in {64, 128}.
 */
RA_API ra_status ring_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                        int B, int H, int Hkv, int L, int d, int n_shards, int causal, int layout,
                        int dtype, void* stream);

/*
 * ring_attn_fwd_f32out -- ring_attn_fwd with the output written in float32 whatever the inputs'
 * dtype: the normalised output before it is rounded to dtype (ring_attn_fwd's out is this array
 * rounded to nearest).  For a backward that takes D = rowsum(dout * out) from the unrounded output
 * (ring_attn_bwd_f32out): with bf16 out, D carries out's rounding, which at the first positions of a
 * causal sequence (a few large, cancelling terms per gradient) moves dq and dk by up to ~1.5e-2.
 *   out: DEVICE float32 [B][H][L][d].  Everything else as ring_attn_fwd.
 */
RA_API ra_status ring_attn_fwd_f32out(const void* q, const void* k, const void* v, float* out, float* lse,
                               int B, int H, int Hkv, int L, int d, int n_shards, int causal, int layout,
                               int dtype, void* stream);

/*
 * ring_attn_ring_step_fwd -- ring step `step` alone, for all shards at once: shard i attends to
 * the K/V of shard (i - step) mod n_shards only (one block_attention of LLM-101-CN section 6.2).
 *   o_part [B][H][L][d] float32 receives each row's attention output normalised by its own sum;
 *   lse_part [B][H][L] float32 its log-sum-exp.  A row that sees no key in that block gets
 *   o_part = 0 and lse_part = -infinity.  Fold the steps together with ring_attn_lse_merge.
 */
RA_API ra_status ring_attn_ring_step_fwd(const void* q, const void* k, const void* v, float* o_part,
                                  float* lse_part, int B, int H, int Hkv, int L, int d,
                                  int n_shards, int step, int causal, int layout, int dtype,
                                  void* stream);

/*
 * ring_attn_ring_step_fwd_accumulate -- ring step `step` folded straight into a running result,
 * in place: the block result of step `step` (as ring_attn_ring_step_fwd computes it) is merged into
 * (o_acc, lse_acc) in the kernel's epilogue, as ring_attn_lse_merge would merge it, without the
 * partial ever going to memory (the running (M, L, O) update of LLM-101-CN section 6.2 across
 * steps).  o_acc [B][H][L][d] and lse_acc [B][H][L] float32: a valid running state -- finite o_acc
 * rows; lse_acc = -infinity marks a row with nothing yet (its o_acc is then ignored).  A row that
 * sees no key at this step is left unchanged.
 */
RA_API ra_status ring_attn_ring_step_fwd_accumulate(const void* q, const void* k, const void* v, float* o_acc,
                                                    float* lse_acc, int B, int H, int Hkv, int L, int d,
                                                    int n_shards, int step, int causal, int layout, int dtype,
                                                    void* stream);

/*
 * ring_attn_lse_merge -- fold one partial result into a running one, in place:
 *   lse = max(a, b) + log(1 + exp(-|a - b|)),  o = exp(a - lse) o_acc + exp(b - lse) o_part,
 * with a = lse_acc, b = lse_part (the online-softmax merge across ring steps, LLM-101-CN 6.2,
 * written for normalised partials).  A partial with lse = -infinity leaves the row unchanged.
 *   o_acc, o_part: [rows][d] float32;  lse_acc, lse_part: [rows] float32;  rows >= 0, d >= 1.
 */
RA_API ra_status ring_attn_lse_merge(float* o_acc, float* lse_acc, const float* o_part,
                              const float* lse_part, long long rows, int d, void* stream);

/*
 * ring_attn_fwd_stepwise -- the ring forward run step by step, as the multi-device algorithm
 * does it: n_shards launches, step 0 writing a float32 running output and lse and every later
 * step folding its block into them (ring_attn_ring_step_fwd_accumulate), then the conversion of
 * the float32 output into `out`.  Same arguments and results as ring_attn_fwd, plus
 *   workspace: device memory of at least ring_attn_fwd_stepwise_workspace_size(...) bytes (the
 *   float32 running output, B * H * L * d * 4 bytes rounded up to 256), 256-byte aligned, owned by
 *   the caller; its contents on entry do not matter.  The running lse is `lse` itself.
 */
RA_API ra_status ring_attn_fwd_stepwise(const void* q, const void* k, const void* v, void* out,
                                 float* lse, int B, int H, int Hkv, int L, int d, int n_shards,
                                 int causal, int layout, int dtype, void* workspace,
                                 size_t workspace_bytes, void* stream);
RA_API size_t ring_attn_fwd_stepwise_workspace_size(int B, int H, int L, int d);

/*
 * ring_attn_fwd_host -- ring_attn_fwd on HOST buffers: q, k, v are read from host memory and out,
 * lse written back to host memory, with the copies overlapped with the compute.  The problem is
 * cut into its B * Hkv kv-head groups (each group: the G = H / Hkv query heads that share a kv
 * head); while group g computes, the inputs of group g + 1 are copied in and the results of group
 * g - 1 copied out on two copy streams of the library (one H2D, one D2H), through two device slots
 * of the workspace.  The groups' kernels alternate between two compute streams of the library, so
 * that one group's kernel starts on the SMs the previous one's last CTAs leave.  Each copy is one
 * cudaMemcpyAsync of a contiguous slice.
 *   q, k, v, out, lse: HOST pointers with the layouts of ring_attn_fwd; page-locked memory lets the
 *   copies run asynchronously and overlap (pageable memory works but serialises them).
 *   workspace: DEVICE, 256-byte aligned, >= ring_attn_fwd_host_workspace_size(H, Hkv, L, d, dtype).
 *   Stream-ordered: when `stream` completes, out and lse are on the host.  One call at a time per
 *   device enqueues (a library mutex); calls on one device run one after another.
 */
RA_API ra_status ring_attn_fwd_host(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                                    int H, int Hkv, int L, int d, int n_shards, int causal, int layout,
                                    int dtype, void* workspace, size_t workspace_bytes, void* stream);
RA_API size_t ring_attn_fwd_host_workspace_size(int H, int Hkv, int L, int d, int dtype);

/*
 * ring_attn_bwd -- gradients of sum(out * dout) with respect to q, k and v, recomputing the
 * attention weights P = exp(s - lse) from the saved lse (the pages give no backward; this is the
 * derivative of the forward definition): D = rowsum(dout * out), dS = P (dout . v - D),
 * dq = dS k / sqrt(d), dk = dS^T q / sqrt(d), dv = P^T dout, with dk and dv summed over the
 * query heads that share a kv head.  Causal blocks that are entirely masked are skipped.
 *   out, lse: the forward's results for the same inputs.  dout: [B][H][L][d] (dtype).
 *   dq [B][H][L][d], dk and dv [B][Hkv][L][d] in grad_dtype (RA_F32 or RA_BF16).
 *   workspace: device memory of at least ring_attn_bwd_workspace_size(...) bytes (256-byte
 *   aligned; contents on entry do not matter), owned by the caller.
 */
RA_API ra_status ring_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                        const float* lse, const void* dout, void* dq, void* dk, void* dv,
                        int grad_dtype, void* workspace, size_t workspace_bytes, int B, int H,
                        int Hkv, int L, int d, int n_shards, int causal, int layout, int dtype,
                        void* stream);
/*
 * ring_attn_bwd_f32out -- ring_attn_bwd with `out` in float32 (from ring_attn_fwd_f32out) while
 * q, k, v, dout are in dtype: D = rowsum(dout * out) is taken from the unrounded output.  Same
 * workspace, arguments and results as ring_attn_bwd otherwise.
 */
RA_API ra_status ring_attn_bwd_f32out(const void* q, const void* k, const void* v, const float* out,
                               const float* lse, const void* dout, void* dq, void* dk, void* dv,
                               int grad_dtype, void* workspace, size_t workspace_bytes, int B, int H,
                               int Hkv, int L, int d, int n_shards, int causal, int layout, int dtype,
                               void* stream);
RA_API size_t ring_attn_bwd_workspace_size(int B, int H, int Hkv, int L, int d, int grad_dtype);

/*
 * ring_attn_bwd_static_scratch -- the backward of ring_attn_bwd for callers that cannot allocate
 * device memory (a host framework that owns all device memory as one pre-sized pool and passes
 * only input and output buffers, or a loop that may not call the allocator).  The pages that
 * define the method have no counterpart to this call: it is an interface convenience, not part
 * of the method.
 * Same arguments and results as ring_attn_bwd without the workspace: the scratch comes from a
 * file-scope device array of ring_attn_bwd_static_scratch_capacity() bytes (64 MiB) that every
 * GPU loading this library holds until the process exits.  Allocates nothing.
 *   - A problem whose ring_attn_bwd_workspace_size exceeds the capacity is rejected with
 *     RA_ERR_INVALID_ARG before anything is enqueued (fp32 gradients need 4 bytes per query row,
 *     bf16 gradients 4 * (d + 1)).
 *   - The first call on a device looks the array's device address up (cudaGetSymbolAddress) with
 *     that device current; make that first call before any stream capture.  The address is kept
 *     for the life of the process: cudaDeviceReset after the first call is not supported.
 *   - Every call on a device shares the array and leaves its contents behind; each call rewrites
 *     or zeroes what it reads.  Calls whose GPU work overlaps (other streams or threads) race.
 */
RA_API ra_status ring_attn_bwd_static_scratch(const void* q, const void* k, const void* v,
                                              const void* out, const float* lse, const void* dout,
                                              void* dq, void* dk, void* dv, int grad_dtype, int B,
                                              int H, int Hkv, int L, int d, int n_shards,
                                              int causal, int layout, int dtype, void* stream);
RA_API size_t ring_attn_bwd_static_scratch_capacity(void);

/*
 * One device of the multi-device ring.  In the pages' setting each device i holds only its own
 * shard -- Q_i, K_i, V_i -- and at ring step r = 0..n-1 computes the attention of Q_i against the
 * K/V block it currently holds, that of shard j = (i - r) mod n, folds it into a running output,
 * and passes the block on to device i + 1 while receiving the next from device i - 1
 * (LLM-101-CN "distributed hands-on code", section 6.2, block_attention and forward; M4-051
 * section 3; "Lecture 30: TP/PP/SP/CP", section 3.2).  These calls are that per-device data path;
 * moving the blocks between devices is the caller's (NCCL or another transport).
 *
 * Local buffers: a device's tensors hold S = L / n_shards rows per head -- rows [i*S, (i+1)*S) of
 * the whole-sequence buffers of the other calls, in the same order (shard i's rows of the layout):
 *   q, dout: [B][H][S][d] (dtype);  k, v: [B][Hkv][S][d] (dtype) of the shard they came from;
 *   o_acc, dq_acc: [B][H][S][d] float32;  lse_acc, lse, D: [B][H][S] float32;
 *   dk, dv: [B][Hkv][S][d] float32, the gradients of the K/V block they travel with.
 * L, n_shards, causal and layout describe the whole sequence: natural positions and the causal
 * mask come from them, so shard_q and shard_kv (0 .. n_shards-1) must name the shards the local
 * buffers hold.  Same requirements on L, n_shards, d and the pointers as ring_attn_fwd.
 */

/*
 * ring_attn_block_fwd -- block attention of the query shard shard_q against the K/V block of shard
 * shard_kv, written to (accumulate = 0) or folded into (accumulate = 1) the running state
 * (o_acc, lse_acc): o_acc holds the output normalised by its own running sum, lse_acc the running
 * log-sum-exp (natural log).  Folding uses the online-softmax merge of ring_attn_lse_merge; a row
 * with lse_acc = -infinity holds nothing yet (its o_acc is not read).  A row that sees no key of
 * this block gets o = 0, lse = -infinity (accumulate = 0) or is left unchanged (accumulate = 1);
 * fully masked causal tiles are skipped.  After the n blocks of the ring, o_acc is the attention
 * output (convert it with ring_attn_f32_convert) and lse_acc its log-sum-exp.
 */
RA_API ra_status ring_attn_block_fwd(const void* q, const void* k, const void* v, float* o_acc, float* lse_acc,
                                     int B, int H, int Hkv, int L, int d, int n_shards, int shard_q, int shard_kv,
                                     int accumulate, int causal, int layout, int dtype, void* stream);

/*
 * ring_attn_block_bwd -- the backward of one block: the contributions of the pairs (query of shard
 * shard_q, key of shard shard_kv) to the gradients, with P = exp(s - lse) recomputed from the
 * query rows' final lse and D = rowsum(dout * out) from ring_attn_bwd_preprocess:
 *   dq_acc += dS k / sqrt(d)          (added to: zero it before the first block),
 *   dk (+)= dS^T q / sqrt(d),  dv (+)= P^T dout,   dS = P (dout . v - D),
 * dk and dv summed over the query heads that share a kv head, and added to (accumulate_kv = 1) or
 * stored (accumulate_kv = 0; a key row that meets no query of this block gets 0).  The sum of
 * the n blocks' contributions is ring_attn_bwd's result.
 */
RA_API ra_status ring_attn_block_bwd(const void* q, const void* k, const void* v, const void* dout,
                                     const float* lse, const float* D, float* dq_acc, float* dk, float* dv, int B,
                                     int H, int Hkv, int L, int d, int n_shards, int shard_q, int shard_kv,
                                     int accumulate_kv, int causal, int layout, int dtype, void* stream);

/*
 * ring_attn_bwd_preprocess -- D[r] = sum_c out[r][c] * dout[r][c] for `rows` rows of d elements
 * (dtype), D float32: the per-row term of the backward, computed once per device before its blocks.
 * ring_attn_f32_zero -- x[0 .. count) = 0 (float32).
 * ring_attn_f32_add -- acc[i] += part[i] for i < count (float32): a device adds its contribution
 *   to the dK / dV accumulators that arrive with a block before passing them on.
 * ring_attn_f32_convert -- dst[i] = src[i] converted to dtype (RA_F32 copies, RA_BF16 rounds to
 *   nearest even): the running output or a gradient accumulator into the caller's dtype.
 * Device pointers, 16-byte aligned; count >= 0 (0 enqueues nothing).
 */
RA_API ra_status ring_attn_bwd_preprocess(const void* out, const void* dout, float* D, long long rows, int d,
                                          int dtype, void* stream);

/*
 * ring_attn_bwd_preprocess_f32out -- ring_attn_bwd_preprocess with out in float32 (the forward's
 * output before rounding, e.g. one device's float32 running output of the ring) and dout in dtype.
 */
RA_API ra_status ring_attn_bwd_preprocess_f32out(const float* out, const void* dout, float* D, long long rows,
                                          int d, int dtype, void* stream);

/*
 * ring_attn_block_rope -- ring_attn_rope on one device's local buffer: x [B][H][S][d] holds shard
 * `shard`'s rows (rows [shard*S, (shard+1)*S) of the whole-sequence layout), and every row turns by
 * the angle of its natural position in the whole sequence, so that the K/V blocks a device passes
 * on carry their positions with them (LLM-101-CN section 6, the questions after 6.2).  Same rotation,
 * arguments and requirements as ring_attn_rope plus shard in [0, n_shards); bit-identical to the
 * same rows of ring_attn_rope on the whole sequence.
 */
RA_API ra_status ring_attn_block_rope(void* x, int B, int H, int L, int d, int n_shards, int shard, int layout,
                                      int dtype, double base, int inverse, void* stream);
RA_API ra_status ring_attn_f32_zero(float* x, long long count, void* stream);
RA_API ra_status ring_attn_f32_add(float* acc, const float* part, long long count, void* stream);
RA_API ra_status ring_attn_f32_convert(const float* src, void* dst, long long count, int dtype, void* stream);

/*
 * ring_attn_shard_tiles -- HOST ONLY, no CUDA call.  For each query shard, the number of
 * (query tile, key tile) pairs of `tile` x `tile` buffer rows (tiles start at each shard's first
 * row) that hold at least one visible (query, key) pair: the per-shard causal work that the
 * contiguous layout leaves unbalanced (device i's work grows with i, M4-051 section 4 item 2) and
 * the zigzag layout equalises.  tiles_per_shard: HOST array of n_shards entries.
 */
RA_API ra_status ring_attn_shard_tiles(int L, int n_shards, int causal, int layout, int tile,
                                long long* tiles_per_shard);

/*
 * ring_attn_fwd_tile_visits / ring_attn_bwd_tile_visits -- ring_attn_fwd / ring_attn_bwd that also
 * count the work the tensor-core kernels do: for every tile pair a kernel computes, 1 is added to
 * visits[i * n_shards + j], i the shard of the query rows and j the shard of the key rows
 * (forward: a 256-row query block of one query head against a 128-row K/V tile; backward: a
 * 128-row query tile of one query head against a 128-row K/V tile).  The causal skip of M4-051
 * section 3 shows as visits[i][j] == 0 for every key shard whose positions all follow the query
 * shard's, and a computed pair always holds at least one visible (query, key) pair.
 *   visits: DEVICE array of n_shards * n_shards unsigned 64-bit counters, 16-byte aligned, added
 *   to (the caller zeroes it).  Other arguments and results as in ring_attn_fwd / ring_attn_bwd.
 *   RA_ERR_UNSUPPORTED when the problem does not take the tensor-core path (ring_attn_*_path).
 */
RA_API ra_status ring_attn_fwd_tile_visits(const void* q, const void* k, const void* v, void* out,
                                           float* lse, int B, int H, int Hkv, int L, int d,
                                           int n_shards, int causal, int layout, int dtype,
                                           unsigned long long* visits, void* stream);
RA_API ra_status ring_attn_bwd_tile_visits(const void* q, const void* k, const void* v,
                                           const void* out, const float* lse, const void* dout,
                                           void* dq, void* dk, void* dv, int grad_dtype,
                                           void* workspace, size_t workspace_bytes, int B, int H,
                                           int Hkv, int L, int d, int n_shards, int causal,
                                           int layout, int dtype, unsigned long long* visits,
                                           void* stream);

/*
 * ring_attn_rope -- rotary position embedding, in place, of a [B][H][L][d] buffer stored in the
 * layout's order (q with its H query heads, or k with its Hkv heads; pass that head count as H).
 * LLM-101-CN "distributed hands-on code", section 6 (the questions after 6.2), asks how positions
 * must be handled when K/V blocks travel round the ring: here row r turns by the angle of its
 * NATURAL position p(r) (its place in the whole sequence, from the layout -- never its buffer row or
 * shard-local index), so the blocks carry their positions with them.  Rotation (RoFormer): for
 * i in [0, d/2), theta_i = base^(-2i/d), the pair (x[2i], x[2i+1]) turns by p * theta_i:
 *   x'[2i] = x[2i] cos - x[2i+1] sin,   x'[2i+1] = x[2i] sin + x[2i+1] cos.
 *   x: DEVICE pointer, dtype RA_BF16 or RA_F32, 16-byte aligned, overwritten.
 *   base > 0 and finite (10000 is the usual value).
 *   inverse != 0 turns by -p * theta_i: applied to dq and dk from ring_attn_bwd (computed with the
 *   rotated q and k) it gives the gradients with respect to the unrotated q and k.
 *   L % n_shards == 0 (zigzag: L % 2n == 0); d in {64, 128}.  Stream-ordered, no host sync.
 */
RA_API ra_status ring_attn_rope(void* x, int B, int H, int L, int d, int n_shards, int layout, int dtype,
                                double base, int inverse, void* stream);

/*
 * DeepSpeed-Ulysses, the other context-parallel design ("Lecture 30: TP/PP/SP/CP", sections 3.3 and
 * 3.4).  Shard i of n holds all heads of its S = L / n tokens; an all-to-all turns that into H / n
 * heads of the whole sequence, each shard runs ordinary attention over the full sequence for its
 * heads, and a second all-to-all brings the output back.  Heads must divide by n: H % n_shards == 0
 * and Hkv % n_shards == 0, else RA_ERR_INVALID_ARG (checked before anything runs).  On one GPU the
 * shards are slices of one allocation and the all-to-alls are row permutations.
 *   Token split (inputs and outputs):  q, out [n][B][S][H][d], k, v [n][B][S][Hkv][d],
 *   lse [n][B][S][H] float32; local token s of shard i is natural position p(i * S + s) under the
 *   layout, as for the ring (contiguous, zigzag or striped).
 *   Head split (inside):  [n][B][H/n][L][d], natural token order, heads h -> shard h / (H/n).
 *
 * ring_attn_ulysses_a2a -- one all-to-all: direction 0 token split -> head split, 1 the reverse.
 *   src, dst: DEVICE, distinct, 16-byte aligned; rows of d elements of dtype (d * size a multiple
 *   of 4 bytes; pass d = 1 with RA_F32 for an lse-shaped tensor); H is that tensor's head count.
 * ring_attn_ulysses_fwd -- the whole forward: three all-to-alls in, attention on every shard, two
 *   back.  Same results as ring_attn_fwd (exact attention), in the token split.
 *   workspace: DEVICE, 256-byte aligned, at least ring_attn_ulysses_workspace_size(...) bytes.
 */
RA_API ra_status ring_attn_ulysses_a2a(const void* src, void* dst, int B, int H, int L, int d, int n_shards,
                                       int layout, int dtype, int direction, void* stream);
RA_API ra_status ring_attn_ulysses_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                                       int B, int H, int Hkv, int L, int d, int n_shards, int causal, int layout,
                                       int dtype, void* workspace, size_t workspace_bytes, void* stream);
RA_API size_t ring_attn_ulysses_workspace_size(int B, int H, int Hkv, int L, int d, int dtype);
/*
 * ring_attn_ulysses_bwd -- the backward of ring_attn_ulysses_fwd: all-to-alls of q, k, v, out,
 *   dout and lse into the head split, the backward of ring_attn_bwd on every shard over the whole
 *   sequence, and all-to-alls of dq, dk, dv back.  All tensors in the token split (lse as returned
 *   by ring_attn_ulysses_fwd); dq [n][B][S][H][d], dk, dv [n][B][S][Hkv][d] in grad_dtype.
 *   workspace: DEVICE, 256-byte aligned, at least ring_attn_ulysses_bwd_workspace_size(...) bytes.
 */
RA_API ra_status ring_attn_ulysses_bwd(const void* q, const void* k, const void* v, const void* out,
                                       const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                       int grad_dtype, void* workspace, size_t workspace_bytes, int B, int H,
                                       int Hkv, int L, int d, int n_shards, int causal, int layout, int dtype,
                                       void* stream);
RA_API size_t ring_attn_ulysses_bwd_workspace_size(int B, int H, int Hkv, int L, int d, int n_shards, int dtype,
                                                   int grad_dtype);

/* Which kernel path ring_attn_fwd / ring_attn_bwd take for these arguments (RA_PATH_*), written
 * to *path (HOST pointer).  Same argument checks as the calls themselves; no CUDA call. */
RA_API ra_status ring_attn_fwd_path(int B, int H, int Hkv, int L, int d, int n_shards, int causal,
                             int layout, int dtype, int* path);
RA_API ra_status ring_attn_bwd_path(int B, int H, int Hkv, int L, int d, int n_shards, int causal,
                             int layout, int dtype, int* path);

/*
 * ring_attn_selftest_bounded_wait -- exercises the failure path of the kernels' bounded waits
 * without a fault: one GPU thread waits, through the kernels' own bounded-wait routine, on an
 * mbarrier that nothing will complete.  After limit_ns (1e3 .. 1e8 ns) the wait gives up, sets
 * RA_DEVICE_TIMEOUT in the device status word (read it with ring_attn_device_status) and the
 * kernel returns; the context stays usable.  *returned (DEVICE pointer to an unsigned int,
 * 16-byte aligned) receives 1 when the wait gave up, 2 if it had completed.
 */
RA_API ra_status ring_attn_selftest_bounded_wait(unsigned long long limit_ns, unsigned int* returned,
                                                 void* stream);

/*
 * The device status word.  There is one word per device, not one per stream or per call: it
 * collects the RA_DEVICE_* bits of every kernel of this library that ran on the device since the
 * word was last read, and reading it clears it for every caller.  A caller that shares the device
 * with others (other threads, streams or libraries using this one) and needs to know whether ITS
 * work timed out must read the word at a point where no other caller's work of this library is in
 * flight on the device; otherwise a bit may belong to another caller, or another caller's read may
 * have cleared a bit that this caller's kernel set.
 *   The device address of the word is looked up once per device, on the first call that needs it,
 * and kept for the life of the process: cudaDeviceReset after that first call is not supported
 * (the module may be reloaded elsewhere).
 *
 * ring_attn_device_status -- reads the word of the current device into *status (HOST pointer; bits
 * RA_DEVICE_*), then clears it.  Synchronises `stream`.
 */
RA_API ra_status ring_attn_device_status(unsigned int* status, void* stream);

/*
 * ring_attn_device_check -- ring_attn_device_status as a status code: synchronises `stream`, reads
 * and clears the word, and returns RA_ERR_TIMEOUT if a bounded wait inside a kernel ran out (that
 * kernel stopped early: its outputs are incomplete and must not be used), RA_ERR_CUDA if a kernel
 * found its shared memory misaligned and did nothing, RA_OK if the word was clear.
 */
RA_API ra_status ring_attn_device_check(void* stream);

/* Message for the calling thread's last non-OK status ("" if none).  Never NULL. */
RA_API const char* ring_attn_last_error(void);

/* ABI version (incremented on any incompatible change). */
RA_API int ring_attn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RINGATTN_H */
