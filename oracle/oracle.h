/*
 * oracle.h -- plain, slow, single-threaded CPU oracle for the emulated-rank
 * gradient collectives.  TEST INFRASTRUCTURE ONLY: nothing in the product
 * library includes, links or calls this code; only the tests, the smoke check
 * and the benchmark's CPU-baseline leg do.  It shares no code, header or
 * table with the CUDA path.
 *
 * Page abbreviations used in the citations below:
 *   [DT]  "Distributed Training for Large Models: Collectives, FSDP/ZeRO,
 *          DeviceMesh, and Multi-Dimensional Parallelism" (zexinliu.github.io)
 *   [AIG] "AI Infra Guide, Chapter 6: Distributed Training Basics"
 *          (theaiera.top, ch06)
 *   [NX]  nxmr.cn news 160867, the article on collective communication and
 *          model parallelism (numbered sub-headings 1.1 .. 7)
 *
 * Precision: the pages fix fp32 for the gradient reduction (FSDP
 * MixedPrecision reduce_dtype=float32, [AIG] 6.3.4; [DT] section 11 notes
 * that frameworks may send low-precision tensors yet sum them in fp32) and
 * for the master weights
 * and Adam moments ([AIG] 6.2.7 Table 6-3).  The oracle therefore computes in
 * fp32 wherever the method does, with every operation rounded once (built
 * with -ffp-contract=off).  int32 sums wrap modulo 2^32.
 *
 * Ranks, chunks and shards: N ranks r = 0..N-1 each hold a full buffer of
 * `count` elements.  Chunk j covers [j*L, min((j+1)*L, count)) with
 * L = ceil(count/N); trailing chunks may be short or empty (torch.chunk-style
 * uneven shards, [DT] section 4 FSDP2, Shard(0) on a dim not divisible by the
 * world size).  Shard j of a reduce-scatter is chunk j reduced over ranks.
 */
#ifndef FSDP_ORACLE_H
#define FSDP_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types and reduction ops of the oracle (its own numbering). */
enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_I32 = 2 };
enum { ORC_SUM = 0, ORC_AVG = 1 };

/* Return codes. */
enum { ORC_OK = 0, ORC_EINVAL = 1, ORC_EUNSUPPORTED = 2, ORC_ENOMEM = 3 };

#define ORC_MAX_RANKS 64

/* ---- chunking -------------------------------------------------------- */
size_t orc_chunk_len(size_t count, int n);
void orc_chunk_bounds(size_t count, int n, int j, size_t* lo, size_t* hi);

/* ---- bf16 <-> f32 ---------------------------------------------------- */
/* Round-to-nearest-even on the fp32 bit pattern; NaN stays a quiet NaN. */
uint16_t orc_f32_to_bf16(float x);
float orc_bf16_to_f32(uint16_t b);
size_t orc_esize(int dtype);
void orc_f32_to_bf16_array(size_t n, const float* x, uint16_t* out);

/* ---- message counters (elements, per rank) --------------------------- */
typedef struct {
  uint64_t sent[ORC_MAX_RANKS];  /* elements sent by each rank           */
  uint64_t recv[ORC_MAX_RANKS];  /* elements received by each rank       */
  int steps;                     /* logical communication steps taken    */
} orc_traffic;

/* ---- ring reduce-scatter, literal message-passing simulation ------------
 * Ring direction r -> r+1.  At step s (1..N-1) rank r sends the partial sum
 * it holds for chunk (r-s) mod N; the receiver adds its own contribution to
 * the same chunk (partial + local).  Chunk j therefore starts at rank j+1
 * and ends at its owner j ([DT] section 2, Reduce-Scatter, the N=4 ring
 * schedule; [NX] 2.2).  Partials are carried in fp32 (int32 for I32).
 * After the last step the epilogue applies AVG (acc / N, fp32 division) and
 * the output cast (bf16 RNE) and writes shard r to out_shards[r].
 *
 * Optional trace (may be NULL), both sized [(N-1)*N], indexed [(s-1)*N + r]:
 *   trace_chunk[(s-1)*N + r] = chunk id rank r sent at step s
 *   trace_value[(s-1)*N + d] = receiver d's partial after its add, first
 *                              element of the chunk, as a double
 */
int orc_ring_reduce_scatter(int n, size_t count, int in_dtype, int op,
                            const void* const* bufs, void* const* out_shards,
                            int out_dtype, orc_traffic* tr, int* trace_chunk,
                            double* trace_value);

/* The same with an explicit chunk length L (chunk j = [j*L, (j+1)*L) cut
 * at count; L*N >= count), for FSDP2's dim-0 shards, whose chunks are
 * whole rows ([DT] section 4, FSDP2 Shard(0)). */
int orc_ring_reduce_scatter_L(int n, size_t count, size_t L, int in_dtype,
                              int op, const void* const* bufs,
                              void* const* out_shards, int out_dtype,
                              orc_traffic* tr, int* trace_chunk,
                              double* trace_value);

/* Low-precision wire ([DT] section 11: frameworks may send tensors in low
 * precision and still accumulate in fp32): the ring reduce-scatter /
 * all-reduce above, except that every message -- the partial sum a rank
 * sends to its neighbour -- is rounded to wire_dtype (ORC_BF16, RNE) before
 * it leaves; the receiver adds its own contribution in fp32.  ORC_F32 gives
 * the ordinary result.  Float inputs only for ORC_BF16. */
int orc_ring_reduce_scatter_wire(int n, size_t count, int in_dtype, int op,
                                 int wire_dtype, const void* const* bufs,
                                 void* const* out_shards, int out_dtype);
int orc_ring_all_reduce_wire(int n, size_t count, int in_dtype, int op,
                             int wire_dtype, const void* const* in,
                             void* const* out, int out_dtype);

/* HSDP gradient reduction ([AIG] 6.3.6; [DT] section 4, a 2-D mesh whose
 * one dimension shards and the other replicates): N = R*S ranks, rank
 * (g, s) at index g*S + s.  A ring reduce-scatter over the S ranks of each
 * group (chunk length ceil(count/S), fp32 partials), then for every shard
 * j a ring all-reduce of the R groups' shard-j partial sums, then AVG
 * (/ N, once) and the output cast.  out_shards[g*S + j] receives shard j;
 * every group holds the same values. */
int orc_hsdp_reduce_scatter(int R, int S, size_t count, int in_dtype, int op,
                            const void* const* bufs, void* const* out_shards,
                            int out_dtype);

/* Closed-form fold with the same association:
 * y_j[e] = ((x_{j+1}[e] + x_{j+2}[e]) + ...) + x_j[e], ranks mod N. */
int orc_fold_reduce_scatter(int n, size_t count, int in_dtype, int op,
                            const void* const* bufs, void* const* out_shards,
                            int out_dtype);

/* The same fold on gathered columns: vals is [nsamp][n] (rank order
 * 0..n-1 for each sample), chunk[i] is the chunk index of sample i. */
int orc_fold_columns(int n, size_t nsamp, int in_dtype, int op,
                     const void* vals, const int* chunk, void* out,
                     int out_dtype);

/* ---- ring all-gather, literal simulation --------------------------------
 * Rank r starts with shard r.  At step s (1..N-1) every rank forwards the
 * shard it received at the previous step (its own at step 1) to r+1
 * ([DT] section 2, All-Reduce second phase, N=4 ring).  Each rank keeps its
 * shards in arrival order and finally rearranges them by shard index into
 * its full buffer.  trace_arrival (may be NULL) is [(N-1)*N]: shard id that
 * rank d received at step s, at [(s-1)*N + d]. */
int orc_ring_all_gather(int n, size_t count, int dtype,
                        const void* const* shards, void* const* bufs,
                        orc_traffic* tr, int* trace_arrival);

int orc_ring_all_gather_L(int n, size_t count, size_t L, int dtype,
                          const void* const* shards, void* const* bufs,
                          orc_traffic* tr, int* trace_arrival);

/* ---- ring all-reduce = ring reduce-scatter then ring all-gather ---------
 * in and out may be the same buffers (in place). */
int orc_ring_all_reduce(int n, size_t count, int in_dtype, int op,
                        const void* const* in, void* const* out,
                        int out_dtype, orc_traffic* tr);

/* Naive reduce-to-root (rank 0 sums ranks 0..N-1 in rank order) followed by
 * a broadcast from the root ([NX] 2.2; [DT] section 2, Reduce). */
int orc_naive_all_reduce(int n, size_t count, int in_dtype, int op,
                         const void* const* in, void* const* out,
                         int out_dtype, orc_traffic* tr);

/* ---- scalar AdamW -------------------------------------------------------
 * Decoupled weight decay (Loshchilov & Hutter; torch.optim.AdamW named in
 * [AIG] 6.8 (FSDP production config) and [DT] section 4 FSDP2 code skeleton).  The pages never print
 * the rule; the textbook form is used, all in fp32:
 *   p <- p * (1 - lr*wd)
 *   m <- b1*m + (1-b1)*g ;  v <- b2*v + (1-b2)*(g*g)
 *   mh = m / (1 - b1^t)  ;  vh = v / (1 - b2^t)
 *   p <- p - lr * (mh / (sqrt(vh) + eps))
 * Scalars derived from the hyper-parameters are formed in double and rounded
 * once to fp32. */
typedef struct {
  double lr, beta1, beta2, eps, weight_decay;
  long step;
} orc_adamw_cfg;

void orc_adamw(size_t n, float* p, float* m, float* v, const float* g,
               const orc_adamw_cfg* cfg);

/* ---- FSDP step ----------------------------------------------------------
 * The FSDP1 flat-parameter lifecycle restricted to one step ([DT] section 4,
 * FSDP1 lifecycle; ZeRO-3 flow steps 5-6): ring reduce-scatter of the bf16
 * grads with fp32 partials and AVG (reduce_dtype fp32, [AIG] 6.3.4), AdamW on
 * each owner's fp32 master/m/v shard, bf16 cast of the updated master shard,
 * ring all-gather of the bf16 shards into every rank's full param buffer.
 * master[j], m[j], v[j] hold shard j (chunk j's length). */
int orc_fsdp_step(int n, size_t count, const uint16_t* const* grads,
                  float* const* master, float* const* m, float* const* v,
                  const orc_adamw_cfg* cfg, uint16_t* const* params);

/* FSDP step with global gradient-norm clipping ([AIG] 6.8, the production
 * loop calls clip_grad_norm_(max_norm=1.0) on the sharded model before the
 * optimizer step).  After the reduce-scatter, the L2 norm of the whole
 * averaged fp32 gradient (all shards) is computed in double, shard by shard
 * in element order; the clip coefficient c = max_norm / (norm + 1e-6),
 * formed in double, capped at 1 and rounded to fp32, multiplies every
 * gradient element (one fp32 multiply) before AdamW.  *norm_out receives
 * the norm. */
int orc_fsdp_step_clipped(int n, size_t count, const uint16_t* const* grads,
                          float* const* master, float* const* m,
                          float* const* v, const orc_adamw_cfg* cfg,
                          double max_norm, uint16_t* const* params,
                          double* norm_out);

/* ---- DDP gradient buckets -----------------------------------------------
 * Plan: tensors are visited in reverse index order (backward order) and
 * appended to the current bucket while its byte size plus the tensor's stays
 * within cap_bytes; otherwise a new bucket starts.  A tensor is never split;
 * one larger than the cap sits alone in its own bucket.  Offsets inside a
 * bucket are contiguous element offsets with no padding ([AIG] 6.2.4 bucket
 * rules; [NX] 5.1; flat layout as in [DT] section 4 FSDP1 FlatParameter).
 * Outputs: tensor_bucket[t], tensor_offset[t] (elements), bucket_numel[b]
 * (caller sizes it ntensors), *nbuckets. */
int orc_bucket_plan(int ntensors, const size_t* numels, size_t esize,
                    size_t cap_bytes, int* tensor_bucket,
                    size_t* tensor_offset, size_t* bucket_numel,
                    int* nbuckets);

/* tensors[r*T + t], buckets[r*B + b]; plain byte copies. */
void orc_bucket_pack(int n, int ntensors, const size_t* numels, size_t esize,
                     const int* tensor_bucket, const size_t* tensor_offset,
                     const void* const* tensors, void* const* buckets);
void orc_bucket_unpack(int n, int ntensors, const size_t* numels,
                       size_t esize, const int* tensor_bucket,
                       const size_t* tensor_offset,
                       const void* const* buckets, void* const* tensors);

/* ---- FSDP2: per-parameter Shard(0) ([DT] section 4, FSDP2) --------------
 * Each parameter p is its own DTensor sharded on dim 0: rank j owns rows
 * [j*Lr, min((j+1)*Lr, dim0)) with Lr = ceil(dim0 / N) (torch.chunk-like,
 * trailing shards short or empty), i.e. chunk length Lr * row_numel
 * elements of the flattened parameter.  The step per parameter is the
 * FSDP step above with that chunking: ring reduce-scatter of the bf16
 * grads (fp32 partials, AVG), AdamW on owner j's fp32 shard, bf16 cast,
 * ring all-gather.  Arrays are indexed [p*N + r] (grads, params: full
 * parameter; master/m/v: shard j of parameter p at [p*N + j]). */
typedef struct {
  size_t dim0;
  size_t row_numel;
} orc_param_shape;

int orc_fsdp2_step(int nparams, const orc_param_shape* shapes, int n,
                   const uint16_t* const* grads, float* const* master,
                   float* const* m, float* const* v, const orc_adamw_cfg* cfg,
                   uint16_t* const* params);

/* ---- gradient accumulation ([AIG] 6.2.6, DDP no_sync) -------------------
 * Micro-steps inside no_sync() only add the new local gradient to the
 * accumulated one, rank by rank, with no communication:
 * acc[e] <- acc[e] + g[e] in fp32 (g of dtype ORC_F32 or ORC_BF16).  The
 * last micro-step adds its gradient and then all-reduces the sum. */
void orc_accumulate(size_t count, float* acc, const void* g, int g_dtype);

/* ---- alpha-beta model ([AIG] 6.1.4; [DT] section 2; [NX] 2.3) -----------
 * T_ring_allreduce = 2(N-1)*alpha + 2(N-1)/N * S / B, seconds. */
double orc_alpha_beta_ring_allreduce(int n, double bytes, double alpha_s,
                                     double bw_bytes_per_s);

#ifdef __cplusplus
}
#endif
#endif
