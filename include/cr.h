/*
 * cr.h -- C ABI of libcr, the emulated-rank gradient collectives for one
 * GB300 GPU.
 *
 * N data-parallel ranks are emulated as N buffers resident in the HBM of one
 * GPU.  Each collective is one (or a few) CUDA kernels that read the rank
 * buffers directly; a "message" of the ring schedule becomes a global load
 * by the thread that reduces that element.  The ring schedule survives as
 * the per-chunk order in which the ranks' contributions are summed, so the
 * result is reproducible and equal, bit for bit, to the ring's.
 *
 * Page abbreviations used in the citations:
 *   [DT]  "Distributed Training for Large Models: Collectives, FSDP/ZeRO,
 *          DeviceMesh, and Multi-Dimensional Parallelism" (zexinliu.github.io)
 *   [AIG] "AI Infra Guide, Chapter 6: Distributed Training Basics"
 *          (theaiera.top, ch06)
 *   [NX]  nxmr.cn news 160867, the article on collective communication and
 *          model parallelism (numbered sub-headings 1.1 .. 7)
 *
 * Conventions shared by every entry point
 *  - Pointer arrays (bufs, out_shards, ...) are HOST arrays of DEVICE
 *    pointers, one per rank; the library copies them into the kernel's
 *    parameters, so the host arrays may be reused as soon as the call returns.
 *  - The caller owns every device buffer.  No entry point allocates device
 *    memory; apart from cr_bucket_plan (the host-side plan the caller
 *    releases with cr_bucket_plan_free), cr_reducer_create (a host object
 *    and CUDA events, released with cr_reducer_destroy) and cr_comm_create
 *    (a host object, released with cr_comm_destroy) nothing allocates at
 *    all, and the library keeps no state between calls beyond cached device
 *    attributes, the static array of cr_fsdp_step_clipped_noalloc and the
 *    device error word of the checked build (cr_check_word).
 *  - Entry points may be called from several host threads at once, on
 *    different buffers: each call's marshalled state and error detail are
 *    per thread, and the cached device attributes are locked.  A reducer
 *    is used by one thread at a time, and calls of
 *    cr_fsdp_step_clipped_noalloc share one static array (see there).
 *  - Every launching call is asynchronous on `stream` (NULL = the legacy
 *    default stream).  Argument errors are detected on the host before any
 *    launch and leave all buffers untouched; a launch (or event record, or
 *    copy) that CUDA refuses returns CR_ERR_CUDA with CUDA's error name and
 *    text in the detail.  If the call's first launch is refused nothing of
 *    the call runs; if a later one is (calls of several launches), the
 *    call's outputs -- and its inputs, where it works in place -- are
 *    undefined.  A refused launch leaves the library usable: the next call
 *    does not see the old error.  cr_last_error() gives the detail of the
 *    last failure on the calling thread.
 *  - Chunking: with L = ceil(count/N), chunk j is the element range
 *    [j*L, min((j+1)*L, count)); trailing chunks may be short or empty, as
 *    with torch.chunk-style uneven Shard(0) shards ([DT] section 4, FSDP2).
 *    Shard j of a reduce-scatter is chunk j reduced over all ranks.
 *  - Reduction order: chunk j is summed starting from rank (j+1) mod N and
 *    ending at its owner j, as the ring reduce-scatter of [DT] section 2
 *    (Reduce-Scatter, N=4 schedule) and [NX] 2.2 do:
 *        y_j = ((x_{j+1} + x_{j+2}) + ... ) + x_j     (ranks mod N)
 *    Partial sums are fp32 for fp32/bf16 inputs (reduce dtype fp32,
 *    [AIG] 6.3.4) and int32 with two's-complement wrap for int32.
 *  - CR_AVG divides the finished fp32 sum by N once ([DT] section 2,
 *    All-Reduce: G = sum_i G_i / N); bf16 outputs are rounded to nearest
 *    even once, after the average.
 *  - Every pointer must be aligned to its element size (CR_ERR_ALIGNMENT).
 *    16-byte aligned buffers take the 128-bit vector path; others a slower
 *    element-wise path with identical results.  Where only the shards are
 *    off the vector grid (a chunk length that is not a multiple of the
 *    vector, or an unaligned shard pointer) the rank buffers are still read
 *    as vectors and the shard elements stored one by one, staged per warp
 *    so that every store covers 32 consecutive elements.
 */
#ifndef CR_H
#define CR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so that no CUDA header is
 * needed to use the library. */
typedef struct CUstream_st* cr_stream_t;

typedef enum {
  CR_OK = 0,
  CR_ERR_INVALID_ARG = 1, /* NULL where a pointer is needed, bad N/count,
                             overlapping buffers that may not overlap    */
  CR_ERR_UNSUPPORTED = 2, /* legal but unimplemented dtype/op combination */
  CR_ERR_ALIGNMENT = 3,   /* pointer not aligned to its element size      */
  CR_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed         */
  CR_ERR_TIMEOUT = 5      /* a rank of a cr_comm_t collective never joined */
} cr_status;

typedef enum { CR_F32 = 0, CR_BF16 = 1, CR_I32 = 2 } cr_dtype;
typedef enum { CR_SUM = 0, CR_AVG = 1 } cr_op;

#define CR_MAX_RANKS 64

/* ---- errors and version ------------------------------------------------ */
const char* cr_status_string(cr_status status);
/* Detail of the last non-OK status returned on this thread ("" if none).
 * The string is owned by the library and valid until the next call. */
const char* cr_last_error(void);
/* Library version, major*10000 + minor*100 + patch. */
int cr_version(void);

/* ---- chunking -------------------------------------------------------------
 * cr_chunk_len: L = ceil(count/nranks) (0 if nranks < 1).
 * cr_shard_range: element range [*lo, *hi) of chunk j.  CR_ERR_INVALID_ARG
 * if nranks is outside [1, CR_MAX_RANKS], j outside [0, nranks) or an output
 * pointer is NULL.  Host only. */
size_t cr_chunk_len(size_t count, int nranks);
cr_status cr_shard_range(size_t count, int nranks, int j, size_t* lo,
                         size_t* hi);

/* ---- reduce-scatter -------------------------------------------------------
 * [DT] section 2, Reduce-Scatter: y_j = sum over source ranks i of x_{j,i},
 * where x_{j,i} is chunk j of rank i's buffer; rank j keeps y_j.
 *   bufs[r]        rank r's input, `count` elements of in_dtype
 *   out_shards[j]  shard j, cr_shard_range(count, nranks, j) length, of
 *                  out_dtype (may be NULL when that shard is empty)
 *   op             CR_SUM or CR_AVG (CR_AVG needs a floating type)
 * Supported (in, out): (F32,F32), (BF16,BF16), (BF16,F32), (I32,I32).
 * In place is allowed when in_dtype == out_dtype and
 * out_shards[j] == (char*)bufs[j] + j*L*esize; any other overlap between an
 * output and an input, or between two outputs, is CR_ERR_INVALID_ARG.
 * Vector path: all pointers 16-byte aligned and L*esize(in) and
 * L*esize(out) multiples of 16. */
cr_status cr_reduce_scatter(const void* const* bufs, int nranks, size_t count,
                            cr_dtype in_dtype, cr_op op,
                            void* const* out_shards, cr_dtype out_dtype,
                            cr_stream_t stream);

/* ---- all-gather -----------------------------------------------------------
 * [DT] section 2, All-Gather: every rank receives concat(p_0, ..., p_{N-1}).
 *   shards[j]  shard j, cr_shard_range length, of dtype (NULL if empty)
 *   bufs[r]    rank r's output, `count` elements:
 *              bufs[r][j*L + k] = shards[j][k] for every r
 * In place is allowed when shards[j] == (char*)bufs[j] + j*L*esize (that
 * store is then skipped); other overlaps are CR_ERR_INVALID_ARG.
 * Vector path: 16-byte aligned pointers and L*esize a multiple of 16. */
cr_status cr_all_gather(const void* const* shards, int nranks, size_t count,
                        cr_dtype dtype, void* const* bufs, cr_stream_t stream);

/* ---- all-reduce -----------------------------------------------------------
 * [DT] section 2, All-Reduce = Reduce-Scatter + All-Gather, fused into one
 * kernel: every element of every output buffer receives the reduced value
 * of that element.  in[r] and out[r], `count` elements each.  in == out per
 * rank (in place) is allowed when in_dtype == out_dtype; other overlaps are
 * CR_ERR_INVALID_ARG.  Supported pairs as for cr_reduce_scatter.
 * Vector path: all pointers 16-byte aligned (any L). */
cr_status cr_all_reduce(const void* const* in, int nranks, size_t count,
                        cr_dtype in_dtype, cr_op op, void* const* out,
                        cr_dtype out_dtype, cr_stream_t stream);

/* ---- all-reduce from host memory, pipelined -------------------------------
 * The all-reduce of cr_all_reduce (in place, in_dtype == out_dtype) for
 * rank buffers that live in host memory.  The range is cut into slices of
 * slice_elems elements; for each slice the call enqueues the host-to-device
 * copies of every rank's slice on h2d_stream, the all-reduce of that slice
 * (same chunks, same ring order as the whole-buffer call, so the result is
 * bit-identical) on compute_stream, and the device-to-host copies of the
 * result on d2h_stream.  Events order the three streams, so slice s+1's
 * upload, slice s's reduction and slice s-1's download run at once over the
 * full-duplex host link.  The call first makes h2d_stream and d2h_stream
 * wait for work already queued on compute_stream, and finally makes
 * compute_stream wait for the last download: synchronising compute_stream
 * waits for the whole operation.
 *   host_in[r]   rank r's input, count elements (pinned host memory for
 *                asynchronous copies; pageable memory works, serialised)
 *   host_out[r]  rank r's result, count elements (may equal host_in[r])
 *   dev_bufs[r]  device staging for rank r, count elements, caller-owned;
 *                holds the reduced values afterwards
 *   slice_elems  0 picks about 16 slices (at least 2^18 elements each);
 *                otherwise rounded up to a multiple of 64
 * The three streams may be the same stream (no overlap then).  Events are
 * created per call and released as they complete; no memory is allocated.
 * Errors as for cr_all_reduce; host buffers must be non-NULL and aligned to
 * the element size, and no two buffers of the same kind may overlap. */
cr_status cr_all_reduce_staged(const void* const* host_in,
                               void* const* host_out, void* const* dev_bufs,
                               int nranks, size_t count, cr_dtype dtype,
                               cr_op op, size_t slice_elems,
                               cr_stream_t compute_stream,
                               cr_stream_t h2d_stream, cr_stream_t d2h_stream);

/* The same all-reduce for rank buffers in pinned host memory, read and
 * written by the kernel itself over the GPU's coherent host link: every
 * input byte crosses the link once towards the GPU, every result byte once
 * back, with no staging copy in HBM (the reduced values go to dev_out as
 * well when it is non-NULL).  On a GB300 the link, not HBM, bounds this
 * call; it moves the same bytes as upload + all-reduce + download, but
 * with both directions in flight at once.
 *   host_in[r], host_out[r]  count elements each, page-locked and mapped
 *                            (cudaHostAlloc, cudaHostRegister or managed);
 *                            host_out[r] == host_in[r] is allowed (in place)
 *   dev_out                  NULL, or nranks device buffers (nranks <= 32)
 * CR_ERR_INVALID_ARG for host memory the GPU cannot address (pageable
 * memory: use cr_all_reduce_staged), otherwise errors as cr_all_reduce. */
cr_status cr_all_reduce_host(const void* const* host_in, void* const* host_out,
                             void* const* dev_out, int nranks, size_t count,
                             cr_dtype dtype, cr_op op, cr_stream_t stream);

/* ---- low-precision wire ---------------------------------------------------
 * [DT] section 11 (precision and distributed communication): a framework
 * may move gradients in low precision while accumulating in fp32.  These
 * are cr_reduce_scatter / cr_all_reduce with the ring's messages carried as
 * wire_dtype: with CR_BF16 the partial sum a rank forwards to its neighbour
 * is rounded to bf16 (nearest even) before the receiver adds its own
 * contribution in fp32, so chunk j becomes
 *     p = x_{j+1};  p = bf16(p) + x_{j+2};  ...;  y_j = bf16(p) + x_j
 * (the owner's last addition is not rounded; CR_AVG and the output cast
 * follow as usual).  The all-gather half of cr_all_reduce_wire moves the
 * finished values in out_dtype, so every rank holds the same result.
 * wire_dtype CR_F32 gives exactly cr_reduce_scatter / cr_all_reduce.
 *   wire_dtype  CR_F32 or CR_BF16 (else CR_ERR_INVALID_ARG); CR_BF16 needs a
 *               floating in_dtype (else CR_ERR_UNSUPPORTED)
 * Every other argument, rule and error as for cr_reduce_scatter and
 * cr_all_reduce. */
cr_status cr_reduce_scatter_wire(const void* const* bufs, int nranks,
                                 size_t count, cr_dtype in_dtype, cr_op op,
                                 cr_dtype wire_dtype, void* const* out_shards,
                                 cr_dtype out_dtype, cr_stream_t stream);
cr_status cr_all_reduce_wire(const void* const* in, int nranks, size_t count,
                             cr_dtype in_dtype, cr_op op, cr_dtype wire_dtype,
                             void* const* out, cr_dtype out_dtype,
                             cr_stream_t stream);

/* ---- HSDP: shard within a group, replicate across groups ------------------
 * [AIG] 6.3.6 (hybrid sharding: shard inside a node, replicate across
 * nodes) and [DT] section 4, FSDP2 (a 2-D mesh, one dimension sharded and the
 * other replicated).  N = R*S ranks on an R x S mesh; rank (g, s) is index
 * g*S + s.  The gradient is reduce-scattered in ring order over the S ranks
 * of each group (shard j = chunk j with L = ceil(count/S)), then each
 * shard is all-reduced in ring order over the R groups (shard j's len_j
 * elements in R chunks of ceil(len_j/R), chunk i summed from group i+1 to
 * group i), all in fp32 partials (int32 wraps); CR_AVG divides by N once.
 *   bufs[g*S + s]        rank (g, s)'s input, `count` elements of in_dtype
 *   out_shards[g*S + j]  shard j as group g holds it (every group receives
 *                        the same values), cr_shard_range(count, S, j)
 *                        length of out_dtype (NULL if empty)
 * R, S >= 1 and R*S <= CR_MAX_RANKS (else CR_ERR_INVALID_ARG).  Supported
 * pairs as for cr_reduce_scatter.  In place is allowed when in_dtype ==
 * out_dtype and out_shards[g*S + j] == (char*)bufs[g*S + j] + j*L*esize;
 * any other overlap is CR_ERR_INVALID_ARG.  R == 1 is cr_reduce_scatter
 * over S ranks; S == 1 is cr_all_reduce over R ranks (outputs only).
 * Vector path: pointers 16-byte aligned and L*esize(in), L*esize(out)
 * multiples of 16. */
cr_status cr_hsdp_reduce_scatter(const void* const* bufs, int R, int S,
                                 size_t count, cr_dtype in_dtype, cr_op op,
                                 void* const* out_shards, cr_dtype out_dtype,
                                 cr_stream_t stream);

/* ---- DDP bucket plan (host) -----------------------------------------------
 * [AIG] 6.2.4: gradients go into buckets (default 25 MB) in the order
 * backward produces them; [AIG] 6.2.6 Horovod Tensor Fusion; [NX] 5.1.
 * Tensors are visited from the last index to the first (backward order) and
 * appended to the current bucket while its bytes plus the tensor's stay
 * within cap_bytes; otherwise a new bucket starts.  A tensor is never split;
 * one larger than the cap gets a bucket of its own.  Tensor offsets inside a
 * bucket are contiguous, in elements, with no padding (the flat layout of
 * [DT] section 4, FSDP1 FlatParameter).
 * On success *plan receives a host object the caller releases with
 * cr_bucket_plan_free.  CR_ERR_INVALID_ARG: ntensors < 0, numels NULL with
 * ntensors > 0, elem_size 0, cap_bytes 0, plan NULL, or byte sizes that
 * overflow size_t. */
typedef struct cr_bucket_plan_t {
  int ntensors;
  int nbuckets;
  size_t elem_size;
  size_t cap_bytes;
  size_t* numels;        /* [ntensors], copy of the input                */
  int* tensor_bucket;    /* [ntensors], bucket holding tensor t          */
  size_t* tensor_offset; /* [ntensors], element offset inside the bucket */
  size_t* bucket_numel;  /* [nbuckets], elements in bucket b             */
} cr_bucket_plan_t;

cr_status cr_bucket_plan(const size_t* numels, int ntensors, size_t elem_size,
                         size_t cap_bytes, cr_bucket_plan_t** plan);
void cr_bucket_plan_free(cr_bucket_plan_t* plan);

/* ---- bucket pack / unpack -------------------------------------------------
 * Byte copies between each rank's tensors and its buckets:
 *   pack:   buckets[r*B + b][off_t + i] = tensors[r*T + t][i]
 *   unpack: tensors[r*T + t][i] = buckets[r*B + b][off_t + i]
 * with b = plan->tensor_bucket[t], off_t = plan->tensor_offset[t],
 * T = plan->ntensors, B = plan->nbuckets.  Pointers may be NULL only for
 * empty tensors; every pointer must be aligned to plan->elem_size.
 * Tensors and buckets must not overlap (not checked).  Any byte offset is
 * handled; the copies run as 16-byte vectors with funnel shifts when the
 * source and destination are mutually misaligned. */
cr_status cr_bucket_pack(const cr_bucket_plan_t* plan, int nranks,
                         const void* const* tensors, void* const* buckets,
                         cr_stream_t stream);
cr_status cr_bucket_unpack(const cr_bucket_plan_t* plan, int nranks,
                           const void* const* buckets, void* const* tensors,
                           cr_stream_t stream);

/* DDP middle step: every bucket of every rank all-reduced in place, with
 * the result cr_all_reduce would give on each bucket (chunks of the
 * bucket's own element count); bucket b of rank r is buckets[r*B + b].
 * All buckets go in one launch (per 128 buckets).  Buckets must not
 * overlap (CR_ERR_INVALID_ARG); supported dtype/op pairs as cr_all_reduce
 * with in == out. */
cr_status cr_bucket_all_reduce(const cr_bucket_plan_t* plan, int nranks,
                               void* const* buckets, cr_dtype dtype, cr_op op,
                               cr_stream_t stream);

/* DDP bucket all-reduce without packing: the result of cr_bucket_pack,
 * cr_bucket_all_reduce and cr_bucket_unpack, bit for bit, computed straight
 * on the gradient tensors ("AI Infra Guide, Chapter 6", 6.2.4,
 * gradient_as_bucket_view: gradients alias the bucket instead of being
 * copied into it).  Element i of tensor t is reduced in the ring order of
 * its bucket position off_t + i within bucket b = plan->tensor_bucket[t]
 * (chunk length ceil(bucket numel / N)), and written back in place to every
 * rank's tensor.  HBM traffic: N reads + N writes per element, a third of
 * the pack / all-reduce / unpack sequence.
 *   tensors[r*T + t]  rank r's tensor t (NULL only if empty), in/out
 * dtype's size must equal plan->elem_size; tensors must not overlap
 * (CR_ERR_INVALID_ARG).  One launch per 128 tensors (per 2048/N tensors
 * when N > 16). */
cr_status cr_bucket_all_reduce_fused(const cr_bucket_plan_t* plan, int nranks,
                                     void* const* tensors, cr_dtype dtype,
                                     cr_op op, cr_stream_t stream);

/* ---- DDP reducer: bucket all-reduce overlapped with backward --------------
 * [AIG] 6.2.4-6.2.5 (figure 6-2): backward produces gradients last layer
 * first; as soon as every gradient of a bucket is ready, that bucket's
 * all-reduce starts on the communication stream while backward goes on.
 * Buckets start strictly in bucket-index order (a bucket that fills early
 * waits for its predecessors), as every rank must issue its collectives in
 * the same order.  Each bucket's all-reduce is cr_bucket_all_reduce_fused
 * restricted to that bucket's tensors, so after a full iteration every
 * tensor holds exactly what cr_bucket_all_reduce_fused gives.
 *
 * cr_reducer_create: validates as cr_bucket_all_reduce_fused (tensors
 *   [r*T + t], N*T pairwise disjoint, aligned), copies the plan and the
 *   pointer table (the caller may free its plan), and creates one CUDA event
 *   per bucket on the current device (host memory and events only; no
 *   device memory).  comm_ctas >= 0 caps the CTAs of every bucket launch
 *   (0: no cap) so that communication leaves SMs to the compute kernels;
 *   results do not depend on it.  comm_stream: where the all-reduces run.
 * cr_reducer_mark_ready: the gradient of tensor t (on all N ranks) has been
 *   enqueued on compute_stream.  For each bucket this makes launchable, in
 *   order: an event is recorded on compute_stream, comm_stream waits for
 *   it, and the bucket's all-reduce is enqueued on comm_stream.
 *   CR_ERR_INVALID_ARG: t outside [0, T), t already marked this iteration.
 * cr_reducer_launched: buckets started so far this iteration (-1 if NULL).
 * cr_reducer_finalize: every tensor must have been marked
 *   (CR_ERR_INVALID_ARG otherwise, nothing enqueued); compute_stream then
 *   waits for all of comm_stream's work, and the next iteration begins.
 * cr_reducer_destroy: releases the object and its events (work already
 *   enqueued is unaffected).
 * The reducer's device must be current for every call.  Not thread-safe.
 * On CR_ERR_CUDA the iteration's state is undefined: destroy the reducer. */
typedef struct cr_reducer cr_reducer_t;

cr_status cr_reducer_create(const cr_bucket_plan_t* plan, int nranks,
                            void* const* tensors, cr_dtype dtype, cr_op op,
                            int comm_ctas, cr_stream_t comm_stream,
                            cr_reducer_t** out);
cr_status cr_reducer_mark_ready(cr_reducer_t* red, int tensor,
                                cr_stream_t compute_stream);
int cr_reducer_launched(const cr_reducer_t* red);
cr_status cr_reducer_finalize(cr_reducer_t* red, cr_stream_t compute_stream);
void cr_reducer_destroy(cr_reducer_t* red);

/* ---- thread-per-rank communicator -----------------------------------------
 * [DT] section 2 and [AIG] 6.1: with real ranks, every rank calls a
 * collective on its own tensor and the collective runs once all ranks have
 * called it.  cr_comm_t gives the emulated ranks that form: each rank's host
 * thread calls cr_comm_<collective>(comm, rank, its buffers...) and blocks
 * until all nranks ranks have joined the same collective; the last to
 * arrive checks that all calls agree (collective, count, dtypes, op) and
 * enqueues the single-kernel collective (cr_all_reduce in place,
 * cr_reduce_scatter, cr_all_gather) over the N ranks' buffers on the
 * communicator's stream.  Every rank then returns that call's status; the
 * work is asynchronous on the stream, as with NCCL.
 * Failures ([AIG] 6.8 and the pages' troubleshooting notes: the NCCL timeout
 * and watchdog, hangs from mismatched calls), decided on the host before
 * any launch:
 *  - a rank that does not join within timeout_ms: every waiting rank returns
 *    CR_ERR_TIMEOUT, nothing is launched, and the communicator is broken --
 *    every later call returns CR_ERR_TIMEOUT at once (cr_comm_broken
 *    reports 1); destroy it, as an aborted NCCL communicator;
 *  - calls that disagree: every rank returns CR_ERR_INVALID_ARG, nothing is
 *    launched, and the next collective may be joined;
 *  - rank outside [0, nranks), or a rank joining the same collective twice:
 *    CR_ERR_INVALID_ARG for that call.
 * The argument checks of the underlying entry point (alignment, overlaps)
 * apply at launch and their status is returned to every rank.  Buffers are
 * device pointers owned by the caller.  cr_comm_create allocates a host
 * object (no CUDA call); cr_comm_destroy releases it (no rank may be inside
 * a call). */
typedef struct cr_comm cr_comm_t;

cr_status cr_comm_create(int nranks, int timeout_ms, cr_stream_t stream,
                         cr_comm_t** out);
cr_status cr_comm_all_reduce(cr_comm_t* comm, int rank, void* buf,
                             size_t count, cr_dtype dtype, cr_op op);
cr_status cr_comm_reduce_scatter(cr_comm_t* comm, int rank, const void* buf,
                                 void* shard, size_t count, cr_dtype in_dtype,
                                 cr_op op, cr_dtype out_dtype);
cr_status cr_comm_all_gather(cr_comm_t* comm, int rank, const void* shard,
                             void* buf, size_t count, cr_dtype dtype);
int cr_comm_broken(const cr_comm_t* comm);
void cr_comm_destroy(cr_comm_t* comm);

/* ---- fused FSDP / ZeRO-3 step ---------------------------------------------
 * One kernel performs the step of [DT] section 4 (ZeRO-3/FSDP flow steps
 * 5-6; FSDP1 unit lifecycle "backward post-hook" then "optimizer step" then
 * the next forward's all-gather) for one flat parameter buffer:
 *   1. reduce-scatter of the bf16 grads, fp32 partials in ring order, / N
 *      (reduce_dtype fp32, keep_low_precision_grads=False, [AIG] 6.3.4);
 *   2. AdamW on owner j's fp32 master/m/v shard with that fp32 gradient;
 *   3. bf16 round-to-nearest-even of the updated master shard;
 *   4. all-gather of the bf16 shards into every rank's param buffer.
 * AdamW (decoupled weight decay; the pages name torch.optim.AdamW but do
 * not print its rule), each operation an individually rounded fp32 op:
 *   p <- p*(1 - lr*wd);  m <- b1*m + (1-b1)*g;  v <- b2*v + (1-b2)*(g*g);
 *   p <- p - lr*((m/(1-b1^t)) / (sqrt(v/(1-b2^t)) + eps))
 * with the scalars 1-lr*wd, 1-b1, 1-b2, 1-b1^t, 1-b2^t formed in double
 * and rounded once to fp32.
 *   grads_bf16[r]   rank r's local full gradient, count bf16
 *   master/m/v[j]   owner j's fp32 shard, cr_shard_range length (in/out)
 *   params_bf16[r]  rank r's full bf16 parameter buffer, count (output)
 * No buffer may overlap another (CR_ERR_INVALID_ARG).  cfg->step >= 1.
 * Vector path: 16-byte aligned pointers and L a multiple of 8. */
typedef struct {
  double lr, beta1, beta2, eps, weight_decay;
  int64_t step;
} cr_adamw_cfg;

cr_status cr_fsdp_step(const void* const* grads_bf16, int nranks,
                       size_t count, float* const* master, float* const* m,
                       float* const* v, const cr_adamw_cfg* cfg,
                       void* const* params_bf16, cr_stream_t stream);

/* ---- range forms: one slab of the element range per GPU -------------------
 * Every output element of a reduce-scatter, all-reduce or FSDP step depends
 * only on the same element of every rank ([DT] section 2, All-Reduce: the
 * sum is element-wise across ranks; AdamW is element-wise too), so the
 * element range [0, count) may be cut into slabs processed independently,
 * e.g. one per GPU, with no exchange between them.  The range calls do the
 * work of the whole-buffer call for elements [begin, end) only, with the
 * WHOLE buffer's chunking -- L = ceil(count / N), element e in chunk e / L,
 * folded in that chunk's ring order -- so every element they write equals,
 * bit for bit, what the whole-buffer call writes there.  (Calling the
 * whole-buffer entry points on a slab would chunk the slab instead, and
 * change the fold order.)  Pointers are slab-local:
 *   in/out/bufs/grads_bf16/params_bf16[r]  rank r's element `begin`; the
 *                    buffer holds end - begin elements
 *   out_shards/master/m/v[j]  the first element of shard j that lies in
 *                    [begin, end), i.e. shard element max(begin, jL) - jL;
 *                    the part holds |[begin, end) intersected with chunk j|
 *                    elements; ignored (may be NULL) if that is empty
 * Dtypes, ops, in-place rules, alignment and errors as the whole-buffer
 * calls; begin <= end <= count (CR_ERR_INVALID_ARG otherwise).  A buffer
 * takes the vector path when its element-0 address (pointer - offset
 * * element size) is 16-byte aligned, as for the whole-buffer calls.
 * The clipped FSDP step has no range form: its global gradient norm needs
 * every slab's sum of squares (one scalar exchange between GPUs).
 * cr_slab_range: slab g of `nslabs` that partition [0, count): whole chunks
 * when nslabs <= nranks (slab g starts at chunk floor(g * N / nslabs)),
 * else 16-element boundaries (slab g starts at element 16 * floor(g *
 * ceil(count / 16) / nslabs)); bounds clamped to count.  Host only. */
cr_status cr_slab_range(size_t count, int nranks, int nslabs, int g,
                        size_t* begin, size_t* end);
cr_status cr_all_reduce_range(const void* const* in, int nranks, size_t count,
                              size_t begin, size_t end, cr_dtype in_dtype,
                              cr_op op, void* const* out, cr_dtype out_dtype,
                              cr_stream_t stream);
cr_status cr_reduce_scatter_range(const void* const* bufs, int nranks,
                                  size_t count, size_t begin, size_t end,
                                  cr_dtype in_dtype, cr_op op,
                                  void* const* out_shards, cr_dtype out_dtype,
                                  cr_stream_t stream);
cr_status cr_fsdp_step_range(const void* const* grads_bf16, int nranks,
                             size_t count, size_t begin, size_t end,
                             float* const* master, float* const* m,
                             float* const* v, const cr_adamw_cfg* cfg,
                             void* const* params_bf16, cr_stream_t stream);

/* cr_fsdp_step with global gradient-norm clipping between the
 * reduce-scatter and AdamW ("AI Infra Guide, Chapter 6", 6.8: the training
 * loop calls clip_grad_norm_(max_norm=1.0) on the sharded model before the
 * optimizer step).  norm = L2 norm of the whole averaged fp32 gradient (all
 * shards: the global norm), squares summed in fp32 batches of 8 and the
 * batches in fp64 (relative error ~1e-7); every gradient element is
 * multiplied (one fp32 multiply) by c = min(1, max_norm / (norm + 1e-6)),
 * formed in double and rounded to fp32, before AdamW.  Three launches: a
 * sum-of-squares pass over the grads that writes one fp64 partial per CTA
 * into `workspace`, one warp that adds the partials in a fixed order (the
 * norm is reproducible run to run) and stores c in the workspace's first 8
 * bytes, then the fused step, which reads c.
 * For N >= 5 on the 128-bit vector path, the first pass also parks every
 * averaged fp32 gradient in the parameter outputs: its low 16 bits at
 * element e of params_bf16[0], its high 16 bits at element e of
 * params_bf16[1] (4 bytes per element).  The update pass reads it back from
 * there, before it overwrites those elements with the bf16 parameters,
 * instead of reading the N bf16 gradients a second time.  The parked value
 * is the fold's own fp32 result, so the update does the same arithmetic on
 * the same values.  The parameters are outputs only -- their contents on
 * entry are ignored -- so nothing else may read params_bf16[0] or [1]
 * while the call runs.
 * Algorithmic bytes per parameter: (4N + 32) with the parked gradient
 * (N >= 5, vector path: 64 at N = 8), else (6N + 24) (the grads are read
 * twice; for N <= 4 this is no more than 4N + 32).
 *   max_norm        finite, > 0 (CR_ERR_INVALID_ARG otherwise)
 *   workspace       caller-owned device scratch, 8-byte aligned, of
 *                   workspace_bytes >= 16 bytes; cr_fsdp_clip_workspace_bytes()
 *                   bytes are always enough (fewer bytes cap the number of
 *                   CTAs of the first pass).  Contents on entry are ignored.
 *   norm_out        device pointer (may be NULL) receiving the norm as fp32
 * Other arguments and errors as cr_fsdp_step; no buffer may overlap another. */
size_t cr_fsdp_clip_workspace_bytes(void);
cr_status cr_fsdp_step_clipped(const void* const* grads_bf16, int nranks,
                               size_t count, float* const* master,
                               float* const* m, float* const* v,
                               const cr_adamw_cfg* cfg, double max_norm,
                               void* workspace, size_t workspace_bytes,
                               void* const* params_bf16, float* norm_out,
                               cr_stream_t stream);

/* cr_fsdp_step_clipped for callers that cannot allocate device memory.
 * The pages have no counterpart: this entry point exists for library users
 * that are handed only their tensors -- for example a plugin of a framework
 * whose own allocator owns the whole device budget, or latency-critical code
 * where a cudaMalloc would synchronise the device -- and so have no
 * workspace to pass.  It runs exactly cr_fsdp_step_clipped (same arguments
 * minus workspace/workspace_bytes, same results and errors) with the
 * workspace (coefficient and sum-of-squares partials) kept in a static
 * device array of 4096 doubles (32 KiB) that the library holds on every GPU
 * that loads it until the process exits.  The first pass uses one partial
 * per CTA and at most 4095 CTAs (the array's partial slots) whatever the
 * element count and the GPU, so no call can need more scratch than the
 * array holds and no size is refused on that account; other arguments are
 * checked and refused exactly as cr_fsdp_step_clipped does.  The first
 * call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it for that
 * device's current context, keyed on the driver's context ID; a context
 * created later on the device (after cudaDeviceReset, say) gets its own
 * lookup at its first call.  Make each such first call before any stream
 * capture.  All calls share the one array: nothing in it needs to start at
 * zero (the first pass writes every partial the second pass reads), but
 * calls that overlap on the GPU -- on different streams, unordered -- race
 * on it and must be serialised by the caller.  Nothing is allocated. */
cr_status cr_fsdp_step_clipped_noalloc(const void* const* grads_bf16,
                                       int nranks, size_t count,
                                       float* const* master, float* const* m,
                                       float* const* v,
                                       const cr_adamw_cfg* cfg,
                                       double max_norm,
                                       void* const* params_bf16,
                                       float* norm_out, cr_stream_t stream);

/* ---- FSDP2: per-parameter Shard(0) ----------------------------------------
 * [DT] section 4, FSDP2: every parameter is its own DTensor with placement
 * Shard(0): of a parameter with dim0 rows of row_numel elements, rank j
 * owns rows [j*Lr, min((j+1)*Lr, dim0)), Lr = ceil(dim0/N) -- uneven, and
 * empty for trailing ranks when dim0 < N.  The step applies cr_fsdp_step's
 * arithmetic to each parameter with that chunking (chunk length
 * Lr*row_numel elements): ring-ordered reduce-scatter of the bf16 grads in
 * fp32, / N, AdamW on owner j's fp32 shard, bf16 cast, all-gather.
 *   shapes[p]                  dim0 and row_numel of parameter p
 *   grads_bf16[p*N + r]        rank r's full gradient of p (dim0*row_numel)
 *   master/m/v[p*N + j]        owner j's fp32 shard of p (NULL if empty)
 *   params_bf16[p*N + r]       rank r's full bf16 parameter p (output)
 * One launch per 64 parameters (per 512/N when N > 8): the pointers travel
 * in the kernel's parameter block; cr_fsdp2_step_planned below makes the
 * whole model one launch.  No buffer may overlap another
 * (CR_ERR_INVALID_ARG).  A parameter whose shard length is
 * a multiple of 8 and whose buffers are 16-byte aligned takes the vector
 * path; any other takes the element-wise one, with identical results. */
typedef struct {
  size_t dim0;
  size_t row_numel;
} cr_param_shape;

cr_status cr_fsdp2_step(const cr_param_shape* shapes, int nparams, int nranks,
                        const void* const* grads_bf16, float* const* master,
                        float* const* m, float* const* v,
                        const cr_adamw_cfg* cfg, void* const* params_bf16,
                        cr_stream_t stream);

/* FSDP2 step in one launch, for a parameter set that stays fixed across
 * steps ([DT] section 4, FSDP2: the sharded parameters and their optimizer
 * state are created once and stepped every iteration).  Same arithmetic and
 * results, bit for bit, as cr_fsdp2_step.
 * cr_fsdp2_plan_create checks every buffer exactly as cr_fsdp2_step does
 * (same arguments, same errors) and builds, on the host, the table the
 * kernel reads: the tile prefix sums, a 48-byte descriptor per non-empty
 * parameter and its 5N device pointers.  On success *plan receives a host
 * object that the caller releases with cr_fsdp2_plan_free; it holds the
 * buffers' addresses, so those buffers must stay allocated, and unmoved,
 * while the plan's table is used.
 * cr_fsdp2_plan_table_bytes: the table's size (0 for a NULL plan).
 * cr_fsdp2_plan_upload copies the table, with one cudaMemcpyAsync on
 * `stream`, into a caller-owned device buffer `table` of table_bytes >=
 * cr_fsdp2_plan_table_bytes(plan), 16-byte aligned (CR_ERR_ALIGNMENT).  The
 * copy is from pageable host memory: the call returns once the bytes are
 * staged, so the plan may be freed right after it.  Upload once per
 * parameter set, not per step, and outside any stream capture: a captured
 * copy would read the plan's host memory again at every replay.
 * cr_fsdp2_step_planned launches the step for the plan's parameters, with
 * the table read from `table` (which must hold this plan's uploaded bytes,
 * unchanged, until the launch completes) and the AdamW configuration given
 * here (the step count may change every call).  One launch, any number of
 * parameters.  The library checks the plan, the table's alignment and cfg;
 * the buffers were checked when the plan was made. */
typedef struct cr_fsdp2_plan cr_fsdp2_plan_t;

cr_status cr_fsdp2_plan_create(const cr_param_shape* shapes, int nparams,
                               int nranks, const void* const* grads_bf16,
                               float* const* master, float* const* m,
                               float* const* v, void* const* params_bf16,
                               cr_fsdp2_plan_t** plan);
size_t cr_fsdp2_plan_table_bytes(const cr_fsdp2_plan_t* plan);
cr_status cr_fsdp2_plan_upload(const cr_fsdp2_plan_t* plan, void* table,
                               size_t table_bytes, cr_stream_t stream);
cr_status cr_fsdp2_step_planned(const cr_fsdp2_plan_t* plan,
                                const void* table, const cr_adamw_cfg* cfg,
                                cr_stream_t stream);
void cr_fsdp2_plan_free(cr_fsdp2_plan_t* plan);

/* ---- DDP gradient accumulation (no_sync) ----------------------------------
 * "AI Infra Guide, Chapter 6", 6.2.6: micro-steps inside model.no_sync()
 * only accumulate their gradient locally; the last one accumulates and then
 * all-reduces the sum.
 * cr_accumulate: acc[r][e] += grads[r][e] for every rank (fp32 addition;
 * grads CR_F32 or CR_BF16), no communication.
 * cr_all_reduce_accumulate: the same addition and, in the same pass, the
 * all-reduce (CR_SUM or CR_AVG) of the N sums in ring order, written back
 * into every acc[r] -- equal, bit for bit, to cr_accumulate followed by
 * cr_all_reduce(acc, ..., CR_F32, op, acc, CR_F32), without the
 * intermediate write and read of the accumulators.
 *   acc[r]    rank r's fp32 accumulator, count elements (in/out)
 *   grads[r]  rank r's new micro-step gradient, count elements
 * Buffers must not overlap (CR_ERR_INVALID_ARG). */
cr_status cr_accumulate(float* const* acc, int nranks, size_t count,
                        const void* const* grads, cr_dtype grad_dtype,
                        cr_stream_t stream);
cr_status cr_all_reduce_accumulate(float* const* acc, int nranks, size_t count,
                                   const void* const* grads,
                                   cr_dtype grad_dtype, cr_op op,
                                   cr_stream_t stream);

/* AdamW alone: as above, on n fp32 elements with an fp32 gradient
 * (for example a shard produced by cr_reduce_scatter with out_dtype F32);
 * param_bf16 (may be NULL) receives the bf16 cast of the updated master.
 * No overlaps allowed. */
cr_status cr_adamw_step(size_t n, float* master, float* m, float* v,
                        const float* grad, const cr_adamw_cfg* cfg,
                        void* param_bf16, cr_stream_t stream);

/* ---- device-side checks (test builds) -------------------------------------
 * The library can be built as a checked variant whose kernels verify, before
 * touching memory, the index arithmetic their accesses rest on (the chunk of
 * an element is a rank, its offset lies inside that rank's shard, a tile
 * belongs to its tensor...).  A failed check sets one bit of a device error
 * word and skips the rest of that thread's work; nothing traps.
 * cr_check_word: the word (0 = no check has failed), cleared afterwards if
 * clear != 0; -1 in the normal build, which has no checks; -2 if reading it
 * failed.  Synchronises with the device.
 * cr_check_selftest: sets bit 31 through the failing-check path (checked
 * build); CR_ERR_UNSUPPORTED in the normal build. */
long long cr_check_word(int clear);
cr_status cr_check_selftest(cr_stream_t stream);

/* ---- communication accounting (host) --------------------------------------
 * Elements rank `rank` sends and receives, and the logical steps taken, in
 * the ring schedule of [DT] section 2 (reduce-scatter N-1 steps, all-gather
 * N-1 steps, all-reduce both) or in the naive schedule of [NX] 2.2
 * (reduce to rank 0, then broadcast from it; all-reduce only).  Multiply by
 * the element size for bytes: with N | count, ring all-reduce gives
 * 2(N-1)/N * count per rank and naive gives 2(N-1) * count at the root.
 * CR_ERR_UNSUPPORTED for a naive reduce-scatter or all-gather. */
typedef enum {
  CR_COLL_REDUCE_SCATTER = 0,
  CR_COLL_ALL_GATHER = 1,
  CR_COLL_ALL_REDUCE = 2
} cr_collective;
typedef enum { CR_SCHED_RING = 0, CR_SCHED_NAIVE = 1 } cr_schedule;

cr_status cr_comm_elems(cr_collective coll, cr_schedule sched, int nranks,
                        size_t count, int rank, uint64_t* sent,
                        uint64_t* recv, int* steps);

#ifdef __cplusplus
}
#endif
#endif /* CR_H */
