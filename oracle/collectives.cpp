/*
 * collectives.cpp -- oracle for chunking, ring reduce-scatter / all-gather /
 * all-reduce and naive reduce+broadcast.  Test infrastructure only (see
 * oracle.h).  Written for obviousness, not speed: every rank's buffers and
 * every ring message are materialised.
 */
#include "oracle.h"

#include <stdlib.h>
#include <string.h>

/* ---- chunking ([DT] section 4 FSDP2 uneven Shard(0); [NX] 2.2) --------- */

size_t orc_chunk_len(size_t count, int n) {
  return (count + (size_t)n - 1) / (size_t)n;
}

void orc_chunk_bounds(size_t count, int n, int j, size_t* lo, size_t* hi) {
  size_t L = orc_chunk_len(count, n);
  size_t a = L * (size_t)j;
  size_t b = a + L;
  if (a > count) a = count;
  if (b > count) b = count;
  *lo = a;
  *hi = b;
}

/* Chunk j of a buffer of count elements cut into chunks of L elements (the
 * last ones short or empty).  Used with L = ceil(count/N) for flat buffers
 * and with L = ceil(dim0/N) * row for FSDP2's dim-0 shards. */
static void bounds_L(size_t count, size_t L, int j, size_t* lo, size_t* hi) {
  size_t a = L * (size_t)j;
  size_t b = a + L;
  if (a > count) a = count;
  if (b > count) b = count;
  *lo = a;
  *hi = b;
}

/* ---- bf16 ------------------------------------------------------------- */

uint16_t orc_f32_to_bf16(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0) {
    /* NaN: keep the sign and top payload bits, force the quiet bit. */
    return (uint16_t)((u >> 16) | 0x0040u);
  }
  /* Round to nearest, ties to even, on the 16 discarded bits. */
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

float orc_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

void orc_f32_to_bf16_array(size_t n, const float* x, uint16_t* out) {
  for (size_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(x[i]);
}

size_t orc_esize(int dtype) {
  switch (dtype) {
    case ORC_F32: return 4;
    case ORC_BF16: return 2;
    case ORC_I32: return 4;
    default: return 0;
  }
}

/* ---- element access helpers -------------------------------------------
 * An accumulator is either an fp32 value (F32/BF16 inputs) or an int32
 * value kept as uint32 so that overflow wraps without undefined behaviour. */

typedef struct {
  float f;
  uint32_t i;
} acc_t;

static int is_int(int dt) { return dt == ORC_I32; }

static acc_t load_acc(const void* buf, int dt, size_t e) {
  acc_t a = {0.0f, 0u};
  if (dt == ORC_F32) {
    a.f = ((const float*)buf)[e];
  } else if (dt == ORC_BF16) {
    a.f = orc_bf16_to_f32(((const uint16_t*)buf)[e]);
  } else {
    a.i = (uint32_t)((const int32_t*)buf)[e];
  }
  return a;
}

static acc_t add_acc(acc_t a, acc_t b, int dt) {
  acc_t r = {0.0f, 0u};
  if (is_int(dt)) r.i = a.i + b.i;
  else r.f = a.f + b.f;
  return r;
}

/* AVG divides the finished fp32 sum by N once ([DT] section 2 All-Reduce,
 * G = sum_i G_i / N; FSDP divides by world_size after the reduce). */
static acc_t finish_acc(acc_t a, int dt, int op, int n) {
  if (!is_int(dt) && op == ORC_AVG) a.f = a.f / (float)n;
  return a;
}

static void store_acc(void* buf, int dt, size_t e, acc_t a) {
  if (dt == ORC_F32) {
    ((float*)buf)[e] = a.f;
  } else if (dt == ORC_BF16) {
    ((uint16_t*)buf)[e] = orc_f32_to_bf16(a.f);
  } else {
    ((int32_t*)buf)[e] = (int32_t)a.i;
  }
}

static double acc_as_double(acc_t a, int dt) {
  return is_int(dt) ? (double)(int32_t)a.i : (double)a.f;
}

/* Legal dtype pairs: float inputs reduce to float outputs, int32 to int32;
 * AVG is defined for float types only. */
static int check_types(int n, int in_dt, int op, int out_dt) {
  if (n < 1 || n > ORC_MAX_RANKS) return ORC_EINVAL;
  if (orc_esize(in_dt) == 0 || orc_esize(out_dt) == 0) return ORC_EINVAL;
  if (op != ORC_SUM && op != ORC_AVG) return ORC_EINVAL;
  if (is_int(in_dt) != is_int(out_dt)) return ORC_EUNSUPPORTED;
  if (is_int(in_dt) && op == ORC_AVG) return ORC_EUNSUPPORTED;
  return ORC_OK;
}

/* ---- ring reduce-scatter: literal simulation ---------------------------
 * [DT] section 2, Reduce-Scatter: ring rank0 -> rank1 -> ... -> rank0; each
 * chunk starts at the rank after its owner and its last hop lands on the
 * owner; step s, rank r sends chunk (r - s) mod N. */

typedef struct {
  int chunk;     /* chunk id this partial belongs to   */
  size_t lo, hi; /* element range of that chunk        */
  acc_t* data;   /* hi - lo accumulators               */
} partial_t;

/* The ring reduce-scatter simulation; wire_dt ORC_BF16 rounds every message
 * (the partial a rank sends) to bf16 before it leaves the sender. */
static int ring_rs_sim(int n, size_t count, size_t L, int in_dt, int op,
                       int wire_dt, const void* const* bufs,
                       void* const* out_shards, int out_dt, orc_traffic* tr,
                       int* trace_chunk, double* trace_value) {
  int rc = check_types(n, in_dt, op, out_dt);
  if (rc) return rc;
  if (L * (size_t)n < count) return ORC_EINVAL;
  if (wire_dt != ORC_F32 && !(wire_dt == ORC_BF16 && !is_int(in_dt))) return ORC_EUNSUPPORTED;
  if (tr) memset(tr, 0, sizeof(*tr));

  /* hold[r]: the partial rank r holds and will send next.
   * inbox[r]: the message rank r receives in the current step. */
  partial_t hold[ORC_MAX_RANKS], inbox[ORC_MAX_RANKS];
  for (int r = 0; r < n; ++r) {
    hold[r].data = (acc_t*)calloc(L ? L : 1, sizeof(acc_t));
    inbox[r].data = (acc_t*)calloc(L ? L : 1, sizeof(acc_t));
    if (!hold[r].data || !inbox[r].data) {
      for (int q = 0; q <= r; ++q) { free(hold[q].data); free(inbox[q].data); }
      return ORC_ENOMEM;
    }
  }

  /* Before step 1 each rank's outgoing partial is its own, unreduced
   * contribution to chunk (r - 1) mod N. */
  for (int r = 0; r < n; ++r) {
    int c = (r - 1 + n) % n;
    hold[r].chunk = c;
    bounds_L(count, L, c, &hold[r].lo, &hold[r].hi);
    for (size_t e = hold[r].lo; e < hold[r].hi; ++e)
      hold[r].data[e - hold[r].lo] = load_acc(bufs[r], in_dt, e);
  }

  for (int s = 1; s <= n - 1; ++s) {
    /* All ranks send at once: rank r's message lands in rank r+1's inbox. */
    for (int r = 0; r < n; ++r) {
      int d = (r + 1) % n;
      size_t len = hold[r].hi - hold[r].lo;
      inbox[d].chunk = hold[r].chunk;
      inbox[d].lo = hold[r].lo;
      inbox[d].hi = hold[r].hi;
      memcpy(inbox[d].data, hold[r].data, len * sizeof(acc_t));
      if (wire_dt == ORC_BF16)  /* the message travels as bf16 */
        for (size_t k = 0; k < len; ++k)
          inbox[d].data[k].f = orc_bf16_to_f32(orc_f32_to_bf16(inbox[d].data[k].f));
      if (tr) { tr->sent[r] += len; tr->recv[d] += len; }
      if (trace_chunk) trace_chunk[(s - 1) * n + r] = hold[r].chunk;
    }
    /* Each receiver adds its own contribution: partial + local. */
    for (int d = 0; d < n; ++d) {
      for (size_t e = inbox[d].lo; e < inbox[d].hi; ++e) {
        acc_t* p = &inbox[d].data[e - inbox[d].lo];
        *p = add_acc(*p, load_acc(bufs[d], in_dt, e), in_dt);
      }
      if (trace_value) {
        trace_value[(s - 1) * n + d] =
            inbox[d].hi > inbox[d].lo ? acc_as_double(inbox[d].data[0], in_dt)
                                      : 0.0;
      }
    }
    /* What a rank just accumulated is what it sends next. */
    for (int d = 0; d < n; ++d) {
      partial_t t = hold[d];
      hold[d] = inbox[d];
      inbox[d] = t;
    }
    if (tr) tr->steps += 1;
  }

  /* After N-1 steps rank r holds chunk r completely reduced. */
  for (int r = 0; r < n; ++r) {
    if (hold[r].chunk != r) {
      rc = ORC_EINVAL; /* cannot happen for a correct schedule */
    }
    for (size_t e = hold[r].lo; e < hold[r].hi; ++e) {
      acc_t a = finish_acc(hold[r].data[e - hold[r].lo], in_dt, op, n);
      store_acc(out_shards[r], out_dt, e - hold[r].lo, a);
    }
  }
  for (int r = 0; r < n; ++r) { free(hold[r].data); free(inbox[r].data); }
  return rc;
}

int orc_ring_reduce_scatter_L(int n, size_t count, size_t L, int in_dt, int op,
                              const void* const* bufs, void* const* out_shards,
                              int out_dt, orc_traffic* tr, int* trace_chunk,
                              double* trace_value) {
  return ring_rs_sim(n, count, L, in_dt, op, ORC_F32, bufs, out_shards, out_dt,
                     tr, trace_chunk, trace_value);
}

int orc_ring_reduce_scatter(int n, size_t count, int in_dt, int op,
                            const void* const* bufs, void* const* out_shards,
                            int out_dt, orc_traffic* tr, int* trace_chunk,
                            double* trace_value) {
  if (n < 1 || n > ORC_MAX_RANKS) return ORC_EINVAL;
  return orc_ring_reduce_scatter_L(n, count, orc_chunk_len(count, n), in_dt, op,
                                   bufs, out_shards, out_dt, tr, trace_chunk,
                                   trace_value);
}

int orc_ring_reduce_scatter_wire(int n, size_t count, int in_dt, int op,
                                 int wire_dt, const void* const* bufs,
                                 void* const* out_shards, int out_dt) {
  if (n < 1 || n > ORC_MAX_RANKS) return ORC_EINVAL;
  return ring_rs_sim(n, count, orc_chunk_len(count, n), in_dt, op, wire_dt, bufs,
                     out_shards, out_dt, NULL, NULL, NULL);
}

int orc_ring_all_reduce_wire(int n, size_t count, int in_dt, int op,
                             int wire_dt, const void* const* in,
                             void* const* out, int out_dt) {
  int rc = check_types(n, in_dt, op, out_dt);
  if (rc) return rc;
  size_t L = orc_chunk_len(count, n);
  size_t es = orc_esize(out_dt);
  void* shards[ORC_MAX_RANKS];
  for (int r = 0; r < n; ++r) {
    shards[r] = malloc((L ? L : 1) * es);
    if (!shards[r]) {
      for (int q = 0; q < r; ++q) free(shards[q]);
      return ORC_ENOMEM;
    }
  }
  rc = orc_ring_reduce_scatter_wire(n, count, in_dt, op, wire_dt, in, shards, out_dt);
  if (rc == ORC_OK)
    rc = orc_ring_all_gather(n, count, out_dt, (const void* const*)shards, out, NULL,
                             NULL);
  for (int r = 0; r < n; ++r) free(shards[r]);
  return rc;
}

/* HSDP: ring reduce-scatter inside each of the R groups of S ranks, then a
 * ring all-reduce of each shard across the R groups, then AVG / cast. */
int orc_hsdp_reduce_scatter(int R, int S, size_t count, int in_dt, int op,
                            const void* const* bufs, void* const* out_shards,
                            int out_dt) {
  if (R < 1 || S < 1 || R * S > ORC_MAX_RANKS) return ORC_EINVAL;
  int rc = check_types(R * S, in_dt, op, out_dt);
  if (rc) return rc;
  const int acc_dt = is_int(in_dt) ? ORC_I32 : ORC_F32;
  const size_t L = orc_chunk_len(count, S);
  /* part[g][j]: group g's sum of shard j over its S ranks (fp32 / int32) */
  void* part[ORC_MAX_RANKS][ORC_MAX_RANKS];
  void* red[ORC_MAX_RANKS];
  int ok = 1;
  for (int g = 0; g < R; ++g)
    for (int j = 0; j < S; ++j) ok = ok && (part[g][j] = malloc((L ? L : 1) * 4)) != NULL;
  for (int g = 0; g < R; ++g) ok = ok && (red[g] = malloc((L ? L : 1) * 4)) != NULL;
  if (!ok) return ORC_ENOMEM;  /* (test sizes only; nothing to free in practice) */
  for (int g = 0; g < R && rc == ORC_OK; ++g)
    rc = orc_ring_reduce_scatter(S, count, in_dt, ORC_SUM, bufs + (size_t)g * S,
                                 part[g], acc_dt, NULL, NULL, NULL);
  for (int j = 0; j < S && rc == ORC_OK; ++j) {
    size_t lo, hi;
    orc_chunk_bounds(count, S, j, &lo, &hi);
    const void* col[ORC_MAX_RANKS];
    for (int g = 0; g < R; ++g) col[g] = part[g][j];
    rc = orc_ring_all_reduce(R, hi - lo, acc_dt, ORC_SUM, col, red, acc_dt, NULL);
    for (int g = 0; g < R && rc == ORC_OK; ++g)
      for (size_t k = 0; k < hi - lo; ++k) {
        acc_t a = load_acc(red[g], acc_dt, k);
        store_acc(out_shards[(size_t)g * S + j], out_dt, k, finish_acc(a, in_dt, op, R * S));
      }
  }
  for (int g = 0; g < R; ++g) {
    for (int j = 0; j < S; ++j) free(part[g][j]);
    free(red[g]);
  }
  return rc;
}

/* ---- closed-form fold --------------------------------------------------- */

int orc_fold_reduce_scatter(int n, size_t count, int in_dt, int op,
                            const void* const* bufs, void* const* out_shards,
                            int out_dt) {
  int rc = check_types(n, in_dt, op, out_dt);
  if (rc) return rc;
  for (int j = 0; j < n; ++j) {
    size_t lo, hi;
    orc_chunk_bounds(count, n, j, &lo, &hi);
    for (size_t e = lo; e < hi; ++e) {
      acc_t a = load_acc(bufs[(j + 1) % n], in_dt, e);
      for (int k = 2; k <= n; ++k)
        a = add_acc(a, load_acc(bufs[(j + k) % n], in_dt, e), in_dt);
      store_acc(out_shards[j], out_dt, e - lo, finish_acc(a, in_dt, op, n));
    }
  }
  return ORC_OK;
}

int orc_fold_columns(int n, size_t nsamp, int in_dt, int op, const void* vals,
                     const int* chunk, void* out, int out_dt) {
  int rc = check_types(n, in_dt, op, out_dt);
  if (rc) return rc;
  for (size_t i = 0; i < nsamp; ++i) {
    int j = chunk[i];
    if (j < 0 || j >= n) return ORC_EINVAL;
    size_t base = i * (size_t)n;
    acc_t a = load_acc(vals, in_dt, base + (size_t)((j + 1) % n));
    for (int k = 2; k <= n; ++k)
      a = add_acc(a, load_acc(vals, in_dt, base + (size_t)((j + k) % n)),
                  in_dt);
    store_acc(out, out_dt, i, finish_acc(a, in_dt, op, n));
  }
  return ORC_OK;
}

/* ---- ring all-gather: literal simulation --------------------------------
 * [DT] section 2 All-Gather and the second phase of All-Reduce: each step
 * every rank forwards one D/N shard to its right neighbour; after N-1 steps
 * each rank rearranges what it holds by shard index. */

int orc_ring_all_gather_L(int n, size_t count, size_t L, int dt,
                          const void* const* shards, void* const* bufs,
                          orc_traffic* tr, int* trace_arrival) {
  if (n < 1 || n > ORC_MAX_RANKS || orc_esize(dt) == 0) return ORC_EINVAL;
  if (L * (size_t)n < count) return ORC_EINVAL;
  if (tr) memset(tr, 0, sizeof(*tr));
  size_t es = orc_esize(dt);

  /* held[r][k]: the k-th shard rank r came to hold (k = 0 is its own),
   * with its id in held_id[r][k]. */
  unsigned char* held[ORC_MAX_RANKS];
  int held_id[ORC_MAX_RANKS][ORC_MAX_RANKS];
  for (int r = 0; r < n; ++r) {
    held[r] = (unsigned char*)malloc((size_t)n * (L ? L : 1) * es);
    if (!held[r]) {
      for (int q = 0; q < r; ++q) free(held[q]);
      return ORC_ENOMEM;
    }
    size_t lo, hi;
    bounds_L(count, L, r, &lo, &hi);
    memcpy(held[r], shards[r], (hi - lo) * es);
    held_id[r][0] = r;
  }

  for (int s = 1; s <= n - 1; ++s) {
    /* Rank r forwards the shard it got at step s-1 (slot s-1); all sends of
     * a step happen at once, so read every sender's slot before writing. */
    for (int r = 0; r < n; ++r) {
      int d = (r + 1) % n;
      int id = held_id[r][s - 1];
      size_t lo, hi;
      bounds_L(count, L, id, &lo, &hi);
      memcpy(held[d] + (size_t)s * L * es, held[r] + (size_t)(s - 1) * L * es,
             (hi - lo) * es);
      held_id[d][s] = id;
      if (tr) { tr->sent[r] += hi - lo; tr->recv[d] += hi - lo; }
      if (trace_arrival) trace_arrival[(s - 1) * n + d] = id;
    }
    if (tr) tr->steps += 1;
  }

  /* Rearrange by shard index into the full buffer. */
  for (int r = 0; r < n; ++r) {
    for (int k = 0; k < n; ++k) {
      int id = held_id[r][k];
      size_t lo, hi;
      bounds_L(count, L, id, &lo, &hi);
      memcpy((unsigned char*)bufs[r] + lo * es, held[r] + (size_t)k * L * es,
             (hi - lo) * es);
    }
    free(held[r]);
  }
  return ORC_OK;
}

int orc_ring_all_gather(int n, size_t count, int dt, const void* const* shards,
                        void* const* bufs, orc_traffic* tr,
                        int* trace_arrival) {
  if (n < 1 || n > ORC_MAX_RANKS) return ORC_EINVAL;
  return orc_ring_all_gather_L(n, count, orc_chunk_len(count, n), dt, shards,
                               bufs, tr, trace_arrival);
}

/* ---- ring all-reduce = reduce-scatter + all-gather ([DT] section 2) ---- */

int orc_ring_all_reduce(int n, size_t count, int in_dt, int op,
                        const void* const* in, void* const* out, int out_dt,
                        orc_traffic* tr) {
  int rc = check_types(n, in_dt, op, out_dt);
  if (rc) return rc;
  size_t L = orc_chunk_len(count, n);
  size_t es = orc_esize(out_dt);
  void* shards[ORC_MAX_RANKS];
  for (int r = 0; r < n; ++r) {
    shards[r] = malloc((L ? L : 1) * es);
    if (!shards[r]) {
      for (int q = 0; q < r; ++q) free(shards[q]);
      return ORC_ENOMEM;
    }
  }
  orc_traffic t1, t2;
  rc = orc_ring_reduce_scatter(n, count, in_dt, op, in, shards, out_dt, &t1,
                               NULL, NULL);
  if (rc == ORC_OK)
    rc = orc_ring_all_gather(n, count, out_dt, (const void* const*)shards, out,
                             &t2, NULL);
  if (rc == ORC_OK && tr) {
    memset(tr, 0, sizeof(*tr));
    for (int r = 0; r < n; ++r) {
      tr->sent[r] = t1.sent[r] + t2.sent[r];
      tr->recv[r] = t1.recv[r] + t2.recv[r];
    }
    tr->steps = t1.steps + t2.steps;
  }
  for (int r = 0; r < n; ++r) free(shards[r]);
  return rc;
}

/* ---- naive reduce-to-root + broadcast ([NX] 2.2) ----------------------- */

int orc_naive_all_reduce(int n, size_t count, int in_dt, int op,
                         const void* const* in, void* const* out, int out_dt,
                         orc_traffic* tr) {
  int rc = check_types(n, in_dt, op, out_dt);
  if (rc) return rc;
  if (tr) memset(tr, 0, sizeof(*tr));
  acc_t* root = (acc_t*)calloc(count ? count : 1, sizeof(acc_t));
  if (!root) return ORC_ENOMEM;
  /* Reduce: the root starts from its own buffer and adds each other rank's
   * full buffer as it arrives, in rank order. */
  for (size_t e = 0; e < count; ++e) root[e] = load_acc(in[0], in_dt, e);
  for (int r = 1; r < n; ++r) {
    for (size_t e = 0; e < count; ++e)
      root[e] = add_acc(root[e], load_acc(in[r], in_dt, e), in_dt);
    if (tr) { tr->sent[r] += count; tr->recv[0] += count; tr->steps += 1; }
  }
  /* Broadcast: the root sends the full result to every other rank. */
  for (int r = 0; r < n; ++r) {
    for (size_t e = 0; e < count; ++e)
      store_acc(out[r], out_dt, e, finish_acc(root[e], in_dt, op, n));
    if (r != 0 && tr) { tr->sent[0] += count; tr->recv[r] += count; tr->steps += 1; }
  }
  free(root);
  return ORC_OK;
}

/* ---- gradient accumulation ([AIG] 6.2.6, no_sync) ------------------------ */

void orc_accumulate(size_t count, float* acc, const void* g, int g_dtype) {
  for (size_t e = 0; e < count; ++e) acc[e] = acc[e] + load_acc(g, g_dtype, e).f;
}

/* ---- alpha-beta model --------------------------------------------------- */

double orc_alpha_beta_ring_allreduce(int n, double bytes, double alpha_s,
                                     double bw_bytes_per_s) {
  double steps = 2.0 * (double)(n - 1);
  return steps * alpha_s + steps / (double)n * bytes / bw_bytes_per_s;
}
