/*
 * adamw_fsdp.cpp -- oracle for the sharded AdamW update and the FSDP step
 * (reduce-scatter -> owner AdamW -> bf16 cast -> all-gather).  Test
 * infrastructure only (see oracle.h).
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* Scalar AdamW with decoupled weight decay; see oracle.h for the rule and
 * the reading of the pages it follows.  One element at a time, every
 * operation an individually rounded fp32 operation. */
void orc_adamw(size_t n, float* p, float* m, float* v, const float* g,
               const orc_adamw_cfg* c) {
  const float lr = (float)c->lr;
  const float eps = (float)c->eps;
  const float b1 = (float)c->beta1;
  const float b2 = (float)c->beta2;
  const float one_minus_b1 = (float)(1.0 - c->beta1);
  const float one_minus_b2 = (float)(1.0 - c->beta2);
  const float decay = (float)(1.0 - c->lr * c->weight_decay);
  const float bc1 = (float)(1.0 - pow(c->beta1, (double)c->step));
  const float bc2 = (float)(1.0 - pow(c->beta2, (double)c->step));
  for (size_t i = 0; i < n; ++i) {
    float gi = g[i];
    float pi = p[i] * decay;
    float mi = b1 * m[i] + one_minus_b1 * gi;
    float vi = b2 * v[i] + one_minus_b2 * (gi * gi);
    float mh = mi / bc1;
    float vh = vi / bc2;
    float denom = sqrtf(vh) + eps;
    pi = pi - lr * (mh / denom);
    p[i] = pi;
    m[i] = mi;
    v[i] = vi;
  }
}

/* FSDP step in the order the pages give for one flat unit:
 * backward post-hook reduce-scatter (fp32 reduce dtype, averaged), the
 * optimizer step on the local shard only, then the all-gather that rebuilds
 * the full bf16 parameter buffer on every rank ([DT] section 4, FSDP1
 * "unit1 lifecycle"; [AIG] 6.3.2 and 6.3.4). */
int orc_fsdp_step(int n, size_t count, const uint16_t* const* grads,
                  float* const* master, float* const* m, float* const* v,
                  const orc_adamw_cfg* cfg, uint16_t* const* params) {
  if (n < 1 || n > ORC_MAX_RANKS) return ORC_EINVAL;
  size_t L = orc_chunk_len(count, n);
  float* gshard[ORC_MAX_RANKS];
  uint16_t* pshard[ORC_MAX_RANKS];
  for (int r = 0; r < n; ++r) {
    gshard[r] = (float*)malloc((L ? L : 1) * sizeof(float));
    pshard[r] = (uint16_t*)malloc((L ? L : 1) * sizeof(uint16_t));
    if (!gshard[r] || !pshard[r]) {
      for (int q = 0; q <= r; ++q) { free(gshard[q]); free(pshard[q]); }
      return ORC_ENOMEM;
    }
  }
  /* 1. reduce-scatter: bf16 grads in, fp32 averaged shard out. */
  int rc = orc_ring_reduce_scatter(n, count, ORC_BF16, ORC_AVG,
                                   (const void* const*)grads,
                                   (void* const*)gshard, ORC_F32, NULL, NULL,
                                   NULL);
  if (rc == ORC_OK) {
    /* 2./3. each owner j updates its own shard and casts it to bf16. */
    for (int j = 0; j < n; ++j) {
      size_t lo, hi;
      orc_chunk_bounds(count, n, j, &lo, &hi);
      orc_adamw(hi - lo, master[j], m[j], v[j], gshard[j], cfg);
      for (size_t k = 0; k < hi - lo; ++k)
        pshard[j][k] = orc_f32_to_bf16(master[j][k]);
    }
    /* 4. all-gather of the bf16 parameter shards. */
    rc = orc_ring_all_gather(n, count, ORC_BF16, (const void* const*)pshard,
                             (void* const*)params, NULL, NULL);
  }
  for (int r = 0; r < n; ++r) { free(gshard[r]); free(pshard[r]); }
  return rc;
}

/* FSDP step with clip_grad_norm_ between the reduce-scatter and AdamW; see
 * oracle.h.  The norm is the global one: every owner's squared shard norm
 * summed over all shards. */
int orc_fsdp_step_clipped(int n, size_t count, const uint16_t* const* grads,
                          float* const* master, float* const* m,
                          float* const* v, const orc_adamw_cfg* cfg,
                          double max_norm, uint16_t* const* params,
                          double* norm_out) {
  if (n < 1 || n > ORC_MAX_RANKS) return ORC_EINVAL;
  size_t L = orc_chunk_len(count, n);
  float* gshard[ORC_MAX_RANKS];
  uint16_t* pshard[ORC_MAX_RANKS];
  for (int r = 0; r < n; ++r) {
    gshard[r] = (float*)malloc((L ? L : 1) * sizeof(float));
    pshard[r] = (uint16_t*)malloc((L ? L : 1) * sizeof(uint16_t));
    if (!gshard[r] || !pshard[r]) {
      for (int q = 0; q <= r; ++q) { free(gshard[q]); free(pshard[q]); }
      return ORC_ENOMEM;
    }
  }
  int rc = orc_ring_reduce_scatter(n, count, ORC_BF16, ORC_AVG,
                                   (const void* const*)grads,
                                   (void* const*)gshard, ORC_F32, NULL, NULL,
                                   NULL);
  if (rc == ORC_OK) {
    /* Global norm: each owner's sum of squares, then the sum over owners. */
    double total = 0.0;
    for (int j = 0; j < n; ++j) {
      size_t lo, hi;
      orc_chunk_bounds(count, n, j, &lo, &hi);
      double local = 0.0;
      for (size_t k = 0; k < hi - lo; ++k)
        local += (double)gshard[j][k] * (double)gshard[j][k];
      total += local;
    }
    double norm = sqrt(total);
    double coef = max_norm / (norm + 1e-6);
    if (coef > 1.0) coef = 1.0;
    float c = (float)coef;
    if (norm_out) *norm_out = norm;
    for (int j = 0; j < n; ++j) {
      size_t lo, hi;
      orc_chunk_bounds(count, n, j, &lo, &hi);
      for (size_t k = 0; k < hi - lo; ++k) gshard[j][k] = gshard[j][k] * c;
      orc_adamw(hi - lo, master[j], m[j], v[j], gshard[j], cfg);
      for (size_t k = 0; k < hi - lo; ++k)
        pshard[j][k] = orc_f32_to_bf16(master[j][k]);
    }
    rc = orc_ring_all_gather(n, count, ORC_BF16, (const void* const*)pshard,
                             (void* const*)params, NULL, NULL);
  }
  for (int r = 0; r < n; ++r) { free(gshard[r]); free(pshard[r]); }
  return rc;
}

/* FSDP2 step, parameter by parameter; see oracle.h. */
int orc_fsdp2_step(int nparams, const orc_param_shape* shapes, int n,
                   const uint16_t* const* grads, float* const* master,
                   float* const* m, float* const* v, const orc_adamw_cfg* cfg,
                   uint16_t* const* params) {
  if (n < 1 || n > ORC_MAX_RANKS || nparams < 0) return ORC_EINVAL;
  for (int p = 0; p < nparams; ++p) {
    const size_t count = shapes[p].dim0 * shapes[p].row_numel;
    const size_t Lr = (shapes[p].dim0 + (size_t)n - 1) / (size_t)n;
    const size_t L = Lr * shapes[p].row_numel;
    float* gshard[ORC_MAX_RANKS];
    uint16_t* pshard[ORC_MAX_RANKS];
    for (int r = 0; r < n; ++r) {
      gshard[r] = (float*)malloc((L ? L : 1) * sizeof(float));
      pshard[r] = (uint16_t*)malloc((L ? L : 1) * sizeof(uint16_t));
      if (!gshard[r] || !pshard[r]) {
        for (int q = 0; q <= r; ++q) { free(gshard[q]); free(pshard[q]); }
        return ORC_ENOMEM;
      }
    }
    int rc = orc_ring_reduce_scatter_L(n, count, L, ORC_BF16, ORC_AVG,
                                       (const void* const*)(grads + (size_t)p * n),
                                       (void* const*)gshard, ORC_F32, NULL, NULL,
                                       NULL);
    if (rc == ORC_OK) {
      for (int j = 0; j < n; ++j) {
        size_t lo = L * (size_t)j, hi = lo + L;
        if (lo > count) lo = count;
        if (hi > count) hi = count;
        const size_t k = (size_t)p * n + j;
        orc_adamw(hi - lo, master[k], m[k], v[k], gshard[j], cfg);
        for (size_t i = 0; i < hi - lo; ++i)
          pshard[j][i] = orc_f32_to_bf16(master[k][i]);
      }
      rc = orc_ring_all_gather_L(n, count, L, ORC_BF16,
                                 (const void* const*)pshard,
                                 (void* const*)(params + (size_t)p * n), NULL,
                                 NULL);
    }
    for (int r = 0; r < n; ++r) { free(gshard[r]); free(pshard[r]); }
    if (rc != ORC_OK) return rc;
  }
  return ORC_OK;
}
