// plan.cpp -- host-only parts of libcr: the DDP bucket planner and the
// communication accounting of the ring and naive schedules.
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "cr.h"

extern "C" {

// Greedy bucket assignment in backward order ("AI Infra Guide, Chapter 6",
// 6.2.4: buckets of ~25 MB filled in the order gradients become ready,
// i.e. reverse registration order; nxmr.cn news 160867, 5.1).
cr_status cr_bucket_plan(const size_t* numels, int ntensors, size_t elem_size,
                         size_t cap_bytes, cr_bucket_plan_t** out) {
  if (!out || ntensors < 0 || elem_size == 0 || cap_bytes == 0 ||
      (ntensors > 0 && !numels))
    return CR_ERR_INVALID_ARG;
  *out = nullptr;
  for (int t = 0; t < ntensors; ++t)
    if (numels[t] > SIZE_MAX / elem_size / 2) return CR_ERR_INVALID_ARG;
  cr_bucket_plan_t* p = static_cast<cr_bucket_plan_t*>(calloc(1, sizeof(cr_bucket_plan_t)));
  if (!p) return CR_ERR_INVALID_ARG;
  const size_t nt = ntensors > 0 ? (size_t)ntensors : 1;
  p->numels = static_cast<size_t*>(malloc(nt * sizeof(size_t)));
  p->tensor_bucket = static_cast<int*>(malloc(nt * sizeof(int)));
  p->tensor_offset = static_cast<size_t*>(malloc(nt * sizeof(size_t)));
  p->bucket_numel = static_cast<size_t*>(malloc(nt * sizeof(size_t)));
  if (!p->numels || !p->tensor_bucket || !p->tensor_offset || !p->bucket_numel) {
    cr_bucket_plan_free(p);
    return CR_ERR_INVALID_ARG;
  }
  p->ntensors = ntensors;
  p->elem_size = elem_size;
  p->cap_bytes = cap_bytes;
  if (ntensors > 0) memcpy(p->numels, numels, (size_t)ntensors * sizeof(size_t));

  int nb = 0;
  size_t bucket_bytes = 0;
  for (int t = ntensors - 1; t >= 0; --t) {
    const size_t bytes = numels[t] * elem_size;
    // A tensor joins the open bucket if it still fits under the cap; an
    // empty bucket takes any tensor, so an oversize one sits alone.
    const bool fits = nb > 0 && (bucket_bytes == 0 || bucket_bytes + bytes <= cap_bytes);
    if (!fits) {
      p->bucket_numel[nb] = 0;
      nb += 1;
      bucket_bytes = 0;
    }
    const int b = nb - 1;
    p->tensor_bucket[t] = b;
    p->tensor_offset[t] = p->bucket_numel[b];
    p->bucket_numel[b] += numels[t];
    bucket_bytes += bytes;
  }
  p->nbuckets = nb;
  *out = p;
  return CR_OK;
}

void cr_bucket_plan_free(cr_bucket_plan_t* p) {
  if (!p) return;
  free(p->numels);
  free(p->tensor_bucket);
  free(p->tensor_offset);
  free(p->bucket_numel);
  free(p);
}

// Closed forms of the schedules' per-rank traffic.  Ring reduce-scatter:
// rank r forwards, at step s, the partial of chunk (r - s) mod N for
// s = 1..N-1, i.e. every chunk except its own, and receives every chunk
// except chunk r-1 ("Distributed Training for Large Models", section 2,
// Reduce-Scatter).  Ring all-gather: rank r forwards shards r, r-1, ...,
// r-N+2, i.e. all but r+1, and receives all but its own (section 2,
// All-Reduce second phase).  Naive all-reduce: the root receives N-1 full
// buffers and sends N-1 full buffers; every other rank sends and receives
// one (nxmr.cn news 160867, 2.2).
cr_status cr_comm_elems(cr_collective coll, cr_schedule sched, int nranks,
                        size_t count, int rank, uint64_t* sent, uint64_t* recv,
                        int* steps) {
  if (nranks < 1 || nranks > CR_MAX_RANKS || rank < 0 || rank >= nranks || !sent ||
      !recv || !steps)
    return CR_ERR_INVALID_ARG;
  const uint64_t n = (uint64_t)nranks;
  const uint64_t L = cr_chunk_len(count, nranks);
  auto len = [&](uint64_t j) -> uint64_t {
    const uint64_t a = L * j < count ? L * j : count;
    const uint64_t b = L * (j + 1) < count ? L * (j + 1) : count;
    return b - a;
  };
  const uint64_t own = len((uint64_t)rank);
  const uint64_t next = len(((uint64_t)rank + 1) % n);
  const uint64_t prev = len(((uint64_t)rank + n - 1) % n);
  if (sched == CR_SCHED_NAIVE) {
    if (coll != CR_COLL_ALL_REDUCE) return CR_ERR_UNSUPPORTED;
    if (rank == 0) {
      *sent = (n - 1) * count;
      *recv = (n - 1) * count;
    } else {
      *sent = count;
      *recv = count;
    }
    *steps = (int)(2 * (n - 1));
    return CR_OK;
  }
  if (sched != CR_SCHED_RING) return CR_ERR_INVALID_ARG;
  const uint64_t rs_sent = count - own, rs_recv = count - prev;
  const uint64_t ag_sent = count - next, ag_recv = count - own;
  switch (coll) {
    case CR_COLL_REDUCE_SCATTER:
      *sent = n > 1 ? rs_sent : 0;
      *recv = n > 1 ? rs_recv : 0;
      *steps = (int)(n - 1);
      return CR_OK;
    case CR_COLL_ALL_GATHER:
      *sent = n > 1 ? ag_sent : 0;
      *recv = n > 1 ? ag_recv : 0;
      *steps = (int)(n - 1);
      return CR_OK;
    case CR_COLL_ALL_REDUCE:
      *sent = n > 1 ? rs_sent + ag_sent : 0;
      *recv = n > 1 ? rs_recv + ag_recv : 0;
      *steps = (int)(2 * (n - 1));
      return CR_OK;
  }
  return CR_ERR_INVALID_ARG;
}

}  // extern "C"
