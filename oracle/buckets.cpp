/*
 * buckets.cpp -- oracle for DDP gradient bucketing: the bucket plan and the
 * pack / unpack copies.  Test infrastructure only (see oracle.h).
 *
 * [AIG] 6.2.4: gradients are grouped into buckets (default 25 MB) in the
 * order backward produces them, so the first gradients ready go into the
 * first buckets; [AIG] 6.2.6 Horovod Tensor Fusion concatenates small
 * tensors into one buffer; [NX] 5.1: fixed-size buckets filled in backward
 * order, each all-reduced as soon as it is full.
 */
#include "oracle.h"

#include <string.h>

int orc_bucket_plan(int ntensors, const size_t* numels, size_t esize,
                    size_t cap_bytes, int* tensor_bucket,
                    size_t* tensor_offset, size_t* bucket_numel,
                    int* nbuckets) {
  if (ntensors < 0 || esize == 0) return ORC_EINVAL;
  int b = -1;
  size_t fill_bytes = 0;
  /* Backward produces the last registered tensor's gradient first. */
  for (int t = ntensors - 1; t >= 0; --t) {
    size_t bytes = numels[t] * esize;
    int start_new = (b < 0) || (fill_bytes > 0 && fill_bytes + bytes > cap_bytes);
    if (start_new) {
      b += 1;
      bucket_numel[b] = 0;
      fill_bytes = 0;
    }
    tensor_bucket[t] = b;
    tensor_offset[t] = bucket_numel[b];
    bucket_numel[b] += numels[t];
    fill_bytes += bytes;
  }
  *nbuckets = b + 1;
  return ORC_OK;
}

void orc_bucket_pack(int n, int ntensors, const size_t* numels, size_t esize,
                     const int* tensor_bucket, const size_t* tensor_offset,
                     const void* const* tensors, void* const* buckets) {
  int nb = 0;
  for (int t = 0; t < ntensors; ++t)
    if (tensor_bucket[t] + 1 > nb) nb = tensor_bucket[t] + 1;
  for (int r = 0; r < n; ++r)
    for (int t = 0; t < ntensors; ++t) {
      unsigned char* dst = (unsigned char*)buckets[r * nb + tensor_bucket[t]];
      memcpy(dst + tensor_offset[t] * esize, tensors[r * ntensors + t],
             numels[t] * esize);
    }
}

void orc_bucket_unpack(int n, int ntensors, const size_t* numels,
                       size_t esize, const int* tensor_bucket,
                       const size_t* tensor_offset,
                       const void* const* buckets, void* const* tensors) {
  int nb = 0;
  for (int t = 0; t < ntensors; ++t)
    if (tensor_bucket[t] + 1 > nb) nb = tensor_bucket[t] + 1;
  for (int r = 0; r < n; ++r)
    for (int t = 0; t < ntensors; ++t) {
      const unsigned char* src =
          (const unsigned char*)buckets[r * nb + tensor_bucket[t]];
      memcpy(tensors[r * ntensors + t], src + tensor_offset[t] * esize,
             numels[t] * esize);
    }
}
