// reducer.cu -- the DDP reducer: bucket all-reduces started as gradients
// become ready, overlapping the rest of the backward pass.
//
// "AI Infra Guide, Chapter 6", 6.2.5 (figure 6-2): when layer L's gradient
// is ready its all-reduce starts while layer L-1's backward runs; the wait
// that remains is only the part of the communication not hidden behind
// compute.  The emulated ranks' backward runs on a compute stream; each
// finished bucket is handed to a communication stream with an event, and
// its all-reduce (the fused, no-pack kernel) runs there on at most
// comm_ctas CTAs -- the SMs a communication library would reserve -- so
// that it can run beside the compute kernels.  Bucket order and readiness
// are tracked by ReducerState (plain C++).
#include <cuda_runtime.h>

#include <cstdio>
#include <vector>

#include "cr_internal.cuh"
#include "reducer_state.h"

struct cr_reducer {
  // Deep copy of the plan (the caller may free its own).
  std::vector<size_t> numels, tensor_offset, bucket_numel;
  std::vector<int> tensor_bucket;
  cr_bucket_plan_t plan;
  std::vector<std::vector<int>> bucket_tensors;  // tensors of each bucket
  std::vector<void*> tensors;                    // [nranks * ntensors]
  int nranks;
  cr_dtype dtype;
  cr_op op;
  uint32_t comm_ctas;
  cudaStream_t comm;
  int device;
  std::vector<cudaEvent_t> ready;  // per bucket: recorded on the compute stream
  cudaEvent_t done;                // recorded on the comm stream by finalize
  cr::ReducerState state;

  cr_reducer(const cr_bucket_plan_t* p)
      : numels(p->numels, p->numels + p->ntensors),
        tensor_offset(p->tensor_offset, p->tensor_offset + p->ntensors),
        bucket_numel(p->bucket_numel, p->bucket_numel + p->nbuckets),
        tensor_bucket(p->tensor_bucket, p->tensor_bucket + p->ntensors),
        bucket_tensors(p->nbuckets),
        state(p->tensor_bucket, p->ntensors, p->nbuckets) {
    plan = *p;
    plan.numels = numels.data();
    plan.tensor_offset = tensor_offset.data();
    plan.bucket_numel = bucket_numel.data();
    plan.tensor_bucket = tensor_bucket.data();
    for (int t = 0; t < p->ntensors; ++t) bucket_tensors[p->tensor_bucket[t]].push_back(t);
  }
};

namespace {

void destroy_events(cr_reducer* red) {
  for (cudaEvent_t e : red->ready)
    if (e) cudaEventDestroy(e);
  red->ready.clear();
  if (red->done) cudaEventDestroy(red->done);
  red->done = nullptr;
}

// The device the reducer was made on must be current for its calls.
cr_status check_device(const cr_reducer* red) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    return cr::report_cuda_error(e, "reducer: cudaGetDevice");
  }
  if (dev != red->device) {
    cr::report_error(CR_ERR_INVALID_ARG, "the reducer's device is not the current device");
    return CR_ERR_INVALID_ARG;
  }
  return CR_OK;
}

}  // namespace

extern "C" {

cr_status cr_reducer_create(const cr_bucket_plan_t* plan, int nranks, void* const* tensors,
                            cr_dtype dtype, cr_op op, int comm_ctas, cr_stream_t comm_stream,
                            cr_reducer_t** out) {
  if (!out) {
    cr::report_error(CR_ERR_INVALID_ARG, "out is NULL");
    return CR_ERR_INVALID_ARG;
  }
  *out = nullptr;
  if (comm_ctas < 0) {
    cr::report_error(CR_ERR_INVALID_ARG, "comm_ctas < 0");
    return CR_ERR_INVALID_ARG;
  }
  cr_status st = cr::bucket_fused_check(plan, nranks, tensors, dtype, op);
  if (st) return st;
  int dev = 0;
  const cudaError_t de = cudaGetDevice(&dev);
  if (de != cudaSuccess) return cr::report_cuda_error(de, "reducer: cudaGetDevice");
  cr_reducer* red = new cr_reducer(plan);
  red->tensors.assign(tensors, tensors + (size_t)nranks * plan->ntensors);
  red->nranks = nranks;
  red->dtype = dtype;
  red->op = op;
  red->comm_ctas = (uint32_t)comm_ctas;
  red->comm = (cudaStream_t)comm_stream;
  red->device = dev;
  red->done = nullptr;
  red->ready.assign(plan->nbuckets, nullptr);
  cudaError_t e = cudaSuccess;
  for (int b = 0; b < plan->nbuckets && e == cudaSuccess; ++b)
    e = cudaEventCreateWithFlags(&red->ready[b], cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&red->done, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    destroy_events(red);
    delete red;
    return cr::report_cuda_error(e, "reducer: cudaEventCreateWithFlags");
  }
  *out = red;
  return CR_OK;
}

cr_status cr_reducer_mark_ready(cr_reducer_t* red, int tensor, cr_stream_t compute_stream) {
  if (!red) {
    cr::report_error(CR_ERR_INVALID_ARG, "reducer is NULL");
    return CR_ERR_INVALID_ARG;
  }
  cr_status st = check_device(red);
  if (st) return st;
  std::vector<int> launch;
  const int rc = red->state.mark(tensor, &launch);
  if (rc == cr::ReducerState::kOutOfRange) {
    cr::report_error(CR_ERR_INVALID_ARG, "tensor index outside the plan");
    return CR_ERR_INVALID_ARG;
  }
  if (rc == cr::ReducerState::kAlreadyReady) {
    cr::report_error(CR_ERR_INVALID_ARG, "tensor already marked ready in this iteration");
    return CR_ERR_INVALID_ARG;
  }
  for (int b : launch) {
    // The comm stream may start bucket b once the compute stream has
    // produced everything enqueued so far (all of b's gradients).
    cudaError_t e = cudaEventRecord(red->ready[b], (cudaStream_t)compute_stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(red->comm, red->ready[b], 0);
    if (e != cudaSuccess) {
      return cr::report_cuda_error(e, "reducer: event record / stream wait");
    }
    const std::vector<int>& ts = red->bucket_tensors[b];
    st = cr::bucket_fused_tensors(&red->plan, red->nranks, red->tensors.data(), red->dtype,
                                  red->op, ts.data(), (int)ts.size(), red->comm_ctas, red->comm);
    if (st) return st;
  }
  return CR_OK;
}

int cr_reducer_launched(const cr_reducer_t* red) { return red ? red->state.launched() : -1; }

cr_status cr_reducer_finalize(cr_reducer_t* red, cr_stream_t compute_stream) {
  if (!red) {
    cr::report_error(CR_ERR_INVALID_ARG, "reducer is NULL");
    return CR_ERR_INVALID_ARG;
  }
  cr_status st = check_device(red);
  if (st) return st;
  if (!red->state.complete()) {
    char msg[128];
    snprintf(msg, sizeof(msg),
             "finalize before every gradient was marked ready (%d of %d buckets launched)",
             red->state.launched(), red->state.nbuckets());
    cr::report_error(CR_ERR_INVALID_ARG, msg);
    return CR_ERR_INVALID_ARG;
  }
  cudaError_t e = cudaEventRecord(red->done, red->comm);
  if (e == cudaSuccess) e = cudaStreamWaitEvent((cudaStream_t)compute_stream, red->done, 0);
  if (e != cudaSuccess) {
    return cr::report_cuda_error(e, "reducer: event record / stream wait");
  }
  red->state.reset();
  return CR_OK;
}

void cr_reducer_destroy(cr_reducer_t* red) {
  if (!red) return;
  destroy_events(red);
  delete red;
}

}  // extern "C"
