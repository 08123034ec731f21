// reducer_state.h -- which DDP buckets may start their all-reduce.
//
// "AI Infra Guide, Chapter 6", 6.2.4-6.2.5: backward produces gradients
// layer by layer, last layer first; DDP groups them into buckets in that
// order and starts a bucket's all-reduce as soon as every gradient in it is
// ready, so that communication overlaps the rest of the backward pass.
// The buckets are launched strictly in bucket-index order (every rank must
// issue its collectives in the same order), so a bucket that fills early
// waits for its predecessors.
//
// This is the host-side bookkeeping alone, in plain C++ (no CUDA): mark()
// records one ready gradient and reports the buckets that may now be
// launched; the caller does the launching.  Compiled by the host compiler
// in the CPU tests.
#pragma once

#include <vector>

namespace cr {

class ReducerState {
 public:
  enum Status { kOk = 0, kOutOfRange = -1, kAlreadyReady = -2 };

  // tensor_bucket[t]: the bucket of tensor t, in [0, nbuckets).
  ReducerState(const int* tensor_bucket, int ntensors, int nbuckets)
      : bucket_of_(tensor_bucket, tensor_bucket + ntensors),
        count_(nbuckets, 0),
        pending_(nbuckets, 0),
        ready_(ntensors, 0) {
    for (int t = 0; t < ntensors; ++t) count_[bucket_of_[t]] += 1;
    reset();
  }

  // Tensor t's gradient is ready.  Appends to *launch, in order, every
  // bucket that can start now: the next unlaunched bucket and its
  // successors, as long as all their tensors are ready.
  int mark(int t, std::vector<int>* launch) {
    if (t < 0 || t >= (int)bucket_of_.size()) return kOutOfRange;
    if (ready_[t]) return kAlreadyReady;
    ready_[t] = 1;
    pending_[bucket_of_[t]] -= 1;
    while (next_ < (int)pending_.size() && pending_[next_] == 0) launch->push_back(next_++);
    return kOk;
  }

  // Buckets launched so far this iteration.
  int launched() const { return next_; }
  bool complete() const { return next_ == (int)pending_.size(); }
  int nbuckets() const { return (int)pending_.size(); }

  // Start a new iteration: no gradient ready, no bucket launched.  Buckets
  // that hold no tensor at all are launchable at once (and launched by the
  // first mark()).
  void reset() {
    pending_ = count_;
    for (auto& r : ready_) r = 0;
    next_ = 0;
  }

 private:
  std::vector<int> bucket_of_;
  std::vector<int> count_;    // tensors per bucket
  std::vector<int> pending_;  // tensors per bucket not yet ready
  std::vector<char> ready_;   // per tensor, this iteration
  int next_ = 0;              // first bucket not yet launched
};

}  // namespace cr
