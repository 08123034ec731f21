// comm.cpp -- a communicator of emulated ranks driven one host thread per
// rank.
//
// With torch.distributed every rank calls all_reduce(tensor) on its own
// tensor, and the collective runs once all ranks have called it
// ("Distributed Training" section 2; "AI Infra Guide, Chapter 6", 6.1).
// Here the N ranks live in one process: each rank's thread calls
// cr_comm_* with its own buffer and blocks until all N have joined the same
// collective; the last one to arrive checks that the N calls agree and
// enqueues the library's single-kernel collective over the N buffers on the
// communicator's stream.  Failures are those the pages describe for real
// ranks (AI Infra Guide 6.8 and the troubleshooting notes: NCCL's timeout
// and watchdog, hangs from mismatched calls): a rank that never joins makes
// every waiting rank return CR_ERR_TIMEOUT after the communicator's timeout
// and leaves the communicator broken, as an aborted NCCL communicator is;
// calls that disagree (kind, count, dtypes, op) fail on every rank with
// CR_ERR_INVALID_ARG.  Neither failure launches anything.
#include <chrono>
#include <condition_variable>
#include <cstdio>
#include <mutex>
#include <string>

#include "cr.h"

namespace cr {
void report_error(cr_status status, const char* msg);
}

namespace {

enum Kind { kAllReduce = 0, kReduceScatter = 1, kAllGather = 2 };

struct Call {
  Kind kind;
  const void* in;  // the rank's input (buffer, or shard for all-gather)
  void* out;       // the rank's output (buffer, shard, or full buffer)
  size_t count;
  cr_dtype in_dtype, out_dtype;
  cr_op op;
};

const char* kind_name(Kind k) {
  return k == kAllReduce ? "all_reduce" : k == kReduceScatter ? "reduce_scatter" : "all_gather";
}

}  // namespace

struct cr_comm {
  int n;
  std::chrono::milliseconds timeout;
  cr_stream_t stream;
  std::mutex mu;
  std::condition_variable cv;
  unsigned long long gen = 0;  // collective currently being joined
  int arrived = 0;
  bool present[CR_MAX_RANKS] = {};
  Call calls[CR_MAX_RANKS];
  bool broken = false;
  cr_status result = CR_OK;  // of the last completed collective
  std::string result_msg;
};

namespace {

cr_status fail(cr_status st, const std::string& msg) {
  cr::report_error(st, msg.c_str());
  return st;
}

// Called by the last rank to arrive, with the lock held: the N calls must
// agree; then the single-kernel collective is enqueued.
cr_status run_collective(cr_comm* c, std::string* msg) {
  const Call& c0 = c->calls[0];
  for (int r = 1; r < c->n; ++r) {
    const Call& x = c->calls[r];
    if (x.kind != c0.kind || x.count != c0.count || x.in_dtype != c0.in_dtype ||
        x.out_dtype != c0.out_dtype || x.op != c0.op) {
      char b[200];
      snprintf(b, sizeof(b),
               "rank %d called %s(count=%zu) but rank 0 called %s(count=%zu), or their "
               "dtypes/op differ",
               r, kind_name(x.kind), x.count, kind_name(c0.kind), c0.count);
      *msg = b;
      return CR_ERR_INVALID_ARG;
    }
  }
  const void* in[CR_MAX_RANKS];
  void* out[CR_MAX_RANKS];
  for (int r = 0; r < c->n; ++r) {
    in[r] = c->calls[r].in;
    out[r] = c->calls[r].out;
  }
  cr_status st = CR_OK;
  switch (c0.kind) {
    case kAllReduce:
      st = cr_all_reduce(in, c->n, c0.count, c0.in_dtype, c0.op, out, c0.out_dtype, c->stream);
      break;
    case kReduceScatter:
      st = cr_reduce_scatter(in, c->n, c0.count, c0.in_dtype, c0.op, out, c0.out_dtype, c->stream);
      break;
    case kAllGather:
      st = cr_all_gather(in, c->n, c0.count, c0.in_dtype, out, c->stream);
      break;
  }
  if (st != CR_OK) *msg = std::string(kind_name(c0.kind)) + ": " + cr_last_error();
  return st;
}

cr_status join(cr_comm* c, int rank, const Call& call) {
  if (!c) return fail(CR_ERR_INVALID_ARG, "communicator is NULL");
  if (rank < 0 || rank >= c->n) {
    char b[96];
    snprintf(b, sizeof(b), "rank %d outside [0, %d)", rank, c->n);
    return fail(CR_ERR_INVALID_ARG, b);
  }
  std::unique_lock<std::mutex> lock(c->mu);
  if (c->broken)
    return fail(CR_ERR_TIMEOUT, "communicator is broken by an earlier timeout; destroy it");
  if (c->present[rank]) {
    char b[96];
    snprintf(b, sizeof(b), "rank %d joined the same collective twice", rank);
    return fail(CR_ERR_INVALID_ARG, b);
  }
  const unsigned long long my_gen = c->gen;
  c->present[rank] = true;
  c->calls[rank] = call;
  c->arrived += 1;
  if (c->arrived == c->n) {
    std::string msg;
    const cr_status st = run_collective(c, &msg);
    c->result = st;
    c->result_msg = msg;
    for (int r = 0; r < c->n; ++r) c->present[r] = false;
    c->arrived = 0;
    c->gen += 1;
    c->cv.notify_all();
    return st == CR_OK ? CR_OK : fail(st, msg);
  }
  const auto deadline = std::chrono::steady_clock::now() + c->timeout;
  const bool done = c->cv.wait_until(lock, deadline, [&] { return c->gen != my_gen || c->broken; });
  if (done && c->gen != my_gen) {
    // The collective completed; the next one cannot complete before every
    // rank of this one has left, so result is still this one's.
    return c->result == CR_OK ? CR_OK : fail(c->result, c->result_msg);
  }
  if (!c->broken) {
    c->broken = true;
    c->cv.notify_all();
  }
  char b[160];
  snprintf(b, sizeof(b), "rank %d: %d of %d ranks joined %s within %lld ms", rank, c->arrived, c->n,
           kind_name(call.kind), (long long)c->timeout.count());
  return fail(CR_ERR_TIMEOUT, b);
}

}  // namespace

extern "C" {

cr_status cr_comm_create(int nranks, int timeout_ms, cr_stream_t stream, cr_comm_t** out) {
  if (!out) return fail(CR_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (nranks < 1 || nranks > CR_MAX_RANKS)
    return fail(CR_ERR_INVALID_ARG, "nranks outside [1, CR_MAX_RANKS]");
  if (timeout_ms < 1) return fail(CR_ERR_INVALID_ARG, "timeout_ms < 1");
  cr_comm* c = new cr_comm();
  c->n = nranks;
  c->timeout = std::chrono::milliseconds(timeout_ms);
  c->stream = stream;
  *out = c;
  return CR_OK;
}

cr_status cr_comm_all_reduce(cr_comm_t* comm, int rank, void* buf, size_t count, cr_dtype dtype,
                             cr_op op) {
  return join(comm, rank, Call{kAllReduce, buf, buf, count, dtype, dtype, op});
}

cr_status cr_comm_reduce_scatter(cr_comm_t* comm, int rank, const void* buf, void* shard,
                                 size_t count, cr_dtype in_dtype, cr_op op, cr_dtype out_dtype) {
  return join(comm, rank, Call{kReduceScatter, buf, shard, count, in_dtype, out_dtype, op});
}

cr_status cr_comm_all_gather(cr_comm_t* comm, int rank, const void* shard, void* buf, size_t count,
                             cr_dtype dtype) {
  return join(comm, rank, Call{kAllGather, shard, buf, count, dtype, dtype, CR_SUM});
}

int cr_comm_broken(const cr_comm_t* comm) {
  if (!comm) return -1;
  cr_comm* c = const_cast<cr_comm*>(comm);
  std::lock_guard<std::mutex> lock(c->mu);
  return c->broken ? 1 : 0;
}

void cr_comm_destroy(cr_comm_t* comm) { delete comm; }

}  // extern "C"
