// cuda_error_check.cu -- a C++ caller of libcr.so (include/cr.h) checking the
// error contract of every launching entry point: a launch that CUDA refuses
// makes the call return CR_ERR_CUDA with the CUDA error's name in
// cr_last_error(), nothing of the call runs, and the library stays usable --
// the next call on a healthy stream succeeds and computes the right result.
//
// The refusal is a real one that involves no GPU fault: while a stream is
// being captured, synchronising it is refused and invalidates the capture,
// after which CUDA refuses every launch, event record and copy enqueued on
// that stream (cudaErrorStreamCaptureInvalidated) until the capture is
// ended.  Every failing call below is enqueued on such a stream; nothing
// reaches the device.
//
// Built with nvcc against the library and run by test_cuda_error_gpu.py;
// prints one line per check and "ALL OK" when every check passed.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstring>
#include <string>
#include <thread>
#include <vector>

#include "cr.h"

static int g_fail = 0;

#define EXPECT(cond, ...)                                    \
  do {                                                       \
    if (!(cond)) {                                           \
      printf("FAIL %s:%d: ", __FILE__, __LINE__);            \
      printf(__VA_ARGS__);                                   \
      printf("\n");                                          \
      ++g_fail;                                              \
    }                                                        \
  } while (0)

#define CK(x)                                                                      \
  do {                                                                             \
    cudaError_t e_ = (x);                                                          \
    if (e_ != cudaSuccess) {                                                       \
      printf("SETUP %s:%d: %s (%s)\n", __FILE__, __LINE__, #x, cudaGetErrorName(e_)); \
      return 2;                                                                    \
    }                                                                              \
  } while (0)

namespace {

constexpr int N = 4;
constexpr size_t C = 4133;                // ragged: no multiple of N or of a vector
constexpr size_t L = (C + N - 1) / N;     // chunk length, 1034
constexpr size_t LH = (C + 1) / 2;        // HSDP 2 x 2: shard length over S = 2

// Every device allocation of the test, with its host snapshot.
struct Arena {
  std::vector<void*> ptrs;
  std::vector<size_t> sizes;
  bool failed = false;
  void* get(size_t bytes) {
    void* p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) {
      failed = true;
      return nullptr;
    }
    ptrs.push_back(p);
    sizes.push_back(bytes);
    return p;
  }
  // Deterministic non-zero bytes everywhere (small integers for int32
  // buffers are set separately).
  bool fill() {
    for (size_t i = 0; i < ptrs.size(); ++i) {
      std::vector<uint8_t> h(sizes[i]);
      for (size_t k = 0; k < h.size(); ++k) h[k] = (uint8_t)((k * 131u + i * 17u + 7u) & 0x3f);
      if (cudaMemcpy(ptrs[i], h.data(), h.size(), cudaMemcpyHostToDevice) != cudaSuccess)
        return false;
    }
    return true;
  }
  std::vector<std::vector<uint8_t>> snapshot() const {
    std::vector<std::vector<uint8_t>> s(ptrs.size());
    for (size_t i = 0; i < ptrs.size(); ++i) {
      s[i].resize(sizes[i]);
      cudaMemcpy(s[i].data(), ptrs[i], sizes[i], cudaMemcpyDeviceToHost);
    }
    return s;
  }
  ~Arena() {
    for (void* p : ptrs) cudaFree(p);
  }
};

bool mentions(const char* text, const char* what) { return text && strstr(text, what) != nullptr; }

// A failing call: CR_ERR_CUDA, and the CUDA error's name in the detail.
void expect_cuda_error(cr_status st, const char* call) {
  const char* detail = cr_last_error();
  EXPECT(st == CR_ERR_CUDA, "%s returned %s (%s), expected CR_ERR_CUDA", call,
         cr_status_string(st), detail);
  if (st == CR_ERR_CUDA)
    EXPECT(mentions(detail, "cudaError"), "%s: detail \"%s\" names no CUDA error", call,
           detail);
  printf("refused  %-34s %s\n", call, detail);
}

void expect_ok(cr_status st, const char* call) {
  EXPECT(st == CR_OK, "%s returned %s (%s) on a healthy stream", call, cr_status_string(st),
         cr_last_error());
  printf("ok       %s\n", call);
}

}  // namespace

int main() {
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev < 1) {
    printf("SETUP: no CUDA device\n");
    return 2;
  }
  Arena A;
  cr_adamw_cfg cfg = {1e-4, 0.9, 0.999, 1e-8, 0.01, 1};

  // ---- buffers ----------------------------------------------------------
  void *xi[N], *shi[N], *gi[N], *hs[N], *sd[N];         // int32 collectives
  float *acc[N], *ms[N], *mm[N], *mv[N], *wo[N];        // fp32
  void *gb[N], *pb[N], *wa[N];                          // bf16
  for (int r = 0; r < N; ++r) {
    xi[r] = A.get(C * 4);
    shi[r] = A.get(L * 4);
    gi[r] = A.get(C * 4);
    hs[r] = A.get(LH * 4);
    sd[r] = A.get(C * 4);
    acc[r] = static_cast<float*>(A.get(C * 4));
    ms[r] = static_cast<float*>(A.get(L * 4));
    mm[r] = static_cast<float*>(A.get(L * 4));
    mv[r] = static_cast<float*>(A.get(L * 4));
    wo[r] = static_cast<float*>(A.get(L * 4));
    gb[r] = A.get(C * 2);
    pb[r] = A.get(C * 2);
    wa[r] = A.get(C * 2);
  }
  float* ams = static_cast<float*>(A.get(L * 4));
  float* amm = static_cast<float*>(A.get(L * 4));
  float* amv = static_cast<float*>(A.get(L * 4));
  float* ag = static_cast<float*>(A.get(L * 4));
  void* ap = A.get(L * 2);
  const size_t wsb = cr_fsdp_clip_workspace_bytes();
  void* ws = A.get(wsb);

  // FSDP2: two parameters, uneven and empty shards (Lr = 2 rows of 3; 1 row of 7).
  const cr_param_shape shapes[2] = {{5, 3}, {2, 7}};
  void* g2[2 * N];
  void* p2[2 * N];
  float *m2[2 * N], *mm2[2 * N], *mv2[2 * N];
  for (int p = 0; p < 2; ++p) {
    const size_t numel = shapes[p].dim0 * shapes[p].row_numel;
    const size_t lr = (shapes[p].dim0 + N - 1) / N;
    for (int r = 0; r < N; ++r) {
      g2[p * N + r] = A.get(numel * 2);
      p2[p * N + r] = A.get(numel * 2);
      size_t lo = lr * r, hi = lr * (r + 1);
      if (lo > shapes[p].dim0) lo = shapes[p].dim0;
      if (hi > shapes[p].dim0) hi = shapes[p].dim0;
      const size_t len = (hi - lo) * shapes[p].row_numel;
      m2[p * N + r] = len ? static_cast<float*>(A.get(len * 4)) : nullptr;
      mm2[p * N + r] = len ? static_cast<float*>(A.get(len * 4)) : nullptr;
      mv2[p * N + r] = len ? static_cast<float*>(A.get(len * 4)) : nullptr;
    }
  }

  // The FSDP2 plan of the same parameters and its device table.
  cr_fsdp2_plan_t* plan2 = nullptr;
  if (cr_fsdp2_plan_create(shapes, 2, N, (const void* const*)g2, m2, mm2, mv2, p2, &plan2) !=
      CR_OK) {
    printf("SETUP: cr_fsdp2_plan_create: %s\n", cr_last_error());
    return 2;
  }
  const size_t tb = cr_fsdp2_plan_table_bytes(plan2);
  void* table = A.get(tb);

  // Range forms: the slab [RB, RE) of every buffer, which cuts chunks 0 and 3.
  constexpr size_t RB = L / 2 + 1, RE = C - 3;
  void *rin[N], *rout[N], *rsh[N], *rg[N], *rp[N];
  float *rms[N], *rmm[N], *rmv[N];
  for (int r = 0; r < N; ++r) {
    const size_t lo = RB > L * r ? RB : L * r;
    const size_t hi0 = L * (r + 1) < C ? L * (r + 1) : C;
    const size_t hi = RE < hi0 ? RE : hi0;
    rin[r] = static_cast<char*>(xi[r]) + RB * 4;    // int32 slabs
    rout[r] = static_cast<char*>(gi[r]) + RB * 4;
    rsh[r] = hi > lo ? static_cast<char*>(shi[r]) + (lo - L * r) * 4 : nullptr;
    rg[r] = static_cast<char*>(gb[r]) + RB * 2;     // bf16 slabs
    rp[r] = static_cast<char*>(pb[r]) + RB * 2;
    rms[r] = hi > lo ? ms[r] + (lo - L * r) : nullptr;
    rmm[r] = hi > lo ? mm[r] + (lo - L * r) : nullptr;
    rmv[r] = hi > lo ? mv[r] + (lo - L * r) : nullptr;
  }

  // Buckets: three bf16 tensors, a 4096-byte cap -> buckets {t2, t1}, {t0}.
  const size_t numels[3] = {1000, 37, 2000};
  cr_bucket_plan_t* plan = nullptr;
  if (cr_bucket_plan(numels, 3, 2, 4096, &plan) != CR_OK) {
    printf("SETUP: cr_bucket_plan: %s\n", cr_last_error());
    return 2;
  }
  const int T = plan->ntensors, B = plan->nbuckets;
  std::vector<void*> bt(N * T), bk(N * B);
  for (int r = 0; r < N; ++r) {
    for (int t = 0; t < T; ++t) bt[r * T + t] = A.get(numels[t] * 2);
    for (int b = 0; b < B; ++b) bk[r * B + b] = A.get(plan->bucket_numel[b] * 2);
  }
  if (A.failed) {
    printf("SETUP: cudaMalloc failed\n");
    return 2;
  }

  // Pinned, mapped host ranks for the host-memory all-reduces.
  void* hin[N];
  for (int r = 0; r < N; ++r) CK(cudaHostAlloc(&hin[r], C * 4, cudaHostAllocMapped));

  // ---- contents -----------------------------------------------------------
  if (!A.fill()) {
    printf("SETUP: fill failed\n");
    return 2;
  }
  std::vector<int32_t> hx(C);
  for (int r = 0; r < N; ++r) {
    for (size_t e = 0; e < C; ++e) hx[e] = (int32_t)((r + 1) * (e % 7 + 1));
    CK(cudaMemcpy(xi[r], hx.data(), C * 4, cudaMemcpyHostToDevice));
    memcpy(hin[r], hx.data(), C * 4);
  }
  cudaStream_t bad, good;
  CK(cudaStreamCreateWithFlags(&bad, cudaStreamNonBlocking));
  CK(cudaStreamCreateWithFlags(&good, cudaStreamNonBlocking));
  // The FSDP2 table, uploaded once before the capture.
  expect_ok(cr_fsdp2_plan_upload(plan2, table, tb, (cr_stream_t)good), "cr_fsdp2_plan_upload");
  CK(cudaStreamSynchronize(good));
  // The no-alloc step looks its static array up on its first call on a
  // device; that call has to come before any capture (as documented).
  expect_ok(cr_fsdp_step_clipped_noalloc((const void* const*)gb, N, C, ms, mm, mv, &cfg, 1.0,
                                         (void* const*)pb, nullptr, (cr_stream_t)good),
            "cr_fsdp_step_clipped_noalloc (first call)");
  CK(cudaDeviceSynchronize());
  const auto before = A.snapshot();
  std::vector<std::vector<uint8_t>> host_before(N);
  for (int r = 0; r < N; ++r)
    host_before[r].assign(static_cast<uint8_t*>(hin[r]), static_cast<uint8_t*>(hin[r]) + C * 4);

  // ---- invalidate a capture on `bad` ---------------------------------------
  CK(cudaStreamBeginCapture(bad, cudaStreamCaptureModeThreadLocal));
  const cudaError_t se = cudaStreamSynchronize(bad);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  CK(cudaStreamIsCapturing(bad, &cs));
  printf("synchronize during capture: %s; capture status %d\n", cudaGetErrorName(se), (int)cs);
  if (se == cudaSuccess || cs != cudaStreamCaptureStatusInvalidated) {
    printf("SETUP: the capture was not invalidated\n");
    cudaGraph_t g = nullptr;
    cudaStreamEndCapture(bad, &g);
    if (g) cudaGraphDestroy(g);
    return 2;
  }
  (void)cudaGetLastError();
  const cr_stream_t sb = (cr_stream_t)bad, sg = (cr_stream_t)good;

  // ---- every launching entry point, refused ---------------------------------
  const void* const* cxi = (const void* const*)xi;
  const void* const* cgb = (const void* const*)gb;
  expect_cuda_error(cr_all_reduce(cxi, N, C, CR_I32, CR_SUM, xi, CR_I32, sb), "cr_all_reduce");
  expect_cuda_error(cr_reduce_scatter(cxi, N, C, CR_I32, CR_SUM, shi, CR_I32, sb),
                    "cr_reduce_scatter");
  expect_cuda_error(cr_all_gather((const void* const*)shi, N, C, CR_I32, gi, sb), "cr_all_gather");
  expect_cuda_error(cr_reduce_scatter_wire(cgb, N, C, CR_BF16, CR_AVG, CR_BF16, (void* const*)wo,
                                           CR_F32, sb),
                    "cr_reduce_scatter_wire");
  expect_cuda_error(cr_all_reduce_wire(cgb, N, C, CR_BF16, CR_AVG, CR_BF16, wa, CR_BF16, sb),
                    "cr_all_reduce_wire");
  expect_cuda_error(cr_hsdp_reduce_scatter(cxi, 2, 2, C, CR_I32, CR_SUM, hs, CR_I32, sb),
                    "cr_hsdp_reduce_scatter");
  expect_cuda_error(cr_all_reduce_host((const void* const*)hin, hin, nullptr, N, C, CR_I32, CR_SUM,
                                       sb),
                    "cr_all_reduce_host");
  expect_cuda_error(cr_all_reduce_staged((const void* const*)hin, hin, sd, N, C, CR_I32, CR_SUM, 0,
                                         sb, sg, sg),
                    "cr_all_reduce_staged");
  expect_cuda_error(cr_accumulate(acc, N, C, cgb, CR_BF16, sb), "cr_accumulate");
  expect_cuda_error(cr_all_reduce_accumulate(acc, N, C, cgb, CR_BF16, CR_SUM, sb),
                    "cr_all_reduce_accumulate");
  expect_cuda_error(cr_fsdp_step(cgb, N, C, ms, mm, mv, &cfg, pb, sb), "cr_fsdp_step");
  expect_cuda_error(cr_fsdp_step_clipped(cgb, N, C, ms, mm, mv, &cfg, 1.0, ws, wsb, pb, nullptr,
                                         sb),
                    "cr_fsdp_step_clipped");
  expect_cuda_error(cr_fsdp_step_clipped_noalloc(cgb, N, C, ms, mm, mv, &cfg, 1.0, pb, nullptr, sb),
                    "cr_fsdp_step_clipped_noalloc");
  expect_cuda_error(cr_adamw_step(L, ams, amm, amv, ag, &cfg, ap, sb), "cr_adamw_step");
  expect_cuda_error(cr_bucket_pack(plan, N, (const void* const*)bt.data(), bk.data(), sb),
                    "cr_bucket_pack");
  expect_cuda_error(cr_bucket_all_reduce(plan, N, bk.data(), CR_BF16, CR_AVG, sb),
                    "cr_bucket_all_reduce");
  expect_cuda_error(cr_bucket_unpack(plan, N, (const void* const*)bk.data(), bt.data(), sb),
                    "cr_bucket_unpack");
  expect_cuda_error(cr_bucket_all_reduce_fused(plan, N, bt.data(), CR_BF16, CR_AVG, sb),
                    "cr_bucket_all_reduce_fused");
  // Reducer: the all-reduce stream refused, then the compute stream refused.
  // Marking bucket 0's tensors in backward order launches nothing until the
  // last of them, whose mark launches the bucket.
  std::vector<int> first_bucket;
  for (int t = T - 1; t >= 0; --t)
    if (plan->tensor_bucket[t] == 0) first_bucket.push_back(t);
  for (int which = 0; which < 2; ++which) {
    cr_reducer_t* red = nullptr;
    const cr_status cst = cr_reducer_create(plan, N, bt.data(), CR_BF16, CR_AVG, 0,
                                            which == 0 ? sb : sg, &red);
    EXPECT(cst == CR_OK, "cr_reducer_create: %s", cr_last_error());
    if (cst != CR_OK) continue;
    const cr_stream_t compute = which == 0 ? sg : sb;
    for (size_t k = 0; k + 1 < first_bucket.size(); ++k)
      EXPECT(cr_reducer_mark_ready(red, first_bucket[k], compute) == CR_OK,
             "marking tensor %d launches nothing: %s", first_bucket[k], cr_last_error());
    EXPECT(cr_reducer_launched(red) == 0, "no bucket may start before bucket 0 is complete");
    expect_cuda_error(cr_reducer_mark_ready(red, first_bucket.back(), compute),
                      which == 0 ? "cr_reducer_mark_ready (comm stream)"
                                 : "cr_reducer_mark_ready (compute stream)");
    cr_reducer_destroy(red);
  }
  // Communicator on the refused stream: every rank gets the launch's status.
  cr_comm_t* comm = nullptr;
  EXPECT(cr_comm_create(2, 20000, sb, &comm) == CR_OK, "cr_comm_create: %s", cr_last_error());
  if (comm) {
    cr_status st[2];
    std::string detail[2];
    std::vector<std::thread> ranks;
    for (int r = 0; r < 2; ++r)
      ranks.emplace_back([&, r] {
        st[r] = cr_comm_all_reduce(comm, r, xi[r], C, CR_I32, CR_SUM);
        detail[r] = cr_last_error();
      });
    for (auto& t : ranks) t.join();
    for (int r = 0; r < 2; ++r) {
      EXPECT(st[r] == CR_ERR_CUDA && mentions(detail[r].c_str(), "cudaError"),
             "cr_comm_all_reduce rank %d returned %s (%s)", r, cr_status_string(st[r]),
             detail[r].c_str());
      printf("refused  cr_comm_all_reduce rank %d         %s\n", r, detail[r].c_str());
    }
    EXPECT(cr_comm_broken(comm) == 0, "a refused launch must not break the communicator");
  }
  expect_cuda_error(cr_all_reduce_range((const void* const*)rin, N, C, RB, RE, CR_I32, CR_SUM,
                                        rout, CR_I32, sb),
                    "cr_all_reduce_range");
  expect_cuda_error(cr_reduce_scatter_range((const void* const*)rin, N, C, RB, RE, CR_I32, CR_SUM,
                                            rsh, CR_I32, sb),
                    "cr_reduce_scatter_range");
  expect_cuda_error(cr_fsdp_step_range((const void* const*)rg, N, C, RB, RE, rms, rmm, rmv, &cfg,
                                       rp, sb),
                    "cr_fsdp_step_range");
  expect_cuda_error(cr_fsdp2_plan_upload(plan2, table, tb, sb), "cr_fsdp2_plan_upload");
  expect_cuda_error(cr_fsdp2_step_planned(plan2, table, &cfg, sb), "cr_fsdp2_step_planned");
  // Last: a chained launch refused, so that the next call's launch would
  // see a stale error in the runtime's last-error word if one were kept.
  expect_cuda_error(cr_fsdp2_step(shapes, 2, N, (const void* const*)g2, m2, mm2, mv2, &cfg, p2, sb),
                    "cr_fsdp2_step");

  // ---- end the capture; nothing may have run --------------------------------
  cudaGraph_t graph = nullptr;
  const cudaError_t ee = cudaStreamEndCapture(bad, &graph);
  EXPECT(ee != cudaSuccess && graph == nullptr, "ending the invalidated capture gave %s",
         cudaGetErrorName(ee));
  if (graph) cudaGraphDestroy(graph);
  (void)cudaGetLastError();
  CK(cudaDeviceSynchronize());
  const auto after = A.snapshot();
  size_t changed = 0;
  for (size_t i = 0; i < before.size(); ++i) changed += before[i] != after[i];
  for (int r = 0; r < N; ++r)
    changed += memcmp(host_before[r].data(), hin[r], C * 4) != 0;
  EXPECT(changed == 0, "%zu buffers changed although every call was refused", changed);
  printf("buffers changed by refused calls: %zu\n", changed);

  // ---- the library stays usable ---------------------------------------------
  expect_ok(cr_all_reduce(cxi, N, C, CR_I32, CR_SUM, xi, CR_I32, sb),
            "cr_all_reduce after the refusals");
  CK(cudaStreamSynchronize(bad));
  size_t wrong = 0;
  for (int r = 0; r < N; ++r) {
    CK(cudaMemcpy(hx.data(), xi[r], C * 4, cudaMemcpyDeviceToHost));
    for (size_t e = 0; e < C; ++e) wrong += hx[e] != (int32_t)(10 * (e % 7 + 1));
  }
  EXPECT(wrong == 0, "%zu all-reduce results differ from the closed form", wrong);
  expect_ok(cr_fsdp2_step(shapes, 2, N, (const void* const*)g2, m2, mm2, mv2, &cfg, p2, sg),
            "cr_fsdp2_step");
  expect_ok(cr_fsdp2_step_planned(plan2, table, &cfg, sg), "cr_fsdp2_step_planned");
  expect_ok(cr_fsdp_step_range((const void* const*)rg, N, C, RB, RE, rms, rmm, rmv, &cfg, rp, sg),
            "cr_fsdp_step_range");
  {
    // the range all-reduce of the closed-form inputs: 10 * (e % 7 + 1)
    // after the all-reduce above, so the slab sums to 40 * (e % 7 + 1)
    expect_ok(cr_all_reduce_range((const void* const*)rin, N, C, RB, RE, CR_I32, CR_SUM, rout,
                                  CR_I32, sg),
              "cr_all_reduce_range");
    CK(cudaStreamSynchronize(good));
    size_t bad_range = 0;
    for (int r = 0; r < N; ++r) {
      CK(cudaMemcpy(hx.data(), gi[r], C * 4, cudaMemcpyDeviceToHost));
      for (size_t e = RB; e < RE; ++e) bad_range += hx[e] != (int32_t)(40 * (e % 7 + 1));
    }
    EXPECT(bad_range == 0, "%zu range all-reduce results differ from the closed form", bad_range);
  }
  expect_ok(cr_bucket_all_reduce_fused(plan, N, bt.data(), CR_BF16, CR_AVG, sg),
            "cr_bucket_all_reduce_fused");
  expect_ok(cr_fsdp_step_clipped(cgb, N, C, ms, mm, mv, &cfg, 1.0, ws, wsb, pb, nullptr, sg),
            "cr_fsdp_step_clipped");
  expect_ok(cr_all_reduce_staged((const void* const*)hin, hin, sd, N, C, CR_I32, CR_SUM, 0, sg, sg,
                                 sg),
            "cr_all_reduce_staged");
  {
    cr_reducer_t* red = nullptr;
    expect_ok(cr_reducer_create(plan, N, bt.data(), CR_BF16, CR_AVG, 0, sb, &red),
              "cr_reducer_create");
    if (red) {
      for (int t = T - 1; t >= 0; --t) expect_ok(cr_reducer_mark_ready(red, t, sg), "mark_ready");
      expect_ok(cr_reducer_finalize(red, sg), "cr_reducer_finalize");
      EXPECT(cr_reducer_launched(red) == 0, "a finalized iteration restarts at bucket 0");
      CK(cudaStreamSynchronize(good));
      cr_reducer_destroy(red);
    }
  }
  if (comm) {
    cr_status st[2];
    std::vector<std::thread> ranks;
    for (int r = 0; r < 2; ++r)
      ranks.emplace_back([&, r] { st[r] = cr_comm_all_reduce(comm, r, xi[r], C, CR_I32, CR_SUM); });
    for (auto& t : ranks) t.join();
    for (int r = 0; r < 2; ++r) expect_ok(st[r], "cr_comm_all_reduce");
    CK(cudaStreamSynchronize(bad));
    wrong = 0;
    for (int r = 0; r < 2; ++r) {
      CK(cudaMemcpy(hx.data(), xi[r], C * 4, cudaMemcpyDeviceToHost));
      for (size_t e = 0; e < C; ++e) wrong += hx[e] != (int32_t)(20 * (e % 7 + 1));
    }
    EXPECT(wrong == 0, "%zu communicator results differ from the closed form", wrong);
    cr_comm_destroy(comm);
  }
  CK(cudaDeviceSynchronize());

  cr_bucket_plan_free(plan);
  cr_fsdp2_plan_free(plan2);
  for (int r = 0; r < N; ++r) cudaFreeHost(hin[r]);
  cudaStreamDestroy(bad);
  cudaStreamDestroy(good);
  if (g_fail) {
    printf("%d checks failed\n", g_fail);
    return 1;
  }
  printf("ALL OK\n");
  return 0;
}
