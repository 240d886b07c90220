// C ABI entry points (include/gptq_fold.h): argument checks, workspace
// carving and the chaining of fold -> ladder -> sweep.  No device memory is
// allocated here; every buffer is the caller's.
#include "common.cuh"

#include <math.h>
#include <string.h>

#include <memory>
#include <mutex>
#include <vector>

namespace gq {
size_t fold_ws_bytes(int n);
size_t sweep_ws_bytes(int rows, int n);
size_t sweep_ws_min_bytes(int rows, int n);
gptq_status fold_run(const float* hp, int n, double lambda, float* U, float* D, float* hdiag,
                     double* lambda_used, void* ws, size_t ws_bytes, cudaStream_t s,
                     const int* perm = nullptr);
gptq_status perm_run(const float* hdiag, int n, int* perm, cudaStream_t s);
gptq_status diag_run(const float* hp, int n, float* hdiag, cudaStream_t s);
size_t sweep_act_ws_bytes(int rows, int n);
gptq_status static_rungs_run(const float* W, int rows, int n, const float* tab, const float* lost,
                             uint8_t* rungs, float* scales, cudaStream_t s);
gptq_status sweep_act_run(const float* W, int rows, int n, const float* Up, const int* perm,
                          const float* tab, const uint8_t* srungs, uint8_t* nib, void* ws,
                          size_t ws_bytes, cudaStream_t s);
gptq_status build_only(const float* hp, int n, double lambda, float* A, float* D, void* ws,
                       size_t ws_bytes, cudaStream_t s);
gptq_status ladder_run(const float* W, int rows, int n, float* tab, float* lost, cudaStream_t s);
gptq_status copy_ladder_run(const float* W, int rows, int n, const float* hdiag, float* wz, float* tab,
                            float* lost, cudaStream_t s);
gptq_status group_run(const float* tile, int rows, const float* ublk, const float* hw,
                      const float* tab, const float* lost, uint8_t* nib, uint8_t* rungs,
                      float* scales, float* E, cudaStream_t s);
gptq_status copy_dead_zeroed(const float* W, int rows, int n, const float* hdiag, float* out,
                             cudaStream_t s);
gptq_status sweep_run(float* W, int rows, int n, const float* U, const float* hw, const float* tab,
                      const float* lost, uint8_t* nib, uint8_t* rungs, float* scales, void* ws,
                      size_t ws_bytes, cudaStream_t s);
gptq_status noalloc_scratch(void** out);
gptq_status fold_enqueue(const float* hp, int n, double lambda, float* U, float* D, float* hdiag,
                         void* ws, size_t ws_bytes, cudaStream_t s, const SideStream& side, unsigned** flag_out);
gptq_status sweep_enqueue(float* W, int rows, int n, const float* U, const float* hw, const float* tab,
                          const float* lost, uint8_t* nib, uint8_t* rungs, float* scales, void* ws,
                          size_t ws_bytes, cudaStream_t s, const SideStream& side, unsigned** status_out);
gptq_status sweep_q2_enqueue(float* W, int rows, int n, const float* U, const float* hw, const float* tab,
                             uint8_t* codes, uint8_t* rungs, float* scales, void* ws, size_t ws_bytes,
                             cudaStream_t s, const SideStream& side, unsigned** status_out);
gptq_status place_q2_run(const float* W, int rows, int n, const float* hw, float* tab, float* lost,
                         float* gscale, cudaStream_t s);
gptq_status group_q2_run(const float* tile, int rows, const float* ublk, const float* hw,
                         const float* tab, uint8_t* codes, uint8_t* rungs, float* scales, float* E,
                         cudaStream_t s);
size_t debias_ws_bytes(int rows, int n);
gptq_status debias_run(int bits, const float* W, int rows, int n, const float* Hp,
                       const uint8_t* codes, const uint8_t* rungs, float* tab, float* lost,
                       float* scales, double* num_den, void* ws, size_t ws_bytes, cudaStream_t s);
gptq_status sweep_q2_run(float* W, int rows, int n, const float* U, const float* hw,
                         const float* tab, uint8_t* codes, uint8_t* rungs, float* scales, void* ws,
                         size_t ws_bytes, cudaStream_t s);
size_t gram_ws_bytes(int n);
gptq_status gram_run(float* Hp, int n, const float* X, int T, void* ws, size_t ws_bytes,
                     cudaStream_t s);
}  // namespace gq

using namespace gq;

namespace {
bool bad_n(int n) { return n <= 0 || n > GPTQ_MAX_N; }
bool bad_rows(int rows) { return rows <= 0 || rows > GPTQ_MAX_ROWS; }
bool ptr_ok(const void* p) { return p != nullptr && aligned16(p); }
bool opt_ok(const void* p) { return p == nullptr || aligned16(p); }
cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
}  // namespace

namespace {

// gptq_quantize_group as a CUDA graph.  Its ~600 launches are dependent
// kernels, each of which, queued on a stream, costs about 2.6 us more in
// launch than as a node of an instantiated graph (measured on this GPU).  A
// call whose arguments (every pointer, size, lambda, the device context and
// the wait limits) were seen once before is captured -- one fold attempt at
// lambda, the ladder on its side stream, the sweep -- instantiated, and from
// then on replayed; the pivot flag and the sweep's status are read once
// after the replay.  A failed attempt (pivot flag) falls back to the
// stream path from the next lambda on.  Calls on a stream that is itself
// being captured, or while per-launch profiling records, take the stream
// path.
struct GroupKey {
  CUcontext ctx;
  int kind;  // 4: q4tp, 2: q2tp
  int dev, n, rows, no_loads;
  unsigned long long wait_ns;
  double lambda;
  size_t ws_bytes;
  const void* p[12];
};

struct GroupGraph {
  GroupKey key;
  cudaGraphExec_t exec;  // null until captured
  long long launches;    // kernels per replay
  unsigned* flag;
  unsigned* status;
  bool failed;           // capture did not work: always the stream path
  unsigned long long used;
};

// The most recently used argument sets; launches and evictions happen under
// the lock, so no replay can meet a destroyed graph.
constexpr size_t kMaxGraphs = 32;
std::mutex g_graph_mu;
std::vector<GroupGraph> g_graphs;
unsigned long long g_graph_clock = 0;

GroupGraph* find_graph(const GroupKey& key) {
  for (GroupGraph& e : g_graphs)
    if (memcmp(&e.key, &key, sizeof(key)) == 0) return &e;
  return nullptr;
}

// Per host thread and device: a stream to capture on and replay on, and the
// side streams the capture forks to.  Made on first use in the device's
// context; made again if that context was replaced (a device reset).
struct ThreadStreams {
  CUcontext ctx = nullptr;
  cudaStream_t st = nullptr;
  cudaEvent_t in = nullptr;
  SideStream ladder, sweep, fold;
  gptq_status init(CUcontext c) {
    if (ctx == c && st != nullptr) return GPTQ_OK;
    // Handles of an old context went with it.
    st = nullptr;
    in = nullptr;
    ladder.forget();
    sweep.forget();
    fold.forget();
    GQ_CUDA(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));
    GQ_CUDA(cudaEventCreateWithFlags(&in, cudaEventDisableTiming));
    GQ_TRY(ladder.init());
    GQ_TRY(sweep.init());
    GQ_TRY(fold.init());
    ctx = c;
    return GPTQ_OK;
  }
};

// One ThreadStreams per device this thread has used, so that a thread that
// moves between devices keeps (and at its exit releases) each device's set.
struct ThreadDeviceStreams {
  std::vector<std::unique_ptr<ThreadStreams>> dev;
  ThreadStreams& get(int d) {
    if (d >= (int)dev.size()) dev.resize((size_t)d + 1);
    if (!dev[(size_t)d]) dev[(size_t)d].reset(new ThreadStreams());
    return *dev[(size_t)d];
  }
};

GroupKey group_key(int kind, const float* H_packed, int n, double lambda, const float* W, int rows,
                   const void* nibbles, const void* rungs, const float* scales, const float* tab, const float* lost,
                   const float* U, const float* D, const float* hdiag, const void* ws, size_t ws_bytes) {
  GroupKey k;
  memset(&k, 0, sizeof(k));  // the comparison is bytewise, padding included
  k.ctx = current_context();
  k.kind = kind;
  cudaGetDevice(&k.dev);
  k.n = n;
  k.rows = rows;
  const WaitCfg wc = wait_cfg();
  k.wait_ns = wc.ns;
  k.no_loads = wc.no_loads;
  k.lambda = lambda;
  k.ws_bytes = ws_bytes;
  const void* p[12] = {H_packed, W, nibbles, rungs, scales, tab, lost, U, D, hdiag, ws, nullptr};
  memcpy(k.p, p, sizeof(p));
  return k;
}

// Runs one group call: the stream path on the first sight of the argument
// set, a capture on the second, replays after that (see GroupKey).
// stream_path(lam0): the whole call on the caller's stream from damping
// lam0 on; enqueue(st, ts, &flag, &status): one attempt at the call's
// damping, forking to ts's side streams and joined back, handing back the
// fold's pivot flag and the sweep's status word.
template <class StreamPath, class Enqueue>
gptq_status run_graphed(const GroupKey& key, cudaStream_t s, double lambda, double* lambda_used,
                        StreamPath& stream_path, Enqueue& enqueue) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (prof_active() || cudaStreamIsCapturing(s, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
    return stream_path(lambda);
  // No lock is held while a path runs.
  bool capture = false, use_stream = false;
  {
    std::lock_guard<std::mutex> lk(g_graph_mu);
    GroupGraph* e = find_graph(key);
    if (e == nullptr) {
      // Seen once: this call takes the stream path.
      if (g_graphs.size() >= kMaxGraphs) {
        size_t lru = 0;
        for (size_t i = 1; i < g_graphs.size(); ++i)
          if (g_graphs[i].used < g_graphs[lru].used) lru = i;
        if (g_graphs[lru].exec) cudaGraphExecDestroy(g_graphs[lru].exec);
        g_graphs.erase(g_graphs.begin() + (long)lru);
      }
      GroupGraph ne{};
      ne.key = key;
      ne.used = ++g_graph_clock;
      g_graphs.push_back(ne);
      use_stream = true;
    } else {
      e->used = ++g_graph_clock;
      use_stream = e->failed;
      capture = e->exec == nullptr;
    }
  }
  if (use_stream) return stream_path(lambda);

  static thread_local ThreadDeviceStreams tds;
  if (key.dev < 0) return stream_path(lambda);
  ThreadStreams& ts = tds.get(key.dev);
  GQ_TRY(ts.init(key.ctx));
  if (capture) {
    // Capture one attempt at lambda and instantiate it.
    const long long l0 = gptq_launch_count();
    unsigned *flag = nullptr, *status = nullptr;
    cudaGraph_t graph = nullptr;
    bool ok = cudaStreamBeginCapture(ts.st, cudaStreamCaptureModeThreadLocal) == cudaSuccess;
    if (ok) {
      const gptq_status e = enqueue(ts.st, ts, &flag, &status);
      // Every capture is ended, whatever the enqueue did.
      ok = cudaStreamEndCapture(ts.st, &graph) == cudaSuccess && e == GPTQ_OK && graph != nullptr;
    }
    cudaGetLastError();  // a refused capture leaves nothing behind to report
    cudaGraphExec_t exec = nullptr;
    if (ok) ok = cudaGraphInstantiate(&exec, graph, 0) == cudaSuccess;
    if (graph) cudaGraphDestroy(graph);
    const long long captured = gptq_launch_count() - l0;
    prof_add_launches(-captured);  // captured, not launched
    {
      std::lock_guard<std::mutex> lk(g_graph_mu);
      GroupGraph* e = find_graph(key);
      if (e == nullptr || e->exec != nullptr || !ok) {
        // Evicted meanwhile, or another thread's capture came first, or no graph.
        if (exec) cudaGraphExecDestroy(exec);
        if (e && !ok) e->failed = true;
        use_stream = !ok || e == nullptr;
      } else {
        e->exec = exec;
        e->launches = captured;
        e->flag = flag;
        e->status = status;
      }
    }
    if (use_stream) return stream_path(lambda);
  }
  // Replay after everything the caller queued on s (launched under the lock,
  // so that no eviction can destroy the graph first), and wait for it.
  unsigned *gflag = nullptr, *gstatus = nullptr;
  cudaError_t le = cudaSuccess;
  {
    std::lock_guard<std::mutex> lk(g_graph_mu);
    GroupGraph* e = find_graph(key);
    if (e == nullptr || e->exec == nullptr) {
      use_stream = true;
    } else {
      le = cudaEventRecord(ts.in, s);
      if (le == cudaSuccess) le = cudaStreamWaitEvent(ts.st, ts.in, 0);
      if (le == cudaSuccess) le = cudaGraphLaunch(e->exec, ts.st);
      if (le == cudaSuccess) prof_add_launches(e->launches);
      gflag = e->flag;
      gstatus = e->status;
    }
  }
  if (use_stream) return stream_path(lambda);
  if (le != cudaSuccess) return GPTQ_ERR_CUDA;
  unsigned hf = 0, hs = 0;
  GQ_CUDA(cudaMemcpyAsync(&hf, gflag, sizeof(unsigned), cudaMemcpyDeviceToHost, ts.st));
  GQ_CUDA(cudaMemcpyAsync(&hs, gstatus, sizeof(unsigned), cudaMemcpyDeviceToHost, ts.st));
  GQ_CUDA(cudaStreamSynchronize(ts.st));
  if ((hf & 2u) || hs) return GPTQ_ERR_TIMEOUT;
  const double lam = lambda > 0.0 ? lambda : 0.0;
  if (hf != 0u) {
    // Not positive definite at lambda: the stream path from the next one.
    const double next = next_lambda(lam);
    if (next > 10.0) return GPTQ_ERR_NOT_SPD;
    return stream_path(next);
  }
  if (lambda_used) *lambda_used = lam;
  return GPTQ_OK;
}

}  // namespace

extern "C" {

const char* gptq_status_string(int status) {
  switch (status) {
    case GPTQ_OK: return "ok";
    case GPTQ_ERR_ARG: return "invalid argument (null/misaligned pointer or non-finite lambda)";
    case GPTQ_ERR_SHAPE: return "invalid shape";
    case GPTQ_ERR_NOMEM: return "workspace too small";
    case GPTQ_ERR_NOT_SPD: return "not positive definite with damping up to lambda = 10";
    case GPTQ_ERR_CUDA: return "CUDA error";
    case GPTQ_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

size_t gptq_fold_workspace_bytes(int n) { return bad_n(n) ? 0 : fold_ws_bytes(n); }

size_t gptq_sweep_workspace_bytes(int rows, int n) {
  if (bad_n(n) || bad_rows(rows)) return 0;
  return sweep_ws_bytes(rows, n);
}

size_t gptq_group_workspace_bytes(int rows, int n) {
  if (bad_n(n) || bad_rows(rows)) return 0;
  const size_t f = fold_ws_bytes(n), sw = sweep_ws_bytes(rows, n);
  const size_t own = round_up((size_t)n * n * 4, 256) + 3 * round_up((size_t)n * 4, 256) +
                     round_up((size_t)rows * n * 4, 256) + round_up((size_t)rows * 32 * 4, 256) +
                     round_up((size_t)rows * 2 * 4, 256) + 1024;
  return own + (f > sw ? f : sw);
}

gptq_status gptq_fold(const float* H_packed, int n, double lambda, float* U, float* D,
                      float* hdiag, double* lambda_used, void* ws, size_t ws_bytes,
                      void* stream) {
  if (bad_n(n)) return GPTQ_ERR_SHAPE;
  if (!ptr_ok(H_packed) || !ptr_ok(U) || !opt_ok(D) || !opt_ok(hdiag) || ws == nullptr)
    return GPTQ_ERR_ARG;
  if (!isfinite(lambda)) return GPTQ_ERR_ARG;
  if (ws_bytes < fold_ws_bytes(n)) return GPTQ_ERR_NOMEM;
  return fold_run(H_packed, n, lambda, U, D, hdiag, lambda_used, ws, ws_bytes, as_stream(stream));
}

gptq_status gptq_build_equilibrated(const float* H_packed, int n, double lambda, float* A,
                                    float* D, void* ws, size_t ws_bytes, void* stream) {
  if (bad_n(n)) return GPTQ_ERR_SHAPE;
  if (!ptr_ok(H_packed) || !ptr_ok(A) || !opt_ok(D) || ws == nullptr) return GPTQ_ERR_ARG;
  if (!isfinite(lambda)) return GPTQ_ERR_ARG;
  if (ws_bytes < fold_ws_bytes(n)) return GPTQ_ERR_NOMEM;
  return build_only(H_packed, n, lambda, A, D, ws, ws_bytes, as_stream(stream));
}

gptq_status gptq_ladder(const float* W, int rows, int n, float* tab, float* lost, void* stream) {
  if (bad_n(n) || bad_rows(rows) || n % GPTQ_GROUP != 0) return GPTQ_ERR_SHAPE;
  if (!ptr_ok(W) || !ptr_ok(tab) || !ptr_ok(lost)) return GPTQ_ERR_ARG;
  return ladder_run(W, rows, n, tab, lost, as_stream(stream));
}

gptq_status gptq_q4tp_group(const float* tile, int rows, const float* ublk, const float* hw,
                            const float* tab, const float* lost, uint8_t* nibbles,
                            uint8_t* rungs, float* scales, float* E, void* stream) {
  if (bad_rows(rows)) return GPTQ_ERR_SHAPE;
  if (!ptr_ok(tile) || !ptr_ok(ublk) || !ptr_ok(hw) || !ptr_ok(tab) || !ptr_ok(lost) ||
      !ptr_ok(nibbles) || rungs == nullptr || !ptr_ok(scales) || !ptr_ok(E))
    return GPTQ_ERR_ARG;
  return group_run(tile, rows, ublk, hw, tab, lost, nibbles, rungs, scales, E, as_stream(stream));
}

gptq_status gptq_q4tp_sweep(float* W, int rows, int n, const float* U, const float* hw,
                            const float* tab, const float* lost, uint8_t* nibbles,
                            uint8_t* rungs, float* scales, void* ws, size_t ws_bytes,
                            void* stream) {
  if (bad_n(n) || bad_rows(rows) || n % GPTQ_GROUP != 0) return GPTQ_ERR_SHAPE;
  if (!ptr_ok(W) || !ptr_ok(U) || !ptr_ok(hw) || !ptr_ok(tab) || !ptr_ok(lost) ||
      !ptr_ok(nibbles) || rungs == nullptr || !ptr_ok(scales) || ws == nullptr)
    return GPTQ_ERR_ARG;
  if (ws_bytes < sweep_ws_min_bytes(rows, n)) return GPTQ_ERR_NOMEM;
  return sweep_run(W, rows, n, U, hw, tab, lost, nibbles, rungs, scales, ws, ws_bytes,
                   as_stream(stream));
}

gptq_status gptq_q4tp_sweep_noalloc(float* W, int rows, int n, const float* U, const float* hw,
                                    const float* tab, const float* lost, uint8_t* nibbles,
                                    uint8_t* rungs, float* scales, void* stream) {
  if (bad_n(n) || bad_rows(rows) || n % GPTQ_GROUP != 0) return GPTQ_ERR_SHAPE;
  if (!ptr_ok(W) || !ptr_ok(U) || !ptr_ok(hw) || !ptr_ok(tab) || !ptr_ok(lost) ||
      !ptr_ok(nibbles) || rungs == nullptr || !ptr_ok(scales))
    return GPTQ_ERR_ARG;
  if (sweep_ws_min_bytes(rows, n) > (size_t)GPTQ_SWEEP_NOALLOC_SCRATCH_BYTES) return GPTQ_ERR_NOMEM;
  void* scratch = nullptr;
  GQ_TRY(noalloc_scratch(&scratch));
  return sweep_run(W, rows, n, U, hw, tab, lost, nibbles, rungs, scales, scratch,
                   (size_t)GPTQ_SWEEP_NOALLOC_SCRATCH_BYTES, as_stream(stream));
}


gptq_status gptq_quantize_group(const float* H_packed, int n, double lambda, const float* W,
                                int rows, uint8_t* nibbles, uint8_t* rungs, float* scales,
                                float* tab, float* lost, float* U, float* D, float* hdiag,
                                double* lambda_used, void* ws, size_t ws_bytes, void* stream) {
  if (bad_n(n) || bad_rows(rows) || n % GPTQ_GROUP != 0) return GPTQ_ERR_SHAPE;
  if (!ptr_ok(H_packed) || !ptr_ok(W) || !ptr_ok(nibbles) || rungs == nullptr ||
      !ptr_ok(scales) || !opt_ok(tab) || !opt_ok(lost) || !opt_ok(U) || !opt_ok(D) ||
      !opt_ok(hdiag) || ws == nullptr)
    return GPTQ_ERR_ARG;
  if (!isfinite(lambda)) return GPTQ_ERR_ARG;
  if (ws_bytes < gptq_group_workspace_bytes(rows, n)) return GPTQ_ERR_NOMEM;
  cudaStream_t s = as_stream(stream);
  Carve c(ws, ws_bytes);
  float* u = U ? U : c.take<float>((size_t)n * n);
  float* d = D ? D : c.take<float>((size_t)n);
  float* hd = hdiag ? hdiag : c.take<float>((size_t)n);
  float* wz = c.take<float>((size_t)rows * n);
  float* tb = tab ? tab : c.take<float>((size_t)rows * 32);
  float* ls = lost ? lost : c.take<float>((size_t)rows * 2);
  float* hd2 = c.take<float>((size_t)n);  // the ladder's own copy of diag(H)
  if (!c.ok) return GPTQ_ERR_NOMEM;
  const size_t off = round_up(c.off, 256);
  void* rest = static_cast<char*>(ws) + off;
  const size_t rest_bytes = ws_bytes - off;
  // The dead-zeroed copy of W and its ladder depend on W and diag(H) alone:
  // they run on a side stream beside the fold (whose one-CTA steps leave
  // the GPU mostly idle), joined before the sweep.
  auto enqueue_ladder = [&](cudaStream_t st, const SideStream& side) -> gptq_status {
    GQ_CUDA(cudaEventRecord(side.fork, st));
    GQ_CUDA(cudaStreamWaitEvent(side.s, side.fork, 0));
    GQ_TRY(diag_run(H_packed, n, hd2, side.s));
    GQ_TRY(copy_ladder_run(W, rows, n, hd2, wz, tb, ls, side.s));
    GQ_CUDA(cudaEventRecord(side.join, side.s));
    return GPTQ_OK;
  };
  auto stream_path = [&](double lam0) -> gptq_status {
    SideStream side;
    GQ_TRY(side.init());
    GQ_TRY(enqueue_ladder(s, side));
    const gptq_status fs = fold_run(H_packed, n, lam0, u, d, hd, lambda_used, rest, rest_bytes, s);
    GQ_CUDA(cudaStreamWaitEvent(s, side.join, 0));
    GQ_TRY(fs);
    return sweep_run(wz, rows, n, u, hd, tb, ls, nibbles, rungs, scales, rest, rest_bytes, s);
  };

  auto enqueue = [&](cudaStream_t st, const ThreadStreams& ts, unsigned** flag, unsigned** status) -> gptq_status {
    GQ_TRY(enqueue_ladder(st, ts.ladder));
    GQ_TRY(fold_enqueue(H_packed, n, lambda, u, d, hd, rest, rest_bytes, st, ts.fold, flag));
    GQ_CUDA(cudaStreamWaitEvent(st, ts.ladder.join, 0));
    return sweep_enqueue(wz, rows, n, u, hd, tb, ls, nibbles, rungs, scales, rest, rest_bytes, st, ts.sweep,
                         status);
  };
  const GroupKey key = group_key(4, H_packed, n, lambda, W, rows, nibbles, rungs, scales, tab, lost, U, D, hdiag,
                                 ws, ws_bytes);
  return run_graphed(key, s, lambda, lambda_used, stream_path, enqueue);
}

gptq_status gptq_q2tp_place(const float* W, int rows, int n, const float* hw, float* tab,
                            float* lost, float* gscale, void* stream) {
  if (bad_n(n) || bad_rows(rows) || n % GPTQ_GROUP != 0) return GPTQ_ERR_SHAPE;
  if (!ptr_ok(W) || !ptr_ok(hw) || !ptr_ok(tab) || !ptr_ok(lost) || !opt_ok(gscale))
    return GPTQ_ERR_ARG;
  return place_q2_run(W, rows, n, hw, tab, lost, gscale, as_stream(stream));
}

gptq_status gptq_q2tp_group(const float* tile, int rows, const float* ublk, const float* hw,
                            const float* tab, uint8_t* codes, uint8_t* rungs, float* scales,
                            float* E, void* stream) {
  if (bad_rows(rows)) return GPTQ_ERR_SHAPE;
  if (!ptr_ok(tile) || !ptr_ok(ublk) || !ptr_ok(hw) || !ptr_ok(tab) || !ptr_ok(codes) ||
      rungs == nullptr || !ptr_ok(scales) || !ptr_ok(E))
    return GPTQ_ERR_ARG;
  return group_q2_run(tile, rows, ublk, hw, tab, codes, rungs, scales, E, as_stream(stream));
}

gptq_status gptq_q2tp_sweep(float* W, int rows, int n, const float* U, const float* hw,
                            const float* tab, uint8_t* codes, uint8_t* rungs, float* scales,
                            void* ws, size_t ws_bytes, void* stream) {
  if (bad_n(n) || bad_rows(rows) || n % GPTQ_GROUP != 0) return GPTQ_ERR_SHAPE;
  if (!ptr_ok(W) || !ptr_ok(U) || !ptr_ok(hw) || !ptr_ok(tab) || !ptr_ok(codes) ||
      rungs == nullptr || !ptr_ok(scales) || ws == nullptr)
    return GPTQ_ERR_ARG;
  if (ws_bytes < sweep_ws_min_bytes(rows, n)) return GPTQ_ERR_NOMEM;
  return sweep_q2_run(W, rows, n, U, hw, tab, codes, rungs, scales, ws, ws_bytes,
                      as_stream(stream));
}

gptq_status gptq_quantize_group_q2tp(const float* H_packed, int n, double lambda, const float* W,
                                     int rows, uint8_t* codes, uint8_t* rungs, float* scales,
                                     float* tab, float* lost, float* U, float* D, float* hdiag,
                                     double* lambda_used, void* ws, size_t ws_bytes, void* stream) {
  if (bad_n(n) || bad_rows(rows) || n % GPTQ_GROUP != 0) return GPTQ_ERR_SHAPE;
  if (!ptr_ok(H_packed) || !ptr_ok(W) || !ptr_ok(codes) || rungs == nullptr || !ptr_ok(scales) ||
      !opt_ok(tab) || !opt_ok(lost) || !opt_ok(U) || !opt_ok(D) || !opt_ok(hdiag) || ws == nullptr)
    return GPTQ_ERR_ARG;
  if (!isfinite(lambda)) return GPTQ_ERR_ARG;
  if (ws_bytes < gptq_group_workspace_bytes(rows, n)) return GPTQ_ERR_NOMEM;
  cudaStream_t s = as_stream(stream);
  Carve c(ws, ws_bytes);
  float* u = U ? U : c.take<float>((size_t)n * n);
  float* d = D ? D : c.take<float>((size_t)n);
  float* hd = hdiag ? hdiag : c.take<float>((size_t)n);
  float* wz = c.take<float>((size_t)rows * n);
  float* tb = tab ? tab : c.take<float>((size_t)rows * 32);
  float* ls = lost ? lost : c.take<float>((size_t)rows * 2);
  float* hd2 = c.take<float>((size_t)n);  // the placement's own copy of diag(H)
  if (!c.ok) return GPTQ_ERR_NOMEM;
  const size_t off = round_up(c.off, 256);
  void* rest = static_cast<char*>(ws) + off;
  const size_t rest_bytes = ws_bytes - off;
  // The dead-zeroed copy of W and its placed ladder depend on W and diag(H)
  // alone: a side stream beside the fold, joined before the sweep.
  auto enqueue_place = [&](cudaStream_t st, const SideStream& side) -> gptq_status {
    GQ_CUDA(cudaEventRecord(side.fork, st));
    GQ_CUDA(cudaStreamWaitEvent(side.s, side.fork, 0));
    GQ_TRY(diag_run(H_packed, n, hd2, side.s));
    GQ_TRY(copy_dead_zeroed(W, rows, n, hd2, wz, side.s));
    GQ_TRY(place_q2_run(wz, rows, n, hd2, tb, ls, nullptr, side.s));
    GQ_CUDA(cudaEventRecord(side.join, side.s));
    return GPTQ_OK;
  };
  auto stream_path = [&](double lam0) -> gptq_status {
    SideStream side;
    GQ_TRY(side.init());
    GQ_TRY(enqueue_place(s, side));
    const gptq_status fs = fold_run(H_packed, n, lam0, u, d, hd, lambda_used, rest, rest_bytes, s);
    GQ_CUDA(cudaStreamWaitEvent(s, side.join, 0));
    GQ_TRY(fs);
    return sweep_q2_run(wz, rows, n, u, hd, tb, codes, rungs, scales, rest, rest_bytes, s);
  };
  auto enqueue = [&](cudaStream_t st, const ThreadStreams& ts, unsigned** flag, unsigned** status) -> gptq_status {
    GQ_TRY(enqueue_place(st, ts.ladder));
    GQ_TRY(fold_enqueue(H_packed, n, lambda, u, d, hd, rest, rest_bytes, st, ts.fold, flag));
    GQ_CUDA(cudaStreamWaitEvent(st, ts.ladder.join, 0));
    return sweep_q2_enqueue(wz, rows, n, u, hd, tb, codes, rungs, scales, rest, rest_bytes, st, ts.sweep,
                            status);
  };
  const GroupKey key = group_key(2, H_packed, n, lambda, W, rows, codes, rungs, scales, tab, lost, U, D, hdiag,
                                 ws, ws_bytes);
  return run_graphed(key, s, lambda, lambda_used, stream_path, enqueue);
}

size_t gptq_debias_workspace_bytes(int rows, int n) {
  if (bad_n(n) || bad_rows(rows)) return 0;
  return debias_ws_bytes(rows, n);
}

gptq_status gptq_debias(int bits, const float* W, int rows, int n, const float* H_packed,
                        const uint8_t* codes, const uint8_t* rungs, float* tab, float* lost,
                        float* scales, double* num_den, void* ws, size_t ws_bytes, void* stream) {
  if (bad_n(n) || bad_rows(rows) || n % GPTQ_GROUP != 0) return GPTQ_ERR_SHAPE;
  if (bits != 2 && bits != 4) return GPTQ_ERR_ARG;
  if (!ptr_ok(W) || !ptr_ok(H_packed) || !ptr_ok(codes) || rungs == nullptr || !ptr_ok(tab) ||
      !ptr_ok(lost) || !ptr_ok(scales) || !opt_ok(num_den) || ws == nullptr)
    return GPTQ_ERR_ARG;
  if (ws_bytes < debias_ws_bytes(rows, n)) return GPTQ_ERR_NOMEM;
  return debias_run(bits, W, rows, n, H_packed, codes, rungs, tab, lost, scales, num_den, ws,
                    ws_bytes, as_stream(stream));
}

size_t gptq_gram_workspace_bytes(int n) { return bad_n(n) ? 0 : gram_ws_bytes(n); }

gptq_status gptq_gram_add(float* H_packed, int n, const float* X, int T, void* ws,
                          size_t ws_bytes, void* stream) {
  if (bad_n(n) || T < 0) return GPTQ_ERR_SHAPE;
  if (!ptr_ok(H_packed) || (T > 0 && !ptr_ok(X)) || ws == nullptr) return GPTQ_ERR_ARG;
  if (ws_bytes < gram_ws_bytes(n)) return GPTQ_ERR_NOMEM;
  if (T == 0) return GPTQ_OK;
  return gram_run(H_packed, n, X, T, ws, ws_bytes, as_stream(stream));
}

gptq_status gptq_act_order_perm(const float* hdiag, int n, int* perm, void* stream) {
  if (bad_n(n)) return GPTQ_ERR_SHAPE;
  if (!ptr_ok(hdiag) || !ptr_ok(perm)) return GPTQ_ERR_ARG;
  return perm_run(hdiag, n, perm, as_stream(stream));
}

gptq_status gptq_fold_permuted(const float* H_packed, int n, double lambda, const int* perm,
                               float* U, float* D, float* hdiag, double* lambda_used, void* ws,
                               size_t ws_bytes, void* stream) {
  if (bad_n(n)) return GPTQ_ERR_SHAPE;
  if (!ptr_ok(H_packed) || !ptr_ok(perm) || !ptr_ok(U) || !opt_ok(D) || !opt_ok(hdiag) ||
      ws == nullptr)
    return GPTQ_ERR_ARG;
  if (!isfinite(lambda)) return GPTQ_ERR_ARG;
  if (ws_bytes < fold_ws_bytes(n)) return GPTQ_ERR_NOMEM;
  return fold_run(H_packed, n, lambda, U, D, hdiag, lambda_used, ws, ws_bytes, as_stream(stream),
                  perm);
}

gptq_status gptq_static_rungs(const float* W, int rows, int n, const float* tab, const float* lost,
                              uint8_t* rungs, float* scales, void* stream) {
  if (bad_n(n) || bad_rows(rows) || n % GPTQ_GROUP != 0) return GPTQ_ERR_SHAPE;
  if (!ptr_ok(W) || !ptr_ok(tab) || !ptr_ok(lost) || rungs == nullptr || !ptr_ok(scales))
    return GPTQ_ERR_ARG;
  return static_rungs_run(W, rows, n, tab, lost, rungs, scales, as_stream(stream));
}

size_t gptq_sweep_act_order_workspace_bytes(int rows, int n) {
  if (bad_n(n) || bad_rows(rows)) return 0;
  return sweep_act_ws_bytes(rows, n);
}

gptq_status gptq_q4tp_sweep_act_order(const float* W, int rows, int n, const float* U,
                                      const int* perm, const float* tab, const uint8_t* rungs,
                                      uint8_t* nibbles, void* ws, size_t ws_bytes, void* stream) {
  if (bad_n(n) || bad_rows(rows) || n % GPTQ_GROUP != 0) return GPTQ_ERR_SHAPE;
  if (!ptr_ok(W) || !ptr_ok(U) || !ptr_ok(perm) || !ptr_ok(tab) || rungs == nullptr ||
      !ptr_ok(nibbles) || ws == nullptr)
    return GPTQ_ERR_ARG;
  if (ws_bytes < sweep_act_ws_bytes(rows, n)) return GPTQ_ERR_NOMEM;
  return sweep_act_run(W, rows, n, U, perm, tab, rungs, nibbles, ws, ws_bytes, as_stream(stream));
}

size_t gptq_group_act_order_workspace_bytes(int rows, int n) {
  if (bad_n(n) || bad_rows(rows)) return 0;
  const size_t f = fold_ws_bytes(n), sw = sweep_act_ws_bytes(rows, n);
  const size_t own = round_up((size_t)n * n * 4, 256) + 4 * round_up((size_t)n * 4, 256) +
                     round_up((size_t)rows * n * 4, 256) + round_up((size_t)rows * 32 * 4, 256) +
                     round_up((size_t)rows * 2 * 4, 256) + 1024;
  return own + (f > sw ? f : sw);
}

gptq_status gptq_quantize_group_act_order(const float* H_packed, int n, double lambda,
                                          const float* W, int rows, uint8_t* nibbles,
                                          uint8_t* rungs, float* scales, int* perm_out, float* U,
                                          double* lambda_used, void* ws, size_t ws_bytes,
                                          void* stream) {
  if (bad_n(n) || bad_rows(rows) || n % GPTQ_GROUP != 0) return GPTQ_ERR_SHAPE;
  if (!ptr_ok(H_packed) || !ptr_ok(W) || !ptr_ok(nibbles) || rungs == nullptr ||
      !ptr_ok(scales) || !opt_ok(perm_out) || !opt_ok(U) || ws == nullptr)
    return GPTQ_ERR_ARG;
  if (!isfinite(lambda)) return GPTQ_ERR_ARG;
  if (ws_bytes < gptq_group_act_order_workspace_bytes(rows, n)) return GPTQ_ERR_NOMEM;
  cudaStream_t s = as_stream(stream);
  Carve c(ws, ws_bytes);
  float* u = U ? U : c.take<float>((size_t)n * n);
  int* perm = perm_out ? perm_out : c.take<int>((size_t)n);
  float* hraw = c.take<float>((size_t)n);
  float* hperm = c.take<float>((size_t)n);
  float* d = c.take<float>((size_t)n);
  float* wz = c.take<float>((size_t)rows * n);
  float* tb = c.take<float>((size_t)rows * 32);
  float* ls = c.take<float>((size_t)rows * 2);
  if (!c.ok) return GPTQ_ERR_NOMEM;
  const size_t off = round_up(c.off, 256);
  void* rest = static_cast<char*>(ws) + off;
  const size_t rest_bytes = ws_bytes - off;
  GQ_TRY(diag_run(H_packed, n, hraw, s));
  GQ_TRY(perm_run(hraw, n, perm, s));
  GQ_TRY(fold_run(H_packed, n, lambda, u, d, hperm, lambda_used, rest, rest_bytes, s, perm));
  GQ_TRY(copy_ladder_run(W, rows, n, hraw, wz, tb, ls, s));
  GQ_TRY(static_rungs_run(wz, rows, n, tb, ls, rungs, scales, s));
  return sweep_act_run(wz, rows, n, u, perm, tb, rungs, nibbles, rest, rest_bytes, s);
}

}  // extern "C"
