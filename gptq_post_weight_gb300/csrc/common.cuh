// Shared definitions for the GB300 GPTQ fold + q4tp sweep kernels.
//
// Citations in these sources: [fold page] = cortiq-engine
// src/gpu_wgpu/gptq_dev.rs (module doc steps 1-5, WGSL kernels, host fns
// fold / fold_inner / sweep); [host page] = cortiq-cli src/gptq.rs (host
// fold gptq_fold_operator_par, host sweeps gptq_quantize_q4tp / _q2tp, the
// debias and calibration functions).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>

#include <mutex>

#include "../../include/gptq_fold.h"

namespace gq {

// Column block of the fold's right-looking Cholesky / inverse.  The working
// matrix is padded to a multiple of it (padding = identity, decoupled).
constexpr int NB = 128;
// Column block of the sweep's lazy trailing update (4 groups of 32).
constexpr int SB = 128;
constexpr int GROUP = 32;

#define GQ_CUDA(expr)                                   \
  do {                                                  \
    cudaError_t _e = (expr);                            \
    if (_e != cudaSuccess) return GPTQ_ERR_CUDA;        \
  } while (0)

#define GQ_LAUNCHED()                                   \
  do {                                                  \
    cudaError_t _e = cudaGetLastError();                \
    if (_e != cudaSuccess) return GPTQ_ERR_CUDA;        \
  } while (0)

#define GQ_TRY(expr)                                    \
  do {                                                  \
    gptq_status _s = (expr);                            \
    if (_s != GPTQ_OK) return _s;                       \
  } while (0)

// Kernel kinds for launch accounting / per-kind timing (gptq_profile_*).
enum Kind : int {
  K_DIAG = 0, K_BUILD, K_POTRF, K_TRSM, K_FOLD_GEMM, K_LADDER, K_SWEEP_BLOCK, K_PREP_UT,
  K_SWEEP_GEMM, K_GROUP, K_COPY, K_GRAM_PREP, K_GRAM_GEMM, K_PLACE, K_DEBIAS, K_DEBIAS_GEMM, K_FOLD_STRIP, K_NKINDS
};

// Every launch site calls prof_begin/prof_end around its <<<>>>: they count
// launches and, while profiling is on, record a CUDA event pair.
void prof_begin(int kind, cudaStream_t s);
void prof_end(int kind, cudaStream_t s);

struct ProfScope {
  int kind;
  cudaStream_t s;
  ProfScope(int k, cudaStream_t st) : kind(k), s(st) { prof_begin(k, st); }
  ~ProfScope() { prof_end(kind, s); }
};
#define GQ_PROF(kind, stream) ::gq::ProfScope _gq_prof_scope_(kind, stream)

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }


// Streaming multiprocessors of the current device (queried once).
int num_sms();

// Limit of every bounded device wait (globaltimer ns) and a test hook:
// with no_loads set, the GEMM producers issue no loads, so the consumers'
// waits run out and the launch reports a timeout (status bit 1) without any
// fault.  wait_cfg() is the current setting (default: 2 s, loads issued),
// changed only by gptq_test_set_wait.
struct WaitCfg {
  unsigned long long ns;
  int no_loads;
};
WaitCfg wait_cfg();

// The calling thread's current CUDA context (driver handle), or null when
// none can be had.  A device reset ends a context; the next one differs.
CUcontext current_context();

// Set-up that must run once per device and context (kernel attributes,
// device symbol addresses): run() calls `f` with the device current, the
// first time it sees the calling thread's (device, context), and again
// after that device's context has changed; concurrent first calls from
// several host threads serialise on the mutex.  A failed `f` is retried on
// the next call.
struct DeviceOnce {
  static constexpr int kMaxDevices = 64;
  std::mutex mu;
  CUcontext ctx[kMaxDevices] = {};
  template <class F>
  gptq_status run(F&& f) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GPTQ_ERR_CUDA;
    std::lock_guard<std::mutex> lk(mu);
    const CUcontext cur = current_context();
    if (cur != nullptr && ctx[dev] == cur) return GPTQ_OK;
    const gptq_status st = f(dev);
    // `f` made the runtime bind the device's context to this thread, if it
    // was not yet; a null context is simply looked up again next time.
    if (st == GPTQ_OK) ctx[dev] = current_context();
    return st;
  }
};

// Bump allocator over the caller's workspace (256-byte aligned pieces).
struct Carve {
  char* base;
  size_t cap;
  size_t off = 0;
  bool ok = true;
  Carve(void* b, size_t c) : base(static_cast<char*>(b)), cap(c) {}
  template <class T>
  T* take(size_t count) {
    size_t o = round_up(off, 256);
    size_t bytes = round_up(count * sizeof(T), 256);
    if (base == nullptr || o + bytes > cap) {
      ok = false;
      off = o + bytes;
      return nullptr;
    }
    off = o + bytes;
    return reinterpret_cast<T*>(base + o);
  }
};

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// GEMM job for the tensor-core kernel: C[r][s] -= sum_t A[r][t] * B[s][t]
// over a set of 128x128 tiles.  A and B are K-major (row-major, contraction
// index contiguous, leading dimension K) and given as TF32 hi/lo pairs
// through TMA tensor maps: OperandMaps.m[a_map] / m[a_map + 1] hold A_hi /
// A_lo, likewise for B; operand row = a_row0 + tile row (b_row0 + tile col).
// C is reached through OperandMaps.c (an f32 tensor map); tile (ti, tj)
// covers C[c_y0 + 128 ti ..][c_x0 + 128 tj ..], and whatever falls outside
// the map's extent is not written (that masks ragged edges).
// mode 0: rectangle of mt x nt tiles; mode 1: lower triangle of an mt x mt
// tile grid (ti >= tj; inside a diagonal tile only r >= s is changed);
// mode 2: rectangle whose tiles with ti == tj are diagonal tiles (a strip
// of a lower triangle starting at its diagonal).
struct TcJob {
  int c_x0, c_y0;
  int a_map, b_map, a_row0, b_row0;
  int mode, mt, nt, M, N, ntiles;
  int add;  // 0: C -= A B^T; 1: C += A B^T
  // SM-pair kernel, rectangles: > 0 walks the tiles in bands of this many
  // tile rows, down each band's columns (tiles running at the same time
  // then share operand panels in L2: for long K); 0 = row by row.
  int band;
  // First column of the contraction in both operands (t = k0 .. k0 + K).
  int k0;
};

struct OperandMaps {
  CUtensorMap m[4];
  CUtensorMap c;
};

inline TcJob tc_rect(int c_x0, int c_y0, int a_map, int a_row0, int b_map, int b_row0, int M,
                     int N) {
  TcJob j{};
  j.c_x0 = c_x0; j.c_y0 = c_y0; j.a_map = a_map; j.b_map = b_map; j.a_row0 = a_row0;
  j.b_row0 = b_row0; j.mode = 0; j.M = M; j.N = N;
  j.mt = (M + 127) / 128; j.nt = (N + 127) / 128;
  j.ntiles = (M > 0 && N > 0) ? j.mt * j.nt : 0;
  return j;
}

// A strip below a diagonal: rows [0, M) by columns [0, N) of C with M >= N,
// whose top N x N square is kept to its lower triangle (tiles above the
// diagonal are not visited, the diagonal tiles are masked).  Single-SM
// kernel only.
inline TcJob tc_strip(int c_x0, int c_y0, int a_map, int a_row0, int b_map, int b_row0, int M,
                      int N) {
  TcJob j = tc_rect(c_x0, c_y0, a_map, a_row0, b_map, b_row0, M, N);
  j.mode = 2;
  if (j.ntiles > 0) j.ntiles = j.mt * j.nt - j.nt * (j.nt - 1) / 2;
  return j;
}

inline TcJob tc_lower(int c_x0, int c_y0, int map, int row0, int M) {
  TcJob j{};
  j.c_x0 = c_x0; j.c_y0 = c_y0; j.a_map = map; j.b_map = map; j.a_row0 = row0; j.b_row0 = row0;
  j.mode = 1; j.M = M; j.N = M;
  j.mt = (M + 127) / 128; j.nt = j.mt;
  j.ntiles = M > 0 ? j.mt * (j.mt + 1) / 2 : 0;
  return j;
}

// Maps of the fold's panel product on the tensor cores (apply_tc.cu): the
// working matrix A (box 32 x 128, as for a C map), the TF32 pair of the
// diagonal block's inverse (NB x NB each, operand maps with boxes of 32
// rows), and the panel buffers P hi/lo, Yp hi/lo (p.m[0..3], operand maps).
struct ApplyMaps {
  CUtensorMap a, lhi, llo;
  OperandMaps p;
};
gptq_status apply_tc_run(const ApplyMaps& am, int k, int s0, int N, int col0, int zero_end, unsigned* flag,
                         float* U, const float* dsg, int n, cudaStream_t s);

// Tensor map over the f32 matrix C [rows][cols] (leading dimension ld) for
// the GEMM's reduce-add epilogue (box 32 x 128, 128-byte swizzle).
gptq_status make_c_map(CUtensorMap* m, float* base, long long rows, long long cols, long long ld);

// Tensor map over a K-major f32 operand array [rows][K] (box 32 x box_rows,
// 128 rows unless given; 128-byte swizzle).  K must be a multiple of 32,
// base 16-byte aligned, box_rows a multiple of 8 up to 256.
gptq_status make_operand_map(CUtensorMap* m, const float* base, long long rows, int K, int box_rows = 128);

// Diagonal-block step fused into an update (fold only): the block at (k, k)
// of the N x N matrix A (leading dimension lda) must be tile 0 of job 0; its
// Cholesky inverse goes, as a TF32 hi/lo pair (row-major), to Lhi / Llo and
// a bad pivot to bit 0 of the status word.
// on: 0 none; kFusedStep: the launch runs the step after tile 0;
// kSkipTile0 (single-SM kernel only): the launch skips tile 0, which another
// launch runs (and the step after it), and leaves that launch one SM.
constexpr int kFusedStep = 1, kSkipTile0 = 2;
struct FusedPotrf {
  const float* A;
  long long lda;
  int k;
  float* Lhi;
  float* Llo;
  int on;
};

// The same on pairs of SMs (gemm_pair.cu): tiles of 256 x 256, each shared by
// the two CTAs of a cluster; for large updates.  Tile 0 of a fused job is
// the 256 x 256 block at the job's origin (its first 128 rows and columns
// hold the diagonal block).
gptq_status gemm_pair_sub(const OperandMaps& maps, const TcJob& j0, const TcJob& j1, int K,
                          const unsigned* flag, unsigned* status, int kind, cudaStream_t s,
                          const FusedPotrf& fp = FusedPotrf{}, int kseg = 0);

// Enqueue C -= A B^T for up to two jobs in one persistent launch.
// `flag`: skip everything when non-zero (may be null).  `status`: bit 1 is
// set if a device-side wait timed out.
// kseg > 0: drain the accumulator to C every kseg (multiple of 32) of K.
gptq_status gemm_tc_sub(const OperandMaps& maps, const TcJob& j0, const TcJob& j1, int K,
                        const unsigned* flag, unsigned* status, int kind, cudaStream_t s,
                        const FusedPotrf& fp = FusedPotrf{}, int kseg = 0);

// A non-blocking side stream and two events for one call (fork: main ->
// side, join: side -> main), released when the call returns; the side
// stream's work is always joined back into the main stream before that.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  gptq_status init() {
    GQ_CUDA(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking));
    GQ_CUDA(cudaEventCreateWithFlags(&fork, cudaEventDisableTiming));
    GQ_CUDA(cudaEventCreateWithFlags(&join, cudaEventDisableTiming));
    return GPTQ_OK;
  }
  // Drops the handles without releasing them (their context is gone).
  void forget() { s = nullptr, fork = join = nullptr; }
  SideStream() = default;
  SideStream(const SideStream&) = delete;
  SideStream& operator=(const SideStream&) = delete;
  ~SideStream() {
    if (join) cudaEventDestroy(join);
    if (fork) cudaEventDestroy(fork);
    if (s) cudaStreamDestroy(s);
  }
};

// The damping schedule after a failed attempt ([fold page] the pivot flag
// and the host retry): 0 -> 1e-4, else x10.
inline double next_lambda(double lam) { return lam == 0.0 ? 1e-4 : lam * 10.0; }

// Whether per-launch profiling is recording (launches must then run one by
// one), and launches replayed from a captured graph, for the launch count.
bool prof_active();
void prof_add_launches(long long n);

// TF32 split: hi = x rounded to TF32 (10-bit mantissa, nearest, ties away),
// lo = (x - hi) rounded to TF32; x - hi is exact in f32.
__device__ __forceinline__ float tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}
// 16-byte global -> shared copy that bypasses registers (both addresses
// 16-byte aligned); completion: cp_async_wait_all() in the issuing thread,
// then a barrier before other threads read it.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

// q2tp level code clamp(round_half_even(clamp(x, -1, 4)), 0, 3) ([fold page]
// WGSL q2_level).  The inner clamp changes no result (rint of anything below
// -1 is <= -1, of anything above 4 is >= 4, and CUDA's fmaxf maps a NaN to 0
// either way), so it is left out.
__device__ __forceinline__ float q2_code(float x) { return fminf(fmaxf(rintf(x), 0.f), 3.f); }

__device__ __forceinline__ void split_tf32(float x, float& hi, float& lo) {
  hi = tf32_rna(x);
  lo = tf32_rna(x - hi);
}

}  // namespace gq
