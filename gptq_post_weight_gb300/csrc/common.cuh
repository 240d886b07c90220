// Shared definitions for the GB300 GPTQ fold + q4tp sweep kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>

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
  K_DIAG = 0, K_BUILD, K_POTRF, K_TRSM_PANEL, K_TRSM_INV, K_FOLD_GEMM, K_LADDER, K_SWEEP_BLOCK,
  K_PREP_UT, K_SWEEP_GEMM, K_GROUP, K_COPY, K_NKINDS
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

// GEMM job: C[r][s] -= sum_t A[r][t] * B[s][t] over a set of 128x128 tiles.
// A and B are K-major (row-major with the contraction index contiguous).
// mode 0: rectangle of mt x nt tiles (row-major order); mode 1: lower
// triangle of an mt x mt tile grid (tiles with ti >= tj; inside a diagonal
// tile only r >= s is written).  Rows >= M or columns >= N are masked.
struct GemmJob {
  float* C;
  const float* A;
  const float* B;
  long long ldc, lda, ldb;
  int mode, mt, nt, M, N, ntiles;
};

inline GemmJob gemm_rect(float* C, long long ldc, const float* A, long long lda, const float* B,
                         long long ldb, int M, int N) {
  GemmJob j{};
  j.C = C; j.A = A; j.B = B; j.ldc = ldc; j.lda = lda; j.ldb = ldb;
  j.mode = 0; j.M = M; j.N = N;
  j.mt = (M + 127) / 128; j.nt = (N + 127) / 128;
  j.ntiles = (M > 0 && N > 0) ? j.mt * j.nt : 0;
  return j;
}

inline GemmJob gemm_lower(float* C, long long ldc, const float* A, long long lda, int M) {
  GemmJob j{};
  j.C = C; j.A = A; j.B = A; j.ldc = ldc; j.lda = lda; j.ldb = lda;
  j.mode = 1; j.M = M; j.N = M;
  j.mt = (M + 127) / 128; j.nt = j.mt;
  j.ntiles = M > 0 ? j.mt * (j.mt + 1) / 2 : 0;
  return j;
}

// Enqueue C -= A B^T for up to two jobs in one launch (K = contraction
// length, multiple of 32).  `flag` (device, may be null): skip all work when
// non-zero.
gptq_status gemm_sub(const GemmJob& j0, const GemmJob& j1, int K, const unsigned* flag,
                     int kind, cudaStream_t s);

}  // namespace gq
