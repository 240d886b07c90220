// The fold operator on the device: U = P X P D^-1 with X = L^-1 and
// L L^T = P D^-1 H_d D^-1 P (cortiq-engine src/gpu_wgpu/gptq_dev.rs, module
// doc steps 1-4).
//
// GB300 layout.  One padded N x N f32 working matrix A (N = n rounded up to
// NB, padding = identity) holds, at once:
//   * its lower triangle: the equilibrated, reversed, damped matrix, updated
//     in place by the right-looking SYRK until each column block is factored;
//   * its strict upper triangle: Y = X^T, the inverse being accumulated.
// Cholesky and inverse run interleaved in one right-looking loop over
// column blocks k (NB wide):
//   potrf(k)      factor the diagonal block (one CTA, shared memory);
//   trsm_panel(k) L[i, k-block] for i below (forward substitution per row)
//                 -> panel buffer P;
//   trsm_inv(k)   X[k-block, c] = L_kk^-1 X[k-block, c] for c < k+NB (rows of
//                 Y) -> panel buffer Yp, and the finished rows of U;
//   update(k)     A[i][j] -= P_i P_j^T (lower tiles, i, j >= k+NB) and
//                 Y[c][i] -= Yp_c P_i^T (c < k+NB <= i): one GEMM launch.
// A pivot that is not positive (or NaN) sets a device flag; every later
// kernel of the attempt returns at once, and the host raises lambda.
#include "common.cuh"

#include <math.h>

namespace gq {
namespace {

constexpr int LDS = NB + 1;

__device__ __forceinline__ long long poff(long long r, long long n) { return r * (2 * n - r + 1) / 2; }

__device__ __forceinline__ bool flagged(const unsigned* flag) {
  return *(volatile const unsigned*)flag != 0u;
}

// Raw diagonal, dead mask and base = max(mean(diag with dead := 1), 1e-12)
// in f64 with a fixed summation order (one CTA).  [fold page] diag_get and
// fold_inner's host lines; [host page] gptq_fold_operator_par.
__global__ void __launch_bounds__(1024) k_diag(const float* __restrict__ hp, int n,
                                               float* __restrict__ hdiag,
                                               double* __restrict__ base_out) {
  __shared__ double part[1024];
  double acc = 0.0;
  for (int i = threadIdx.x; i < n; i += 1024) {
    float h = hp[poff(i, n)];
    hdiag[i] = h;
    acc += (h > 0.f) ? (double)h : 1.0;
  }
  part[threadIdx.x] = acc;
  __syncthreads();
  for (int s = 512; s > 0; s >>= 1) {
    if (threadIdx.x < s) part[threadIdx.x] += part[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    double mean = part[0] / (double)n;
    *base_out = mean > 1e-12 ? mean : 1e-12;
  }
}

// One row i of A: lower part = equilibrated reversed damped H, upper part
// zero (initial Y), padding rows identity.  [fold page] build_a.
__global__ void __launch_bounds__(256) k_build(const float* __restrict__ hp, int n, int N,
                                               const float* __restrict__ hdiag,
                                               const double* __restrict__ base, double lam,
                                               float* __restrict__ A, long long lda,
                                               float* __restrict__ Dsigned, float* __restrict__ dabs,
                                               int write_upper) {
  const int i = blockIdx.x;
  const double damp = lam * (*base);
  const float dampf = (float)damp;
  float* arow = A + (long long)i * lda;
  if (i >= n) {
    for (int j = threadIdx.x; j < N; j += blockDim.x)
      if (write_upper || j <= i) arow[j] = (j == i) ? 1.f : 0.f;
    return;
  }
  const int ii = n - 1 - i;
  const float hii = hdiag[ii];
  const bool dead_i = !(hii > 0.f);
  if (threadIdx.x == 0) {
    float d = dead_i ? -(float)sqrt(1.0 + damp) : (float)sqrt((double)hii + damp);
    if (Dsigned) Dsigned[ii] = d;
    dabs[ii] = fabsf(d);
  }
  const float di = dead_i ? 1.f : (float)sqrt((double)hii + damp);
  const long long prow = poff(ii, n);
  for (int j = threadIdx.x; j < N; j += blockDim.x) {
    float v = 0.f;
    if (j <= i) {
      const int jj = n - 1 - j;  // jj >= ii
      const float hjj = hdiag[jj];
      const bool dead_j = !(hjj > 0.f);
      if (dead_i || dead_j) {
        v = (ii == jj) ? 1.f : 0.f;
      } else {
        float h = hp[prow + (jj - ii)];
        if (ii == jj) h = __fadd_rn(h, dampf);
        const float dj = (float)sqrt((double)hjj + damp);
        v = __fdiv_rn(h, __fmul_rn(di, dj));
      }
    } else if (!write_upper) {
      continue;
    }
    arow[j] = v;
  }
}

// Cholesky of the NB x NB diagonal block at k (lower), in shared memory:
// 32-column sub-panels, each factored by one warp, then a triangular solve
// of the rows below and a rank-32 update, all inside the CTA.  Pivot test of
// the fold page's chol_diag: !(piv > 0) (NaN included) -> flag, piv := 1.
// Output: Lkk (NB x NB, zeros above the diagonal).
__global__ void __launch_bounds__(256) k_potrf(const float* __restrict__ A, long long lda, int k,
                                               float* __restrict__ Lkk, unsigned* flag) {
  if (flagged(flag)) return;
  extern __shared__ float S[];  // [NB][LDS]
  __shared__ int bad;
  const int tid = threadIdx.x;
  if (tid == 0) bad = 0;
  for (int e = tid; e < NB * NB; e += 256) {
    const int r = e / NB, c = e % NB;
    S[r * LDS + c] = (c <= r) ? A[(long long)(k + r) * lda + k + c] : 0.f;
  }
  __syncthreads();
  for (int p = 0; p < NB; p += 32) {
    if (tid < 32) {
      const int lane = tid;
      for (int c = 0; c < 32; ++c) {
        float piv = S[(p + c) * LDS + p + c];
        if (!(piv > 0.f)) {
          piv = 1.f;
          if (lane == 0) bad = 1;
        }
        const float l = sqrtf(piv);
        __syncwarp();
        if (lane == c) S[(p + c) * LDS + p + c] = l;
        if (lane > c) S[(p + lane) * LDS + p + c] = __fdiv_rn(S[(p + lane) * LDS + p + c], l);
        __syncwarp();
        if (lane > c) {
          const float lr = S[(p + lane) * LDS + p + c];
          for (int s = c + 1; s <= lane; ++s)
            S[(p + lane) * LDS + p + s] = fmaf(-lr, S[(p + s) * LDS + p + c], S[(p + lane) * LDS + p + s]);
        }
        __syncwarp();
      }
    }
    __syncthreads();
    for (int r = p + 32 + tid; r < NB; r += 256) {
      for (int t = 0; t < 32; ++t) {
        float s = S[r * LDS + p + t];
        for (int u = 0; u < t; ++u) s = fmaf(-S[r * LDS + p + u], S[(p + t) * LDS + p + u], s);
        S[r * LDS + p + t] = __fdiv_rn(s, S[(p + t) * LDS + p + t]);
      }
    }
    __syncthreads();
    const int m = NB - p - 32;
    for (int e = tid; e < m * m; e += 256) {
      const int rr = e / m, ss = e % m;
      if (ss > rr) continue;
      const int r = p + 32 + rr, s2 = p + 32 + ss;
      float acc = 0.f;
#pragma unroll 8
      for (int t = 0; t < 32; ++t) acc = fmaf(S[r * LDS + p + t], S[s2 * LDS + p + t], acc);
      S[r * LDS + s2] -= acc;
    }
    __syncthreads();
  }
  if (bad && tid == 0) atomicOr(flag, 1u);
  for (int e = tid; e < NB * NB; e += 256) {
    const int r = e / NB, c = e % NB;
    Lkk[e] = (c <= r) ? S[r * LDS + c] : 0.f;
  }
}

// Forward substitution L_kk z = v for 128 row vectors per CTA (one thread
// each, v in registers).  MODE 0 (Cholesky panel, fold page chol_panel):
// rows i >= k+NB, v = A[i][k..k+NB), z -> P[i][*].  MODE 1 (inverse block
// row, fold page inv_diag + inv_rows): rows c < k+NB, v = Y[c][k..k+NB)
// (the unit vector e_{c-k} when c is in block k), z -> Yp[c][*] and the
// finished entries of U: U[n-1-i][n-1-c] = X[i][c] / |d_{n-1-c}|
// ([fold page] make_u), i = k + t.  z is stored as its TF32 hi/lo split,
// the operand format of the update GEMM.
template <int MODE>
__global__ void __launch_bounds__(128) k_trsm(const float* __restrict__ A, long long lda, int k,
                                              int row0, int nrows, const float* __restrict__ Lkk,
                                              float* __restrict__ out_hi, float* __restrict__ out_lo,
                                              const unsigned* flag,
                                              float* __restrict__ U, const float* __restrict__ dabs,
                                              int n) {
  if (flagged(flag)) return;
  extern __shared__ __align__(16) float Ls[];  // [NB][NB]
  for (int e = threadIdx.x; e < NB * NB / 4; e += 128)
    reinterpret_cast<float4*>(Ls)[e] = reinterpret_cast<const float4*>(Lkk)[e];
  __syncthreads();
  const int r = row0 + blockIdx.x * 128 + threadIdx.x;
  if (r >= row0 + nrows) return;
  float x[NB];
  const int unit = (MODE == 1 && r >= k) ? r - k : -1;
  if (unit >= 0) {
#pragma unroll
    for (int t = 0; t < NB; ++t) x[t] = (t == unit) ? 1.f : 0.f;
  } else {
    const float4* src = reinterpret_cast<const float4*>(A + (long long)r * lda + k);
#pragma unroll
    for (int t = 0; t < NB / 4; ++t) {
      float4 v = src[t];
      x[4 * t] = v.x; x[4 * t + 1] = v.y; x[4 * t + 2] = v.z; x[4 * t + 3] = v.w;
    }
  }
#pragma unroll
  for (int t = 0; t < NB; ++t) {
    float s = x[t];
    const float4* lrow = reinterpret_cast<const float4*>(Ls + t * NB);
#pragma unroll
    for (int u4 = 0; u4 < t / 4; ++u4) {
      float4 l = lrow[u4];
      s = fmaf(-l.x, x[4 * u4], s);
      s = fmaf(-l.y, x[4 * u4 + 1], s);
      s = fmaf(-l.z, x[4 * u4 + 2], s);
      s = fmaf(-l.w, x[4 * u4 + 3], s);
    }
#pragma unroll
    for (int u = (t / 4) * 4; u < t; ++u) s = fmaf(-Ls[t * NB + u], x[u], s);
    x[t] = __fdiv_rn(s, Ls[t * NB + t]);
  }
  if (unit >= 0) {
#pragma unroll
    for (int t = 0; t < NB; ++t)
      if (t < unit) x[t] = 0.f;
  }
  float4* dh = reinterpret_cast<float4*>(out_hi + (long long)r * NB);
  float4* dl = reinterpret_cast<float4*>(out_lo + (long long)r * NB);
#pragma unroll
  for (int t = 0; t < NB / 4; ++t) {
    float4 h, l;
    split_tf32(x[4 * t], h.x, l.x);
    split_tf32(x[4 * t + 1], h.y, l.y);
    split_tf32(x[4 * t + 2], h.z, l.z);
    split_tf32(x[4 * t + 3], h.w, l.w);
    dh[t] = h;
    dl[t] = l;
  }
  if (MODE == 1 && r < n) {
    const int m = n - 1 - r;
    const float dm = dabs[m];
#pragma unroll
    for (int t = 0; t < NB; ++t) {
      const int i = k + t;
      if (i < n) U[(long long)(n - 1 - i) * n + m] = __fdiv_rn(x[t], dm);
    }
  }
}

}  // namespace

struct FoldWs {
  int n, N;
  float* A;       // N x N
  float* P_hi;    // N x NB   (L panel of the current step, TF32 hi/lo)
  float* P_lo;
  float* Yp_hi;   // N x NB   (Y panel of the current step, TF32 hi/lo)
  float* Yp_lo;
  float* Lkk;     // NB x NB
  float* hdiag;   // n
  float* dabs;    // n
  double* base;   // 1
  unsigned* flag; // 1 (+pad)
};

static bool carve_fold(Carve& c, int n, FoldWs& w) {
  w.n = n;
  w.N = (int)round_up((size_t)n, NB);
  const size_t N = (size_t)w.N;
  w.A = c.take<float>(N * N);
  w.P_hi = c.take<float>(N * NB);
  w.P_lo = c.take<float>(N * NB);
  w.Yp_hi = c.take<float>(N * NB);
  w.Yp_lo = c.take<float>(N * NB);
  w.Lkk = c.take<float>((size_t)NB * NB);
  w.hdiag = c.take<float>((size_t)n);
  w.dabs = c.take<float>((size_t)n);
  w.base = c.take<double>(1);
  w.flag = c.take<unsigned>(4);
  return c.ok;
}

size_t fold_ws_bytes(int n) {
  Carve c(nullptr, 0);
  FoldWs w;
  carve_fold(c, n, w);
  return c.off + 256;
}

static gptq_status init_attrs() {
  static bool done = false;
  if (done) return GPTQ_OK;
  GQ_CUDA(cudaFuncSetAttribute(k_potrf, cudaFuncAttributeMaxDynamicSharedMemorySize, NB * LDS * 4));
  GQ_CUDA(cudaFuncSetAttribute(k_trsm<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, NB * NB * 4));
  GQ_CUDA(cudaFuncSetAttribute(k_trsm<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, NB * NB * 4));
  done = true;
  return GPTQ_OK;
}

// One factorisation attempt at damping lam: build, interleaved Cholesky +
// inverse, U.  The pivot flag is left on the device.
static gptq_status fold_attempt(const float* hp, const FoldWs& w, const OperandMaps& maps,
                                double lam, float* U, float* D, cudaStream_t s) {
  const int n = w.n, N = w.N;
  const long long ld = N;
  GQ_CUDA(cudaMemsetAsync(w.flag, 0, sizeof(unsigned), s));
  {
    GQ_PROF(K_BUILD, s);
    k_build<<<N, 256, 0, s>>>(hp, n, N, w.hdiag, w.base, lam, w.A, ld, D, w.dabs, 1);
    GQ_LAUNCHED();
  }
  for (int k = 0; k < N; k += NB) {
    const int s0 = k + NB;
    {
      GQ_PROF(K_POTRF, s);
      k_potrf<<<1, 256, NB * LDS * 4, s>>>(w.A, ld, k, w.Lkk, w.flag);
      GQ_LAUNCHED();
    }
    if (s0 < N) {
      GQ_PROF(K_TRSM_PANEL, s);
      k_trsm<0><<<(N - s0) / 128, 128, NB * NB * 4, s>>>(w.A, ld, k, s0, N - s0, w.Lkk, w.P_hi,
                                                         w.P_lo, w.flag, nullptr, nullptr, n);
      GQ_LAUNCHED();
    }
    {
      GQ_PROF(K_TRSM_INV, s);
      k_trsm<1><<<s0 / 128, 128, NB * NB * 4, s>>>(w.A, ld, k, 0, s0, w.Lkk, w.Yp_hi, w.Yp_lo,
                                                   w.flag, U, w.dabs, n);
      GQ_LAUNCHED();
    }
    if (s0 < N) {
      // maps: 0/1 = P hi/lo, 2/3 = Yp hi/lo.
      const TcJob syrk = tc_lower(w.A + (long long)s0 * ld + s0, ld, 0, s0, N - s0);
      const TcJob inv = tc_rect(w.A + s0, ld, 2, 0, 0, s0, s0, N - s0);
      GQ_TRY(gemm_tc_sub(maps, syrk, inv, NB, w.flag, w.flag, K_FOLD_GEMM, s));
    }
  }
  return GPTQ_OK;
}

gptq_status fold_run(const float* hp, int n, double lambda, float* U, float* D, float* hdiag,
                     double* lambda_used, void* ws, size_t ws_bytes, cudaStream_t s) {
  GQ_TRY(init_attrs());
  Carve c(ws, ws_bytes);
  FoldWs w;
  if (!carve_fold(c, n, w)) return GPTQ_ERR_NOMEM;
  {
    GQ_PROF(K_DIAG, s);
    k_diag<<<1, 1024, 0, s>>>(hp, n, w.hdiag, w.base);
    GQ_LAUNCHED();
  }
  if (hdiag) GQ_CUDA(cudaMemcpyAsync(hdiag, w.hdiag, (size_t)n * 4, cudaMemcpyDeviceToDevice, s));
  GQ_CUDA(cudaMemsetAsync(U, 0, (size_t)n * n * 4, s));
  OperandMaps maps;
  GQ_TRY(make_operand_map(&maps.m[0], w.P_hi, w.N, NB));
  GQ_TRY(make_operand_map(&maps.m[1], w.P_lo, w.N, NB));
  GQ_TRY(make_operand_map(&maps.m[2], w.Yp_hi, w.N, NB));
  GQ_TRY(make_operand_map(&maps.m[3], w.Yp_lo, w.N, NB));
  double lam = lambda > 0.0 ? lambda : 0.0;
  for (;;) {
    GQ_TRY(fold_attempt(hp, w, maps, lam, U, D, s));
    unsigned hflag = 0;
    GQ_CUDA(cudaMemcpyAsync(&hflag, w.flag, sizeof(unsigned), cudaMemcpyDeviceToHost, s));
    GQ_CUDA(cudaStreamSynchronize(s));
    if (hflag & 2u) return GPTQ_ERR_TIMEOUT;
    if (hflag == 0u) break;
    lam = (lam == 0.0) ? 1e-4 : lam * 10.0;
    if (lam > 10.0) return GPTQ_ERR_NOT_SPD;
  }
  if (lambda_used) *lambda_used = lam;
  return GPTQ_OK;
}

gptq_status build_only(const float* hp, int n, double lambda, float* A, float* D, void* ws,
                       size_t ws_bytes, cudaStream_t s) {
  Carve c(ws, ws_bytes);
  FoldWs w;
  if (!carve_fold(c, n, w)) return GPTQ_ERR_NOMEM;
  {
    GQ_PROF(K_DIAG, s);
    k_diag<<<1, 1024, 0, s>>>(hp, n, w.hdiag, w.base);
    GQ_LAUNCHED();
  }
  // Rows of the caller's n x n matrix, lower triangle only.
  GQ_PROF(K_BUILD, s);
  k_build<<<n, 256, 0, s>>>(hp, n, n, w.hdiag, w.base, lambda > 0 ? lambda : 0.0, A, n, D, w.dabs, 0);
  GQ_LAUNCHED();
  return GPTQ_OK;
}

}  // namespace gq
