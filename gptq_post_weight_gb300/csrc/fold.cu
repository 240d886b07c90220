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
//   potrf(k)      factor and invert the diagonal block (one CTA, shared
//                 memory) -> L_kk^-1 as a TF32 pair;
//   apply(k)      both triangular solves as one tensor-core product with
//                 that inverse (apply_tc.cu): the panel L[i, k-block] for i
//                 below -> panel buffer P; the inverse's block row
//                 X[k-block, c] for c < k+NB (rows of Y) -> panel buffer Yp,
//                 and the finished entries of U;
//   update(k)     A[i][j] -= P_i P_j^T (lower tiles, i, j >= k+NB) and
//                 Y[c][i] -= Yp_c P_i^T (c < k+NB <= i): one GEMM launch.
// A pivot that is not positive (or NaN) sets a device flag; every later
// kernel of the attempt returns at once, and the host raises lambda.
#include "common.cuh"
#include "potrf.cuh"

#include <math.h>

namespace gq {
namespace {


__device__ __forceinline__ long long poff(long long r, long long n) { return r * (2 * n - r + 1) / 2; }

__device__ __forceinline__ bool flagged(const unsigned* flag) {
  return *(volatile const unsigned*)flag != 0u;
}

// Raw diagonal and dead mask, one channel per thread, and each CTA's part of
// the f64 sum behind base = max(mean(diag with dead := 1), 1e-12), summed
// in a fixed order.  [fold page] diag_get and fold_inner's host lines;
// [host page] gptq_fold_operator_par.
// With a permutation (act order), position i holds channel perm[i].
constexpr int DIAG_T = 256;

__global__ void __launch_bounds__(DIAG_T) k_diag(const float* __restrict__ hp, int n,
                                                 const int* __restrict__ perm,
                                                 float* __restrict__ hdiag,
                                                 double* __restrict__ part) {
  __shared__ double red[DIAG_T];
  const int i = blockIdx.x * DIAG_T + threadIdx.x;
  double v = 0.0;
  if (i < n) {
    const int ch = perm ? perm[i] : i;
    const float h = hp[poff(ch, n)];
    hdiag[i] = h;
    v = (h > 0.f) ? (double)h : 1.0;
  }
  red[threadIdx.x] = v;
  __syncthreads();
  for (int s = DIAG_T / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) part[blockIdx.x] = red[0];
}

// base from k_diag's parts (fixed order); every CTA of k_dvec forms it.
__device__ double diag_base(const double* __restrict__ part, int n) {
  __shared__ double red[DIAG_T];
  const int nparts = (n + DIAG_T - 1) / DIAG_T;
  double acc = 0.0;
  for (int p = threadIdx.x; p < nparts; p += DIAG_T) acc += part[p];
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int s = DIAG_T / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  const double mean = red[0] / (double)n;
  return mean > 1e-12 ? mean : 1e-12;
}

// U's strict lower block triangle, the entries no panel-product store
// reaches: U row u holds fold row i = n-1-u of block k = NB floor(i / NB),
// whose store writes the columns from n - k - NB on.
__global__ void __launch_bounds__(256) k_zero_lower(float* __restrict__ U, int n, int vec4) {
  const int u = blockIdx.x;
  const int i = n - 1 - u;
  const int end = n - (i / NB) * NB - NB;  // columns [0, end)
  if (end <= 0) return;
  float* row = U + (long long)u * n;
  int c0 = 0;
  if (vec4) {
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    c0 = end & ~3;
    for (int c = 4 * threadIdx.x; c < c0; c += 4 * blockDim.x) __stcs(reinterpret_cast<float4*>(row + c), z);
  }
  for (int c = c0 + threadIdx.x; c < end; c += blockDim.x) row[c] = 0.f;
}

// Per attempt: d_k = sqrt(H_kk + damp) and, for a dead channel, the fold
// page's signed D: -sqrt(1 + damp) (make_u divides by |d|; the builder
// never uses |d| of a dead row/column).  The working copy keeps the sign,
// so one load tells the builder both |d| and deadness.
__global__ void __launch_bounds__(DIAG_T) k_dvec(int n, const float* __restrict__ hdiag,
                                                 const double* __restrict__ part, double lam,
                                                 float* __restrict__ Dsigned, float* __restrict__ dsg,
                                                 double* __restrict__ base_out) {
  const double base = diag_base(part, n);
  if (blockIdx.x == 0 && threadIdx.x == 0) *base_out = base;
  const int i = blockIdx.x * DIAG_T + threadIdx.x;
  if (i >= n) return;
  const double damp = lam * base;
  const float h = hdiag[i];
  const bool dead = !(h > 0.f);
  const float d = dead ? -(float)sqrt(1.0 + damp) : (float)sqrt((double)h + damp);
  if (Dsigned) Dsigned[i] = d;
  dsg[i] = d;
}

// One row i of A: lower part = equilibrated reversed damped H, upper part
// zero (initial Y), padding rows identity.  [fold page] build_a.  With a
// permutation (act order, host page's permute_sym) the matrix is
// H[perm][perm]: its entries are gathered from the packed triangle.
// Each thread fills four consecutive columns per pass (their packed-H and
// d loads in flight together) and stores them as one float4; the packed
// row is read once (streaming) and A written once (streaming).
__global__ void __launch_bounds__(256) k_build(const float* __restrict__ hp, int n, int N,
                                               const int* __restrict__ perm,
                                               const double* __restrict__ base, double lam,
                                               const float* __restrict__ dsg,
                                               float* __restrict__ A, long long lda,
                                               int write_upper) {
  const int i = blockIdx.x;
  float* arow = A + (long long)i * lda;
  if (i >= n) {
    for (int j = threadIdx.x; j < N; j += blockDim.x)
      if (write_upper || j <= i) arow[j] = (j == i) ? 1.f : 0.f;
    return;
  }
  const float dampf = (float)(lam * (*base));
  const int ii = n - 1 - i;
  const float sdi = dsg[ii];
  const bool dead_i = sdi < 0.f;
  const float di = fabsf(sdi);
  const long long prow = poff(ii, n);
  const int jend = write_upper ? N : i + 1;
  // Columns j > i are zero (the upper part and the padding); the lower part
  // needs H[ii][jj], jj = n-1-j >= ii.
  auto entry = [&](int j) -> float {
    if (j > i) return 0.f;
    const int jj = n - 1 - j;  // jj >= ii
    const float sdj = dsg[jj];
    if (dead_i || sdj < 0.f) return (ii == jj) ? 1.f : 0.f;
    float h;
    if (perm) {
      const int pa = perm[ii], pb = perm[jj];
      const int a = pa < pb ? pa : pb, b = pa < pb ? pb : pa;
      h = __ldcs(hp + poff(a, n) + (b - a));
    } else {
      h = __ldcs(hp + prow + (jj - ii));
    }
    if (ii == jj) h = __fadd_rn(h, dampf);
    return __fdiv_rn(h, __fmul_rn(di, sdj));
  };
  if ((lda & 3) == 0) {
    // Four columns per thread and pass; lda is a multiple of 4, so the
    // float4 stores are aligned.
    for (int j0 = 4 * threadIdx.x; j0 < jend; j0 += 4 * blockDim.x) {
      float4 v;
      v.x = entry(j0);
      v.y = j0 + 1 < jend ? entry(j0 + 1) : 0.f;
      v.z = j0 + 2 < jend ? entry(j0 + 2) : 0.f;
      v.w = j0 + 3 < jend ? entry(j0 + 3) : 0.f;
      if (j0 + 3 < jend) {
        __stcs(reinterpret_cast<float4*>(arow + j0), v);
      } else {
        arow[j0] = v.x;
        if (j0 + 1 < jend) arow[j0 + 1] = v.y;
        if (j0 + 2 < jend) arow[j0 + 2] = v.z;
      }
    }
  } else {
    for (int j = threadIdx.x; j < jend; j += blockDim.x) arow[j] = entry(j);
  }
}

// Standalone launch of the diagonal-block step.
__global__ void __launch_bounds__(256) k_potrf(const float* __restrict__ A, long long lda, int k,
                                               float* __restrict__ Lhi, float* __restrict__ Llo,
                                               unsigned* flag) {
  if (flagged(flag)) return;
  extern __shared__ float S[];
  potrf_inverse_block(A + (long long)k * lda + k, lda, Lhi, Llo, flag, S);
}

// Steps go in groups of up to FG blocks: the panel buffers hold a group's
// panels side by side (step i of the group in columns [i NB, (i+1) NB)), so
// that the trailing matrix is updated once per group with K = FG NB.  The
// panel product that fills them is apply_tc.cu.
constexpr int FG = 4;
constexpr int PW = FG * NB;

// Act-order channel order ([host page] act_order_perm): descending H_ii in
// Rust's total order on f32 (NaN and -0.0 ordered), ties by ascending index.
// Each thread ranks one channel against all others (keys staged in shared
// memory) and writes perm[rank] = channel.
__device__ __forceinline__ int total_key(float x) {
  const int b = __float_as_int(x);
  return b < 0 ? (b ^ 0x7FFFFFFF) : b;
}

__global__ void __launch_bounds__(256) k_perm_rank(const float* __restrict__ hdiag, int n,
                                                   int* __restrict__ perm) {
  __shared__ int keys[2048];
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const int ki = i < n ? total_key(hdiag[i]) : 0;
  int rank = 0;
  for (int base = 0; base < n; base += 2048) {
    const int m = (n - base) < 2048 ? (n - base) : 2048;
    __syncthreads();
    for (int e = threadIdx.x; e < m; e += blockDim.x) keys[e] = total_key(hdiag[base + e]);
    __syncthreads();
    if (i < n) {
      for (int e = 0; e < m; ++e) {
        const int kj = keys[e], j = base + e;
        rank += (kj > ki) || (kj == ki && j < i);
      }
    }
  }
  if (i < n) perm[rank] = i;
}

}  // namespace

namespace {
__global__ void k_hdiag(const float* __restrict__ hp, int n, float* __restrict__ hdiag) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) hdiag[i] = hp[poff(i, n)];
}
}  // namespace

gptq_status diag_run(const float* hp, int n, float* hdiag, cudaStream_t s) {
  GQ_PROF(K_DIAG, s);
  k_hdiag<<<(n + 255) / 256, 256, 0, s>>>(hp, n, hdiag);
  GQ_LAUNCHED();
  return GPTQ_OK;
}

gptq_status perm_run(const float* hdiag, int n, int* perm, cudaStream_t s) {
  GQ_PROF(K_COPY, s);
  k_perm_rank<<<(n + 255) / 256, 256, 0, s>>>(hdiag, n, perm);
  GQ_LAUNCHED();
  return GPTQ_OK;
}

struct FoldWs {
  int n, N;
  float* A;       // N x N
  float* P_hi;    // N x PW   (L panels of the current group of steps, TF32 hi/lo)
  float* P_lo;
  float* Yp_hi;   // N x PW   (Y panels of the current group of steps, TF32 hi/lo)
  float* Yp_lo;
  float* Lhi;     // NB x NB: inverse of the current diagonal block of L, TF32 hi
  float* Llo;     //          and lo parts, row-major
  float* hdiag;   // n
  float* dsg;     // n: d with a dead channel's sign (see k_dvec)
  double* base;   // 1
  double* part;   // ceil(n / DIAG_T): k_diag's per-CTA sums
  unsigned* flag; // 1 (+pad)
};

static bool carve_fold(Carve& c, int n, FoldWs& w) {
  w.n = n;
  w.N = (int)round_up((size_t)n, NB);
  const size_t N = (size_t)w.N;
  w.A = c.take<float>(N * N);
  w.P_hi = c.take<float>(N * PW);
  w.P_lo = c.take<float>(N * PW);
  w.Yp_hi = c.take<float>(N * PW);
  w.Yp_lo = c.take<float>(N * PW);
  w.Lhi = c.take<float>((size_t)NB * NB);
  w.Llo = c.take<float>((size_t)NB * NB);
  w.hdiag = c.take<float>((size_t)n);
  w.dsg = c.take<float>((size_t)n);
  w.base = c.take<double>(1);
  w.part = c.take<double>((size_t)(n + DIAG_T - 1) / DIAG_T);
  w.flag = c.take<unsigned>(4);
  return c.ok;
}

size_t fold_ws_bytes(int n) {
  Carve c(nullptr, 0);
  FoldWs w;
  carve_fold(c, n, w);
  return c.off + 256;
}

constexpr int POTRF_SMEM = POTRF_SMEM_BYTES;

static gptq_status init_attrs() {
  static DeviceOnce once;
  return once.run([](int) -> gptq_status {
    GQ_CUDA(cudaFuncSetAttribute(k_potrf, cudaFuncAttributeMaxDynamicSharedMemorySize, POTRF_SMEM));
    return GPTQ_OK;
  });
}

// One factorisation attempt at damping lam: build, interleaved Cholesky +
// inverse, U.  The pivot flag is left on the device.
static gptq_status fold_attempt(const float* hp, const FoldWs& w, const ApplyMaps& am,
                                double lam, float* U, float* D, cudaStream_t s, const int* perm,
                                const SideStream& side) {
  const OperandMaps& maps = am.p;
  const int n = w.n, N = w.N;
  const long long ld = N;
  GQ_CUDA(cudaMemsetAsync(w.flag, 0, sizeof(unsigned), s));
  {
    GQ_PROF(K_BUILD, s);
    k_dvec<<<(n + DIAG_T - 1) / DIAG_T, DIAG_T, 0, s>>>(n, w.hdiag, w.part, lam, D, w.dsg, w.base);
    GQ_LAUNCHED();
    k_build<<<N, 256, 0, s>>>(hp, n, N, perm, w.base, lam, w.dsg, w.A, ld, 1);
    GQ_LAUNCHED();
  }
  // Steps go in groups of FG blocks k_0 .. k_{G-1} (k_i = k + i NB; fewer
  // at the end), s = k + G NB:
  //   apply(k_i) -> panel columns [i NB, (i+1) NB), and zeros into the Yp
  //   entries of the group's later rows (X is lower triangular);
  //   then, if a block of the group remains, the strip update of the
  //   group's remaining block columns [k_{i+1}, s) by panel i alone (K = NB):
  //   the SYRK rows from k_{i+1} down (top square kept to its lower
  //   triangle) and the inverse's rows above k_{i+1}; then the diagonal-block
  //   step of block k_{i+1};
  //   one trailing update with K = G NB (every panel of the group) for
  //   everything right of / below the group.
  // The diagonal-block step of a group's first block rides in the update
  // GEMM that finishes it (tile 0 of that GEMM is exactly that block).  A
  // later block's step runs alone on the side stream, right after a
  // one-tile launch of the strip's tile 0 (that block), while the strip's
  // other tiles run on the main stream: alone, the step's code stays warm
  // (fused into a strip it ran a quarter slower from cold instruction
  // caches).  The very first step runs alone.
  auto apply = [&](int k, int col0, int zero_end) -> gptq_status {
    return apply_tc_run(am, k, k + NB, N, col0, zero_end, w.flag, U, w.dsg, n, s);
  };
  auto fused = [&](int k) { return FusedPotrf{w.A, ld, k, w.Lhi, w.Llo, kFusedStep}; };
  auto potrf_alone = [&](int k, cudaStream_t st) -> gptq_status {
    GQ_PROF(K_POTRF, st);
    k_potrf<<<1, 256, POTRF_SMEM, st>>>(w.A, ld, k, w.Lhi, w.Llo, w.flag);
    GQ_LAUNCHED();
    return GPTQ_OK;
  };
  GQ_TRY(potrf_alone(0, s));
  // maps: 0/1 = P hi/lo, 2/3 = Yp hi/lo (K = PW wide).
  int k = 0;
  while (k < N) {
    const int G = (N - k) / NB < FG ? (N - k) / NB : FG;
    const int sg = k + G * NB;
    for (int i = 0; i < G; ++i) {
      const int ki = k + i * NB, kn = ki + NB;
      GQ_TRY(apply(ki, i * NB, sg));
      if (kn < sg) {
        const int wdt = sg - kn;
        TcJob syrk = tc_strip(kn, kn, 0, kn, 0, kn, N - kn, wdt);
        TcJob inv = tc_rect(kn, 0, 2, 0, 0, kn, kn, wdt);
        syrk.k0 = inv.k0 = i * NB;
        // Side stream: the strip's tile 0 (the diagonal block kn) and the
        // step on it, alone (its code stays warm in a small kernel); main
        // stream: the strip's other tiles; joined before the next panel
        // product.
        TcJob diag = tc_lower(kn, kn, 0, kn, NB);
        diag.k0 = i * NB;
        GQ_CUDA(cudaEventRecord(side.fork, s));
        GQ_CUDA(cudaStreamWaitEvent(side.s, side.fork, 0));
        GQ_TRY(gemm_tc_sub(maps, diag, TcJob{}, NB, w.flag, w.flag, K_FOLD_STRIP, side.s));
        GQ_TRY(potrf_alone(kn, side.s));
        GQ_CUDA(cudaEventRecord(side.join, side.s));
        FusedPotrf skip0 = fused(kn);
        skip0.on = kSkipTile0;
        GQ_TRY(gemm_tc_sub(maps, syrk, inv, NB, w.flag, w.flag, K_FOLD_STRIP, s, skip0));
        GQ_CUDA(cudaStreamWaitEvent(s, side.join, 0));
      }
    }
    if (sg < N) {
      const TcJob syrk = tc_lower(sg, sg, 0, sg, N - sg);
      const TcJob inv = tc_rect(sg, 0, 2, 0, 0, sg, sg, N - sg);
      if (G > 1) {
        GQ_TRY(gemm_pair_sub(maps, syrk, inv, G * NB, w.flag, w.flag, K_FOLD_GEMM, s, fused(sg)));
      } else {
        GQ_TRY(gemm_tc_sub(maps, syrk, inv, NB, w.flag, w.flag, K_FOLD_GEMM, s, fused(sg)));
      }
    }
    k = sg;
  }
  return GPTQ_OK;
}

// The set-up every attempt shares: diag(H), the caller's copy of it, the
// zeros of U's lower block triangle (the panel products store every other
// entry), the tensor maps of the workspace.
static gptq_status fold_setup(const float* hp, int n, float* U, float* hdiag, void* ws, size_t ws_bytes,
                              cudaStream_t s, const int* perm, FoldWs& w, ApplyMaps& am) {
  GQ_TRY(init_attrs());
  Carve c(ws, ws_bytes);
  if (!carve_fold(c, n, w)) return GPTQ_ERR_NOMEM;
  {
    GQ_PROF(K_DIAG, s);
    k_diag<<<(n + DIAG_T - 1) / DIAG_T, DIAG_T, 0, s>>>(hp, n, perm, w.hdiag, w.part);
    GQ_LAUNCHED();
  }
  if (hdiag) GQ_CUDA(cudaMemcpyAsync(hdiag, w.hdiag, (size_t)n * 4, cudaMemcpyDeviceToDevice, s));
  {
    GQ_PROF(K_DIAG, s);
    const int vec4 = (n % 4 == 0) && (reinterpret_cast<uintptr_t>(U) % 16 == 0);
    k_zero_lower<<<n, 256, 0, s>>>(U, n, vec4);
    GQ_LAUNCHED();
  }
  OperandMaps& maps = am.p;
  GQ_TRY(make_operand_map(&maps.m[0], w.P_hi, w.N, PW));
  GQ_TRY(make_operand_map(&maps.m[1], w.P_lo, w.N, PW));
  GQ_TRY(make_operand_map(&maps.m[2], w.Yp_hi, w.N, PW));
  GQ_TRY(make_operand_map(&maps.m[3], w.Yp_lo, w.N, PW));
  GQ_TRY(make_c_map(&maps.c, w.A, w.N, w.N, w.N));
  am.a = maps.c;  // the panel product loads A's vectors in the same boxes
  GQ_TRY(make_operand_map(&am.lhi, w.Lhi, NB, NB, 32));
  GQ_TRY(make_operand_map(&am.llo, w.Llo, NB, NB, 32));
  return GPTQ_OK;
}

gptq_status fold_run(const float* hp, int n, double lambda, float* U, float* D, float* hdiag,
                     double* lambda_used, void* ws, size_t ws_bytes, cudaStream_t s,
                     const int* perm) {
  FoldWs w;
  ApplyMaps am;
  GQ_TRY(fold_setup(hp, n, U, hdiag, ws, ws_bytes, s, perm, w, am));
  SideStream side;
  GQ_TRY(side.init());
  double lam = lambda > 0.0 ? lambda : 0.0;
  for (;;) {
    GQ_TRY(fold_attempt(hp, w, am, lam, U, D, s, perm, side));
    unsigned hflag = 0;
    GQ_CUDA(cudaMemcpyAsync(&hflag, w.flag, sizeof(unsigned), cudaMemcpyDeviceToHost, s));
    GQ_CUDA(cudaStreamSynchronize(s));
    if (hflag & 2u) return GPTQ_ERR_TIMEOUT;
    if (hflag == 0u) break;
    lam = next_lambda(lam);
    if (lam > 10.0) return GPTQ_ERR_NOT_SPD;
  }
  if (lambda_used) *lambda_used = lam;
  return GPTQ_OK;
}

gptq_status fold_enqueue(const float* hp, int n, double lambda, float* U, float* D, float* hdiag,
                         void* ws, size_t ws_bytes, cudaStream_t s, const SideStream& side, unsigned** flag_out) {
  FoldWs w;
  ApplyMaps am;
  GQ_TRY(fold_setup(hp, n, U, hdiag, ws, ws_bytes, s, nullptr, w, am));
  GQ_TRY(fold_attempt(hp, w, am, lambda > 0.0 ? lambda : 0.0, U, D, s, nullptr, side));
  *flag_out = w.flag;
  return GPTQ_OK;
}

gptq_status build_only(const float* hp, int n, double lambda, float* A, float* D, void* ws,
                       size_t ws_bytes, cudaStream_t s) {
  Carve c(ws, ws_bytes);
  FoldWs w;
  if (!carve_fold(c, n, w)) return GPTQ_ERR_NOMEM;
  {
    GQ_PROF(K_DIAG, s);
    k_diag<<<(n + DIAG_T - 1) / DIAG_T, DIAG_T, 0, s>>>(hp, n, nullptr, w.hdiag, w.part);
    GQ_LAUNCHED();
  }
  // Rows of the caller's n x n matrix, lower triangle only.
  GQ_PROF(K_BUILD, s);
  const double lam = lambda > 0 ? lambda : 0.0;
  k_dvec<<<(n + DIAG_T - 1) / DIAG_T, DIAG_T, 0, s>>>(n, w.hdiag, w.part, lam, D, w.dsg, w.base);
  GQ_LAUNCHED();
  k_build<<<n, 256, 0, s>>>(hp, n, n, nullptr, w.base, lam, w.dsg, A, n, 0);
  GQ_LAUNCHED();
  return GPTQ_OK;
}

}  // namespace gq
