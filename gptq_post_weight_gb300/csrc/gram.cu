// Device Gram accumulation into the packed Hessian: H += X^T X, X [T, n]
// (tokens x channels, row-major f32), H the upper triangle by rows (the fold
// page's poff layout).  This is the calibration step in front of the fold
// (host page's calibration pass: gram_alloc / gram_add_dev per linear input).
//
// GB300 layout: tokens are taken in chunks of up to KC; each chunk is
// transposed into K-major TF32 hi/lo operands (channels x tokens), and the
// tensor-core GEMM accumulates the lower triangle of a dense N x N f32
// scratch G with C += A A^T (3xTF32, K = the chunk).  At the end the lower
// triangle of G is added, transposed through shared memory, into H_packed.
#include "common.cuh"

namespace gq {
namespace {

constexpr int KC = 4096;  // tokens per chunk (multiple of 32)
// Tokens accumulated in tensor memory before the partial sums are added to
// G (round-to-nearest): the tensor cores' f32 accumulation rounds toward
// zero, which over thousands of same-sign terms (the diagonal) would drift by
// ~1e-5..1e-4 relative; 128 tokens (48 MMAs) keep it near 3e-6.
constexpr int KSEG = 128;

__device__ __forceinline__ long long poff(long long r, long long n) { return r * (2 * n - r + 1) / 2; }

// Xt[i][t] = X[c0 + t][i] for t < kc, i < n; zero for t in [kc, K) or
// i in [n, N).  Written as the TF32 split.
__global__ void k_gram_transpose(const float* __restrict__ X, int n, int c0, int kc, int K, int N,
                                 float* __restrict__ Xt_hi, float* __restrict__ Xt_lo) {
  __shared__ float tile[32][33];
  const int i0 = blockIdx.x * 32, t0 = blockIdx.y * 32;
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int t = t0 + r, i = i0 + threadIdx.x;
    tile[r][threadIdx.x] = (t < kc && i < n) ? X[(long long)(c0 + t) * n + i] : 0.f;
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int i = i0 + r, t = t0 + threadIdx.x;
    if (i < N && t < K) {
      float h, l;
      split_tf32(tile[threadIdx.x][r], h, l);
      Xt_hi[(long long)i * KC + t] = h;
      Xt_lo[(long long)i * KC + t] = l;
    }
  }
}

// H_packed[poff(i) + j - i] += G[j][i] for i <= j < n (lower triangle of G,
// transposed through a 32 x 32 shared tile so both sides are coalesced).
__global__ void k_gram_pack(const float* __restrict__ G, long long ldg, int n,
                            float* __restrict__ Hp) {
  __shared__ float tile[32][33];
  const int i0 = blockIdx.x * 32, j0 = blockIdx.y * 32;  // tile rows j of G, cols i
  if (j0 + 31 < i0) return;  // entirely above the diagonal: nothing to add
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int j = j0 + r, i = i0 + threadIdx.x;
    tile[r][threadIdx.x] = (j < n && i < n && j >= i) ? G[(long long)j * ldg + i] : 0.f;
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int i = i0 + r, j = j0 + threadIdx.x;
    if (i < n && j < n && j >= i) Hp[poff(i, n) + (j - i)] += tile[threadIdx.x][r];
  }
}

}  // namespace

size_t gram_ws_bytes(int n) {
  const size_t N = round_up((size_t)n, NB);
  return round_up(N * N * 4, 256) + 2 * round_up(N * KC * 4, 256) + 1024;
}

gptq_status gram_run(float* Hp, int n, const float* X, int T, void* ws, size_t ws_bytes,
                     cudaStream_t s) {
  const int N = (int)round_up((size_t)n, NB);
  Carve c(ws, ws_bytes);
  float* G = c.take<float>((size_t)N * N);
  float* Xt_hi = c.take<float>((size_t)N * KC);
  float* Xt_lo = c.take<float>((size_t)N * KC);
  unsigned* status = c.take<unsigned>(4);
  if (!c.ok) return GPTQ_ERR_NOMEM;
  GQ_CUDA(cudaMemsetAsync(status, 0, sizeof(unsigned), s));
  GQ_CUDA(cudaMemsetAsync(G, 0, (size_t)N * N * 4, s));
  OperandMaps maps;  // 0/1 = Xt hi/lo (2/3 unused)
  GQ_TRY(make_operand_map(&maps.m[0], Xt_hi, N, KC));
  GQ_TRY(make_operand_map(&maps.m[1], Xt_lo, N, KC));
  maps.m[2] = maps.m[0];
  maps.m[3] = maps.m[1];
  GQ_TRY(make_c_map(&maps.c, G, N, N, N));
  const TcJob none{};
  for (int c0 = 0; c0 < T; c0 += KC) {
    const int kc = (T - c0) < KC ? (T - c0) : KC;
    const int K = (int)round_up((size_t)kc, 32);
    {
      GQ_PROF(K_GRAM_PREP, s);
      dim3 grid(N / 32, K / 32);
      k_gram_transpose<<<grid, dim3(32, 8), 0, s>>>(X, n, c0, kc, K, N, Xt_hi, Xt_lo);
      GQ_LAUNCHED();
    }
    TcJob j = tc_lower(0, 0, 0, 0, N);
    j.add = 1;  // C += A A^T
    GQ_TRY(gemm_pair_sub(maps, j, none, K, status, status, K_GRAM_GEMM, s, FusedPotrf{}, KSEG));
  }
  {
    GQ_PROF(K_GRAM_PREP, s);
    dim3 grid((n + 31) / 32, (n + 31) / 32);
    k_gram_pack<<<grid, dim3(32, 8), 0, s>>>(G, N, n, Hp);
    GQ_LAUNCHED();
  }
  unsigned hs = 0;
  GQ_CUDA(cudaMemcpyAsync(&hs, status, sizeof(unsigned), cudaMemcpyDeviceToHost, s));
  GQ_CUDA(cudaStreamSynchronize(s));
  return hs ? GPTQ_ERR_TIMEOUT : GPTQ_OK;
}

}  // namespace gq
