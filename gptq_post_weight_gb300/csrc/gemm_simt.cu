// C -= A B^T on 128x128 tiles with f32 FMA on the CUDA cores.
//
// This is the rank-K update that every hot loop of the path reduces to: the
// Cholesky's trailing SYRK and the inverse's block update (fold page,
// chol_update / inv_update) and the sweep's trailing GEMM (q4tp_trail).
#include "common.cuh"

namespace gq {
namespace {

constexpr int TM = 128, TK = 32, PAD = 4;

__device__ __forceinline__ void tile_of(const GemmJob& J, int t, int& ti, int& tj) {
  if (J.mode == 1) {
    int i = (int)((sqrtf(8.0f * (float)t + 1.0f) - 1.0f) * 0.5f);
    while ((i + 1) * (i + 2) / 2 <= t) ++i;
    while (i * (i + 1) / 2 > t) --i;
    ti = i;
    tj = t - i * (i + 1) / 2;
  } else {
    ti = t / J.nt;
    tj = t % J.nt;
  }
}

__global__ void __launch_bounds__(256) k_gemm_simt(GemmJob j0, GemmJob j1, int K,
                                                  const unsigned* flag) {
  if (flag != nullptr && *(volatile const unsigned*)flag != 0u) return;
  int t = blockIdx.x;
  const bool second = t >= j0.ntiles;
  const GemmJob& J = second ? j1 : j0;
  if (second) t -= j0.ntiles;
  int ti, tj;
  tile_of(J, t, ti, tj);
  const int r0 = ti * TM, s0 = tj * TM;

  __shared__ __align__(16) float As[TK][TM + PAD];
  __shared__ __align__(16) float Bs[TK][TM + PAD];

  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < K; k0 += TK) {
    // 128 rows x 32 k of A and of B: 4096 floats each, 16 per thread.
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      int e = (tid + q * 256);  // float4 index, 8 per row
      int row = e >> 3, kk = (e & 7) * 4;
      float4 va = make_float4(0.f, 0.f, 0.f, 0.f), vb = va;
      if (r0 + row < J.M) va = *reinterpret_cast<const float4*>(J.A + (long long)(r0 + row) * J.lda + k0 + kk);
      if (s0 + row < J.N) vb = *reinterpret_cast<const float4*>(J.B + (long long)(s0 + row) * J.ldb + k0 + kk);
      As[kk + 0][row] = va.x; As[kk + 1][row] = va.y; As[kk + 2][row] = va.z; As[kk + 3][row] = va.w;
      Bs[kk + 0][row] = vb.x; Bs[kk + 1][row] = vb.y; Bs[kk + 2][row] = vb.z; Bs[kk + 3][row] = vb.w;
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < TK; ++kk) {
      float a[8], b[8];
      float4 a0 = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      float4 a1 = *reinterpret_cast<const float4*>(&As[kk][64 + ty * 4]);
      float4 b0 = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      float4 b1 = *reinterpret_cast<const float4*>(&Bs[kk][64 + tx * 4]);
      a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w; a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
      b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w; b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = r0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
    if (r >= J.M) continue;
    float* crow = J.C + (long long)r * J.ldc;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int s = s0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
      if (s >= J.N) continue;
      if (J.mode == 1 && ti == tj && s > r) continue;
      crow[s] -= acc[i][j];
    }
  }
}

}  // namespace

gptq_status gemm_sub(const GemmJob& j0, const GemmJob& j1, int K, const unsigned* flag,
                     int kind, cudaStream_t s) {
  const int total = j0.ntiles + j1.ntiles;
  if (total <= 0) return GPTQ_OK;
  GQ_PROF(kind, s);
  k_gemm_simt<<<total, 256, 0, s>>>(j0, j1, K, flag);
  GQ_LAUNCHED();
  return GPTQ_OK;
}

}  // namespace gq
