// Cholesky factor and inverse of one NB x NB diagonal block (the fold's
// diagonal-block step), shared by the standalone kernel (first block) and
// the update GEMM, which runs it on the block its first tile just finished.
#pragma once

#include "common.cuh"

namespace gq {

constexpr int LDS = NB + 1;
constexpr int POTRF_SMEM_BYTES = 3 * NB * LDS * 4;

// Cholesky of the NB x NB diagonal block at k (lower) in shared memory, and
// its inverse.  Factorization in 32-column panels: warp 0 factors the
// panel's 32 x 32 diagonal block in registers (lane = row; the pivot column
// travels by shuffles; reciprocal square root, no divisions), the rows below
// are solved against it (one thread per row), then a rank-32 update of the
// rest of the block (4 x 4 register tiles).  Pivot test of the fold page's
// chol_diag: !(piv > 0) (NaN included) -> flag, piv := 1.
// Inverse ([fold page] inv_diag, blocked): each 32 x 32 diagonal block comes
// out of its panel's triangular solve (identity rows solved beside the rows
// below), then the off-diagonal blocks by block diagonals: X_ij = -X_ii
// sum_{j <= m < i} L_im X_mj, as register-tiled block products.  Loops stay
// rolled where unrolling buys little: the step runs once per block column on
// whichever SM its CTA lands on, mostly from a cold instruction cache.
// Output: Linv itself as its TF32 hi/lo split (NB x NB row-major each):
// the K-major operand of the panel product on the tensor cores.  Only the
// 32 x 32 blocks on and below the block diagonal are written (zeros above
// the diagonal inside the diagonal blocks); the rest is never read.
// Runs on the whole CTA (any multiple of 32 threads >= 128); S is at least
// POTRF_SMEM_BYTES of shared memory.  The block starts at Ablk (leading
// dimension lda); it is read with L1-bypassing loads.
static __device__ __noinline__ void potrf_inverse_block(const float* __restrict__ Ablk, long long lda,
                                                 float* __restrict__ Lhi, float* __restrict__ Llo,
                                                 unsigned* flag, float* S) {
  float* Li = S + NB * LDS;
  float* T = Li + NB * LDS;
  __shared__ float rinv[NB];
  __shared__ __align__(16) float colbuf[2][32];
  __shared__ int bad;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int NT = blockDim.x;
  if (tid == 0) bad = 0;
  // Up to 24 float4 loads per thread, all in flight before the first store.
  {
#pragma unroll 1
    for (int b0 = 0; b0 < NB * NB / 4; b0 += 24 * NT) {
      float4 v[24];
#pragma unroll
      for (int i = 0; i < 24; ++i) {
        const int e = b0 + tid + NT * i, r = e / (NB / 4), c4 = e % (NB / 4);
        if (e < NB * NB / 4) v[i] = __ldcg(reinterpret_cast<const float4*>(Ablk + (long long)r * lda + 4 * c4));
      }
#pragma unroll
      for (int i = 0; i < 24; ++i) {
        const int e = b0 + tid + NT * i, r = e / (NB / 4), c = 4 * (e % (NB / 4));
        if (e >= NB * NB / 4) continue;
        float* dst = S + r * LDS + c;
        dst[0] = (c <= r) ? v[i].x : 0.f;
        dst[1] = (c + 1 <= r) ? v[i].y : 0.f;
        dst[2] = (c + 2 <= r) ? v[i].z : 0.f;
        dst[3] = (c + 3 <= r) ? v[i].w : 0.f;
      }
    }
  }
  __syncthreads();
  for (int p = 0; p < NB; p += 32) {
    if (warp == 0) {
      float a[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) a[j] = S[(p + lane) * LDS + p + j];
      // Column c needs only column c-1's update of itself before its pivot
      // (one shuffle); column c-1's updates of columns c+1.. are issued after
      // that pivot's exchange, in the latency of its reciprocal square root,
      // reading column c-1 from a shared buffer (float4 broadcasts).  Every
      // entry still receives its updates in column order.
      // The next pivot (lane c+1's own entry minus its own square) does not
      // wait for the exchange that the other lanes need.  Lanes above a
      // column's diagonal update their (never stored) upper entries too,
      // which saves the per-entry lane test.
      float lprev = 0.f, pn = a[0];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float piv = __shfl_sync(0xffffffffu, pn, c);
        if (c > 0) {
          const float* cb = colbuf[(c - 1) & 1];
#pragma unroll
          for (int j4 = (c + 1) / 4; j4 < 8; ++j4) {
            const float4 l4 = *reinterpret_cast<const float4*>(cb + 4 * j4);
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const int j = 4 * j4 + jj;
              if (j >= c + 1) a[j] = fmaf(-lprev, lv[jj], a[j]);  // lanes < j: unused upper entries
            }
          }
        }
        if (!(piv > 0.f)) {
          piv = 1.f;
          if (lane == 0) bad = 1;
        }
        const float rs = rsqrtf(piv);
        const float lic = (lane == c) ? piv * rs : a[c] * rs;
        if (lane >= c) a[c] = lic;
        if (lane == c) rinv[p + c] = rs;
        colbuf[c & 1][lane] = lic;
        if (c + 1 < 32) {
          pn = fmaf(-lic, lic, a[c + 1]);
          const float lnc = __shfl_sync(0xffffffffu, lic, c + 1);
          a[c + 1] = (lane == c + 1) ? pn : fmaf(-lic, lnc, a[c + 1]);
        }
        __syncwarp();
        lprev = lic;
      }
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j <= lane) S[(p + lane) * LDS + p + j] = a[j];
    }
    __syncthreads();
    // Rows below the panel, L_rp = A_rp L_pp^-T, and after them 32 identity
    // rows e_t0, whose solutions are the rows of L_pp^-T, i.e. the columns of
    // X_pp = L_pp^-1 (the inverse's diagonal block, zeros above its diagonal):
    // one code path for both.
    const int nbelow = NB - p - 32;
    for (int v = tid; v < nbelow + 32; v += NT) {
      const bool unit = v >= nbelow;
      const int r = p + 32 + v, t0 = v - nbelow;
      float x[32];
#pragma unroll
      for (int t = 0; t < 32; ++t) x[t] = unit ? (t == t0 ? 1.f : 0.f) : S[r * LDS + p + t];
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int u = 0; u + 1 < t; u += 2) {
          a0 = fmaf(x[u], S[(p + t) * LDS + p + u], a0);
          a1 = fmaf(x[u + 1], S[(p + t) * LDS + p + u + 1], a1);
        }
        if (t & 1) a0 = fmaf(x[t - 1], S[(p + t) * LDS + p + t - 1], a0);
        x[t] = (x[t] - (a0 + a1)) * rinv[p + t];
      }
      if (unit) {
#pragma unroll
        for (int t = 0; t < 32; ++t) Li[(p + t) * LDS + p + t0] = x[t];
      } else {
#pragma unroll
        for (int t = 0; t < 32; ++t) S[r * LDS + p + t] = x[t];
      }
    }
    __syncthreads();
    const int m = NB - p - 32;  // rows/cols of the remaining block
    const int mt = m / 4;
    const int ntile = mt * (mt + 1) / 2;
    for (int e = tid; e < ntile; e += NT) {
      int ti = (int)((sqrtf(8.0f * (float)e + 1.0f) - 1.0f) * 0.5f);
      while ((ti + 1) * (ti + 2) / 2 <= e) ++ti;
      while (ti * (ti + 1) / 2 > e) --ti;
      const int tj = e - ti * (ti + 1) / 2;
      const int r0 = p + 32 + 4 * ti, c0 = p + 32 + 4 * tj;
      float acc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 8
      for (int t = 0; t < 32; ++t) {
        float ra[4], rb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          ra[i] = S[(r0 + i) * LDS + p + t];
          rb[i] = S[(c0 + i) * LDS + p + t];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ra[i], rb[j], acc[i][j]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (c0 + j <= r0 + i) S[(r0 + i) * LDS + c0 + j] -= acc[i][j];
    }
    __syncthreads();
  }
  if (bad && tid == 0) atomicOr(flag, 1u);
  // Off-diagonal blocks, one block diagonal d at a time: for block (i, j),
  // i = j + d, the products L_im X_mj (m = j .. i-1, each 32 x 32 x 32) go
  // to partials P in T, then X_ij = -X_ii (P_j + P_j+1 + ...), partials
  // summed in m order.  Every product is cut into 64 register tiles of
  // 4 x 4; the zero upper halves of X_jj and X_ii are simply multiplied.
  constexpr int PS = 33;  // partial row stride
#pragma unroll 1
  for (int d = 1; d < 4; ++d) {
    const int nblk = 4 - d;
    for (int tix = tid; tix < nblk * d * 64; tix += NT) {
      const int pr = tix / 64, tt = tix % 64;
      const int j = pr / d, i = j + d, m = j + pr % d;
      const int r0 = (tt / 8) * 4, c0 = (tt % 8) * 4;
      const float* Lb = S + (32 * i + r0) * LDS + 32 * m;
      const float* Xb = Li + (32 * m) * LDS + 32 * j + c0;
      float acc[4][4];
#pragma unroll
      for (int ii = 0; ii < 4; ++ii)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) acc[ii][jj] = 0.f;
#pragma unroll 8
      for (int k = 0; k < 32; ++k) {
        float av[4], bv[4];
#pragma unroll
        for (int ii = 0; ii < 4; ++ii) av[ii] = Lb[ii * LDS + k];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) bv[jj] = Xb[k * LDS + jj];
#pragma unroll
        for (int ii = 0; ii < 4; ++ii)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) acc[ii][jj] = fmaf(av[ii], bv[jj], acc[ii][jj]);
      }
      float* P = T + pr * 32 * PS;
#pragma unroll
      for (int ii = 0; ii < 4; ++ii)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) P[(r0 + ii) * PS + c0 + jj] = acc[ii][jj];
    }
    __syncthreads();
    for (int tix = tid; tix < nblk * 64; tix += NT) {
      const int j = tix / 64, tt = tix % 64, i = j + d;
      const int r0 = (tt / 8) * 4, c0 = (tt % 8) * 4;
      const float* Xa = Li + (32 * i + r0) * LDS + 32 * i;
      const float* P = T + j * d * 32 * PS + c0;
      float acc[4][4];
#pragma unroll
      for (int ii = 0; ii < 4; ++ii)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) acc[ii][jj] = 0.f;
#pragma unroll 4
      for (int k = 0; k < 32; ++k) {
        float av[4], bv[4];
#pragma unroll
        for (int ii = 0; ii < 4; ++ii) av[ii] = Xa[ii * LDS + k];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          float t = P[k * PS + jj];
#pragma unroll
          for (int q = 1; q < 3; ++q)
            if (q < d) t += P[q * 32 * PS + k * PS + jj];
          bv[jj] = t;
        }
#pragma unroll
        for (int ii = 0; ii < 4; ++ii)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) acc[ii][jj] = fmaf(av[ii], bv[jj], acc[ii][jj]);
      }
#pragma unroll
      for (int ii = 0; ii < 4; ++ii)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) Li[(32 * i + r0 + ii) * LDS + 32 * j + c0 + jj] = -acc[ii][jj];
    }
    __syncthreads();
  }
  // The ten 32 x 32 blocks on and below the block diagonal, four columns of
  // a row per item; the diagonal blocks hold exact zeros above the diagonal
  // (their identity rows' substitution starts with zeros).  The six blocks
  // above are never read: the panel product loads, for each 32-wide slice
  // of u, only the rows of Linv at or below that slice's diagonal block.
  for (int e = tid; e < 10 * 32 * 8; e += NT) {
    const int b = e >> 8, w = e & 255;
    const int bi = b >= 6 ? 3 : b >= 3 ? 2 : b >= 1 ? 1 : 0;
    const int bj = b - bi * (bi + 1) / 2;
    const int r = 32 * bi + (w >> 3), c = 32 * bj + 4 * (w & 7);
    const float* src = Li + r * LDS + c;
    float4 h, l;
    split_tf32(src[0], h.x, l.x);
    split_tf32(src[1], h.y, l.y);
    split_tf32(src[2], h.z, l.z);
    split_tf32(src[3], h.w, l.w);
    *reinterpret_cast<float4*>(Lhi + r * NB + c) = h;
    *reinterpret_cast<float4*>(Llo + r * NB + c) = l;
  }
}


}  // namespace gq
