// The q2tp "placed" rule's own kernels: the ladder placement and the group
// rule on given tiles.  The sweep itself is the q4tp sweep's pipeline with
// the q2tp rule in its block kernel (sweep.cu).
//
// Placement ([host page] Q2tpRule::Placed, gptq_quantize_q2tp_dev: "ladders
// placed on the host from the dead-zeroed weights" at "the H_ii-weighted
// MSE-optimal group scales"; the placement and ladder functions themselves
// are not on the pages).  Reading: the group scale is the exact minimiser
// over s > 0 of E(s) = sum_t h_t (|w_t| - l_t s)^2, l_t = 1.5 if |w_t| > s
// else 0.5 (the four levels +-0.5 s, +-1.5 s of q2_level), h = H_ii clipped
// at 0.  E is continuous and piecewise quadratic; each piece is convex and
// each kink concave, so the minimum is the stationary point of one piece,
//   s_O = (0.5 sum_t h|w| + sum_O h|w|) / (0.25 sum_t h + 2 sum_O h),
// for an outer set O = the k largest |w| (k = 0..32).  The kernel scores the
// pieces in f32 and recomputes the winner's scale in f64; when the two best
// f32 scores are within the f32 error of each other, both are scored again
// in f64 (ties: the smaller scale).  A group takes part only if some
// channel has h > 0 and w != 0.  The row's ladder: lo = f16(log2 min s*),
// step = f16(max(0, (log2 max s* - lo) / 30)) (0 if min == max), rung 0 = 0,
// rung c >= 1 = f32(2^(lo + (c-1) step)); no group taking part: all zero.
#include "common.cuh"

#include <cuda_fp16.h>
#include <math.h>

namespace gq {
namespace {

constexpr int PLACE_THREADS = 128;

__device__ __forceinline__ float hclip(float h) { return h > 0.f ? h : 0.f; }

// Sort (a, h) by a, descending, in registers (bitonic network, every index
// a compile-time constant).
__device__ __forceinline__ void sort_desc(float (&a)[GROUP], float (&h)[GROUP]) {
#pragma unroll
  for (int k = 2; k <= GROUP; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
      for (int i = 0; i < GROUP; ++i) {
        const int l = i ^ j;
        if (l > i) {
          const bool sw = ((i & k) == 0) ? (a[i] < a[l]) : (a[i] > a[l]);
          const float ai = a[i], al = a[l], hi = h[i], hl = h[l];
          a[i] = sw ? al : ai;
          a[l] = sw ? ai : al;
          h[i] = sw ? hl : hi;
          h[l] = sw ? hi : hl;
        }
      }
    }
  }
}

// f64 stationary scale of the outer set = the first k of the sorted group.
__device__ double top_scale_f64(const float (&a)[GROUP], const float (&h)[GROUP], int k) {
  double ta = 0.0, th = 0.0, oa = 0.0, oh = 0.0;
#pragma unroll
  for (int t = 0; t < GROUP; ++t) {
    const double ht = h[t], ha = ht * (double)a[t];
    ta += ha;
    th += ht;
    if (t < k) {
      oa += ha;
      oh += ht;
    }
  }
  return (0.5 * ta + oa) / (0.25 * th + 2.0 * oh);
}

// E(s) in f64 (levels by |w| > s).
__device__ double err_f64(const float (&a)[GROUP], const float (&h)[GROUP], double s) {
  double e = 0.0;
#pragma unroll
  for (int t = 0; t < GROUP; ++t) {
    const double at = a[t];
    const double d = at - (at > s ? 1.5 : 0.5) * s;
    e += (double)h[t] * d * d;
  }
  return e;
}

// One block per row; thread k places groups k, k + 128, ... .  Per group:
// sort |w| (with h) descending; the piece with the k largest outer has
// B_k = sum h|w| l = 0.5 sum h|w| + sum_top-k h|w|, C_k = sum h l^2 = 0.25
// sum h + 2 sum_top-k h, stationary point s_k = B_k / C_k and there
// E = sum h w^2 - B_k s_k; it counts when s_k lies in its piece,
// a_(k+1) <= s_k <= a_(k).  The smallest f32 E wins; the winner's scale is
// recomputed in f64, and if the runner-up is within the f32 error both are
// scored again in f64.
__global__ void __launch_bounds__(PLACE_THREADS) k_q2tp_place(const float* __restrict__ W, int n,
                                                              const float* __restrict__ hw,
                                                              float* __restrict__ tab,
                                                              float* __restrict__ lost,
                                                              float* __restrict__ gscale) {
  __shared__ double smin[PLACE_THREADS / 32], smax[PLACE_THREADS / 32];
  __shared__ int scnt[PLACE_THREADS / 32];
  __shared__ float slo, sst;
  __shared__ int sc_all;
  const int r = blockIdx.x, tid = threadIdx.x;
  const int gpr = n / GROUP;
  const float* wr = W + (long long)r * n;
  double dmin = INFINITY, dmax = 0.0;
  int cnt = 0;
  for (int g = tid; g < gpr; g += PLACE_THREADS) {
    float a[GROUP], h[GROUP];
    bool part = false;
#pragma unroll
    for (int q = 0; q < GROUP / 4; ++q) {
      const float4 v = reinterpret_cast<const float4*>(wr + g * GROUP)[q];
      const float4 u = reinterpret_cast<const float4*>(hw + g * GROUP)[q];
      a[4 * q] = fabsf(v.x); a[4 * q + 1] = fabsf(v.y); a[4 * q + 2] = fabsf(v.z); a[4 * q + 3] = fabsf(v.w);
      h[4 * q] = hclip(u.x); h[4 * q + 1] = hclip(u.y); h[4 * q + 2] = hclip(u.z); h[4 * q + 3] = hclip(u.w);
    }
#pragma unroll
    for (int t = 0; t < GROUP; ++t) part |= (h[t] > 0.f && a[t] > 0.f);
    double sd = 0.0;
    if (part) {
      sort_desc(a, h);
      float ta = 0.f, th = 0.f, aa = 0.f;
#pragma unroll
      for (int t = 0; t < GROUP; ++t) {
        ta += h[t] * a[t];
        th += h[t];
        aa += h[t] * a[t] * a[t];
      }
      float e1 = INFINITY, e2 = INFINITY, s1 = 0.f;
      int k1 = 0, k2 = 0;
      float pa = 0.f, ph = 0.f;
#pragma unroll
      for (int k = 0; k <= GROUP; ++k) {
        const float B = 0.5f * ta + pa, C = 0.25f * th + 2.f * ph;
        const float sc = B / C;
        const float up = k == 0 ? INFINITY : a[k - 1];
        const float dn = k == GROUP ? 0.f : a[k];
        if (sc <= up && sc >= dn) {
          const float e = aa - B * sc;
          if (e < e1) {
            if (sc != s1) {
              e2 = e1;
              k2 = k1;
            }
            e1 = e;
            s1 = sc;
            k1 = k;
          } else if (e < e2 && sc != s1) {
            e2 = e;
            k2 = k;
          }
        }
        if (k < GROUP) {
          pa += h[k] * a[k];
          ph += h[k];
        }
      }
      sd = top_scale_f64(a, h, k1);
      if (e2 - e1 <= 1e-4f * fabsf(e1) + 1e-5f * aa) {
        const double sd2 = top_scale_f64(a, h, k2);
        const double ea1 = err_f64(a, h, sd), ea2 = err_f64(a, h, sd2);
        if (ea2 < ea1 || (ea2 == ea1 && sd2 < sd)) sd = sd2;
      }
      dmin = fmin(dmin, sd);
      dmax = fmax(dmax, sd);
      ++cnt;
    }
    if (gscale) gscale[(long long)r * gpr + g] = (float)sd;
  }
  for (int o = 16; o > 0; o >>= 1) {
    dmin = fmin(dmin, __shfl_xor_sync(0xffffffffu, dmin, o));
    dmax = fmax(dmax, __shfl_xor_sync(0xffffffffu, dmax, o));
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  }
  const int wid = tid / 32, lane = tid % 32;
  if (lane == 0) {
    smin[wid] = dmin;
    smax[wid] = dmax;
    scnt[wid] = cnt;
  }
  __syncthreads();
  if (tid == 0) {
    double mn = smin[0], mx = smax[0];
    int c = scnt[0];
    for (int i = 1; i < PLACE_THREADS / 32; ++i) {
      mn = fmin(mn, smin[i]);
      mx = fmax(mx, smax[i]);
      c += scnt[i];
    }
    float lo = 0.f, st = 0.f;
    if (c > 0) {
      lo = __half2float(__double2half(log2(mn)));
      if (mx > mn) {
        const double sd = (log2(mx) - (double)lo) / 30.0;
        st = __half2float(__double2half(sd > 0.0 ? sd : 0.0));
      }
    }
    slo = lo;
    sst = st;
    sc_all = c;
    lost[2 * r] = lo;
    lost[2 * r + 1] = st;
  }
  __syncthreads();
  if (tid < 32) {
    const int c = tid;
    tab[r * 32 + c] = (sc_all > 0 && c > 0) ? (float)exp2((double)slo + (double)(c - 1) * (double)sst) : 0.f;
  }
}

// The q2tp group rule on given tiles, one thread per row ([fold page] WGSL
// q2tp_group, step by step): rung 0 for an all-zero tile, else the first of
// rungs 1..31 with the smallest sum_t h_t d_t d_t (d_t = w_t -
// (q2_level(w_t (1/s) + 1.5) - 1.5) s, summed in column order; rungs with
// s <= 0 skipped; start (3.4e38, rung 1)); then per column j the code
// q2_level(w_j / s + 1.5) (0 if s <= 0), e_j = (w_j - (q - 1.5) s) / U_jj (0
// if U_jj <= 0) and w_t -= e_j U_jt for t > j.  One rounding per operation.
__global__ void __launch_bounds__(128) k_group_q2(const float* __restrict__ tile, int rows,
                                                  const float* __restrict__ ublk,
                                                  const float* __restrict__ hw,
                                                  const float* __restrict__ tab,
                                                  uint8_t* __restrict__ codes,
                                                  uint8_t* __restrict__ rungs,
                                                  float* __restrict__ scales, float* __restrict__ E) {
  __shared__ float Us[GROUP * GROUP];
  __shared__ float hws[GROUP];
  for (int e = threadIdx.x; e < GROUP * GROUP; e += blockDim.x) Us[e] = ublk[e];
  if (threadIdx.x < GROUP) hws[threadIdx.x] = hclip(hw[threadIdx.x]);
  __syncthreads();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= rows) return;
  const float* tabrow = tab + (long long)r * 32;
  float w[GROUP];
  float amax = 0.f;
#pragma unroll
  for (int t = 0; t < GROUP; ++t) {
    w[t] = tile[(long long)r * GROUP + t];
    amax = fmaxf(amax, fabsf(w[t]));
  }
  int best_c = 0;
  if (amax > 0.f) {
    float best_e = 3.4e38f;
    best_c = 1;
#pragma unroll 1
    for (int cand = 1; cand < 32; ++cand) {
      const float sc = tabrow[cand];
      if (!(sc > 0.f)) continue;
      const float iv = __fdiv_rn(1.0f, sc);
      float err = 0.f;
#pragma unroll
      for (int t = 0; t < GROUP; ++t) {
        const float q = q2_code(__fadd_rn(__fmul_rn(w[t], iv), 1.5f));
        const float d = __fsub_rn(w[t], __fmul_rn(__fsub_rn(q, 1.5f), sc));
        err = __fadd_rn(err, __fmul_rn(__fmul_rn(hws[t], d), d));
      }
      if (err < best_e) {
        best_e = err;
        best_c = cand;
      }
    }
  }
  const float s = tabrow[best_c];
  uint32_t words[2] = {0u, 0u};
#pragma unroll
  for (int j = 0; j < GROUP; ++j) {
    const float q = s > 0.f ? q2_code(__fadd_rn(__fdiv_rn(w[j], s), 1.5f)) : 0.f;
    words[j / 16] |= (uint32_t)q << (2 * (j % 16));
    const float dj = Us[j * GROUP + j];
    float ej = 0.f;
    if (dj > 0.f) ej = __fdiv_rn(__fsub_rn(w[j], __fmul_rn(__fsub_rn(q, 1.5f), s)), dj);
    E[(long long)r * GROUP + j] = ej;
    if (ej != 0.f) {
#pragma unroll
      for (int t = j + 1; t < GROUP; ++t) w[t] = __fsub_rn(w[t], __fmul_rn(ej, Us[j * GROUP + t]));
    }
  }
  reinterpret_cast<uint2*>(codes)[r] = make_uint2(words[0], words[1]);
  rungs[r] = (uint8_t)best_c;
  scales[r] = s;
}

}  // namespace

gptq_status place_q2_run(const float* W, int rows, int n, const float* hw, float* tab, float* lost,
                         float* gscale, cudaStream_t s) {
  GQ_PROF(K_PLACE, s);
  k_q2tp_place<<<rows, PLACE_THREADS, 0, s>>>(W, n, hw, tab, lost, gscale);
  GQ_LAUNCHED();
  return GPTQ_OK;
}

gptq_status group_q2_run(const float* tile, int rows, const float* ublk, const float* hw,
                         const float* tab, uint8_t* codes, uint8_t* rungs, float* scales, float* E,
                         cudaStream_t s) {
  GQ_PROF(K_GROUP, s);
  k_group_q2<<<(rows + 127) / 128, 128, 0, s>>>(tile, rows, ublk, hw, tab, codes, rungs, scales, E);
  GQ_LAUNCHED();
  return GPTQ_OK;
}

}  // namespace gq
