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
// pieces in f32 with compensated sums; when a group's two best f32 scores
// are within their f32 error of each other both are scored again in f64
// (scores within 1e-12 sum h w^2 of each other are a tie: the smaller
// scale), and the scales that set the row's ladder (its
// extremes) are recomputed in f64.  A group takes part only if some
// channel has h > 0 and w != 0.  The row's ladder: lo = f16(log2 min s*),
// step = f16(max(0, (log2 max s* - lo) / 30)) (0 if min == max), rung 0 = 0,
// rung c >= 1 = f32(2^(lo + (c-1) step)); no group taking part: all zero.
#include "common.cuh"

#include <cuda_fp16.h>
#include <math.h>

namespace gq {
namespace {

constexpr int PLACE_THREADS = 128;
// Two pieces' f64 scores closer than this times sum_t h_t w_t^2 count as a
// tie (an f64 score of 32 terms is exact to about 1e-16 of that sum); the
// smaller scale is taken.  A group whose weights all share one magnitude a
// has two exact optima, a/1.5 and 2a, that only rounding tells apart.
constexpr double PLACE_TIE_REL = 1e-12;

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

// s + e == a + b exactly (Knuth's two-sum; no contraction, no reordering).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// (hi, lo) += x * y, the product's own rounding error kept (fmaf).
__device__ __forceinline__ void acc_prod(float& hi, float& lo, float x, float y) {
  const float p = __fmul_rn(x, y);
  const float pe = fmaf(x, y, -p);
  float e;
  two_sum(hi, p, hi, e);
  lo = __fadd_rn(lo, __fadd_rn(e, pe));
}
__device__ __forceinline__ void acc(float& hi, float& lo, float x) {
  float e;
  two_sum(hi, x, hi, e);
  lo = __fadd_rn(lo, e);
}

// The f32 search of one group (a sorted descending, h with it): the piece
// whose k largest weights sit on the outer levels has B_k = sum h|w| l =
// 0.5 sum h|w| + sum_top-k h|w| and C_k = sum h l^2 = 0.25 sum h +
// 2 sum_top-k h; its stationary point is s_k = B_k / C_k, where E = sum h w^2
// - B_k s_k; it counts when it lies in its piece, a_(k+1) <= s_k <= a_(k).
// The sums are compensated (two-sum, exact products), so B_k and C_k carry
// about one rounding each and the f32 E of two pieces differ from their
// exact difference by less than 1e-6 sum h w^2; the runner-up within 2e-6
// of the best is a tie, left to f64.  thr1 / thr2 = the smallest outer
// weight of the best / runner-up piece (+inf for no outer weight).
struct PlaceSearch {
  float s, thr1, thr2;
  bool tie;
};

__device__ __forceinline__ PlaceSearch place_search(const float (&a)[GROUP], const float (&h)[GROUP]) {
  float tah = 0.f, tal = 0.f, thh = 0.f, thl = 0.f, aa = 0.f;
#pragma unroll
  for (int t = 0; t < GROUP; ++t) {
    acc_prod(tah, tal, h[t], a[t]);
    acc(thh, thl, h[t]);
    aa += h[t] * a[t] * a[t];
  }
  float e1 = INFINITY, e2 = INFINITY, s1 = 0.f, thr1 = INFINITY, thr2 = INFINITY;
  float pah = 0.f, pal = 0.f, phh = 0.f, phl = 0.f;
#pragma unroll
  for (int k = 0; k <= GROUP; ++k) {
    float bs, be, cs, ce;
    two_sum(0.5f * tah, pah, bs, be);
    two_sum(0.25f * thh, 2.f * phh, cs, ce);
    const float B = bs + (be + (0.5f * tal + pal));
    const float C = cs + (ce + (0.25f * thl + 2.f * phl));
    const float sc = B / C;
    const float up = k == 0 ? INFINITY : a[k - 1];
    const float dn = k == GROUP ? 0.f : a[k];
    if (sc <= up && sc >= dn) {
      const float e = aa - B * sc;
      if (e < e1) {
        if (sc != s1) {
          e2 = e1;
          thr2 = thr1;
        }
        e1 = e;
        s1 = sc;
        thr1 = up;
      } else if (e < e2 && sc != s1) {
        e2 = e;
        thr2 = up;
      }
    }
    if (k < GROUP) {
      acc_prod(pah, pal, h[k], a[k]);
      acc(phh, phl, h[k]);
    }
  }
  PlaceSearch r;
  r.s = s1;
  r.thr1 = thr1;
  r.thr2 = thr2;
  r.tie = e2 - e1 <= 2e-6f * aa;
  return r;
}

// Load group g (|w|, clipped h); false if it does not take part.
__device__ __forceinline__ bool place_load(const float* wr, const float* hw, int g, float (&a)[GROUP],
                                           float (&h)[GROUP]) {
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
  return part;
}

__device__ __forceinline__ double warp_sum_f64(double x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// f64 scale of group g's piece whose outer weights are {t : |w_t| >= thr},
// one element per lane (the whole warp calls it for the same group).
__device__ double warp_scale_f64(float a, float h, float thr) {
  const double hd = h, ha = hd * (double)a;
  const bool o = a >= thr;
  const double ta = warp_sum_f64(ha), th = warp_sum_f64(hd);
  const double oa = warp_sum_f64(o ? ha : 0.0), oh = warp_sum_f64(o ? hd : 0.0);
  return (0.5 * ta + oa) / (0.25 * th + 2.0 * oh);
}

__device__ double warp_err_f64(float a, float h, double s) {
  const double ad = a;
  const double d = ad - (ad > s ? 1.5 : 0.5) * s;
  return warp_sum_f64((double)h * d * d);
}

constexpr int PLACE_MAX_GPR = GPTQ_MAX_N / GROUP;

// One block per row.  Phase 1: thread k places groups k, k + 128, ... in
// f32 (sort, piece search).  Phase 2: the groups whose two best pieces tie
// in f32 are decided in f64 by a whole warp (one element per lane).  Only
// the row's extreme scales set the ladder, so phase 3 recomputes in f64 just
// the groups within 1e-4 (relative) of the f32 minimum or maximum -- far
// above the f32 scale's error -- and the ladder comes from their f64
// scales.  gscale gets the f32 scales (0 for groups that do not take part).
__global__ void __launch_bounds__(PLACE_THREADS, 3) k_q2tp_place(const float* __restrict__ W, int n,
                                                              const float* __restrict__ hw,
                                                              float* __restrict__ tab,
                                                              float* __restrict__ lost,
                                                              float* __restrict__ gscale) {
  __shared__ float gs[PLACE_MAX_GPR], thr1s[PLACE_MAX_GPR], thr2s[PLACE_MAX_GPR];
  __shared__ uint8_t ties[PLACE_MAX_GPR];
  __shared__ float fmn[PLACE_THREADS / 32], fmx[PLACE_THREADS / 32];
  __shared__ double smin[PLACE_THREADS / 32], smax[PLACE_THREADS / 32];
  __shared__ int scnt[PLACE_THREADS / 32];
  __shared__ float slo, sst;
  const int r = blockIdx.x, tid = threadIdx.x;
  const int wid = tid / 32, lane = tid % 32;
  constexpr int NW = PLACE_THREADS / 32;
  const int gpr = n / GROUP;
  const float* wr = W + (long long)r * n;
  for (int g = tid; g < gpr; g += PLACE_THREADS) {
    float a[GROUP], h[GROUP];
    float sf = 0.f, t1 = INFINITY, t2 = INFINITY;
    bool tie = false;
    if (place_load(wr, hw, g, a, h)) {
      sort_desc(a, h);
      const PlaceSearch ps = place_search(a, h);
      sf = ps.s;
      t1 = ps.thr1;
      t2 = ps.thr2;
      tie = ps.tie;
    }
    gs[g] = sf;
    thr1s[g] = t1;
    thr2s[g] = t2;
    ties[g] = tie;
  }
  __syncthreads();
  // Phase 2: f32 ties, one warp per group.
  for (int g0 = wid * 32; g0 < gpr; g0 += PLACE_THREADS) {
    unsigned m = __ballot_sync(0xffffffffu, g0 + lane < gpr && ties[g0 + lane]);
    while (m) {
      const int g = g0 + __ffs(m) - 1;
      m &= m - 1;
      const float a = fabsf(wr[g * GROUP + lane]), h = hclip(hw[g * GROUP + lane]);
      const double s1 = warp_scale_f64(a, h, thr1s[g]), s2 = warp_scale_f64(a, h, thr2s[g]);
      const double e1 = warp_err_f64(a, h, s1), e2 = warp_err_f64(a, h, s2);
      // Scores within PLACE_TIE_REL * sum h w^2 are equal: the smaller scale.
      const double band = PLACE_TIE_REL * warp_sum_f64((double)h * (double)a * (double)a);
      const bool tied = fabs(e1 - e2) <= band;
      const bool take2 = tied ? s2 < s1 : e2 < e1;
      __syncwarp();
      if (lane == 0) {
        gs[g] = (float)(take2 ? s2 : s1);
        if (take2) thr1s[g] = thr2s[g];
      }
    }
  }
  __syncthreads();
  float mnf = INFINITY, mxf = 0.f;
  int cnt = 0;
  for (int g = tid; g < gpr; g += PLACE_THREADS) {
    const float sf = gs[g];
    if (gscale) gscale[(long long)r * gpr + g] = sf;
    if (sf > 0.f) {
      mnf = fminf(mnf, sf);
      mxf = fmaxf(mxf, sf);
      ++cnt;
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    mnf = fminf(mnf, __shfl_xor_sync(0xffffffffu, mnf, o));
    mxf = fmaxf(mxf, __shfl_xor_sync(0xffffffffu, mxf, o));
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  }
  if (lane == 0) {
    fmn[wid] = mnf;
    fmx[wid] = mxf;
    scnt[wid] = cnt;
  }
  __syncthreads();
  mnf = fmn[0];
  mxf = fmx[0];
  cnt = scnt[0];
  for (int i = 1; i < NW; ++i) {
    mnf = fminf(mnf, fmn[i]);
    mxf = fmaxf(mxf, fmx[i]);
    cnt += scnt[i];
  }
  // Phase 3: the candidates for the extremes, in f64, one warp per group.
  double dmin = INFINITY, dmax = 0.0;
  if (cnt > 0) {
    const float lo_cut = mnf * (1.f + 1e-4f), hi_cut = mxf * (1.f - 1e-4f);
    for (int g0 = wid * 32; g0 < gpr; g0 += PLACE_THREADS) {
      const float sl = g0 + lane < gpr ? gs[g0 + lane] : 0.f;
      unsigned m = __ballot_sync(0xffffffffu, sl > 0.f && (sl <= lo_cut || sl >= hi_cut));
      while (m) {
        const int g = g0 + __ffs(m) - 1;
        m &= m - 1;
        const float a = fabsf(wr[g * GROUP + lane]), h = hclip(hw[g * GROUP + lane]);
        const double sd = warp_scale_f64(a, h, thr1s[g]);
        dmin = fmin(dmin, sd);
        dmax = fmax(dmax, sd);
      }
    }
  }
  if (lane == 0) {
    smin[wid] = dmin;
    smax[wid] = dmax;
  }
  __syncthreads();
  if (tid == 0) {
    double mn = smin[0], mx = smax[0];
    for (int i = 1; i < NW; ++i) {
      mn = fmin(mn, smin[i]);
      mx = fmax(mx, smax[i]);
    }
    float lo = 0.f, st = 0.f;
    if (cnt > 0) {
      lo = __half2float(__double2half(log2(mn)));
      if (mx > mn) {
        const double sd = (log2(mx) - (double)lo) / 30.0;
        st = __half2float(__double2half(sd > 0.0 ? sd : 0.0));
      }
    }
    slo = lo;
    sst = st;
    lost[2 * r] = lo;
    lost[2 * r + 1] = st;
  }
  __syncthreads();
  if (tid < 32) {
    const int c = tid;
    tab[r * 32 + c] = (cnt > 0 && c > 0) ? (float)exp2((double)slo + (double)(c - 1) * (double)sst) : 0.f;
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
