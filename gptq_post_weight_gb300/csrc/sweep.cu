// The q4tp sweep on the device (cortiq-engine src/gpu_wgpu/gptq_dev.rs,
// module doc step 5 and WGSL q4tp_group / q4tp_trail; the same rule as the
// host page's gptq_quantize_q4tp).
//
// Lazy blocks of SB = 128 columns (4 groups): one kernel runs the four
// groups of a block out of shared memory (rung choice, rounding, in-group
// feedback, then the group's residuals into the rest of the block), and
// GEMMs apply the residuals to every later column:
// W[:, b1:] -= E_blk U[b0:b1, b1:].  Blocks go in groups of four: before
// each block of a group, a thin update (K = 128, 256, 384) brings its
// columns up to date with the group's earlier blocks, and after the last
// one update with K = 512 (all four blocks' residuals) covers everything to
// the right, so W is read and written once per 512 columns.  With SB = 32
// and groups of one this is the fold page's per-group q4tp_trail; the wider
// blocks are the same mathematics with the residual sums taken in a
// different order.
//
// The same pipeline runs the q2tp "placed" rule ([fold page] WGSL q2_level /
// q2tp_group; [host page] gptq_quantize_q2tp_dev): a full rung search and
// 2-bit codes in the block kernel, everything else unchanged.
//
// The per-group rule uses one rounding per operation (no contraction) so it
// reproduces the pages' f32 arithmetic bit for bit.
#include "common.cuh"

#include <cuda_fp16.h>
#include <math.h>

#include <mutex>

namespace gq {
namespace {

// The rung / rounding rule of one (row, group) tile ([fold page] q4tp_group;
// [host page] gptq_quantize_q4tp), one thread per row:
//  * nominal = clamp(round_half_away((log2(amax/7) - lo) / step), 0, 31)
//    (0 if amax == 0 or step <= 0; log2 = the f64 value rounded to f32);
//  * rung = best of nominal-2..min(nominal+1, 31) by sum_t hw_t (w_t - q_t s)^2
//    with q_t = clamp(rne(w_t * (1/s)), -8, 7), summed in column order,
//    strict '<' over ascending rungs, rungs with s <= 0 skipped;
//  * per column j: q_j = clamp(rne(w_j / s), -8, 7) (0 if s <= 0), nibble
//    q_j + 8, e_j = (w_j - q_j s) / U_jj (0 if U_jj <= 0), w_t -= e_j U_jt
//    for t > j.
// One rounding per operation (no contraction), so the f32 results are the
// pages' bit for bit.  The up to four candidate rungs are evaluated side by
// side (independent sums), which changes no result.
// Nominal rung clamp(round_half_away((l2 - lo) / st), 0, 31) of x = amax/7
// (amax > 0, st > 0), l2 = log2(x) taken in f64 and rounded to f32.  The
// f32 log2f (CUDA documents at most 1 ulp of error) decides the integer
// unless its quotient lands within a margin of a rounding boundary k + 1/2
// (0 <= k <= 30); only then is the f64 value computed, so the result is the
// f64 reading's exactly.  The margin covers 8 ulps of l2 (log2f's error plus
// l2's own rounding, with room), one ulp for the subtraction and two for the
// division, each scaled to the quotient.
__device__ __forceinline__ int nominal_rung(float x, float lo, float st) {
  const float l2a = log2f(x);
  const float tta = __fdiv_rn(__fsub_rn(l2a, lo), st);
  const float bnd = fminf(fmaxf(floorf(tta) + 0.5f, 0.5f), 30.5f);
  const float margin =
      (fabsf(l2a) * 9.6e-7f + (fabsf(l2a) + fabsf(lo)) * 1.2e-7f) / st + fabsf(tta) * 2.4e-7f + 1e-6f;
  float tt = tta;
  if (!(fabsf(tta - bnd) > margin)) {  // near a boundary, or NaN
    const float l2 = (float)log2((double)x);
    tt = __fdiv_rn(__fsub_rn(l2, lo), st);
  }
  return (int)fminf(fmaxf(roundf(tt), 0.f), 31.f);
}

__device__ __forceinline__ int q4tp_pick(const float (&w)[GROUP], const float* hw,
                                         const float* tabrow, float lo, float st) {
  float amax = 0.f;
#pragma unroll
  for (int t = 0; t < GROUP; ++t) amax = fmaxf(amax, fabsf(w[t]));
  const int nominal = (amax > 0.f && st > 0.f) ? nominal_rung(__fdiv_rn(amax, 7.0f), lo, st) : 0;
  int best_c = nominal;
  if (amax > 0.f) {
    const int lo_c = nominal >= 2 ? nominal - 2 : 0;
    const int hi_c = nominal + 1 < 31 ? nominal + 1 : 31;
    float sc[4], iv[4], err[4];
    bool valid[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int cand = lo_c + k;
      sc[k] = cand <= hi_c ? tabrow[cand] : 0.f;
      valid[k] = cand <= hi_c && sc[k] > 0.f;
      iv[k] = __fdiv_rn(1.0f, valid[k] ? sc[k] : 1.f);
      err[k] = 0.f;
    }
#pragma unroll
    for (int t = 0; t < GROUP; ++t) {
      const float h = hw[t];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float q = fminf(fmaxf(rintf(__fmul_rn(w[t], iv[k])), -8.f), 7.f);
        const float d = __fsub_rn(w[t], __fmul_rn(q, sc[k]));
        err[k] = __fadd_rn(err[k], __fmul_rn(__fmul_rn(h, d), d));
      }
    }
    float best_e = INFINITY;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (valid[k] && err[k] < best_e) {
        best_e = err[k];
        best_c = lo_c + k;
      }
    }
  }
  return best_c;
}

__device__ __forceinline__ void q4tp_round(float (&w)[GROUP], float s, const float* U, int ldu,
                                           uint32_t (&words)[4], float (&e)[GROUP]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) words[i] = 0u;
#pragma unroll
  for (int j = 0; j < GROUP; ++j) {
    float q = 0.f;
    if (s > 0.f) q = fminf(fmaxf(rintf(__fdiv_rn(w[j], s)), -8.f), 7.f);
    const uint32_t nb = (uint32_t)((int)q + 8) & 15u;
    words[j / 8] |= nb << (4 * (j % 8));
    const float dj = U[j * ldu + j];
    float ej = 0.f;
    if (dj > 0.f) ej = __fdiv_rn(__fsub_rn(w[j], __fmul_rn(q, s)), dj);
    e[j] = ej;
    if (ej != 0.f) {
#pragma unroll
      for (int t = j + 1; t < GROUP; ++t) w[t] = __fsub_rn(w[t], __fmul_rn(ej, U[j * ldu + t]));
    }
  }
}

// Per-row ladder ([host page] gptq_quantize_q4tp_dev's tab / lost; the
// converter itself is not on the pages -- reading in the header).  With DZ
// the kernel also writes the dead-zeroed copy of W ([host page]
// gptq_quantize_q4tp_dev: "zero the dead columns", !(H_ii > 0)) and takes
// the ladder from it: W is read once and its copy written once.
// One CTA per row, streaming: consecutive threads take consecutive float4s
// of the row (four passes in flight per thread), so the eight float4s of a
// group sit in eight consecutive lanes and its absmax is a three-step
// shuffle reduction.
constexpr int LADDER_THREADS = 256;
template <bool DZ>
__global__ void __launch_bounds__(LADDER_THREADS) k_ladder(const float* __restrict__ W, int n,
                                                           float* __restrict__ tab, float* __restrict__ lost,
                                                           const float* __restrict__ hdiag,
                                                           float* __restrict__ wz) {
  const int r = blockIdx.x;
  const float4* wr = reinterpret_cast<const float4*>(W + (long long)r * n);
  const float4* h4 = reinterpret_cast<const float4*>(hdiag);
  float4* o4 = reinterpret_cast<float4*>(wz + (long long)r * n);
  const int nv = n / 4;  // n % 32 == 0: whole groups of eight float4s
  float xmin = INFINITY, xmax = 0.f;
  int cnt = 0;
  const int lane8 = threadIdx.x & 31;
  const bool head = (threadIdx.x & 7) == 0;
  // The trip count is the same for every lane of a warp (the shuffles below
  // need the whole warp); lanes past the row's end load nothing.
#pragma unroll 4
  for (int v0 = threadIdx.x & ~31; v0 < nv; v0 += LADDER_THREADS) {
    const int v = v0 + lane8;
    const bool ok = v < nv;
    float4 x = ok ? __ldcs(wr + v) : make_float4(0.f, 0.f, 0.f, 0.f);
    if (DZ && ok) {
      const float4 h = h4[v];
      x.x = h.x > 0.f ? x.x : 0.f;
      x.y = h.y > 0.f ? x.y : 0.f;
      x.z = h.z > 0.f ? x.z : 0.f;
      x.w = h.w > 0.f ? x.w : 0.f;
      __stcs(o4 + v, x);
    }
    float a = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
    // The group's eight float4s are lanes 8m .. 8m+7 of this warp (n is a
    // multiple of 32, so a group is wholly inside or wholly past the row).
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
    if (ok && head && a > 0.f) {
      const float xg = __fdiv_rn(a, 7.0f);
      xmin = fminf(xmin, xg);
      xmax = fmaxf(xmax, xg);
      ++cnt;
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    xmin = fminf(xmin, __shfl_xor_sync(0xffffffffu, xmin, o));
    xmax = fmaxf(xmax, __shfl_xor_sync(0xffffffffu, xmax, o));
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  }
  __shared__ float smin[LADDER_THREADS / 32], smax[LADDER_THREADS / 32];
  __shared__ int scnt[LADDER_THREADS / 32];
  __shared__ float slo, sst;
  const int wid = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (lane == 0) {
    smin[wid] = xmin;
    smax[wid] = xmax;
    scnt[wid] = cnt;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float mn = smin[0], mx = smax[0];
    int c = scnt[0];
    for (int i = 1; i < LADDER_THREADS / 32; ++i) {
      mn = fminf(mn, smin[i]);
      mx = fmaxf(mx, smax[i]);
      c += scnt[i];
    }
    float lo = 0.f, st = 0.f;
    if (c > 0) {
      lo = __half2float(__double2half(log2((double)mn)));
      if (mx > mn) {
        double sd = (log2((double)mx) - (double)lo) / 31.0;
        st = __half2float(__double2half(sd > 0.0 ? sd : 0.0));
      }
    }
    slo = lo;
    sst = st;
    lost[2 * r] = lo;
    lost[2 * r + 1] = st;
    scnt[0] = c;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int c = threadIdx.x;
    tab[r * 32 + c] = scnt[0] > 0 ? (float)exp2((double)slo + (double)c * (double)sst) : 0.f;
  }
}

// The group rule on given tiles (one thread per row; the same device code as
// the sweep's block kernel).
__global__ void __launch_bounds__(128) k_group(const float* __restrict__ tile, int rows,
                                               const float* __restrict__ ublk,
                                               const float* __restrict__ hw,
                                               const float* __restrict__ tab,
                                               const float* __restrict__ lost,
                                               uint8_t* __restrict__ nib, uint8_t* __restrict__ rungs,
                                               float* __restrict__ scales, float* __restrict__ E) {
  __shared__ float Us[GROUP * GROUP];
  __shared__ float hws[GROUP];
  for (int e = threadIdx.x; e < GROUP * GROUP; e += blockDim.x) Us[e] = ublk[e];
  if (threadIdx.x < GROUP) hws[threadIdx.x] = hw[threadIdx.x];
  __syncthreads();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= rows) return;
  float w[GROUP], e[GROUP];
#pragma unroll
  for (int t = 0; t < GROUP; ++t) w[t] = tile[(long long)r * GROUP + t];
  const int c = q4tp_pick(w, hws, tab + (long long)r * 32, lost[2 * r], lost[2 * r + 1]);
  const float s = tab[(long long)r * 32 + c];
  uint32_t words[4];
  q4tp_round(w, s, Us, GROUP, words, e);
  reinterpret_cast<uint4*>(nib)[r] = make_uint4(words[0], words[1], words[2], words[3]);
  rungs[r] = (uint8_t)c;
  scales[r] = s;
#pragma unroll
  for (int t = 0; t < GROUP; ++t) E[(long long)r * GROUP + t] = e[t];
}

constexpr int SWEEP_ROWS = 40;                 // 5 warps: 5120 rows fill 128 CTAs, one wave
constexpr int SWEEP_THREADS = 4 * SWEEP_ROWS;  // a quad of lanes per row
constexpr int LW = SB + 16;  // W block row stride: float4 rows, two rows per phase conflict-free
// Blocks whose residuals one trailing update applies (K = GMAX * SB); a
// workspace too small for that runs groups of GMIN blocks.
constexpr int GMAX = 4, GMIN = 2;
constexpr int SWEEP_SMEM = (SB * SB + SB + SWEEP_ROWS * LW + SWEEP_ROWS * 32) * 4;


// One lazy block [b0, b0+B) (B <= SB, a multiple of 32) for 40 rows per CTA.
// The block's U (B x B), the rung weights and the rows' block of W sit in
// shared memory.  Each row belongs to a quad of four lanes of one warp (8
// rows per warp), and a warp carries its rows through the whole block
// without waiting on the other warps:
//  * rung choice: lane k of the quad evaluates candidate nominal-2+k over
//    the group's 32 columns (its own sum, in column order), the quad swaps
//    the four sums and every lane takes the same pick;
//  * rounding: every lane of the quad runs the row's 32 columns in full
//    (no exchange on the sequential path).  Per column the critical path is
//    the code, the residual and the next column's update; the updates of
//    the later columns by the previous residual are issued after the
//    column's first division, in its latency.  Each column still receives
//    e_0, e_1, ... in order with one rounding per operation, so codes and
//    residuals are the one-thread rule's bit for bit;
//  * the group's residuals go to E (TF32 hi/lo, the trailing GEMM's
//    operand) and into the block's later columns (w_c -= sum_j e_j U_jc),
//    lane k taking the 4-column chunks 4k, 4k+16, ... .
// MODE_Q4_ACT (act order): W and U are in permuted channel order, the rungs
// are given (static, per original group) and each column takes the scale of
// its original group; codes go to `codes` (int8, permuted order) instead of
// the nibble plane.
// MODE_Q2 (the q2tp "placed" rule, [fold page] WGSL q2_level / q2tp_group):
// rungs 1..31 searched in full (lane k of the quad takes rungs 1+k, 5+k, ...;
// each lane keeps its lowest best rung, the quad then takes the lowest rung
// of the smallest error, which is the one-thread ascending strict-'<' scan
// from (3.4e38, rung 1)); an all-zero tile takes rung 0; codes
// q2_level(w/s + 1.5) into the 2-bit plane (8 bytes a tile); residual
// (w - (q - 1.5) s) / U_jj; rung weights H_ii clipped at 0.
enum SweepMode : int { MODE_Q4 = 0, MODE_Q4_ACT = 1, MODE_Q2 = 2 };

template <int MODE>
__global__ void __launch_bounds__(SWEEP_THREADS) k_sweep_block(
    const float* __restrict__ W, int rows, int n, int b0, int B, const float* __restrict__ U,
    const float* __restrict__ hw, const float* __restrict__ tab, const float* __restrict__ lost,
    uint8_t* __restrict__ nib, uint8_t* __restrict__ rungs, float* __restrict__ scales,
    float* __restrict__ E_hi, float* __restrict__ E_lo, int ecol0, int ew,
    const int* __restrict__ perm, int8_t* __restrict__ codes) {
  constexpr bool ACT = MODE == MODE_Q4_ACT;
  constexpr bool Q2 = MODE == MODE_Q2;
  constexpr int NWORDS = ACT ? GROUP / 4 : (Q2 ? GROUP / 16 : GROUP / 8);
  extern __shared__ __align__(16) float sm[];
  float* Us = sm;             // [SB][SB]
  float* hws = Us + SB * SB;  // [SB]
  float* Ws = hws + SB;       // [SWEEP_ROWS][LW]
  float* Ts = Ws + SWEEP_ROWS * LW;  // [SWEEP_ROWS][32]: the rows' rung tables
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int r0 = blockIdx.x * SWEEP_ROWS;
  {
    // The rows' block of W and the first group's rows of the block's U by
    // asynchronous 16-byte copies (one commit group), then the rest of U
    // (a second group, which lands while group 0 is worked); rows past the
    // end are filled with ones.
    const int q4 = B / 4;
#pragma unroll 4
    for (int e = tid; e < SWEEP_ROWS * q4; e += SWEEP_THREADS) {
      const int rr = e / q4, c4 = e % q4;
      float* dst = Ws + rr * LW + 4 * c4;
      if (r0 + rr < rows)
        cp_async16(dst, W + (long long)(r0 + rr) * n + b0 + 4 * c4);
      else  // rows past the end round ones (a zero dividend sends a division down its slow path)
        *reinterpret_cast<float4*>(dst) = make_float4(1.f, 1.f, 1.f, 1.f);
    }
#pragma unroll 4
    for (int e = tid; e < GROUP * q4; e += SWEEP_THREADS)
      cp_async16(Us + (e / q4) * SB + 4 * (e % q4), U + (long long)(b0 + e / q4) * n + b0 + 4 * (e % q4));
    // The rows' rung tables (a row past the end takes the last row's).
    for (int e = tid; e < SWEEP_ROWS * 8; e += SWEEP_THREADS) {
      const int rr = e / 8, rsrc = r0 + rr < rows ? r0 + rr : rows - 1;
      cp_async16(Ts + rr * 32 + 4 * (e % 8), tab + (long long)rsrc * 32 + 4 * (e % 8));
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
#pragma unroll 4
    for (int e = GROUP * q4 + tid; e < B * q4; e += SWEEP_THREADS)
      cp_async16(Us + (e / q4) * SB + 4 * (e % q4), U + (long long)(b0 + e / q4) * n + b0 + 4 * (e % q4));
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 1;" ::: "memory");
  }
  for (int e = tid; e < B; e += SWEEP_THREADS) {
    const float h = ACT ? 0.f : hw[b0 + e];
    hws[e] = Q2 ? (h > 0.f ? h : 0.f) : h;
  }
  __syncthreads();
  const int sub = lane & 3, qbase = lane & ~3;
  const int rl = warp * 8 + (lane >> 2);
  const int r = r0 + rl;
  const bool live = r < rows;
  const int rs = live ? r : rows - 1;  // rows past the end compute on a real row, store nothing
  const int gpr = n / GROUP;
  const float* tabrow = Ts + rl * 32;
  float* wrow = Ws + rl * LW;
  float lo = 0.f, st = 0.f;
  if (MODE == MODE_Q4) {
    lo = lost[2 * rs];
    st = lost[2 * rs + 1];
  }
  for (int g = 0; g < B / GROUP; ++g) {
    const int gc = g * GROUP;
    if (g == 1) {
      // The rest of the block's U (group 0 needed only its own rows).
      asm volatile("cp.async.wait_group 0;" ::: "memory");
      __syncthreads();
    }
    float w[GROUP];
#pragma unroll
    for (int q = 0; q < GROUP / 4; ++q) {
      const float4 v = *reinterpret_cast<const float4*>(wrow + gc + 4 * q);
      w[4 * q] = v.x;
      w[4 * q + 1] = v.y;
      w[4 * q + 2] = v.z;
      w[4 * q + 3] = v.w;
    }
    float s = 0.f;
    int best_c = 0;
    float sc[ACT ? GROUP : 1];
    if (ACT) {
#pragma unroll
      for (int t = 0; t < GROUP; ++t) sc[t] = tabrow[rungs[(long long)rs * gpr + perm[b0 + gc + t] / GROUP]];
    } else if (Q2) {
      float amax = 0.f;
#pragma unroll
      for (int t = 0; t < GROUP; ++t) amax = fmaxf(amax, fabsf(w[t]));
      const bool any = amax > 0.f;
      float be = 3.4e38f;
      int bc = 64;  // none below 3.4e38 yet
      if (any) {
        // Two candidates side by side in packed f32x2 arithmetic (each lane
        // of a packed operation rounds like the scalar one; w - p is taken
        // as w + (-p), the same IEEE result).
        const float* hg = hws + gc;
        const float2 c15 = make_float2(1.5f, 1.5f), m15 = make_float2(-1.5f, -1.5f);
#pragma unroll 1
        for (int k = 0; k < 8; k += 2) {
          const int ca = 1 + sub + 4 * k, cb = ca + 4;
          if (ca > 31) break;
          const float sa = tabrow[ca], sb = cb <= 31 ? tabrow[cb] : 0.f;
          const bool va = sa > 0.f, vb = sb > 0.f;
          if (!va && !vb) continue;
          const float2 iv = make_float2(__fdiv_rn(1.0f, va ? sa : 1.f), __fdiv_rn(1.0f, vb ? sb : 1.f));
          const float2 ns = make_float2(-sa, -sb);
          float2 err = make_float2(0.f, 0.f);
#pragma unroll
          for (int t = 0; t < GROUP; ++t) {
            const float2 w2 = make_float2(w[t], w[t]);
            const float2 x = __fadd2_rn(__fmul2_rn(w2, iv), c15);
            const float2 lev = __fadd2_rn(make_float2(q2_code(x.x), q2_code(x.y)), m15);
            const float2 d = __fadd2_rn(w2, __fmul2_rn(lev, ns));
            const float2 hd = __fmul2_rn(make_float2(hg[t], hg[t]), d);
            err = __fadd2_rn(err, __fmul2_rn(hd, d));
          }
          if (va && err.x < be) {
            be = err.x;
            bc = ca;
          }
          if (vb && err.y < be) {
            be = err.y;
            bc = cb;
          }
        }
      }
      // Every lane reaches the exchange (rows differ in amax).
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        const float oe = __shfl_xor_sync(0xffffffffu, be, o);
        const int oc = __shfl_xor_sync(0xffffffffu, bc, o);
        if (oe < be || (oe == be && oc < bc)) {
          be = oe;
          bc = oc;
        }
      }
      best_c = any ? (bc < 32 ? bc : 1) : 0;
      s = tabrow[best_c];
    } else {
      // Rung rule, one candidate per lane.
      float amax = 0.f;
#pragma unroll
      for (int t = 0; t < GROUP; ++t) amax = fmaxf(amax, fabsf(w[t]));
      const int nominal = (amax > 0.f && st > 0.f) ? nominal_rung(__fdiv_rn(amax, 7.0f), lo, st) : 0;
      // Every lane of the warp reaches the exchange below (rows differ in
      // amax, the four lanes of a quad do not); a row with amax == 0 has no
      // valid candidate and keeps the nominal rung.
      best_c = nominal;
      const bool any = amax > 0.f;
      const int lo_c = nominal >= 2 ? nominal - 2 : 0;
      const int hi_c = nominal + 1 < 31 ? nominal + 1 : 31;
      const int cand = lo_c + sub;
      const float sck = (any && cand <= hi_c) ? tabrow[cand] : 0.f;
      const bool valid = any && cand <= hi_c && sck > 0.f;
      float err = 0.f;
      if (any) {
        const float iv = __fdiv_rn(1.0f, valid ? sck : 1.f);
        const float* hg = hws + gc;
#pragma unroll
        for (int t = 0; t < GROUP; ++t) {
          const float q = fminf(fmaxf(rintf(__fmul_rn(w[t], iv)), -8.f), 7.f);
          const float d = __fsub_rn(w[t], __fmul_rn(q, sck));
          err = __fadd_rn(err, __fmul_rn(__fmul_rn(hg[t], d), d));
        }
      }
      float best_e = INFINITY;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float ek = __shfl_sync(0xffffffffu, err, qbase | k);
        const int vk = __shfl_sync(0xffffffffu, (int)valid, qbase | k);
        if (vk && ek < best_e) {
          best_e = ek;
          best_c = lo_c + k;
        }
      }
      s = tabrow[best_c];
    }
    // Rounding with in-group feedback (software-pipelined, see above).
    const float* Ug = Us + gc * SB + gc;
    uint32_t words[NWORDS];
#pragma unroll
    for (int i = 0; i < NWORDS; ++i) words[i] = 0u;
    // The chain's own U entries (diagonal and first superdiagonal) in
    // registers before it starts, and the residuals kept in registers (every
    // lane of the quad computes every e_j): no shared-memory store inside the
    // chain, so nothing orders its loads behind one.
    float ud[GROUP], u1[GROUP], e[GROUP];
#pragma unroll
    for (int j = 0; j < GROUP; ++j) {
      ud[j] = Ug[j * SB + j];
      u1[j] = j + 1 < GROUP ? Ug[j * SB + j + 1] : 0.f;
    }
    float eprev = 0.f;
#pragma unroll
    for (int j = 0; j < GROUP; ++j) {
      const float x = w[j];  // current: e_{j-1} reached it at the end of the last step
      const float sj = ACT ? sc[j] : s;
      const float t1 = sj > 0.f ? __fdiv_rn(x, sj) : 0.f;
      if (j > 0) {
        // w_t -= e_{j-1} U_{j-1,t}, two columns per packed instruction:
        // w + (-e) U is w - e U bit for bit (one rounding each, as before).
        const float* ur = Ug + (j - 1) * SB;
        if ((j + 1) & 1) w[j + 1] = __fsub_rn(w[j + 1], __fmul_rn(eprev, ur[j + 1]));
        const float2 ne = make_float2(-eprev, -eprev);
#pragma unroll
        for (int t = (j + 2) & ~1; t + 1 < GROUP; t += 2) {
          const float2 u2 = *reinterpret_cast<const float2*>(ur + t);
          const float2 w2 = __fadd2_rn(make_float2(w[t], w[t + 1]), __fmul2_rn(ne, u2));
          w[t] = w2.x;
          w[t + 1] = w2.y;
        }
      }
      float q, lev;
      if (Q2) {
        q = sj > 0.f ? q2_code(__fadd_rn(t1, 1.5f)) : 0.f;
        lev = __fsub_rn(q, 1.5f);
      } else {
        q = sj > 0.f ? fminf(fmaxf(rintf(t1), -8.f), 7.f) : 0.f;
        lev = q;
      }
      const float dj = ud[j];
      float ej = 0.f;
      if (dj > 0.f) ej = __fdiv_rn(__fsub_rn(x, __fmul_rn(lev, sj)), dj);
      e[j] = ej;
      if (ACT)
        words[j / 4] |= ((uint32_t)(int)q & 255u) << (8 * (j % 4));
      else if (Q2)
        words[j / 16] |= (uint32_t)q << (2 * (j % 16));
      else
        words[j / 8] |= ((uint32_t)((int)q + 8) & 15u) << (4 * (j % 8));
      if (j + 1 < GROUP) w[j + 1] = __fsub_rn(w[j + 1], __fmul_rn(ej, u1[j]));
      eprev = ej;
    }
    if (live) {
      if (ACT) {
        // Lane k stores the int8 codes of columns 8k .. 8k+7.
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (sub == c)
            *reinterpret_cast<uint2*>(codes + (long long)r * n + b0 + gc + 8 * c) =
                make_uint2(words[2 * c], words[2 * c + 1]);
      } else if (sub == 0) {
        const long long tix = (long long)r * gpr + b0 / GROUP + g;
        if constexpr (Q2)
          reinterpret_cast<uint2*>(nib)[tix] = make_uint2(words[0], words[1]);
        else
          reinterpret_cast<uint4*>(nib)[tix] = make_uint4(words[0], words[1], words[2], words[3]);
        rungs[tix] = (uint8_t)best_c;
        scales[tix] = s;
      }
      float* eh = E_hi + (long long)r * ew + ecol0 + gc;
      float* el = E_lo + (long long)r * ew + ecol0 + gc;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (sub != c) continue;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          float4 h, l;
          split_tf32(e[8 * c + 4 * t], h.x, l.x);
          split_tf32(e[8 * c + 4 * t + 1], h.y, l.y);
          split_tf32(e[8 * c + 4 * t + 2], h.z, l.z);
          split_tf32(e[8 * c + 4 * t + 3], h.w, l.w);
          reinterpret_cast<float4*>(eh + 8 * c)[t] = h;
          reinterpret_cast<float4*>(el + 8 * c)[t] = l;
        }
      }
    }
    // The group's residuals into the rest of the block.
    const int rest = B - gc - GROUP;
#pragma unroll 2
    for (int m = 0; m < rest / 16; ++m) {
      const int c = gc + GROUP + 16 * m + 4 * sub;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < GROUP; ++j) {
        const float4 u = *reinterpret_cast<const float4*>(Us + (gc + j) * SB + c);
        acc.x = fmaf(e[j], u.x, acc.x);
        acc.y = fmaf(e[j], u.y, acc.y);
        acc.z = fmaf(e[j], u.z, acc.z);
        acc.w = fmaf(e[j], u.w, acc.w);
      }
      float4 v = *reinterpret_cast<float4*>(wrow + c);
      v.x -= acc.x;
      v.y -= acc.y;
      v.z -= acc.z;
      v.w -= acc.w;
      *reinterpret_cast<float4*>(wrow + c) = v;
    }
    __syncwarp();
  }
}

// Ut[c][t] = U[b0 + t][b1 + c], t < kt (one or two blocks' rows of U),
// c < n - b1: the block rows of U to the right of the first block, K-major
// for the GEMM, stored as their TF32 hi/lo split.  Rows b1 + c of U below
// the diagonal are zero, so the same stripe serves the thin update of the
// second block (c < SB, first SB of t) and the pair's trailing update.
// One CTA per 32 columns c x 128 rows t of the stripe: float4 loads of U's
// rows into shared memory, float4 stores of Ut's rows (c fixed, 128
// consecutive t) from it.
constexpr int PREP_T = 128;
__global__ void __launch_bounds__(256) k_prep_ut(const float* __restrict__ U, int n, int b0, int b1, int kt,
                                                 int ew, float* __restrict__ Ut_hi, float* __restrict__ Ut_lo) {
  __shared__ float tile[PREP_T][33];
  const int c0 = blockIdx.x * 32, t0 = blockIdx.y * PREP_T;
  const int ncol = n - b1, tid = threadIdx.x;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int tt = tid / 8 + 32 * i, c4 = tid % 8;
    const int t = t0 + tt, c = c0 + 4 * c4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < kt && c < ncol) v = *reinterpret_cast<const float4*>(U + (long long)(b0 + t) * n + b1 + c);
    tile[tt][4 * c4] = v.x;
    tile[tt][4 * c4 + 1] = v.y;
    tile[tt][4 * c4 + 2] = v.z;
    tile[tt][4 * c4 + 3] = v.w;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int cc = tid / 32 + 8 * i, t4 = tid % 32;
    const int c = c0 + cc, t = t0 + 4 * t4;
    if (c >= ncol || t >= kt) continue;
    float4 h, l;
    split_tf32(tile[4 * t4][cc], h.x, l.x);
    split_tf32(tile[4 * t4 + 1][cc], h.y, l.y);
    split_tf32(tile[4 * t4 + 2][cc], h.z, l.z);
    split_tf32(tile[4 * t4 + 3][cc], h.w, l.w);
    *reinterpret_cast<float4*>(Ut_hi + (long long)c * ew + t) = h;
    *reinterpret_cast<float4*>(Ut_lo + (long long)c * ew + t) = l;
  }
}

// W copy with dead channels (!(H_ii > 0)) zeroed ([host page]
// gptq_quantize_q4tp_dev: "zero the dead columns").
__global__ void k_copy_dz(const float* __restrict__ W, long long total, int n,
                          const float* __restrict__ hdiag, float* __restrict__ out) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(i % n);
    out[i] = (hdiag[c] > 0.f) ? W[i] : 0.f;
  }
}

}  // namespace

static size_t sweep_ws_bytes_g(int rows, int n, int g) {
  const size_t ew = (size_t)g * SB;
  return 2 * round_up((size_t)rows * ew * 4, 256) + 2 * round_up((size_t)n * ew * 4, 256) + 1024;
}
size_t sweep_ws_bytes(int rows, int n) { return sweep_ws_bytes_g(rows, n, GMAX); }
size_t sweep_ws_min_bytes(int rows, int n) { return sweep_ws_bytes_g(rows, n, GMIN); }

static gptq_status sweep_attrs() {
  static DeviceOnce once;
  return once.run([](int) -> gptq_status {
    GQ_CUDA(cudaFuncSetAttribute(k_sweep_block<MODE_Q4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SWEEP_SMEM));
    GQ_CUDA(cudaFuncSetAttribute(k_sweep_block<MODE_Q4_ACT>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, SWEEP_SMEM));
    GQ_CUDA(cudaFuncSetAttribute(k_sweep_block<MODE_Q2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SWEEP_SMEM));
    return GPTQ_OK;
  });
}

gptq_status ladder_run(const float* W, int rows, int n, float* tab, float* lost, cudaStream_t s) {
  GQ_PROF(K_LADDER, s);
  k_ladder<false><<<rows, LADDER_THREADS, 0, s>>>(W, n, tab, lost, nullptr, nullptr);
  GQ_LAUNCHED();
  return GPTQ_OK;
}

gptq_status copy_ladder_run(const float* W, int rows, int n, const float* hdiag, float* wz, float* tab,
                            float* lost, cudaStream_t s) {
  GQ_PROF(K_LADDER, s);
  k_ladder<true><<<rows, LADDER_THREADS, 0, s>>>(W, n, tab, lost, hdiag, wz);
  GQ_LAUNCHED();
  return GPTQ_OK;
}

gptq_status group_run(const float* tile, int rows, const float* ublk, const float* hw,
                      const float* tab, const float* lost, uint8_t* nib, uint8_t* rungs,
                      float* scales, float* E, cudaStream_t s) {
  GQ_PROF(K_GROUP, s);
  k_group<<<(rows + 127) / 128, 128, 0, s>>>(tile, rows, ublk, hw, tab, lost, nib, rungs, scales, E);
  GQ_LAUNCHED();
  return GPTQ_OK;
}

gptq_status copy_dead_zeroed(const float* W, int rows, int n, const float* hdiag, float* out,
                             cudaStream_t s) {
  const long long total = (long long)rows * n;
  GQ_PROF(K_COPY, s);
  k_copy_dz<<<152 * 8, 256, 0, s>>>(W, total, n, hdiag, out);
  GQ_LAUNCHED();
  return GPTQ_OK;
}

// Scratch for gptq_q4tp_sweep_noalloc: a file-scope device array, so that a
// caller that must not allocate device memory can still run the sweep.  Its
// host-side name is only a stand-in, never a device address: the address
// comes from cudaGetSymbolAddress, looked up with the device current on the
// first call in each device's context (again after a device reset, whose
// new context places the array anew), and kept for later calls.
namespace {
__device__ __align__(256) unsigned char g_noalloc_scratch[GPTQ_SWEEP_NOALLOC_SCRATCH_BYTES];
DeviceOnce g_noalloc_once;
void* g_noalloc_ptr[DeviceOnce::kMaxDevices] = {};
}  // namespace

gptq_status noalloc_scratch(void** out) {
  GQ_TRY(g_noalloc_once.run([](int dev) -> gptq_status {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return GPTQ_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
    return GPTQ_OK;
  }));
  int dev = 0;
  GQ_CUDA(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lk(g_noalloc_once.mu);
  *out = g_noalloc_ptr[dev];
  return *out != nullptr ? GPTQ_OK : GPTQ_ERR_CUDA;
}

// side_in: a side stream made by the caller (null: one of the call's own);
// status_out: null to read the status word back and wait for the stream
// (the call's result), else only enqueue and hand back the device status
// word (bit 1: a wait timed out).
static gptq_status sweep_core(int mode, float* W, int rows, int n, const float* U, const float* hw,
                              const float* tab, const float* lost, uint8_t* nib, uint8_t* rungs,
                              float* scales, void* ws, size_t ws_bytes, cudaStream_t s,
                              const int* perm, int8_t* codes, const SideStream* side_in = nullptr,
                              unsigned** status_out = nullptr) {
  GQ_TRY(sweep_attrs());
  const int G = ws_bytes >= sweep_ws_bytes_g(rows, n, GMAX) ? GMAX : GMIN;
  const int ew = G * SB;
  Carve c(ws, ws_bytes);
  float* E_hi = c.take<float>((size_t)rows * ew);
  float* E_lo = c.take<float>((size_t)rows * ew);
  float* Ut_hi = c.take<float>((size_t)n * ew);
  float* Ut_lo = c.take<float>((size_t)n * ew);
  unsigned* status = c.take<unsigned>(4);
  if (!c.ok) return GPTQ_ERR_NOMEM;
  GQ_CUDA(cudaMemsetAsync(status, 0, sizeof(unsigned), s));
  OperandMaps maps;  // 0/1 = Ut hi/lo, 2/3 = E hi/lo
  GQ_TRY(make_operand_map(&maps.m[0], Ut_hi, n, ew));
  GQ_TRY(make_operand_map(&maps.m[1], Ut_lo, n, ew));
  GQ_TRY(make_operand_map(&maps.m[2], E_hi, rows, ew));
  GQ_TRY(make_operand_map(&maps.m[3], E_lo, rows, ew));
  GQ_TRY(make_c_map(&maps.c, W, rows, n, n));
  const int smem = SWEEP_SMEM;
  const TcJob none{};
  const int grid_rows = (rows + SWEEP_ROWS - 1) / SWEEP_ROWS;
  auto block = [&](int b0, int B, int ecol0) -> gptq_status {
    GQ_PROF(K_SWEEP_BLOCK, s);
    if (mode == MODE_Q4_ACT)
      k_sweep_block<MODE_Q4_ACT><<<grid_rows, SWEEP_THREADS, smem, s>>>(
          W, rows, n, b0, B, U, hw, tab, lost, nib, rungs, scales, E_hi, E_lo, ecol0, ew, perm, codes);
    else if (mode == MODE_Q2)
      k_sweep_block<MODE_Q2><<<grid_rows, SWEEP_THREADS, smem, s>>>(
          W, rows, n, b0, B, U, hw, tab, lost, nib, rungs, scales, E_hi, E_lo, ecol0, ew, nullptr,
          nullptr);
    else
      k_sweep_block<MODE_Q4><<<grid_rows, SWEEP_THREADS, smem, s>>>(
          W, rows, n, b0, B, U, hw, tab, lost, nib, rungs, scales, E_hi, E_lo, ecol0, ew, nullptr,
          nullptr);
    GQ_LAUNCHED();
    return GPTQ_OK;
  };
  // A group's Ut stripe depends on U alone, so it is built on a side stream
  // beside the group's first block (which leaves SMs and issue slots free):
  // it waits for the previous group's update (the last reader of Ut) and the
  // group's first thin update waits for it.
  SideStream own;
  if (side_in == nullptr) GQ_TRY(own.init());
  const SideStream& side = side_in ? *side_in : own;
  auto prep = [&](int b0, int b1, int kt) -> gptq_status {
    GQ_CUDA(cudaEventRecord(side.fork, s));
    GQ_CUDA(cudaStreamWaitEvent(side.s, side.fork, 0));
    {
      GQ_PROF(K_PREP_UT, side.s);
      dim3 grid((n - b1 + 31) / 32, (kt + PREP_T - 1) / PREP_T);
      k_prep_ut<<<grid, 256, 0, side.s>>>(U, n, b0, b1, kt, ew, Ut_hi, Ut_lo);
      GQ_LAUNCHED();
    }
    GQ_CUDA(cudaEventRecord(side.join, side.s));
    return GPTQ_OK;
  };
  // Groups of up to G blocks from b0: each block in turn; after block i a
  // thin update (K = SB, block i's residuals, contraction columns
  // i SB .. (i+1) SB) brings every later column of the group up to date, so
  // the group's next block starts from current weights; then one update
  // with K = (blocks) * SB for every column right of the group.
  // Ut[c][t] = U[b0 + t][b0 + SB + c] (TF32 split), E[r][t] = the group's
  // residuals, t < K.
  // maps: 0/1 = Ut hi/lo, 2/3 = E hi/lo.
  int b0 = 0;
  while (b0 < n) {
    const int left = (n - b0 + SB - 1) / SB;
    const int nb = left < G ? left : G;
    const int b1 = b0 + SB;
    const int kt = (nb * SB < n - b0) ? nb * SB : n - b0;  // rows of U the group reads
    int bend = b0;
    if (b1 < n) GQ_TRY(prep(b0, b1, kt));
    for (int i = 0; i < nb; ++i) {
      const int bi = b0 + i * SB;
      const int Bi = (n - bi) < SB ? (n - bi) : SB;
      GQ_TRY(block(bi, Bi, i * SB));
      bend = bi + Bi;
      if (i == 0 && b1 < n) GQ_CUDA(cudaStreamWaitEvent(s, side.join, 0));
      if (i + 1 < nb) {
        const int bn = bi + SB;
        TcJob thin = tc_rect(bn, 0, 2, 0, 0, bn - b1, rows, b0 + kt - bn);
        thin.k0 = i * SB;
        GQ_TRY(gemm_tc_sub(maps, thin, none, SB, status, status, K_SWEEP_GEMM, s));
      }
    }
    if (bend < n)
      GQ_TRY(gemm_pair_sub(maps, tc_rect(bend, 0, 2, 0, 0, bend - b1, rows, n - bend), none, nb * SB,
                           status, status, K_SWEEP_GEMM, s));
    b0 = bend;
  }
  if (status_out) {
    *status_out = status;
    return GPTQ_OK;
  }
  unsigned hs = 0;
  GQ_CUDA(cudaMemcpyAsync(&hs, status, sizeof(unsigned), cudaMemcpyDeviceToHost, s));
  GQ_CUDA(cudaStreamSynchronize(s));
  return hs ? GPTQ_ERR_TIMEOUT : GPTQ_OK;
}

gptq_status sweep_run(float* W, int rows, int n, const float* U, const float* hw, const float* tab,
                      const float* lost, uint8_t* nib, uint8_t* rungs, float* scales, void* ws,
                      size_t ws_bytes, cudaStream_t s) {
  return sweep_core(MODE_Q4, W, rows, n, U, hw, tab, lost, nib, rungs, scales, ws, ws_bytes, s,
                    nullptr, nullptr);
}

gptq_status sweep_enqueue(float* W, int rows, int n, const float* U, const float* hw, const float* tab,
                          const float* lost, uint8_t* nib, uint8_t* rungs, float* scales, void* ws,
                          size_t ws_bytes, cudaStream_t s, const SideStream& side, unsigned** status_out) {
  return sweep_core(MODE_Q4, W, rows, n, U, hw, tab, lost, nib, rungs, scales, ws, ws_bytes, s,
                    nullptr, nullptr, &side, status_out);
}

// The q2tp "placed" sweep: the same blocks and updates with the q2tp rule in
// the block kernel; `codes` is the 2-bit plane (8 bytes a tile).
gptq_status sweep_q2_run(float* W, int rows, int n, const float* U, const float* hw,
                         const float* tab, uint8_t* codes, uint8_t* rungs, float* scales, void* ws,
                         size_t ws_bytes, cudaStream_t s) {
  return sweep_core(MODE_Q2, W, rows, n, U, hw, tab, nullptr, codes, rungs, scales, ws, ws_bytes, s,
                    nullptr, nullptr);
}

gptq_status sweep_q2_enqueue(float* W, int rows, int n, const float* U, const float* hw, const float* tab,
                             uint8_t* codes, uint8_t* rungs, float* scales, void* ws, size_t ws_bytes,
                             cudaStream_t s, const SideStream& side, unsigned** status_out) {
  return sweep_core(MODE_Q2, W, rows, n, U, hw, tab, nullptr, codes, rungs, scales, ws, ws_bytes, s,
                    nullptr, nullptr, &side, status_out);
}

namespace {

// Static rung of every (row, group): the rung rule with unit weights on the
// (dead-zeroed) original weights -- the reading of the converter's own
// choice that act order keeps fixed.
__global__ void k_static_rungs(const float* __restrict__ W, int rows, int n,
                               const float* __restrict__ tab, const float* __restrict__ lost,
                               uint8_t* __restrict__ rungs, float* __restrict__ scales) {
  __shared__ float ones[GROUP];
  if (threadIdx.x < GROUP) ones[threadIdx.x] = 1.f;
  __syncthreads();
  const int gpr = n / GROUP;
  const long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (idx >= (long long)rows * gpr) return;
  const int r = (int)(idx / gpr), g = (int)(idx % gpr);
  float w[GROUP];
  const float4* src = reinterpret_cast<const float4*>(W + (long long)r * n + g * GROUP);
#pragma unroll
  for (int q = 0; q < GROUP / 4; ++q) {
    const float4 v = src[q];
    w[4 * q] = v.x; w[4 * q + 1] = v.y; w[4 * q + 2] = v.z; w[4 * q + 3] = v.w;
  }
  const float* tabrow = tab + (long long)r * 32;
  const int c = q4tp_pick(w, ones, tabrow, lost[2 * r], lost[2 * r + 1]);
  rungs[idx] = (uint8_t)c;
  scales[idx] = tabrow[c];
}

// Wp[r][a] = W[r][perm[a]].
__global__ void k_gather_cols(const float* __restrict__ W, int rows, int n, const int* __restrict__ perm,
                              float* __restrict__ Wp) {
  const long long total = (long long)rows * n;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / n;
    const int a = (int)(i % n);
    Wp[i] = W[r * n + perm[a]];
  }
}

__global__ void k_invperm(const int* __restrict__ perm, int n, int* __restrict__ inv) {
  const int a = blockIdx.x * blockDim.x + threadIdx.x;
  if (a < n) inv[perm[a]] = a;
}

// Nibble tile (r, g) from the permuted codes: column c of the group is
// channel c, found at permuted position inv[c].
__global__ void k_pack_nibbles(const int8_t* __restrict__ codes, int rows, int n,
                               const int* __restrict__ inv, uint8_t* __restrict__ nib) {
  const int gpr = n / GROUP;
  const long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (idx >= (long long)rows * gpr) return;
  const long long r = idx / gpr;
  const int g = (int)(idx % gpr);
  uint32_t words[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int j = 0; j < GROUP; ++j) {
    const int q = codes[r * n + inv[g * GROUP + j]];
    words[j / 8] |= ((uint32_t)(q + 8) & 15u) << (4 * (j % 8));
  }
  reinterpret_cast<uint4*>(nib)[idx] = make_uint4(words[0], words[1], words[2], words[3]);
}

}  // namespace

size_t sweep_act_ws_bytes(int rows, int n) {
  return sweep_ws_bytes(rows, n) + round_up((size_t)rows * n * 4, 256) +
         round_up((size_t)rows * n, 256) + round_up((size_t)n * 4, 256) + 1024;
}

gptq_status static_rungs_run(const float* W, int rows, int n, const float* tab, const float* lost,
                             uint8_t* rungs, float* scales, cudaStream_t s) {
  const long long tot = (long long)rows * (n / GROUP);
  GQ_PROF(K_LADDER, s);
  k_static_rungs<<<(unsigned)((tot + 127) / 128), 128, 0, s>>>(W, rows, n, tab, lost, rungs, scales);
  GQ_LAUNCHED();
  return GPTQ_OK;
}

// The act-order sweep ([host page] gptq_quantize_q4tp_act_order): W (original
// order, dead columns zeroed) is gathered into permuted order, swept against
// the permuted operator with the static rungs, and the codes are packed back
// into the original nibble plane.
gptq_status sweep_act_run(const float* W, int rows, int n, const float* Up, const int* perm,
                          const float* tab, const uint8_t* srungs, uint8_t* nib, void* ws,
                          size_t ws_bytes, cudaStream_t s) {
  Carve c(ws, ws_bytes);
  float* Wp = c.take<float>((size_t)rows * n);
  int8_t* codes = c.take<int8_t>((size_t)rows * n);
  int* inv = c.take<int>((size_t)n);
  if (!c.ok) return GPTQ_ERR_NOMEM;
  const size_t off = round_up(c.off, 256);
  {
    GQ_PROF(K_COPY, s);
    k_gather_cols<<<152 * 8, 256, 0, s>>>(W, rows, n, perm, Wp);
    GQ_LAUNCHED();
    k_invperm<<<(n + 255) / 256, 256, 0, s>>>(perm, n, inv);
    GQ_LAUNCHED();
  }
  GQ_TRY(sweep_core(MODE_Q4_ACT, Wp, rows, n, Up, nullptr, tab, nullptr, nullptr,
                    const_cast<uint8_t*>(srungs),
                    nullptr, static_cast<char*>(ws) + off, ws_bytes - off, s, perm, codes));
  const long long tot = (long long)rows * (n / GROUP);
  GQ_PROF(K_COPY, s);
  k_pack_nibbles<<<(unsigned)((tot + 127) / 128), 128, 0, s>>>(codes, rows, n, inv, nib);
  GQ_LAUNCHED();
  return GPTQ_OK;
}

}  // namespace gq
