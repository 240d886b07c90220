// The q4tp sweep on the device (cortiq-engine src/gpu_wgpu/gptq_dev.rs,
// module doc step 5 and WGSL q4tp_group / q4tp_trail; the same rule as the
// host page's gptq_quantize_q4tp).
//
// Lazy blocks of SB = 128 columns (4 groups): one kernel runs the four
// groups of a block for 64 rows per CTA out of shared memory (rung choice,
// rounding, in-group feedback, then the group's residuals into the rest of
// the block), then one GEMM applies the block's residuals to every later
// column: W[:, b1:] -= E_blk U[b0:b1, b1:].  With SB = 32 this is the fold
// page's per-group q4tp_trail; a wider block is the same mathematics with
// the residual sums taken in a different order.
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
// [host page] gptq_quantize_q4tp), one warp per row:
//  * nominal = clamp(round_half_away((log2(amax/7) - lo) / step), 0, 31)
//    (0 if amax == 0 or step <= 0; log2 = the f64 value rounded to f32);
//  * rung = best of nominal-2..min(nominal+1, 31) by sum_t hw_t (w_t - q_t s)^2
//    with q_t = clamp(rne(w_t * (1/s)), -8, 7), strict '<', s <= 0 skipped;
//  * per column j: q_j = clamp(rne(w_j / s), -8, 7) (0 if s <= 0), nibble
//    q_j + 8, e_j = (w_j - q_j s) / U_jj (0 if U_jj <= 0), w_t -= e_j U_jt
//    for t > j.
// One rounding per operation (no contraction), so the f32 results are the
// pages' bit for bit.
// Lane t holds column t of the group.  Every floating-point step is taken in
// the pages' order: the
// candidate errors are summed sequentially over t (the terms are gathered by
// shuffles in column order), and the feedback is applied column by column.
// `wl` holds this lane's value of the group; `wlater[k]` its values of the
// later groups in the same block (nl of them), which get the same per-column
// update w -= e_j U[j][c] (one rounding for the product, one for the
// difference), as the host page's full-row update does.  Returns the rung;
// q, e are this lane's code and residual.
template <int NLATER>
__device__ __forceinline__ int q4tp_group_warp(float& wl, float (&wlater)[NLATER], int nl,
                                               float hwl, const float* tabrow, float lo, float st,
                                               const float* U, int ldu, int lane, float& s_out,
                                               float& q_out, float& e_out) {
  float amax = fabsf(wl);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  int nominal = 0;
  if (amax > 0.f && st > 0.f) {
    const float x = __fdiv_rn(amax, 7.0f);
    const float l2 = (float)log2((double)x);
    const float tt = __fdiv_rn(__fsub_rn(l2, lo), st);
    nominal = (int)fminf(fmaxf(roundf(tt), 0.f), 31.f);
  }
  int best_c = nominal;
  if (amax > 0.f) {
    const int lo_c = nominal >= 2 ? nominal - 2 : 0;
    const int hi_c = nominal + 1 < 31 ? nominal + 1 : 31;
    float term[4], err[4];
    bool valid[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int cand = lo_c + k;
      const float sc = cand <= hi_c ? tabrow[cand] : 0.f;
      valid[k] = cand <= hi_c && sc > 0.f;
      const float iv = __fdiv_rn(1.0f, valid[k] ? sc : 1.f);
      const float q = fminf(fmaxf(rintf(__fmul_rn(wl, iv)), -8.f), 7.f);
      const float d = __fsub_rn(wl, __fmul_rn(q, sc));
      term[k] = __fmul_rn(__fmul_rn(hwl, d), d);
      err[k] = 0.f;
    }
#pragma unroll
    for (int t = 0; t < GROUP; ++t) {
#pragma unroll
      for (int k = 0; k < 4; ++k) err[k] = __fadd_rn(err[k], __shfl_sync(0xffffffffu, term[k], t));
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
  const float s = tabrow[best_c];
  float myq = 0.f, mye = 0.f;
#pragma unroll 4
  for (int j = 0; j < GROUP; ++j) {
    float e = 0.f;
    if (lane == j) {
      float q = 0.f;
      if (s > 0.f) q = fminf(fmaxf(rintf(__fdiv_rn(wl, s)), -8.f), 7.f);
      const float dj = U[j * ldu + j];
      if (dj > 0.f) e = __fdiv_rn(__fsub_rn(wl, __fmul_rn(q, s)), dj);
      myq = q;
      mye = e;
    }
    e = __shfl_sync(0xffffffffu, e, j);
    if (e != 0.f) {
      const float* urow = U + j * ldu;
      if (lane > j) wl = __fsub_rn(wl, __fmul_rn(e, urow[lane]));
#pragma unroll
      for (int k = 0; k < NLATER; ++k)
        if (k < nl) wlater[k] = __fsub_rn(wlater[k], __fmul_rn(e, urow[GROUP * (k + 1) + lane]));
    }
  }
  s_out = s;
  q_out = myq;
  e_out = mye;
  return best_c;
}

// Packs the 32 codes of a warp into the tile's 4 words (byte j/2, low nibble
// for even j) and writes them: lanes 0..3 store one word each.
__device__ __forceinline__ void store_nibbles_warp(float q, int lane, uint32_t* dst) {
  const uint32_t nb = (uint32_t)((int)q + 8) & 15u;
  uint32_t word = 0u;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t v = __shfl_sync(0xffffffffu, nb, (lane & 3) * 8 + i);
    word |= v << (4 * i);
  }
  if (lane < 4) dst[lane] = word;
}

// Per-row ladder ([host page] gptq_quantize_q4tp_dev's tab / lost; the
// converter itself is not on the pages -- reading in the header).
__global__ void __launch_bounds__(128) k_ladder(const float* __restrict__ W, int n,
                                                float* __restrict__ tab, float* __restrict__ lost) {
  const int r = blockIdx.x;
  const float* wr = W + (long long)r * n;
  const int gpr = n / GROUP;
  float xmin = INFINITY, xmax = 0.f;
  int cnt = 0;
  for (int g = threadIdx.x; g < gpr; g += blockDim.x) {
    const float4* p = reinterpret_cast<const float4*>(wr + g * GROUP);
    float a = 0.f;
#pragma unroll
    for (int q = 0; q < GROUP / 4; ++q) {
      float4 v = p[q];
      a = fmaxf(a, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    if (a > 0.f) {
      const float x = __fdiv_rn(a, 7.0f);
      xmin = fminf(xmin, x);
      xmax = fmaxf(xmax, x);
      ++cnt;
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    xmin = fminf(xmin, __shfl_xor_sync(0xffffffffu, xmin, o));
    xmax = fmaxf(xmax, __shfl_xor_sync(0xffffffffu, xmax, o));
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  }
  __shared__ float smin[4], smax[4];
  __shared__ int scnt[4];
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
    for (int i = 1; i < 4; ++i) {
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

// The group rule on given tiles, one warp per row (the same device code as
// the sweep's block kernel).
__global__ void __launch_bounds__(256) k_group(const float* __restrict__ tile, int rows,
                                               const float* __restrict__ ublk,
                                               const float* __restrict__ hw,
                                               const float* __restrict__ tab,
                                               const float* __restrict__ lost,
                                               uint8_t* __restrict__ nib, uint8_t* __restrict__ rungs,
                                               float* __restrict__ scales, float* __restrict__ E) {
  __shared__ float Us[GROUP * GROUP];
  for (int e = threadIdx.x; e < GROUP * GROUP; e += blockDim.x) Us[e] = ublk[e];
  __syncthreads();
  const int lane = threadIdx.x % 32;
  const int r = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (r >= rows) return;
  float wl = tile[(long long)r * GROUP + lane];
  float none[1] = {0.f};
  float s, q, e;
  const int c = q4tp_group_warp<1>(wl, none, 0, hw[lane], tab + (long long)r * 32, lost[2 * r],
                                   lost[2 * r + 1], Us, GROUP, lane, s, q, e);
  store_nibbles_warp(q, lane, reinterpret_cast<uint32_t*>(nib + (long long)r * 16));
  if (lane == 0) {
    rungs[r] = (uint8_t)c;
    scales[r] = s;
  }
  E[(long long)r * GROUP + lane] = e;
}

constexpr int SWEEP_WARPS = 16;

// One lazy block [b0, b0+B) (B <= SB): one warp per row, rows strided over
// the grid's warps.  The block's U (B x B) and rung weights sit in shared
// memory; each lane keeps its column of every group of the block in
// registers.  Group by group: the rung rule, codes, residuals and the
// per-column feedback into the rest of the group and the later groups of the
// block; then nibbles, rung, scale and the residuals E (TF32 hi/lo, the
// trailing GEMM's operand) go out.
__global__ void __launch_bounds__(SWEEP_WARPS * 32) k_sweep_block(
    const float* __restrict__ W, int rows, int n, int b0, int B, const float* __restrict__ U,
    const float* __restrict__ hw, const float* __restrict__ tab, const float* __restrict__ lost,
    uint8_t* __restrict__ nib, uint8_t* __restrict__ rungs, float* __restrict__ scales,
    float* __restrict__ E_hi, float* __restrict__ E_lo) {
  extern __shared__ __align__(16) float sm[];
  float* Us = sm;            // [SB][SB]
  float* hws = Us + SB * SB; // [SB]
  // The block's U rows as float4 (B is a multiple of 32), 8 loads in flight
  // per thread per batch.
  {
    const int q4 = B / 4;
    const int tot = B * q4;
#pragma unroll 1
    for (int b = 0; b < tot; b += 8 * SWEEP_WARPS * 32) {
      float4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = b + threadIdx.x + i * SWEEP_WARPS * 32;
        if (e < tot)
          v[i] = *reinterpret_cast<const float4*>(U + (long long)(b0 + e / q4) * n + b0 + 4 * (e % q4));
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = b + threadIdx.x + i * SWEEP_WARPS * 32;
        if (e < tot) *reinterpret_cast<float4*>(Us + (e / q4) * SB + 4 * (e % q4)) = v[i];
      }
    }
  }
  for (int e = threadIdx.x; e < B; e += blockDim.x) hws[e] = hw[b0 + e];
  __syncthreads();
  const int lane = threadIdx.x % 32;
  const int ng = B / GROUP;
  const int gpr = n / GROUP;
  for (int r = blockIdx.x * SWEEP_WARPS + threadIdx.x / 32; r < rows; r += gridDim.x * SWEEP_WARPS) {
    const float* wrow = W + (long long)r * n + b0;
    float wv[SB / GROUP];
#pragma unroll
    for (int g = 0; g < SB / GROUP; ++g) wv[g] = g < ng ? wrow[g * GROUP + lane] : 0.f;
    const float lo = lost[2 * r], st = lost[2 * r + 1];
    const float* tabrow = tab + (long long)r * 32;
#pragma unroll
    for (int g = 0; g < SB / GROUP; ++g) {
      if (g >= ng) break;
      float later[SB / GROUP - 1];
#pragma unroll
      for (int k = 0; k < SB / GROUP - 1; ++k) later[k] = (g + 1 + k < SB / GROUP) ? wv[(g + 1 + k) % (SB / GROUP)] : 0.f;
      float s, q, e;
      const int c = q4tp_group_warp<SB / GROUP - 1>(wv[g], later, ng - g - 1, hws[g * GROUP + lane], tabrow,
                                                    lo, st, Us + g * GROUP * SB + g * GROUP, SB, lane, s,
                                                    q, e);
#pragma unroll
      for (int k = 0; k < SB / GROUP - 1; ++k)
        if (g + 1 + k < SB / GROUP) wv[(g + 1 + k) % (SB / GROUP)] = later[k];
      const long long tix = (long long)r * gpr + b0 / GROUP + g;
      store_nibbles_warp(q, lane, reinterpret_cast<uint32_t*>(nib + tix * 16));
      if (lane == 0) {
        rungs[tix] = (uint8_t)c;
        scales[tix] = s;
      }
      float h, l;
      split_tf32(e, h, l);
      E_hi[(long long)r * SB + g * GROUP + lane] = h;
      E_lo[(long long)r * SB + g * GROUP + lane] = l;
    }
  }
}

// Ut[c][t] = U[b0 + t][b1 + c]: the block row of U, K-major for the GEMM,
// stored as its TF32 hi/lo split.
__global__ void k_prep_ut(const float* __restrict__ U, int n, int b0, int b1,
                          float* __restrict__ Ut_hi, float* __restrict__ Ut_lo) {
  __shared__ float tile[32][33];
  const int c0 = blockIdx.x * 32, t0 = blockIdx.y * 32;
  const int ncol = n - b1;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int c = c0 + threadIdx.x;
    tile[i][threadIdx.x] = (c < ncol) ? U[(long long)(b0 + t0 + i) * n + b1 + c] : 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int c = c0 + i;
    if (c < ncol) {
      float h, l;
      split_tf32(tile[threadIdx.x][i], h, l);
      Ut_hi[(long long)c * SB + t0 + threadIdx.x] = h;
      Ut_lo[(long long)c * SB + t0 + threadIdx.x] = l;
    }
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

size_t sweep_ws_bytes(int rows, int n) {
  return 2 * round_up((size_t)rows * SB * 4, 256) + 2 * round_up((size_t)n * SB * 4, 256) + 1024;
}

static gptq_status sweep_attrs() {
  static bool done = false;
  if (done) return GPTQ_OK;
  GQ_CUDA(cudaFuncSetAttribute(k_sweep_block, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (SB * SB + SB) * 4));
  done = true;
  return GPTQ_OK;
}

gptq_status ladder_run(const float* W, int rows, int n, float* tab, float* lost, cudaStream_t s) {
  GQ_PROF(K_LADDER, s);
  k_ladder<<<rows, 128, 0, s>>>(W, n, tab, lost);
  GQ_LAUNCHED();
  return GPTQ_OK;
}

gptq_status group_run(const float* tile, int rows, const float* ublk, const float* hw,
                      const float* tab, const float* lost, uint8_t* nib, uint8_t* rungs,
                      float* scales, float* E, cudaStream_t s) {
  GQ_PROF(K_GROUP, s);
  k_group<<<(rows + 7) / 8, 256, 0, s>>>(tile, rows, ublk, hw, tab, lost, nib, rungs, scales, E);
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
// host-side name is only a stand-in; the device address comes from
// cudaGetSymbolAddress, looked up once per device (on that device's first
// call) and cached.
namespace {
__device__ __align__(256) unsigned char g_noalloc_scratch[GPTQ_SWEEP_NOALLOC_SCRATCH_BYTES];
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};
}  // namespace

gptq_status noalloc_scratch(void** out) {
  int dev = 0;
  GQ_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return GPTQ_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return GPTQ_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return GPTQ_OK;
}

gptq_status sweep_run(float* W, int rows, int n, const float* U, const float* hw, const float* tab,
                      const float* lost, uint8_t* nib, uint8_t* rungs, float* scales, void* ws,
                      size_t ws_bytes, cudaStream_t s) {
  GQ_TRY(sweep_attrs());
  Carve c(ws, ws_bytes);
  float* E_hi = c.take<float>((size_t)rows * SB);
  float* E_lo = c.take<float>((size_t)rows * SB);
  float* Ut_hi = c.take<float>((size_t)n * SB);
  float* Ut_lo = c.take<float>((size_t)n * SB);
  unsigned* status = c.take<unsigned>(4);
  if (!c.ok) return GPTQ_ERR_NOMEM;
  GQ_CUDA(cudaMemsetAsync(status, 0, sizeof(unsigned), s));
  OperandMaps maps;  // 0/1 = Ut hi/lo, 2/3 = E hi/lo
  GQ_TRY(make_operand_map(&maps.m[0], Ut_hi, n, SB));
  GQ_TRY(make_operand_map(&maps.m[1], Ut_lo, n, SB));
  GQ_TRY(make_operand_map(&maps.m[2], E_hi, rows, SB));
  GQ_TRY(make_operand_map(&maps.m[3], E_lo, rows, SB));
  GQ_TRY(make_c_map(&maps.c, W, rows, n, n));
  const int smem = (SB * SB + SB) * 4;
  const TcJob none{};
  int sms = 0, dev = 0;
  GQ_CUDA(cudaGetDevice(&dev));
  GQ_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int want = (rows + SWEEP_WARPS - 1) / SWEEP_WARPS;
  const int blocks = want < 2 * sms ? want : 2 * sms;
  for (int b0 = 0; b0 < n; b0 += SB) {
    const int B = (n - b0) < SB ? (n - b0) : SB;
    const int b1 = b0 + B;
    {
      GQ_PROF(K_SWEEP_BLOCK, s);
      k_sweep_block<<<blocks, SWEEP_WARPS * 32, smem, s>>>(
          W, rows, n, b0, B, U, hw, tab, lost, nib, rungs, scales, E_hi, E_lo);
      GQ_LAUNCHED();
    }
    if (b1 < n) {
      {
        GQ_PROF(K_PREP_UT, s);
        dim3 grid((n - b1 + 31) / 32, SB / 32);
        k_prep_ut<<<grid, dim3(32, 8), 0, s>>>(U, n, b0, b1, Ut_hi, Ut_lo);
        GQ_LAUNCHED();
      }
      GQ_TRY(gemm_tc_sub(maps, tc_rect(b1, 0, 2, 0, 0, 0, rows, n - b1), none, SB, status,
                         status, K_SWEEP_GEMM, s));
    }
  }
  unsigned hs = 0;
  GQ_CUDA(cudaMemcpyAsync(&hs, status, sizeof(unsigned), cudaMemcpyDeviceToHost, s));
  GQ_CUDA(cudaStreamSynchronize(s));
  return hs ? GPTQ_ERR_TIMEOUT : GPTQ_OK;
}

}  // namespace gq
