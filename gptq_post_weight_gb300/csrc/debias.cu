// Output debias of a quantized matrix ([host page] q2tp_debias_gemm /
// q4tp_debias_gemm, the GEMM form of q2tp_debias_hessian): per row r the
// slope b = (W^ H W^T)_rr / (W H W^T)_rr of the quantized outputs on the
// original ones is removed through the row's f16 lo; codes, rungs and the
// step stay.  The page leaves the lo update (q2tp_unshrink_row) unshown;
// reading: lo' = f16(lo + log2(den / num)) when num > 0 and den > 0, rungs
// rebuilt from (lo', step), each (row, group) scale = its rung's new value.
//
// GB300 layout: H is unpacked into a dense TF32 hi/lo pair (rows of H are its
// columns: H is symmetric), W is split likewise, and Y = W H runs on the
// tensor cores (SM-pair 3xTF32 GEMM, C += A B^T with A = W, B = H, the
// accumulator drained into Y every KSEG of K).  One block per row then
// forms num = W^_r . Y_r and den = W_r . Y_r with compensated f32 sums
// (exact products, two-sum), combines them in f64 and rewrites the row's
// lo, ladder and scales.
#include "common.cuh"

#include <cuda_fp16.h>
#include <math.h>

namespace gq {
namespace {

constexpr int KSEG = 128;  // K per accumulator drain (the tensor cores' f32 sums round toward zero)
constexpr int DB_THREADS = 256;

__device__ __forceinline__ long long poff(long long r, long long n) { return r * (2 * n - r + 1) / 2; }

// Hh/Hl[s][t] = TF32 split of H[s][t], from the packed upper triangle.  One
// 32 x 32 tile per block; a tile below the diagonal is read along the
// packed rows (its transpose) and turned through shared memory.
__global__ void k_unpack_split_h(const float* __restrict__ Hp, int n, float* __restrict__ Hh,
                                 float* __restrict__ Hl) {
  __shared__ float tile[32][33];
  const int t0 = blockIdx.x * 32, s0 = blockIdx.y * 32;
  const int tx = threadIdx.x;
  for (int ty = threadIdx.y; ty < 32; ty += blockDim.y) {
    if (t0 >= s0) {  // on or above the diagonal: row s = s0 + ty, column t = t0 + tx
      const int s = s0 + ty, t = t0 + tx;
      const int a = s < t ? s : t, b = s < t ? t : s;
      tile[ty][tx] = Hp[poff(a, n) + (b - a)];
    } else {  // below: H[s][t] = H[t][s], packed row t = t0 + ty, column s = s0 + tx
      const int t = t0 + ty, s = s0 + tx;
      tile[tx][ty] = Hp[poff(t, n) + (s - t)];
    }
  }
  __syncthreads();
  for (int ty = threadIdx.y; ty < 32; ty += blockDim.y) {
    float h, l;
    split_tf32(tile[ty][tx], h, l);
    const long long o = (long long)(s0 + ty) * n + t0 + tx;
    Hh[o] = h;
    Hl[o] = l;
  }
}

__global__ void k_split(const float* __restrict__ X, long long total4, float* __restrict__ Xh,
                        float* __restrict__ Xl) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total4;
       i += (long long)gridDim.x * blockDim.x) {
    const float4 v = reinterpret_cast<const float4*>(X)[i];
    float4 h, l;
    split_tf32(v.x, h.x, l.x);
    split_tf32(v.y, h.y, l.y);
    split_tf32(v.z, h.z, l.z);
    split_tf32(v.w, h.w, l.w);
    reinterpret_cast<float4*>(Xh)[i] = h;
    reinterpret_cast<float4*>(Xl)[i] = l;
  }
}

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// (hi, lo) += x * y with the product's rounding error kept.
__device__ __forceinline__ void acc_prod(float& hi, float& lo, float x, float y) {
  const float p = __fmul_rn(x, y);
  const float pe = fmaf(x, y, -p);
  float e;
  two_sum(hi, p, hi, e);
  lo = __fadd_rn(lo, __fadd_rn(e, pe));
}

__device__ __forceinline__ double block_sum_f64(double x, double* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  const int wid = threadIdx.x / 32, lane = threadIdx.x % 32;
  __syncthreads();
  if (lane == 0) red[wid] = x;
  __syncthreads();
  double t = 0.0;
  for (int i = 0; i < DB_THREADS / 32; ++i) t += red[i];
  return t;
}

// One block per row: num, den, then lo', the ladder and the scales.
template <bool TWO_BIT>
__global__ void __launch_bounds__(DB_THREADS) k_debias_rows(
    const float* __restrict__ W, const float* __restrict__ Y, int n, const uint8_t* __restrict__ codes,
    const uint8_t* __restrict__ rungs, float* __restrict__ tab, float* __restrict__ lost,
    float* __restrict__ scales, double* __restrict__ num_den) {
  __shared__ double red[DB_THREADS / 32];
  __shared__ float stab[32];
  __shared__ int s_update;
  const int r = blockIdx.x, tid = threadIdx.x;
  const int gpr = n / GROUP;
  const float* wr = W + (long long)r * n;
  const float* yr = Y + (long long)r * n;
  const float* sr = scales + (long long)r * gpr;
  float nh = 0.f, nl = 0.f, dh = 0.f, dl = 0.f;
  for (int i = 4 * tid; i < n; i += 4 * DB_THREADS) {
    const float4 w = *reinterpret_cast<const float4*>(wr + i);
    const float4 y = *reinterpret_cast<const float4*>(yr + i);
    const float s = sr[i / GROUP];
    float lev[4];
    if (TWO_BIT) {
      const uint32_t b = codes[(long long)r * (n / 4) + i / 4];
#pragma unroll
      for (int j = 0; j < 4; ++j) lev[j] = (float)((b >> (2 * j)) & 3u) - 1.5f;
    } else {
      const uint32_t b = *reinterpret_cast<const uint16_t*>(codes + (long long)r * (n / 2) + i / 2);
#pragma unroll
      for (int j = 0; j < 4; ++j) lev[j] = (float)((b >> (4 * j)) & 15u) - 8.f;
    }
    acc_prod(nh, nl, __fmul_rn(lev[0], s), y.x);
    acc_prod(nh, nl, __fmul_rn(lev[1], s), y.y);
    acc_prod(nh, nl, __fmul_rn(lev[2], s), y.z);
    acc_prod(nh, nl, __fmul_rn(lev[3], s), y.w);
    acc_prod(dh, dl, w.x, y.x);
    acc_prod(dh, dl, w.y, y.y);
    acc_prod(dh, dl, w.z, y.z);
    acc_prod(dh, dl, w.w, y.w);
  }
  const double num = block_sum_f64((double)nh + (double)nl, red);
  const double den = block_sum_f64((double)dh + (double)dl, red);
  if (tid == 0) {
    const float lo = lost[2 * r], st = lost[2 * r + 1];
    int upd = 0;
    if (num > 0.0 && den > 0.0) {
      const float lo2 = __half2float(__double2half((double)lo + log2(den / num)));
      lost[2 * r] = lo2;
      upd = 0;
      for (int c = 0; c < 32; ++c) upd |= tab[r * 32 + c] > 0.f;
      if (upd) {
        for (int c = 0; c < 32; ++c) {
          const double e = TWO_BIT ? (double)lo2 + (double)(c - 1) * (double)st
                                   : (double)lo2 + (double)c * (double)st;
          stab[c] = (TWO_BIT && c == 0) ? 0.f : (float)exp2(e);
        }
      }
    }
    s_update = upd;
    if (num_den) {
      num_den[2 * r] = num;
      num_den[2 * r + 1] = den;
    }
  }
  __syncthreads();
  if (!s_update) return;
  if (tid < 32) tab[r * 32 + tid] = stab[tid];
  for (int g = tid; g < gpr; g += DB_THREADS)
    scales[(long long)r * gpr + g] = stab[rungs[(long long)r * gpr + g] & 31];
}

}  // namespace

size_t debias_ws_bytes(int rows, int n) {
  return 2 * round_up((size_t)n * n * 4, 256) + 3 * round_up((size_t)rows * n * 4, 256) + 1024;
}

gptq_status debias_run(int bits, const float* W, int rows, int n, const float* Hp,
                       const uint8_t* codes, const uint8_t* rungs, float* tab, float* lost,
                       float* scales, double* num_den, void* ws, size_t ws_bytes, cudaStream_t s) {
  Carve c(ws, ws_bytes);
  float* Hh = c.take<float>((size_t)n * n);
  float* Hl = c.take<float>((size_t)n * n);
  float* Wh = c.take<float>((size_t)rows * n);
  float* Wl = c.take<float>((size_t)rows * n);
  float* Y = c.take<float>((size_t)rows * n);
  unsigned* status = c.take<unsigned>(4);
  if (!c.ok) return GPTQ_ERR_NOMEM;
  GQ_CUDA(cudaMemsetAsync(status, 0, sizeof(unsigned), s));
  GQ_CUDA(cudaMemsetAsync(Y, 0, (size_t)rows * n * 4, s));
  {
    GQ_PROF(K_DEBIAS, s);
    k_unpack_split_h<<<dim3(n / 32, n / 32), dim3(32, 8), 0, s>>>(Hp, n, Hh, Hl);
    GQ_LAUNCHED();
  }
  {
    GQ_PROF(K_DEBIAS, s);
    k_split<<<num_sms() * 8, 256, 0, s>>>(W, (long long)rows * n / 4, Wh, Wl);
    GQ_LAUNCHED();
  }
  OperandMaps maps;  // 0/1 = W hi/lo, 2/3 = H hi/lo
  GQ_TRY(make_operand_map(&maps.m[0], Wh, rows, n));
  GQ_TRY(make_operand_map(&maps.m[1], Wl, rows, n));
  GQ_TRY(make_operand_map(&maps.m[2], Hh, n, n));
  GQ_TRY(make_operand_map(&maps.m[3], Hl, n, n));
  GQ_TRY(make_c_map(&maps.c, Y, rows, n, n));
  TcJob j = tc_rect(0, 0, 0, 0, 2, 0, rows, n);
  j.add = 1;   // Y += W H^T (= W H)
  j.band = 8;  // 76 concurrent tiles ~ 8 x 9.5: about 17 operand panels in flight instead of 70
  GQ_TRY(gemm_pair_sub(maps, j, TcJob{}, n, status, status, K_DEBIAS_GEMM, s, FusedPotrf{}, KSEG));
  {
    GQ_PROF(K_DEBIAS, s);
    if (bits == 2)
      k_debias_rows<true><<<rows, DB_THREADS, 0, s>>>(W, Y, n, codes, rungs, tab, lost, scales, num_den);
    else
      k_debias_rows<false><<<rows, DB_THREADS, 0, s>>>(W, Y, n, codes, rungs, tab, lost, scales, num_den);
    GQ_LAUNCHED();
  }
  unsigned hs = 0;
  GQ_CUDA(cudaMemcpyAsync(&hs, status, sizeof(unsigned), cudaMemcpyDeviceToHost, s));
  GQ_CUDA(cudaStreamSynchronize(s));
  return hs ? GPTQ_ERR_TIMEOUT : GPTQ_OK;
}

}  // namespace gq
