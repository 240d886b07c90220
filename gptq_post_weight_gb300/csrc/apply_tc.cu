// Both triangular solves of one fold step as one product on the tensor
// cores: Z = V Linv^T, Linv = L_kk^-1 (the step's diagonal block inverted).
//
//  * rows r >= s0 = k + NB: the Cholesky panel ([fold page] chol_panel),
//    v = A[r][k .. k+NB), z -> the panel buffer P;
//  * rows r < s0: the inverse's block row ([fold page] inv_rows),
//    v = Y[r][k .. k+NB) (for the rows of block k itself the unit vector
//    e_{r-k}: that row of Z is a column of Linv), z -> the buffer Yp, and
//    the finished entries of U ([fold page] make_u):
//    U[n-1-i][n-1-r] = X[i][r] / |d_{n-1-r}|, i = k + c (d given with a dead
//    channel's sign), taken as X times
//    the rounded reciprocal (within a rounding of the quotient);
//  * rows of the next block (s0 <= r < zero_end): their Yp entries in this
//    half are zero (X is lower triangular).
// z goes out as its TF32 hi/lo split, the operand format of the update
// GEMM, in columns [col0, col0 + NB) of the 2 NB-wide panel buffers.
//
// One CTA per 128-row tile (persistent over tiles when there are more tiles
// than SMs), 6 warps.  A CTA holds about one tile, so the kernel is shaped
// for latency: every load of a tile is in flight at once.  Linv is lower
// triangular, so slice kc of u (32 wide) meets only the columns c >= 32 kc
// of Z: its MMAs run with N = NB - 32 kc into the accumulator's columns
// from 32 kc, and only Linv's rows c >= 32 kc are loaded (boxes of 32
// rows).  That keeps the whole tile's operands in 208 KB of shared memory.
//   warp 0      TMA producers, lane kc for slice kc: the tile's raw f32
//               vectors (a 128 x 32 box of A, 128-byte swizzle) and the rows
//               of the TF32 pair of Linv the slice meets;
//   warps 2-5   split each slice's raw vectors into their TF32 pair in place
//               (the unit rows of block k written directly), then, once the
//               product is in tensor memory, the epilogue: tcgen05.ld of one
//               row per thread, TF32 split into swizzled staging slices (in
//               the operand area, free once the MMAs are done) stored by
//               TMA, U's entries straight from registers (one warp
//               instruction covers 32 consecutive columns of a U row);
//   warp 1      allocates 128 TMEM columns and issues the 3xTF32 MMAs
//               (V_lo Linv_hi + V_hi Linv_lo + V_hi Linv_hi, f32 accumulate).
// Every wait is bounded (WaitCfg); on expiry the kernel stops, lets what it
// started land, frees its tensor memory and sets bit 1 of the flag word.
#include "common.cuh"
#include "tcgen05.cuh"

namespace gq {
namespace {

constexpr int AM = 128;              // rows per tile
constexpr int AK = 32;               // u per slice
constexpr int ANCH = NB / AK;        // slices per tile
constexpr int A_BOX = AM * AK * 4;   // 16 KB: one 128 x 32 f32 box
constexpr int L_BOX = 32 * AK * 4;   // 4 KB: 32 rows of Linv, one slice of u
constexpr int V_AREA = ANCH * 2 * A_BOX;                     // V hi, V lo per slice: 128 KB
constexpr int L_ROWS = NB * ANCH - AK * (ANCH * (ANCH - 1) / 2);  // 128 + 96 + 64 + 32
constexpr int L_AREA = L_ROWS * AK * 4;                      // one part (hi or lo): 40 KB
constexpr int A_SMEM = V_AREA + 2 * L_AREA + 1024;
constexpr int A_THREADS = 192;
constexpr uint32_t A_TMEM_COLS = NB;

// Byte offset of slice kc's Linv rows (c >= 32 kc) inside one part.
__host__ __device__ constexpr int l_off(int kc) { return (NB * kc - AK * (kc * (kc - 1) / 2)) * AK * 4; }

// kind::tf32, D f32, A and B TF32 K-major, M = AM, N = nn.
__device__ __forceinline__ uint32_t idesc_n(int nn) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(nn >> 3) << 17) | ((uint32_t)(AM >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32_1(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                           uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}

__device__ __forceinline__ float4 split4(float4 x, float4& lo) {
  float4 hi;
  split_tf32(x.x, hi.x, lo.x);
  split_tf32(x.y, hi.y, lo.y);
  split_tf32(x.z, hi.z, lo.z);
  split_tf32(x.w, hi.w, lo.w);
  return hi;
}

__global__ void __launch_bounds__(A_THREADS, 1)
    k_apply_tc(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap lhi_map,
               const __grid_constant__ CUtensorMap llo_map, const __grid_constant__ CUtensorMap phi_map,
               const __grid_constant__ CUtensorMap plo_map, const __grid_constant__ CUtensorMap yhi_map,
               const __grid_constant__ CUtensorMap ylo_map, int k, int s0, int N, int col0, int zero_end,
               unsigned* flag, float* __restrict__ U, const float* __restrict__ dsg, int n, WaitCfg wc) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  // full[kc]: slice kc landed; conv[kc]: slice kc split; tfull: the tile's
  // product is in tensor memory; ofree: the epilogue is done with the
  // operand area and tensor memory (the next tile may load).
  __shared__ __align__(8) uint64_t full[ANCH], conv[ANCH], tfull, ofree, drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh, skip_sh, issued_sh[ANCH];
  if (threadIdx.x == 0) skip_sh = (*(volatile const unsigned*)flag != 0u) ? 1 : 0;
  __syncthreads();
  if (skip_sh) return;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int ntiles = N / AM;
  if (threadIdx.x == 0) {
    for (int c = 0; c < ANCH; ++c) {
      mbar_init(&full[c], 1);
      mbar_init(&conv[c], 128);
    }
    mbar_init(&tfull, 1);
    mbar_init(&ofree, 1);
    mbar_init(&drain, 1);
    abort_sh = 0;
    for (int c = 0; c < ANCH; ++c) issued_sh[c] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_base_sh)),
                 "r"(A_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  volatile int* abort = &abort_sh;
  uint8_t* const larea = smem + V_AREA;  // Linv hi part, then lo part

  if (warp == 0) {
    if (lane < ANCH) {
      // Lane kc issues slice kc's loads (the four slices' loads go out side
      // by side).
      const int kc = lane;
      int it = 0;
      // wc.no_loads (a test hook): issue nothing; the waits below run out.
      for (int t = blockIdx.x; t < ntiles && !*abort && !wc.no_loads; t += gridDim.x, ++it) {
        if (it > 0 && !mbar_wait(&ofree, (uint32_t)((it - 1) & 1), abort, wc.ns)) break;
        const int r0 = t * AM;
        mbar_expect_tx(&full[kc], A_BOX + 2 * (ANCH - kc) * L_BOX);
        tma_load_2d(smem_u32(smem + kc * 2 * A_BOX), &amap, k + kc * AK, r0, &full[kc]);
#pragma unroll 1
        for (int cb = kc; cb < ANCH; ++cb) {
          const uint32_t o = (uint32_t)(l_off(kc) + (cb - kc) * L_BOX);
          tma_load_2d(smem_u32(larea + o), &lhi_map, kc * AK, cb * 32, &full[kc]);
          tma_load_2d(smem_u32(larea + L_AREA + o), &llo_map, kc * AK, cb * 32, &full[kc]);
        }
        issued_sh[kc] = it + 1;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int it = 0;
      for (int t = blockIdx.x; t < ntiles && !*abort; t += gridDim.x, ++it) {
        bool ok = true;
        for (int kc = 0; kc < ANCH; ++kc) {
          if (!mbar_wait(&conv[kc], (uint32_t)(it & 1), abort, wc.ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t v_hi = smem_u32(smem + kc * 2 * A_BOX), v_lo = v_hi + A_BOX;
          const uint32_t l_hi = smem_u32(larea + l_off(kc)), l_lo = l_hi + L_AREA;
          const uint32_t d = tmem + (uint32_t)(kc * AK);  // columns c >= 32 kc
          const uint32_t id = idesc_n(NB - kc * AK);
#pragma unroll
          for (int kk = 0; kk < AK / 8; ++kk) {
            const uint32_t off = (uint32_t)kk * 32u;
            mma_tf32_1(d, sdesc(v_lo + off), sdesc(l_hi + off), id, (kc || kk) ? 1u : 0u);
            mma_tf32_1(d, sdesc(v_hi + off), sdesc(l_lo + off), id, 1u);
            mma_tf32_1(d, sdesc(v_hi + off), sdesc(l_hi + off), id, 1u);
          }
        }
        if (!ok) break;
        mma_commit(&tfull);
      }
      // Every MMA issued has completed once `drain` flips.
      mma_commit(&drain);
      if (!mbar_wait(&drain, 0u, abort, wc.ns)) {
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(&drain, 0u) && globaltimer() - t0 < wc.ns) {
        }
      }
    }
  } else {
    const int et = threadIdx.x - 64;  // 0..127
    const int q = warp & 3;           // TMEM lane quarter this warp may read
    const int rr = q * 32 + lane;     // the tile row this thread drains
    const bool leader = threadIdx.x == 64;
    int chunk = 0, it = 0;
    bool go = true;
    for (int t = blockIdx.x; go && t < ntiles; t += gridDim.x, ++it) {
      const int r0 = t * AM;
      const bool unit = r0 == k;  // the rows of block k: unit vectors
      for (int kc = 0; kc < ANCH; ++kc) {
        if (!epi_all(mbar_wait(&full[kc], (uint32_t)(it & 1), abort, wc.ns))) {
          go = false;
          break;
        }
        float4* vh = reinterpret_cast<float4*>(smem + kc * 2 * A_BOX);
        float4* vl = reinterpret_cast<float4*>(smem + kc * 2 * A_BOX + A_BOX);
#pragma unroll
        for (int i = 0; i < A_BOX / 16 / 128; ++i) {
          const int e = et + 128 * i;  // float4 slot of the swizzled box
          float4 x;
          if (unit) {
            const int row = e >> 3, c4 = (e & 7) ^ (row & 7);  // logical 16-byte chunk
            const int u0 = kc * AK + 4 * c4;
            x = make_float4(u0 == row ? 1.f : 0.f, u0 + 1 == row ? 1.f : 0.f, u0 + 2 == row ? 1.f : 0.f,
                            u0 + 3 == row ? 1.f : 0.f);
          } else {
            x = vh[e];
          }
          float4 lo;
          const float4 hi = split4(x, lo);
          vh[e] = hi;
          vl[e] = lo;
        }
        fence_proxy_async_smem();
        mbar_arrive(&conv[kc]);
      }
      if (!go) break;
      if (!epi_all(mbar_wait(&tfull, (uint32_t)(it & 1), abort, wc.ns))) {
        go = false;
        break;
      }
      tc_fence_after();
      const int r = r0 + rr;
      const bool panel = r0 >= s0;
      const CUtensorMap* mh = panel ? &phi_map : &yhi_map;
      const CUtensorMap* ml = panel ? &plo_map : &ylo_map;
      const bool uok = !panel && r < n;
      const float rdm = uok ? __frcp_rn(fabsf(dsg[n - 1 - r])) : 0.f;
      float* ucol = U + (n - 1 - r);  // column n-1-r of U
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int cc = 0; cc < NB; cc += 32) {
        uint32_t v[32];
        tmem_ld32(tbase + (uint32_t)cc, v);
        tmem_ld_wait();
        // Staging: the first two slices' V areas (hi slice, then lo slice).
        uint8_t* buf = smem + (chunk & 1) * 2 * A_BOX;
        if (leader && chunk >= 2) bulk_wait_read1();  // the stores that last read `buf` are done
        epi_sync();
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 z = make_float4(__uint_as_float(v[4 * c4]), __uint_as_float(v[4 * c4 + 1]),
                                       __uint_as_float(v[4 * c4 + 2]), __uint_as_float(v[4 * c4 + 3]));
          float4 lo;
          const float4 hi = split4(z, lo);
          const int off = rr * 128 + ((c4 ^ (rr & 7)) * 16);
          *reinterpret_cast<float4*>(buf + off) = hi;
          *reinterpret_cast<float4*>(buf + A_BOX + off) = lo;
        }
        if (uok) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int i = k + cc + j;
            if (i < n) ucol[(long long)(n - 1 - i) * n] = __fmul_rn(__uint_as_float(v[j]), rdm);
          }
        }
        fence_proxy_async_smem();
        epi_sync();
        if (leader) {
          tma_store_2d(mh, smem_u32(buf), col0 + cc, r0);
          tma_store_2d(ml, smem_u32(buf + A_BOX), col0 + cc, r0);
          bulk_commit();
        }
        ++chunk;
      }
      if (panel && r0 < zero_end) {
        // The next block's rows: zeros into their Yp entries of this half.
        uint8_t* buf = smem + (chunk & 1) * 2 * A_BOX;
        if (leader) bulk_wait_read1();
        epi_sync();
#pragma unroll
        for (int i = 0; i < A_BOX / 16 / 128; ++i)
          reinterpret_cast<float4*>(buf)[et + 128 * i] = make_float4(0.f, 0.f, 0.f, 0.f);
        fence_proxy_async_smem();
        epi_sync();
        if (leader) {
#pragma unroll 1
          for (int cc = 0; cc < NB; cc += 32) {
            tma_store_2d(&yhi_map, smem_u32(buf), col0 + cc, r0);
            tma_store_2d(&ylo_map, smem_u32(buf), col0 + cc, r0);
          }
          bulk_commit();
        }
        ++chunk;
      }
      // The operand area and tensor memory are free once every store has
      // read its staging slice.
      tc_fence_before();
      if (leader) bulk_wait_read0();
      epi_sync();
      if (leader) mbar_arrive(&ofree);
      chunk = 0;
    }
    if (leader) bulk_wait_all();
  }

  __syncthreads();
  if (threadIdx.x == 0 && abort_sh) {
    // Loads issued for a slice's last tile may still target this CTA's
    // shared memory: wait (bounded) for each to land before the CTA exits.
    for (int kc = 0; kc < ANCH; ++kc) {
      const int ti = issued_sh[kc];
      if (ti == 0) continue;
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(&full[kc], (uint32_t)((ti - 1) & 1)) && globaltimer() - t0 < wc.ns) {
      }
    }
    atomicOr(flag, 2u);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(A_TMEM_COLS)
                 : "memory");
  }
}

DeviceOnce g_apply_attr;

}  // namespace

gptq_status apply_tc_run(const ApplyMaps& am, int k, int s0, int N, int col0, int zero_end, unsigned* flag,
                         float* U, const float* dsg, int n, cudaStream_t s) {
  GQ_TRY(g_apply_attr.run([](int) -> gptq_status {
    GQ_CUDA(cudaFuncSetAttribute(k_apply_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, A_SMEM));
    return GPTQ_OK;
  }));
  if (N % AM != 0 || k % NB != 0 || s0 != k + NB || col0 % 32 != 0) return GPTQ_ERR_ARG;
  const int ntiles = N / AM;
  const int grid = ntiles < num_sms() ? ntiles : num_sms();
  GQ_PROF(K_TRSM, s);
  k_apply_tc<<<grid, A_THREADS, A_SMEM, s>>>(am.a, am.lhi, am.llo, am.p.m[0], am.p.m[1], am.p.m[2], am.p.m[3],
                                            k, s0, N, col0, zero_end, flag, U, dsg, n, wait_cfg());
  GQ_LAUNCHED();
  return GPTQ_OK;
}

}  // namespace gq
