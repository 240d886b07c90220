// C -= A B^T on the 5th-generation tensor cores (tcgen05, kind::tf32) with
// the 3xTF32 split: A = A_hi + A_lo, B = B_hi + B_lo (each part exactly a
// TF32 value), and C -= A_lo B_hi + A_hi B_lo + A_hi B_hi accumulated in f32
// in tensor memory.  That keeps the products at about f32 accuracy, which the
// fold needs (the pages compute in f32).
//
// This is the rank-K update every hot loop of the path reduces to: the
// Cholesky's trailing SYRK and the inverse's block update (fold page,
// chol_update / inv_update) and the sweep's trailing GEMM (q4tp_trail).
//
// Persistent kernel, one CTA per SM, 6 warps:
//   warp 0      TMA producer: 128x32 f32 boxes of A_hi, A_lo, B_hi, B_lo
//               (128-byte swizzle) into a 3-stage shared-memory ring;
//   warp 1      allocates 256 TMEM columns (two 128x128 f32 accumulators)
//               and issues the MMAs from one thread; tcgen05.commit frees a
//               stage / publishes a finished accumulator;
//   warps 2-5   epilogue: tcgen05.ld of one accumulator row per thread,
//               -acc into a 128x32 swizzled staging slice (two, alternating),
//               then one TMA reduce-add of the slice into C (the L2 does the
//               read-modify-write, so no SM ever waits on reading C); the
//               accumulator buffer is released after its last slice, so the
//               epilogue of tile i overlaps the MMAs of tile i+1.
// Every wait is bounded (about 2 s of globaltimer); on expiry the kernel
// stops issuing, drains what it started, frees TMEM and sets bit 1 of the
// status word.
// Fused diagonal-block step: in the fold every update's first tile is the
// next 128 x 128 diagonal block.  With `fp.on`, CTA 0 computes only that
// tile (the other CTAs share the rest), waits for its reduce-add to land,
// then factors and inverts the block in its own shared memory while the
// other CTAs finish the update.
#include "common.cuh"
#include "potrf.cuh"
#include "tcgen05.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

namespace gq {
namespace {

constexpr int BM = 128, BN = 128, BK = 32, STAGES = 3;
constexpr int TILE_A = BM * BK * 4;  // 16 KB
constexpr int TILE_B = BN * BK * 4;  // 16 KB
constexpr int STAGE_BYTES = 2 * TILE_A + 2 * TILE_B;
constexpr int CSLICE = BM * 32 * 4;  // 16 KB: 128 rows x 32 columns of C
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 2 * CSLICE + 1024;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 2 * BN;

// Instruction descriptor, kind::tf32: D f32 (bits 4-5 = 1), A and B TF32
// (bits 7-9, 10-12 = 2), both K-major (bits 15, 16 = 0), N >> 3 at bit 17,
// M >> 4 at bit 24.
constexpr uint32_t IDESC = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(BN >> 3) << 17) |
                           ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(IDESC), "r"(accum)
      : "memory");
}

// Tile t of a job: mode 1 walks a lower triangle by rows; mode 2 (a strip
// whose top nt x nt tiles straddle the diagonal) walks that top triangle by
// rows, then the full rows below it; mode 0 walks a rectangle by rows.
__device__ __forceinline__ void tile_of(const TcJob& J, int t, int& ti, int& tj) {
  const int tri = J.mode == 1 ? J.ntiles : J.mode == 2 ? J.nt * (J.nt + 1) / 2 : 0;
  if (t < tri) {
    int i = (int)((sqrtf(8.0f * (float)t + 1.0f) - 1.0f) * 0.5f);
    while ((i + 1) * (i + 2) / 2 <= t) ++i;
    while (i * (i + 1) / 2 > t) --i;
    ti = i;
    tj = t - i * (i + 1) / 2;
  } else {
    const int u = t - tri, r0 = J.mode == 2 ? J.nt : 0;
    ti = r0 + u / J.nt;
    tj = u % J.nt;
  }
}

__global__ void __launch_bounds__(THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap m0, const __grid_constant__ CUtensorMap m1,
              const __grid_constant__ CUtensorMap m2, const __grid_constant__ CUtensorMap m3,
              const __grid_constant__ CUtensorMap cmap, TcJob j0, TcJob j1, int K, int kseg,
              const unsigned* flag, unsigned* status, FusedPotrf fp, WaitCfg wc) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment by an offset on the shared array itself (not an
  // integer round trip), so that accesses through `smem` stay shared-memory
  // instructions, here and in the diagonal-block step that reuses it.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int issued_sh, consumed_sh;
  __shared__ int skip_sh;
  // One read of the skip flag, shared by the whole CTA (uniform exit).
  if (threadIdx.x == 0) skip_sh = (flag != nullptr && *(volatile const unsigned*)flag != 0u) ? 1 : 0;
  __syncthreads();
  if (skip_sh) return;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int total = j0.ntiles + j1.ntiles;
  const int nk = K / BK;
  // Split-K within a tile: the accumulator is drained to C (reduce-add,
  // round-to-nearest in L2) every `segc` chunks, which bounds how many MMAs
  // accumulate into one f32 TMEM value before it is rounded properly.
  const int segc = (kseg > 0 && kseg / BK < nk) ? kseg / BK : nk;
  const int nseg = (nk + segc - 1) / segc;
  // Tile sequence of this CTA: t0, t0 + tstride, ...
  int t0 = blockIdx.x, tstride = gridDim.x;
  if (fp.on == kFusedStep) {
    if (blockIdx.x == 0) {
      tstride = total;  // tile 0 only
    } else {
      tstride = gridDim.x - 1;
    }
  } else if (fp.on == kSkipTile0) {
    t0 = blockIdx.x + 1;  // tile 0 is run elsewhere
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 128);
    }
    mbar_init(&drain, 1);
    abort_sh = 0;
    issued_sh = 0;
    consumed_sh = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_base_sh)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  volatile int* abort = &abort_sh;

  if (warp == 0) {
    if (lane == 0) {
      const CUtensorMap* maps[4] = {&m0, &m1, &m2, &m3};
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      // wc.no_loads (a test hook): issue nothing, so that the MMA and
      // epilogue waits below run out and report a timeout.
      for (int t = t0; t < total && !*abort && !wc.no_loads; t += tstride) {
        const bool second = t >= j0.ntiles;
        const TcJob& J = second ? j1 : j0;
        int ti, tj;
        tile_of(J, second ? t - j0.ntiles : t, ti, tj);
        const int ay = J.a_row0 + ti * BM, by = J.b_row0 + tj * BN;
        const CUtensorMap* ahi = maps[J.a_map];
        const CUtensorMap* alo = maps[J.a_map + 1];
        const CUtensorMap* bhi = maps[J.b_map];
        const CUtensorMap* blo = maps[J.b_map + 1];
        for (int c = 0; c < nk; ++c) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort, wc.ns)) break;
          const uint32_t sb = smem_u32(smem + stage * STAGE_BYTES);
          mbar_expect_tx(&full[stage], STAGE_BYTES);
          const int kx = J.k0 + c * BK;
          tma_load_2d(sb, ahi, kx, ay, &full[stage]);
          tma_load_2d(sb + TILE_A, alo, kx, ay, &full[stage]);
          tma_load_2d(sb + 2 * TILE_A, bhi, kx, by, &full[stage]);
          tma_load_2d(sb + 2 * TILE_A + TILE_B, blo, kx, by, &full[stage]);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      issued_sh = issued;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0, acc = 0, consumed = 0;
      uint32_t phase = 0, aphase = 0;
      for (int t = t0; t < total && !*abort; t += tstride) {
        bool ok = true;
        for (int sg = 0; sg < nseg && ok; ++sg) {
          if (!mbar_wait(&tempty[acc], aphase ^ 1u, abort, wc.ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(acc * BN);
          const int cend = (sg + 1) * segc < nk ? (sg + 1) * segc : nk;
          for (int c = sg * segc; c < cend; ++c) {
            if (!mbar_wait(&full[stage], phase, abort, wc.ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_hi = smem_u32(smem + stage * STAGE_BYTES);
            const uint32_t a_lo = a_hi + TILE_A, b_hi = a_hi + 2 * TILE_A, b_lo = b_hi + TILE_B;
#pragma unroll
            for (int kk = 0; kk < BK / 8; ++kk) {
              const uint32_t off = (uint32_t)kk * 32u;
              mma_tf32(d, sdesc(a_lo + off), sdesc(b_hi + off), (c > sg * segc || kk) ? 1u : 0u);
              mma_tf32(d, sdesc(a_hi + off), sdesc(b_lo + off), 1u);
              mma_tf32(d, sdesc(a_hi + off), sdesc(b_hi + off), 1u);
            }
            mma_commit(&empty[stage]);
            ++consumed;
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit(&tfull[acc]);
          if (++acc == 2) {
            acc = 0;
            aphase ^= 1u;
          }
        }
        if (!ok) break;
      }
      consumed_sh = consumed;
      // Every MMA this thread issued has completed once `drain` flips.
      mma_commit(&drain);
      if (!mbar_wait(&drain, 0u, abort, wc.ns)) {
        // Give the drain a last bounded chance even after an abort.
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(&drain, 0u) && globaltimer() - t0 < wc.ns) {
        }
      }
    }
  } else {
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    const bool leader = threadIdx.x == 64;
    uint8_t* cstage = smem + STAGES * STAGE_BYTES;
    int acc = 0, chunk = 0;
    uint32_t aphase = 0;
    bool go = true;
    for (int w = t0 * nseg; go && w < total * nseg; w += (w % nseg == nseg - 1) ? (tstride - 1) * nseg + 1 : 1) {
      const int t = w / nseg;
      // All 128 epilogue threads agree before any of them reaches the
      // .sync.aligned loads or the named barriers below.
      if (!epi_all(mbar_wait(&tfull[acc], aphase, abort, wc.ns))) {
        go = false;
        break;
      }
      tc_fence_after();
      const bool second = t >= j0.ntiles;
      const TcJob& J = second ? j1 : j0;
      int ti, tj;
      tile_of(J, second ? t - j0.ntiles : t, ti, tj);
      const int rr = q * 32 + lane;  // row inside the tile
      const bool diag = (J.mode != 0) && (ti == tj);
      const uint32_t tbase = tmem + (uint32_t)(acc * BN) + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int cc = 0; cc < BN; cc += 32) {
        uint32_t v[32];
        tmem_ld32(tbase + (uint32_t)cc, v);
        tmem_ld_wait();
        uint8_t* buf = cstage + (chunk & 1) * CSLICE;
        if (leader) bulk_wait_read1();  // the reduce that last read `buf` is done
        epi_sync();
        uint8_t* rowp = buf + rr * 128;
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          float4 o;
          o.x = J.add ? __uint_as_float(v[4 * c4]) : -__uint_as_float(v[4 * c4]);
          o.y = J.add ? __uint_as_float(v[4 * c4 + 1]) : -__uint_as_float(v[4 * c4 + 1]);
          o.z = J.add ? __uint_as_float(v[4 * c4 + 2]) : -__uint_as_float(v[4 * c4 + 2]);
          o.w = J.add ? __uint_as_float(v[4 * c4 + 3]) : -__uint_as_float(v[4 * c4 + 3]);
          if (diag) {  // lower triangle only: add nothing above the diagonal
            const int c0 = cc + 4 * c4;
            if (c0 > rr) o.x = 0.f;
            if (c0 + 1 > rr) o.y = 0.f;
            if (c0 + 2 > rr) o.z = 0.f;
            if (c0 + 3 > rr) o.w = 0.f;
          }
          *reinterpret_cast<float4*>(rowp + ((c4 ^ (rr & 7)) * 16)) = o;
        }
        fence_proxy_async_smem();
        epi_sync();
        if (leader) {
          tma_reduce_add_2d(&cmap, smem_u32(buf), J.c_x0 + tj * BN + cc, J.c_y0 + ti * BM);
          bulk_commit();
        }
        ++chunk;
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        aphase ^= 1u;
      }
    }
    if (leader) bulk_wait_all();
  }

  __syncthreads();
  if (threadIdx.x == 0 && abort_sh) {
    // Loads issued but never consumed still target this CTA's shared memory:
    // wait (bounded) for them to land before the CTA exits.
    for (int i = consumed_sh; i < issued_sh; ++i) {
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(&full[i % STAGES], (uint32_t)((i / STAGES) & 1)) &&
             globaltimer() - t0 < wc.ns) {
      }
    }
    atomicOr(status, 2u);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                 : "memory");
  }
  if (fp.on == kFusedStep && blockIdx.x == 0 && !abort_sh) {
    // The epilogue leader waited for its reduce-adds (wait_group 0); make
    // the tensor core's global writes visible to plain loads, then run the
    // diagonal-block step on the finished tile (shared memory is free: every
    // load has landed and every MMA has retired).
    if (threadIdx.x == 64) asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncthreads();
    potrf_inverse_block(fp.A + (long long)fp.k * fp.lda + fp.k, fp.lda, fp.Lhi, fp.Llo, status,
                        reinterpret_cast<float*>(smem));
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  // A function-local static: initialised once, thread-safe.
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<CtxGetCurrentFn>(p);
    return static_cast<CtxGetCurrentFn>(nullptr);
  }();
  return fn;
}

DeviceOnce g_tc_attr;

}  // namespace

CUcontext current_context() {
  const auto fn = ctx_get_current_fn();
  CUcontext c = nullptr;
  if (fn == nullptr || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

int num_sms() {
  static std::mutex mu;
  static int sms[DeviceOnce::kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= DeviceOnce::kMaxDevices) dev = 0;
  std::lock_guard<std::mutex> lk(mu);
  if (sms[dev] <= 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
    sms[dev] = v;
  }
  return sms[dev];
}


gptq_status make_operand_map(CUtensorMap* m, const float* base, long long rows, int K, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return GPTQ_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0 || K % BK != 0) return GPTQ_ERR_ARG;
  if (box_rows <= 0 || box_rows > 256 || box_rows % 8 != 0) return GPTQ_ERR_ARG;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 4u};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GPTQ_OK : GPTQ_ERR_CUDA;
}

gptq_status make_c_map(CUtensorMap* m, float* base, long long rows, long long cols, long long ld) {
  auto fn = encode_fn();
  if (fn == nullptr) return GPTQ_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0 || (ld * 4) % 16 != 0) return GPTQ_ERR_ARG;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 4u};
  cuuint32_t box[2] = {32u, (cuuint32_t)BM};
  cuuint32_t es[2] = {1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GPTQ_OK : GPTQ_ERR_CUDA;
}

gptq_status gemm_tc_sub(const OperandMaps& maps, const TcJob& j0, const TcJob& j1, int K,
                        const unsigned* flag, unsigned* status, int kind, cudaStream_t s,
                        const FusedPotrf& fp, int kseg) {
  GQ_TRY(g_tc_attr.run([](int) -> gptq_status {
    GQ_CUDA(cudaFuncSetAttribute(k_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES));
    return GPTQ_OK;
  }));
  if (K % BK != 0 || K <= 0) return GPTQ_ERR_ARG;
  const int total = j0.ntiles + j1.ntiles;
  if (total <= 0) return GPTQ_OK;
  // kSkipTile0: one tile fewer, and one SM left to the launch that runs it.
  const int skip = fp.on == kSkipTile0 ? 1 : 0;
  if (total - skip <= 0) return GPTQ_OK;
  const int grid = total - skip < num_sms() - skip ? total - skip : num_sms() - skip;
  GQ_PROF(kind, s);
  k_gemm_tc<<<grid, THREADS, SMEM_BYTES, s>>>(maps.m[0], maps.m[1], maps.m[2], maps.m[3], maps.c, j0,
                                              j1, K, kseg, flag, status, fp, wait_cfg());
  GQ_LAUNCHED();
  return GPTQ_OK;
}

}  // namespace gq
