// C -= A B^T (3xTF32, as in gemm_tc.cu) on pairs of SMs: tcgen05.mma with
// cta_group::2 and tiles of 256 x 256.
//
// A cluster of two CTAs shares every tile.  CTA r of the pair holds rows
// 128 r .. 128 r + 127 of the tile's A panel and of its B panel in its own
// shared memory (a 3-stage ring of 128 x 32 f32 boxes, hi and lo), and rows
// 128 r .. of the 256 x 256 accumulator in its own tensor memory (two
// accumulators: all 512 columns).  One thread of the even CTA (the leader)
// issues the MMAs for both; each MMA reads half of A and half of B from each
// SM, so per flop an SM's shared memory feeds the tensor core half of what a
// single-SM 128 x 128 tile needs -- the tensor core of a lone SM is held back
// by exactly that bandwidth.  Both CTAs' TMA loads complete on the leader's
// stage barrier, MMA completions are multicast to both CTAs, and both
// epilogues (each its own 128 rows) release an accumulator on the leader's
// barrier.  Waits are bounded as in the single-SM kernel.
// Fused diagonal-block step: pair 0 computes only tile 0 (its leader's rows
// hold the next 128 x 128 diagonal block), then the leader factors and
// inverts that block while the other pairs finish the update.
#include "common.cuh"
#include "potrf.cuh"
#include "tcgen05.cuh"

namespace gq {
namespace {

constexpr int PM = 256, PN = 256, HM = 128, HN = 128, PBK = 32, PSTAGES = 3;
constexpr int P_TILE_A = HM * PBK * 4;  // 16 KB
constexpr int P_TILE_B = HN * PBK * 4;  // 16 KB
constexpr int P_STAGE = 2 * P_TILE_A + 2 * P_TILE_B;
constexpr int P_CSLICE = HM * 32 * 4;  // 128 rows x 32 columns of C
constexpr int P_SMEM = PSTAGES * P_STAGE + 2 * P_CSLICE + 1024;
constexpr int P_THREADS = 192;
constexpr uint32_t P_TMEM_COLS = 512;
// kind::tf32, D f32, K-major A and B; M = 256 (both CTAs), N = 256.
constexpr uint32_t P_IDESC = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(PN >> 3) << 17) |
                             ((uint32_t)(PM >> 4) << 24);

__device__ __forceinline__ void mma_tf32_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(P_IDESC), "r"(accum)
      : "memory");
}

// A job with its tile counts in units of 256 x 256.
struct PJob {
  TcJob j;
  int mt, nt, ntiles;
};

__device__ __forceinline__ void ptile_of(const PJob& J, int t, int& ti, int& tj) {
  if (J.j.mode == 1) {
    int i = (int)((sqrtf(8.0f * (float)t + 1.0f) - 1.0f) * 0.5f);
    while ((i + 1) * (i + 2) / 2 <= t) ++i;
    while (i * (i + 1) / 2 > t) --i;
    ti = i;
    tj = t - i * (i + 1) / 2;
  } else if (J.j.band > 0) {
    const int per = J.j.band * J.nt;
    const int g = t / per, r = t - g * per;
    const int rows = min(J.j.band, J.mt - g * J.j.band);
    ti = g * J.j.band + r % rows;
    tj = r / rows;
  } else {
    ti = t / J.nt;
    tj = t % J.nt;
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(P_THREADS, 1)
    k_gemm_pair(const __grid_constant__ CUtensorMap m0, const __grid_constant__ CUtensorMap m1,
                const __grid_constant__ CUtensorMap m2, const __grid_constant__ CUtensorMap m3,
                const __grid_constant__ CUtensorMap cmap, PJob j0, PJob j1, int K, int kseg,
                const unsigned* flag, unsigned* status, FusedPotrf fp, WaitCfg wc) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t full[PSTAGES], empty[PSTAGES], tfull[2], tempty[2], drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh, skip_sh;
  if (threadIdx.x == 0) skip_sh = (flag != nullptr && *(volatile const unsigned*)flag != 0u) ? 1 : 0;
  __syncthreads();
  if (skip_sh) return;  // the same flag in both CTAs of a pair: both leave

  const uint32_t rank = cluster_rank();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
  const int total = j0.ntiles + j1.ntiles;
  const int nk = K / PBK;
  const int segc = (kseg > 0 && kseg / PBK < nk) ? kseg / PBK : nk;
  const int nseg = (nk + segc - 1) / segc;
  int t0 = pair, tstride = npairs;
  if (fp.on == kFusedStep) tstride = (pair == 0) ? total : npairs - 1;
  if (threadIdx.x == 0) {
    for (int s = 0; s < PSTAGES; ++s) {
      mbar_init(&full[s], 1);   // the leader's expect_tx; bytes from both CTAs
      mbar_init(&empty[s], 1);  // multicast MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 256);  // both CTAs' epilogue threads (leader's copy)
    }
    mbar_init(&drain, 1);
    abort_sh = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {  // one warp of each CTA of the pair, together
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_base_sh)),
                 "r"(P_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers initialized, TMEM allocated
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  volatile int* abort = &abort_sh;

  if (warp == 0) {
    if (lane == 0) {
      const CUtensorMap* maps[4] = {&m0, &m1, &m2, &m3};
      const uint64_t keep = l2_evict_last();  // operand panels: reread by many tiles
      int stage = 0;
      uint32_t phase = 0;
      // wc.no_loads (a test hook): issue nothing, so that the waits of the
      // MMA thread and of both epilogues run out and report a timeout.
      for (int t = t0; t < total && !*abort && !wc.no_loads; t += tstride) {
        const bool second = t >= j0.ntiles;
        const PJob& J = second ? j1 : j0;
        int ti, tj;
        ptile_of(J, second ? t - j0.ntiles : t, ti, tj);
        const int ay = J.j.a_row0 + ti * PM + (int)rank * HM;
        const int by = J.j.b_row0 + tj * PN + (int)rank * HN;
        const CUtensorMap* ahi = maps[J.j.a_map];
        const CUtensorMap* alo = maps[J.j.a_map + 1];
        const CUtensorMap* bhi = maps[J.j.b_map];
        const CUtensorMap* blo = maps[J.j.b_map + 1];
        for (int c = 0; c < nk; ++c) {
          if (!mbar_wait_cl(&empty[stage], phase ^ 1u, abort, wc.ns)) break;
          const uint32_t sb = smem_u32(smem + stage * P_STAGE);
          const uint32_t fb = mapa_u32(smem_u32(&full[stage]), 0);
          if (rank == 0) mbar_expect_tx(&full[stage], 2 * P_STAGE);
          const int kx = J.j.k0 + c * PBK;
          tma_load_2d_pair_hint(sb, ahi, kx, ay, fb, keep);
          tma_load_2d_pair_hint(sb + P_TILE_A, alo, kx, ay, fb, keep);
          tma_load_2d_pair_hint(sb + 2 * P_TILE_A, bhi, kx, by, fb, keep);
          tma_load_2d_pair_hint(sb + 2 * P_TILE_A + P_TILE_B, blo, kx, by, fb, keep);
          if (++stage == PSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, aphase = 0;
      for (int t = t0; t < total && !*abort; t += tstride) {
        bool ok = true;
        for (int sg = 0; sg < nseg && ok; ++sg) {
          if (!mbar_wait_cl(&tempty[acc], aphase ^ 1u, abort, wc.ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(acc * PN);
          const int cend = (sg + 1) * segc < nk ? (sg + 1) * segc : nk;
          for (int c = sg * segc; c < cend; ++c) {
            if (!mbar_wait_cl(&full[stage], phase, abort, wc.ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_hi = smem_u32(smem + stage * P_STAGE);
            const uint32_t a_lo = a_hi + P_TILE_A, b_hi = a_hi + 2 * P_TILE_A, b_lo = b_hi + P_TILE_B;
#pragma unroll
            for (int kk = 0; kk < PBK / 8; ++kk) {
              const uint32_t off = (uint32_t)kk * 32u;
              mma_tf32_pair(d, sdesc(a_lo + off), sdesc(b_hi + off), (c > sg * segc || kk) ? 1u : 0u);
              mma_tf32_pair(d, sdesc(a_hi + off), sdesc(b_lo + off), 1u);
              mma_tf32_pair(d, sdesc(a_hi + off), sdesc(b_hi + off), 1u);
            }
            mma_commit_pair(&empty[stage]);
            if (++stage == PSTAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit_pair(&tfull[acc]);
          if (++acc == 2) {
            acc = 0;
            aphase ^= 1u;
          }
        }
        if (!ok) break;
      }
      // Every MMA issued has completed once `drain` flips.
      mma_commit_pair(&drain);
      if (!mbar_wait_cl(&drain, 0u, abort, wc.ns)) {
        const uint64_t tt = globaltimer();
        while (!mbar_try_wait_cl(&drain, 0u) && globaltimer() - tt < wc.ns) {
        }
      }
    }
  } else {
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    const bool leader = threadIdx.x == 64;
    const uint64_t stream_c = l2_evict_first();  // C passes through once per update
    uint8_t* cstage = smem + PSTAGES * P_STAGE;
    const uint32_t tempty_cl[2] = {mapa_u32(smem_u32(&tempty[0]), 0), mapa_u32(smem_u32(&tempty[1]), 0)};
    int acc = 0, chunk = 0;
    uint32_t aphase = 0;
    bool go = true;
    for (int w = t0 * nseg; go && w < total * nseg;
         w += (w % nseg == nseg - 1) ? (tstride - 1) * nseg + 1 : 1) {
      const int t = w / nseg;
      if (!epi_all(mbar_wait_cl(&tfull[acc], aphase, abort, wc.ns))) {
        go = false;
        break;
      }
      tc_fence_after();
      const bool second = t >= j0.ntiles;
      const PJob& J = second ? j1 : j0;
      int ti, tj;
      ptile_of(J, second ? t - j0.ntiles : t, ti, tj);
      const int rr = q * 32 + lane;
      const int rabs = ti * PM + (int)rank * HM + rr;  // row inside the job
      const bool rowin = rabs < J.j.M;
      const bool diagband = (J.j.mode != 0) && (ti == tj);
      const uint32_t tbase = tmem + (uint32_t)(acc * PN) + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int cc = 0; cc < PN; cc += 32) {
        uint32_t v[32];
        tmem_ld32(tbase + (uint32_t)cc, v);
        tmem_ld_wait();
        uint8_t* buf = cstage + (chunk & 1) * P_CSLICE;
        if (leader) bulk_wait_read1();  // the reduce that last read `buf` is done
        epi_sync();
        uint8_t* rowp = buf + rr * 128;
        const int cb = tj * PN + cc;  // first column of the slice inside the job
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          float4 o;
          o.x = J.j.add ? __uint_as_float(v[4 * c4]) : -__uint_as_float(v[4 * c4]);
          o.y = J.j.add ? __uint_as_float(v[4 * c4 + 1]) : -__uint_as_float(v[4 * c4 + 1]);
          o.z = J.j.add ? __uint_as_float(v[4 * c4 + 2]) : -__uint_as_float(v[4 * c4 + 2]);
          o.w = J.j.add ? __uint_as_float(v[4 * c4 + 3]) : -__uint_as_float(v[4 * c4 + 3]);
          // Outside the job (a 256 tile past its edge) or above the diagonal
          // of a triangular job: add nothing.
          const int c0 = cb + 4 * c4;
          const int lim = diagband ? (rabs < J.j.N - 1 ? rabs : J.j.N - 1) : J.j.N - 1;
          if (!rowin || c0 > lim) o.x = 0.f;
          if (!rowin || c0 + 1 > lim) o.y = 0.f;
          if (!rowin || c0 + 2 > lim) o.z = 0.f;
          if (!rowin || c0 + 3 > lim) o.w = 0.f;
          *reinterpret_cast<float4*>(rowp + ((c4 ^ (rr & 7)) * 16)) = o;
        }
        fence_proxy_async_smem();
        epi_sync();
        if (leader) {
          tma_reduce_add_2d_hint(&cmap, smem_u32(buf), J.j.c_x0 + cb, J.j.c_y0 + ti * PM + (int)rank * HM,
                                 stream_c);
          bulk_commit();
        }
        ++chunk;
      }
      tc_fence_before();
      mbar_arrive_cluster(tempty_cl[acc]);
      if (++acc == 2) {
        acc = 0;
        aphase ^= 1u;
      }
    }
    if (leader) bulk_wait_all();
  }

  __syncthreads();
  if (threadIdx.x == 0 && abort_sh) {
    // Loads still in flight into this CTA's shared memory complete on the
    // leader's barriers: give them time to land (bounded), then report.
    const uint64_t tt = globaltimer();
    while (globaltimer() - tt < 200000ull) {
    }
    atomicOr(status, 2u);
  }
  // Neither CTA frees TMEM or leaves while the leader's MMAs may still read
  // the peer's shared memory or write either CTA's accumulators.
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(P_TMEM_COLS)
                 : "memory");
  }
  if (fp.on == kFusedStep && pair == 0 && rank == 0 && !abort_sh) {
    // The epilogue leader waited for its reduce-adds; make them visible to
    // plain loads, then run the diagonal-block step on the finished block.
    if (threadIdx.x == 64) asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncthreads();
    potrf_inverse_block(fp.A + (long long)fp.k * fp.lda + fp.k, fp.lda, fp.Lhi, fp.Llo, status,
                        reinterpret_cast<float*>(smem));
  }
}

PJob to_pjob(const TcJob& j) {
  PJob p{};
  p.j = j;
  if (j.M <= 0 || j.N <= 0 || j.ntiles <= 0) return p;
  p.mt = (j.M + PM - 1) / PM;
  p.nt = (j.N + PN - 1) / PN;
  p.ntiles = j.mode == 1 ? p.mt * (p.mt + 1) / 2 : p.mt * p.nt;
  return p;
}

}  // namespace

gptq_status gemm_pair_sub(const OperandMaps& maps, const TcJob& j0, const TcJob& j1, int K,
                          const unsigned* flag, unsigned* status, int kind, cudaStream_t s,
                          const FusedPotrf& fp, int kseg) {
  static DeviceOnce attr;
  GQ_TRY(attr.run([](int) -> gptq_status {
    GQ_CUDA(cudaFuncSetAttribute(k_gemm_pair, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM));
    return GPTQ_OK;
  }));
  if (K % PBK != 0 || K <= 0) return GPTQ_ERR_ARG;
  const PJob p0 = to_pjob(j0), p1 = to_pjob(j1);
  const int total = p0.ntiles + p1.ntiles;
  if (total <= 0) return GPTQ_OK;
  int pairs = num_sms() / 2;
  if (pairs > total) pairs = total;
  if (fp.on == kFusedStep && total > 1 && pairs < 2) pairs = 2;  // pair 0 takes tile 0 only
  if (pairs < 1) pairs = 1;
  GQ_PROF(kind, s);
  k_gemm_pair<<<2 * pairs, P_THREADS, P_SMEM, s>>>(maps.m[0], maps.m[1], maps.m[2], maps.m[3], maps.c, p0,
                                                   p1, K, kseg, flag, status, fp, wait_cfg());
  GQ_LAUNCHED();
  return GPTQ_OK;
}

}  // namespace gq
