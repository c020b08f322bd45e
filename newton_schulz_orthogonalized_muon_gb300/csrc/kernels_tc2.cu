// CTA-pair tensor-core Newton-Schulz GEMMs (tcgen05.mma.cta_group::2).
//
// The products of kernels_tc.cu (SYRK, POLY, UPDATE, FINAL of the standard
// method; G_R0, G_P, G_PROD of the Gram method) with the same epilogues, on
// 256 x 256 output tiles computed by a cluster of two CTAs on two SMs:
//   * each CTA loads its own 128 rows of the A operand and its half (128 of
//     256 columns) of the B operand per K step, 32 KB per stage instead of
//     the 48 KB a single CTA needs for a 128 x 256 tile, so six stages (five
//     beside FINAL's epilogue buffers) fit in shared memory and
//     each SM pulls a third less data through L2;
//   * the leader CTA (cluster rank 0) issues tcgen05.mma.cta_group::2
//     (M = 256 across the pair, N = 256, K = 16); the hardware reads the
//     peer's operand halves from the peer's shared memory and writes each
//     CTA's 128 accumulator rows into that CTA's TMEM;
//   * both CTAs' TMA loads signal the leader's "full" barrier; the leader's
//     MMA commits are multicast to the "empty" and "tmem full" barriers of
//     both CTAs; both CTAs' epilogues read their own TMEM and report to the
//     leader's "tmem empty" barrier.
// Every wait is bounded as in the one-CTA kernel; both CTAs meet at a
// cluster barrier before TMEM is released and the kernel exits.
#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace muon {
namespace {

using namespace tc;

constexpr int PBM = 256;       // rows of the pair's tile (128 per CTA)
constexpr int PBN = 256;       // columns of the tile = N of the pair MMA (128 loaded per CTA)
// UPDATE / FINAL input blocks in flight per epilogue warp: UPDATE takes one
// 3 KB slot (two measured no faster on long K); FINAL keeps two, as one slot
// costs it register spills.  XS overrides the default: UPDATE with two slots
// serves short K (m <= 1024), where the epilogue's input latency, not the
// main loop, bounds a tile; the five-stage ring leaves room for it.
template <int MODE>
struct PairSlots {
  static constexpr int v = MODE == MODE_FINAL ? 2 : 1;
};

template <int MODE, int AP, int BP, int XS = PairSlots<MODE>::v>
struct PairCfg {
  static constexpr int A_BYTES = 128 * BK * 2;           // one plane of this CTA's 128 rows of A
  static constexpr int B_BYTES = 128 * BK * 2;           // one plane of this CTA's half of B
  static constexpr int STAGE_BYTES = AP * A_BYTES + BP * B_BYTES;   // 32 KB with one plane each
  static constexpr int EPI_BYTES = EpiLayout<MODE, XS>::BYTES + SymEpi<MODE>::BYTES;
  static constexpr int BAR_BYTES = 512;
  // shared memory: [stages][epilogue buffers][barriers], + 1024 alignment slack
  static constexpr int STAGES_FIT = (MAX_DYN_SMEM - 1024 - BAR_BYTES - EPI_BYTES) / STAGE_BYTES;
  // At most five stages although six fit beside the one-slot epilogues: under
  // the GPU's power cap the sixth stage bought no cycles (the same cycle count
  // per launch at ~1.4 GHz, where memory latency spans fewer cycles) and the
  // clock settled ~5% lower with it.
  static constexpr int STAGES_MAX = 5;
  static constexpr int STAGES = STAGES_FIT < STAGES_MAX ? STAGES_FIT : STAGES_MAX;
  static constexpr int TMEM_COLS = 2 * PBN;              // double-buffered 256-column accumulator
  static constexpr size_t SMEM = static_cast<size_t>(STAGES) * STAGE_BYTES + EPI_BYTES + BAR_BYTES + 1024;
  static_assert(STAGES >= 2 && SMEM <= MAX_DYN_SMEM, "shared memory");
};

template <int MODE, int AP, int BP, int XS = PairSlots<MODE>::v>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(TC_THREADS, 1)
    ns_gemm_pair_kernel(const __grid_constant__ CUtensorMap map_a0, const __grid_constant__ CUtensorMap map_a1,
                        const __grid_constant__ CUtensorMap map_b0, const __grid_constant__ CUtensorMap map_b1,
                        const __grid_constant__ CUtensorMap map_xh, const __grid_constant__ CUtensorMap map_xl,
                        const __grid_constant__ CUtensorMap map_xo, const NsGemmParams p) {
  using C = PairCfg<MODE, AP, BP, XS>;
  using L = EpiLayout<MODE, XS>;
  constexpr bool kUpd = ModeTraits<MODE>::kMN;
  // symmetric products with one B plane: a tile of the ragged last column
  // block with at most 128 valid columns runs N = 128, each CTA loading 64
  // rows of B through map_b1 (the same operand with 64-row boxes)
  constexpr bool kN128 = ModeTraits<MODE>::kSym && BP == 1;
  static_assert(MODE != MODE_G_FINAL, "the element-wise G_FINAL runs on the one-CTA kernel");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* epi = smem + C::STAGES * C::STAGE_BYTES;                 // 1024-aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(epi + C::EPI_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* xfull = drain + 1;                                        // [EPI_WARPS][2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xfull + 2 * EPI_WARPS);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  static_assert(8 * (2 * 8 + 5 + 2 * EPI_WARPS) + 8 <= C::BAR_BYTES, "barrier block");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();           // 0: leader, issues the MMAs
  const int pair = static_cast<int>(cluster_id_x());
  const int npairs = static_cast<int>(num_clusters_x());

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);      // leader: its expect_tx arrival (+ both CTAs' bytes)
      mbar_init(&empty[s], 1);     // the leader's multicast commit
    }
    mbar_init(&tfull[0], 1);
    mbar_init(&tfull[1], 1);
    mbar_init(&tempty[0], 2 * EPI_WARPS);   // leader: every epilogue warp of both CTAs
    mbar_init(&tempty[1], 2 * EPI_WARPS);
    mbar_init(drain, 1);
    for (int w = 0; w < 2 * EPI_WARPS; ++w) mbar_init(&xfull[w], 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
  if (warp == 1 && lane == 0) {
    tma_prefetch_map(&map_a0);
    tma_prefetch_map(&map_b0);
    if (AP == 2) tma_prefetch_map(&map_a1);
    if (BP == 2 || (kN128 && p.sym_n128 != 0)) tma_prefetch_map(&map_b1);
    if (L::kLoadX) {
      tma_prefetch_map(&map_xh);
      tma_prefetch_map(&map_xl);
    }
    if (MODE == MODE_UPDATE || SymEpi<MODE>::kTma) tma_prefetch_map(&map_xo);
    if (ModeTraits<MODE>::kPlanesOut) tma_prefetch_map(&map_xl);
  }
  tc_fence_before();
  cluster_sync_all();      // the peer's barriers are initialised and TMEM is allocated in both CTAs
  tc_fence_after();
  // operands, outputs and descriptors are written or read by earlier kernels
  pdl_wait();
  pdl_launch_dependents();
  const uint32_t tmem_base = *tmem_slot;
  const int num_kb = ((ModeTraits<MODE>::kKn ? p.n : p.m) + BK - 1) / BK;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ producer
      int s = 0, issued = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = pair; ok && t < p.num_tiles; t += npairs) {
        int b, i, j;
        decode_tile<MODE>(p, t, b, i, j);
        const bool n128 = kN128 && p.sym_n128 != 0 && p.m - j * PBN <= 128;
        const int arow = i * PBM + static_cast<int>(rank) * 128;     // this CTA's rows of A
        const int bcol = j * PBN + static_cast<int>(rank) * (n128 ? 64 : 128);   // this CTA's half of B
        const uint32_t stage_tx = n128 ? 2 * (C::STAGE_BYTES - C::B_BYTES / 2) : 2 * C::STAGE_BYTES;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait_bounded(&empty[s], ph ^ 1u, abort, p.timeout_ns)) {
            raise_timeout(abort, p.err);
            ok = false;
            break;
          }
          const uint32_t sa = smem_u32(smem + s * C::STAGE_BYTES);
          const uint32_t sb = sa + AP * C::A_BYTES;
          const uint32_t fb = mapa_shared(smem_u32(&full[s]), 0);   // the leader's full barrier
          if (rank == 0) mbar_arrive_expect_tx(&full[s], stage_tx);
#pragma unroll
          for (int pa = 0; pa < AP; ++pa) {
            const CUtensorMap* ma = pa == 0 ? &map_a0 : &map_a1;
            tma_load_3d_pair(sa + pa * C::A_BYTES, ma, fb, kb * BK, arow, b);        // one 128-row box
          }
#pragma unroll
          for (int pb = 0; pb < BP; ++pb) {
            const CUtensorMap* mb = pb == 0 ? &map_b0 : &map_b1;
            if (kUpd) {      // X^ read MN-major: 64 columns x 64 K rows per box
              tma_load_3d_pair(sb + pb * C::B_BYTES, mb, fb, bcol, kb * BK, b);
              tma_load_3d_pair(sb + pb * C::B_BYTES + BOX_BYTES, mb, fb, bcol + 64, kb * BK, b);
            } else if (n128) {   // K-major, N = 128: this CTA's 64 rows of B
              tma_load_3d_pair(sb, &map_b1, fb, kb * BK, bcol, b);
            } else {         // K-major: this CTA's 128 rows of B in one box
              tma_load_3d_pair(sb + pb * C::B_BYTES, mb, fb, kb * BK, bcol, b);
            }
          }
          ++issued;
          if (++s == C::STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // drain (leader): its full barriers count both CTAs' bytes, so once the
      // last armed phase of every stage completed, no load of the pair is in flight
      if (rank == 0) {
        for (int st = 0; st < C::STAGES && st < issued; ++st) {
          const int last = ((issued - 1 - st) / C::STAGES) * C::STAGES + st;
          mbar_wait_bounded(&full[st], static_cast<uint32_t>((last / C::STAGES) & 1), nullptr, DRAIN_NS);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ----------------------------------------------- MMA issuer (leader)
      const uint32_t idesc256 = idesc_bf16_f32(PBM, PBN, kUpd ? 1 : 0);
      const uint32_t idesc128 = idesc_bf16_f32(PBM, 128, kUpd ? 1 : 0);
      int s = 0, acc = 0;
      uint32_t ph = 0, acc_ph = 0;
      bool ok = true;
      for (int t = pair; ok && t < p.num_tiles; t += npairs) {
        bool n128 = false;
        if (kN128 && p.sym_n128 != 0) {
          int b, i, j;
          decode_tile<MODE>(p, t, b, i, j);
          n128 = p.m - j * PBN <= 128;
        }
        const uint32_t idesc = n128 ? idesc128 : idesc256;
        if (!mbar_wait_bounded(&tempty[acc], acc_ph ^ 1u, abort, p.timeout_ns)) {
          raise_timeout(abort, p.err);
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * PBN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait_bounded(&full[s], ph, abort, p.timeout_ns)) {
            raise_timeout(abort, p.err);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * C::STAGE_BYTES);
          const uint32_t sb = sa + AP * C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t a0 = sdesc_sw128(sa + kk * 32, 16, 1024);
            // K-major B: 32 bytes per K = 16 step; MN-major B: 2 KB per step,
            // 8 KB between the two 64-column boxes
            const uint64_t b0 = kUpd ? sdesc_sw128(sb + kk * 2048, BOX_BYTES, 1024) : sdesc_sw128(sb + kk * 32, 16, 1024);
            umma_bf16_pair(d, a0, b0, idesc, (kb | kk) != 0 ? 1u : 0u);
            if (BP == 2)     // hi(A) * lo(B)
              umma_bf16_pair(d, a0, sdesc_sw128(sb + C::B_BYTES + kk * 32, 16, 1024), idesc, 1u);
            if (AP == 2)     // lo(A) * hi(B)
              umma_bf16_pair(d, sdesc_sw128(sa + C::A_BYTES + kk * 32, 16, 1024), b0, idesc, 1u);
          }
          umma_commit_pair_mc(&empty[s], 0x3);
          if (++s == C::STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair_mc(&tfull[acc], 0x3);
        acc ^= 1;
        if (acc == 0) acc_ph ^= 1u;
      }
      // drain: every pair MMA issued by this thread has completed
      umma_commit_pair_mc(drain, 0x1);
      mbar_wait_bounded(drain, 0, nullptr, DRAIN_NS);
    }
  } else if constexpr (SymEpi<MODE>::kTma) {
    // --------------------------------------------------------- epilogue
    // symmetric products: each CTA stages its 128 rows of the tile block by
    // block and writes them (and their mirror) with TMA bulk stores
    EpiTiles et{};
    et.t0 = pair;
    et.tstep = npairs;
    et.row_off = static_cast<int>(rank) * 128;
    et.remote = true;
    et.tempty = nullptr;
    et.tempty_remote[0] = mapa_shared(smem_u32(&tempty[0]), 0);
    et.tempty_remote[1] = mapa_shared(smem_u32(&tempty[1]), 0);
    sym_epilogue<MODE, PBN, PBM>(p, &map_xo, &map_xl, &map_xl, epi + (warp - 2) * SYM_WARP_BYTES, tfull, et, abort,
                                 tmem_base, warp, lane);
  } else {
    // --------------------------------------------------------- epilogue
    // UPDATE / FINAL: each CTA drains its own 128 accumulator rows of the
    // 256 x 256 tile through the TMA epilogue; the accumulator is handed
    // back to the leader's "tmem empty" barrier.
    EpiTiles et{};
    et.t0 = pair;
    et.tstep = npairs;
    et.row_off = static_cast<int>(rank) * 128;
    et.remote = true;
    et.tempty = nullptr;
    et.tempty_remote[0] = mapa_shared(smem_u32(&tempty[0]), 0);
    et.tempty_remote[1] = mapa_shared(smem_u32(&tempty[1]), 0);
    mn_epilogue<MODE, PBN, PBM, XS>(p, &map_xh, &map_xl, &map_xo, epi + (warp - 2) * L::WARP_BYTES,
                                xfull + 2 * (warp - 2), tfull, et, abort, tmem_base, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();      // no CTA leaves while its peer may still read its operands or signal it
  tc_fence_after();
  if (warp == 0) {
    __syncwarp();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

template <int MODE, int AP, int BP, int XS = PairSlots<MODE>::v>
cudaError_t launch_pair(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0, const CUtensorMap& b1,
                        const CUtensorMap& xh, const CUtensorMap& xl, const CUtensorMap& xo, const NsGemmParams& p,
                        int pairs, cudaStream_t s) {
  auto kern = ns_gemm_pair_kernel<MODE, AP, BP, XS>;
  using C = PairCfg<MODE, AP, BP, XS>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const cudaError_t e = launch_k(pdl_level() >= 1, kern, dim3(2 * pairs), dim3(TC_THREADS), C::SMEM, s, a0, a1, b0, b1, xh, xl, xo, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

// Number of CTA pairs of this kernel that fit on the device at once (the
// UPDATE instantiation has the largest shared-memory footprint).
int ns_gemm_pair_max_pairs() {
  static int cached = -1;
  if (cached < 0) {
    auto kern = ns_gemm_pair_kernel<MODE_UPDATE, 1, 1>;
    using C = PairCfg<MODE_UPDATE, 1, 1>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM)) !=
        cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(TC_THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cached = n;
  }
  return cached;
}

cudaError_t launch_ns_gemm_pair(int mode, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& so,
                               const CUtensorMap& so_lo, const NsGemmParams& p, int pairs, cudaStream_t s,
                               const CUtensorMap* b64) {
  if (p.num_tiles == 0) return cudaSuccess;
  NsGemmParams q = p;
  q.sym_n128 = (b64 != nullptr && (mode == MODE_SYRK || mode == MODE_POLY)) ? 1 : 0;
  const CUtensorMap& b1 = q.sym_n128 ? *b64 : b;
  switch (mode) {
    case MODE_SYRK: return launch_pair<MODE_SYRK, 1, 1>(a, a, b, b1, b, b, so, q, pairs, s);
    case MODE_POLY: return launch_pair<MODE_POLY, 1, 1>(a, a, b, b1, b, b, so, q, pairs, s);
    case MODE_G_R0: return launch_pair<MODE_G_R0, 1, 1>(a, a, b, b, b, so_lo, so, p, pairs, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_ns_gemm_pair_update(int mode, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& xh,
                                      const CUtensorMap& xl, const CUtensorMap& xo, const NsGemmParams& p, int pairs,
                                      cudaStream_t s, int slots) {
  if (p.num_tiles == 0) return cudaSuccess;
  switch (mode) {
    case MODE_UPDATE:
      return slots == 2 ? launch_pair<MODE_UPDATE, 1, 1, 2>(a, a, b, b, xh, xl, xo, p, pairs, s)
                        : launch_pair<MODE_UPDATE, 1, 1>(a, a, b, b, xh, xl, xo, p, pairs, s);
    case MODE_FINAL: return launch_pair<MODE_FINAL, 1, 1>(a, a, b, b, xh, xl, xo, p, pairs, s);
    case MODE_FINAL_T: return launch_pair<MODE_FINAL_T, 1, 1>(a, a, b, b, xh, xl, xo, p, pairs, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_ns_gemm_pair_gram_final(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b,
                                           const NsGemmParams& p, int pairs, cudaStream_t s) {
  if (p.num_tiles == 0) return cudaSuccess;
  return launch_pair<MODE_G_FINAL_T, 2, 1>(a0, a1, b, b, b, b, b, p, pairs, s);
}

cudaError_t launch_ns_gemm_pair_planes(int mode, const CUtensorMap& a0, const CUtensorMap& a1,
                                      const CUtensorMap& b0, const CUtensorMap& b1, const CUtensorMap& so,
                                      const CUtensorMap& so_lo, const NsGemmParams& p, int pairs, cudaStream_t s) {
  if (p.num_tiles == 0) return cudaSuccess;
  switch (mode) {
    case MODE_G_P: return launch_pair<MODE_G_P, 2, 2>(a0, a1, b0, b1, b0, so_lo, so, p, pairs, s);
    case MODE_G_PROD: return launch_pair<MODE_G_PROD, 2, 2>(a0, a1, b0, b1, b0, so_lo, so, p, pairs, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace muon
