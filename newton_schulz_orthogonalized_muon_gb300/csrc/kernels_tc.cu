// Tensor-core Newton-Schulz GEMMs for sm_103a (tcgen05 + TMA + TMEM).
//
// One quintic NS iteration on X (m x n, m <= n) is X <- P X with
//   A = X X^T,  P = a I + b A + c A A
// ("Muon Optimizer and the Distributed Implementation", §Newton-Schulz
// Iteration: phi(X) = (a + b XX^T + c (XX^T)^2) X; "DeepSpeed 集成 Muon 优化器
// 实战", §核心算子, coefficients (3.4445, -4.7750, 2.0315)).  Each product is
// one launch of the persistent kernel below in one of four modes:
//
//   SYRK   A = s^2 X X^T    K = n, both operands K-major rows of X (bf16);
//                           only tiles touching the upper triangle are
//                           computed, each element c >= r is written to
//                           (r, c) and mirrored to (c, r).
//   POLY   P = a I + b A + c A A
//                           K = m, A symmetric so A A = A A^T: same operand
//                           form as SYRK; the b*A term is read back in the
//                           epilogue; symmetric bf16 output as above, and
//                           the fp32 diagonal P_rr stored on the side.
//   UPDATE X = s (P^ X^ + P_rr X - P^_rr X^)
//                           K = m, A operand = rows of P^ = bf16(P)
//                           (K-major), B operand = X^ = bf16(X) read MN-major
//                           (n contiguous).  The diagonal of P carries the
//                           large coefficient a = 3.4445 while a + (bA+cA^2)_rr
//                           is O(1): rounding P's diagonal to bf16 would be
//                           amplified by that cancellation, so the epilogue
//                           swaps the rounded diagonal term P^_rr X^ in the
//                           accumulator for the exact one P_rr X (fp32 master
//                           X).  Writes the new fp32 master and its bf16 copy.
//   FINAL  like UPDATE, but the result goes straight into its destination
//          (the parameter: W <- (1 - lr wd) W - lr 0.2 sqrt(max(A,B)) O,
//          transposed back where the NS ran on W^T; or the caller's matrix).
//
// s = 1/||U||_F on the first iteration (the normalisation X0 = U/||U||_F is
// folded into the first SYRK and UPDATE epilogues), 1 afterwards.
//
// The Gram method ("DeepSpeed 集成 Muon 优化器实战", §核心算子: iterate on the
// small square R = XX^T) reuses the same kernel with operands held as two
// bf16 planes (hi, lo): a product of two plane pairs issues three MMAs per
// K step (hi*hi + hi*lo + lo*hi) into one fp32 accumulator, which keeps the
// m x m iteration at about 16 mantissa bits.  Modes G_R0, G_P, G_PROD write
// symmetric plane pairs; G_FINAL applies Q (two planes) to X0 (one plane).
//
// CTA layout (320 threads, 1 CTA per SM, persistent over output tiles):
//   warp 0  lane 0: TMA producer (64 x 64 bf16 boxes, 128-byte swizzle)
//   warp 1  lane 0: MMA issuer, tcgen05.mma.cta_group::1.kind::f16,
//                   M = 128, N = BN, K = 16, fp32 accumulator in TMEM
//   warps 2-9     : epilogue, two warps per TMEM lane quadrant (one per
//                   column half), one TMEM lane (= output row) per thread;
//                   in UPDATE / FINAL each warp streams its blocks of the
//                   fp32 master in and out with TMA (tc_common.cuh)
// The accumulator is double buffered in TMEM (2 x BN columns), so the
// epilogue of one tile overlaps the main loop of the next.
//
// Every barrier wait is bounded (time limit): on expiry the kernel records
// ERRBIT_TIMEOUT, drains its own MMAs and TMA copies (again bounded), frees
// TMEM and returns.
#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace muon {
namespace {

using namespace tc;


// UPDATE / FINAL input blocks in flight per epilogue warp: UPDATE takes one
// 3 KB slot, which leaves room for a fourth main-loop stage at BN = 256;
// FINAL keeps two 4 KB slots, FINAL_T one (5 KB), G_FINAL_T two 2 KB slots
// (free: the stage count is the same with one).
template <int MODE>
struct OneSlots {
  static constexpr int v = (MODE == MODE_FINAL || MODE == MODE_G_FINAL_T) ? 2 : 1;
};

template <int MODE, int BN, int AP, int BP>
struct Cfg {
  static constexpr int A_BYTES = BM * BK * 2;            // one plane of the A tile
  static constexpr int B_BYTES = BN * BK * 2;            // one plane of the B tile
  static constexpr int STAGE_BYTES = AP * A_BYTES + BP * B_BYTES;
  static constexpr int EPI_BYTES = EpiLayout<MODE, OneSlots<MODE>::v>::BYTES + SymEpi<MODE>::BYTES;
  static constexpr int BAR_BYTES = 512;
  // shared memory: [stages][epilogue buffers][barriers], + 1024 alignment slack
  static constexpr int STAGES_FIT = (MAX_DYN_SMEM - 1024 - BAR_BYTES - EPI_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT < 8 ? STAGES_FIT : 8;
  static constexpr int TMEM_COLS = 2 * BN * AccParts<MODE>::v;   // two tiles in flight, each of AccParts parts
  static constexpr size_t SMEM = static_cast<size_t>(STAGES) * STAGE_BYTES + EPI_BYTES + BAR_BYTES + 1024;
  static_assert(STAGES >= 2, "pipeline needs two stages");
  static_assert(SMEM <= MAX_DYN_SMEM, "shared memory");
};

// --------------------------------------------------------------- kernel
template <int MODE, int BN, int AP, int BP>
__global__ void __launch_bounds__(TC_THREADS, 1)
    ns_gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a0, const __grid_constant__ CUtensorMap map_a1,
                      const __grid_constant__ CUtensorMap map_a2, const __grid_constant__ CUtensorMap map_b0,
                      const __grid_constant__ CUtensorMap map_b1, const __grid_constant__ CUtensorMap map_b2,
                      const __grid_constant__ CUtensorMap map_xh, const __grid_constant__ CUtensorMap map_xl,
                      const __grid_constant__ CUtensorMap map_xo, const NsGemmParams p) {
  static_assert(AP <= 3 && BP <= 3 && (AP < 3 || BP == 3), "operand planes");
  using C = Cfg<MODE, BN, AP, BP>;
  using L = EpiLayout<MODE, OneSlots<MODE>::v>;
  constexpr bool kUpd = ModeTraits<MODE>::kMN;
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

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&tfull[0], 1);
    mbar_init(&tfull[1], 1);
    mbar_init(&tempty[0], EPI_WARPS);
    mbar_init(&tempty[1], EPI_WARPS);
    mbar_init(drain, 1);
    for (int w = 0; w < 2 * EPI_WARPS; ++w) mbar_init(&xfull[w], 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, C::TMEM_COLS);
  if (warp == 1 && lane == 0) {
    tma_prefetch_map(&map_a0);
    tma_prefetch_map(&map_b0);
    if (AP >= 2) tma_prefetch_map(&map_a1);
    if (AP >= 3) tma_prefetch_map(&map_a2);
    if (BP >= 2) tma_prefetch_map(&map_b1);
    if (BP >= 3) tma_prefetch_map(&map_b2);
    if (L::kLoadX) {
      tma_prefetch_map(&map_xh);
      tma_prefetch_map(&map_xl);
    }
    if (MODE == MODE_UPDATE || SymEpi<MODE>::kTma) tma_prefetch_map(&map_xo);
    if (ModeTraits<MODE>::kOutPlanes >= 2) tma_prefetch_map(&map_xl);
    if (ModeTraits<MODE>::kOutPlanes >= 3) tma_prefetch_map(&map_xh);
  }
  tc_fence_before();
  __syncthreads();
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
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        int b, i, j;
        decode_tile<MODE>(p, t, b, i, j);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait_bounded(&empty[s], ph ^ 1u, abort, p.timeout_ns)) {
            raise_timeout(abort, p.err);
            ok = false;
            break;
          }
          const uint32_t sa = smem_u32(smem + s * C::STAGE_BYTES);
          const uint32_t sb = sa + AP * C::A_BYTES;
          mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
#pragma unroll
          for (int pa = 0; pa < AP; ++pa) {
            const CUtensorMap* ma = pa == 0 ? &map_a0 : pa == 1 ? &map_a1 : &map_a2;
            tma_load_3d(sa + pa * C::A_BYTES, ma, &full[s], kb * BK, i * BM, b);     // one 128-row box
          }
#pragma unroll
          for (int pb = 0; pb < BP; ++pb) {
            const CUtensorMap* mb = pb == 0 ? &map_b0 : pb == 1 ? &map_b1 : &map_b2;
#pragma unroll
            for (int q = 0; q < BN / 64; ++q) {
              if (kUpd)        // MN-major: 64 columns x 64 K rows per box
                tma_load_3d(sb + pb * C::B_BYTES + q * BOX_BYTES, mb, &full[s], j * BN + q * 64, kb * BK, b);
              else if ((q & 1) == 0)   // K-major: one 128-row box per two 64-row halves
                tma_load_3d(sb + pb * C::B_BYTES + q * BOX_BYTES, mb, &full[s], kb * BK, j * BN + q * 64, b);
            }
          }
          ++issued;
          if (++s == C::STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // drain: the last armed phase of every stage must have landed
      for (int st = 0; st < C::STAGES && st < issued; ++st) {
        const int last = ((issued - 1 - st) / C::STAGES) * C::STAGES + st;
        mbar_wait_bounded(&full[st], static_cast<uint32_t>((last / C::STAGES) & 1), nullptr, DRAIN_NS);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------- MMA issuer
      const uint32_t idesc = idesc_bf16_f32(BM, BN, kUpd ? 1 : 0);
      int s = 0, acc = 0;
      uint32_t ph = 0, acc_ph = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        if (!mbar_wait_bounded(&tempty[acc], acc_ph ^ 1u, abort, p.timeout_ns)) {
          raise_timeout(abort, p.err);
          break;
        }
        tc_fence_after();
        constexpr int kParts = AccParts<MODE>::v;
        const uint32_t dt = tmem_base + static_cast<uint32_t>(acc * BN * kParts);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait_bounded(&full[s], ph, abort, p.timeout_ns)) {
            raise_timeout(abort, p.err);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * C::STAGE_BYTES);
          const uint32_t sb = sa + AP * C::A_BYTES;
          // with two accumulator parts, even K steps go to the first, odd to the second
          const uint32_t d = dt + static_cast<uint32_t>((kParts == 2 && (kb & 1)) ? BN : 0);
          const int kfirst = kParts == 2 ? (kb >> 1) : kb;   // 0: the part's first K step
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t a0 = sdesc_sw128(sa + kk * 32, 16, 1024);
            const uint32_t boff = kUpd ? kk * 2048 : kk * 32;
            const uint64_t b0 = kUpd ? sdesc_sw128(sb + boff, BOX_BYTES, 1024) : sdesc_sw128(sb + boff, 16, 1024);
            umma_bf16(d, a0, b0, idesc, (kfirst | kk) != 0 ? 1u : 0u);
            // plane q of A / B in this stage
            auto adesc = [&](int q) { return sdesc_sw128(sa + q * C::A_BYTES + kk * 32, 16, 1024); };
            auto bdesc = [&](int q) {
              const uint32_t sbq = sb + q * C::B_BYTES + boff;
              return kUpd ? sdesc_sw128(sbq, BOX_BYTES, 1024) : sdesc_sw128(sbq, 16, 1024);
            };
            if (BP >= 2) umma_bf16(d, a0, bdesc(1), idesc, 1u);          // p0(A) * p1(B)
            if (AP >= 2) umma_bf16(d, adesc(1), b0, idesc, 1u);          // p1(A) * p0(B)
            if (AP == 3) {                                               // the terms of order 2^-16
              umma_bf16(d, a0, bdesc(2), idesc, 1u);                     // p0(A) * p2(B)
              umma_bf16(d, adesc(1), bdesc(1), idesc, 1u);               // p1(A) * p1(B)
              umma_bf16(d, adesc(2), b0, idesc, 1u);                     // p2(A) * p0(B)
            }
          }
          umma_commit(&empty[s]);
          if (++s == C::STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_ph ^= 1u;
      }
      // drain: every MMA issued by this thread has completed
      umma_commit(drain);
      mbar_wait_bounded(drain, 0, nullptr, DRAIN_NS);
    }
  } else if constexpr (SymEpi<MODE>::kTma) {
    // --------------------------------------------------------- epilogue
    // symmetric products: blocks staged in shared memory, TMA bulk stores
    // (map_xo / map_xl carry the output's 32 x 32 maps: the matrix, or the
    // hi / lo planes of a Gram-method matrix)
    EpiTiles et{};
    et.t0 = blockIdx.x;
    et.tstep = gridDim.x;
    et.row_off = 0;
    et.remote = false;
    et.tempty = tempty;
    sym_epilogue<MODE, BN, BM>(p, &map_xo, &map_xl, &map_xh, epi + (warp - 2) * SYM_WARP_BYTES, tfull, et, abort,
                               tmem_base, warp, lane);
  } else {
    // --------------------------------------------------------- epilogue
    EpiTiles et{};
    et.t0 = blockIdx.x;
    et.tstep = gridDim.x;
    et.row_off = 0;
    et.remote = false;
    et.tempty = tempty;
    mn_epilogue<MODE, BN, BM, OneSlots<MODE>::v>(p, &map_xh, &map_xl, &map_xo, epi + (warp - 2) * L::WARP_BYTES, xfull + 2 * (warp - 2),
                              tfull, et, abort, tmem_base, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    __syncwarp();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <int MODE, int BN, int AP, int BP>
cudaError_t launch_one(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0, const CUtensorMap& b1,
                       const CUtensorMap& xh, const CUtensorMap& xl, const CUtensorMap& xo, const NsGemmParams& p,
                       int grid, cudaStream_t s, const CUtensorMap* a2 = nullptr, const CUtensorMap* b2 = nullptr) {
  auto kern = ns_gemm_tc_kernel<MODE, BN, AP, BP>;
  using C = Cfg<MODE, BN, AP, BP>;
  static bool configured = false;   // per instantiation; the attribute is per device function
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const cudaError_t e = launch_k(pdl_level() >= 1, kern, dim3(grid), dim3(TC_THREADS), C::SMEM, s, a0, a1, a2 ? *a2 : a1, b0, b1,
                                 b2 ? *b2 : b1, xh, xl, xo, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_ns_gemm_tc(int mode, int bn, const CUtensorMap& ma, const CUtensorMap& mb,
                              const CUtensorMap& mso, const CUtensorMap& mso_lo, const NsGemmParams& p, int grid,
                              cudaStream_t s) {
  if (p.num_tiles == 0) return cudaSuccess;
  if (bn == 256) {
    switch (mode) {
      case MODE_SYRK: return launch_one<MODE_SYRK, 256, 1, 1>(ma, ma, mb, mb, mb, mb, mso, p, grid, s);
      case MODE_POLY: return launch_one<MODE_POLY, 256, 1, 1>(ma, ma, mb, mb, mb, mb, mso, p, grid, s);
      case MODE_G_R0: return launch_one<MODE_G_R0, 256, 1, 1>(ma, ma, mb, mb, mb, mso_lo, mso, p, grid, s);
    }
  } else if (bn == 128) {
    switch (mode) {
      case MODE_SYRK: return launch_one<MODE_SYRK, 128, 1, 1>(ma, ma, mb, mb, mb, mb, mso, p, grid, s);
      case MODE_POLY: return launch_one<MODE_POLY, 128, 1, 1>(ma, ma, mb, mb, mb, mb, mso, p, grid, s);
      case MODE_G_R0: return launch_one<MODE_G_R0, 128, 1, 1>(ma, ma, mb, mb, mb, mso_lo, mso, p, grid, s);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_ns_gemm_tc_update(int mode, int bn, const CUtensorMap& ma, const CUtensorMap& mb,
                                     const CUtensorMap& mxh, const CUtensorMap& mxl, const CUtensorMap& mxo,
                                     const NsGemmParams& p, int grid, cudaStream_t s) {
  if (p.num_tiles == 0) return cudaSuccess;
  if (bn == 256) {
    switch (mode) {
      case MODE_UPDATE: return launch_one<MODE_UPDATE, 256, 1, 1>(ma, ma, mb, mb, mxh, mxl, mxo, p, grid, s);
      case MODE_FINAL: return launch_one<MODE_FINAL, 256, 1, 1>(ma, ma, mb, mb, mxh, mxl, mxo, p, grid, s);
      case MODE_FINAL_T: return launch_one<MODE_FINAL_T, 256, 1, 1>(ma, ma, mb, mb, mxh, mxl, mxo, p, grid, s);
    }
  } else if (bn == 128) {
    switch (mode) {
      case MODE_UPDATE: return launch_one<MODE_UPDATE, 128, 1, 1>(ma, ma, mb, mb, mxh, mxl, mxo, p, grid, s);
      case MODE_FINAL: return launch_one<MODE_FINAL, 128, 1, 1>(ma, ma, mb, mb, mxh, mxl, mxo, p, grid, s);
      case MODE_FINAL_T: return launch_one<MODE_FINAL_T, 128, 1, 1>(ma, ma, mb, mb, mxh, mxl, mxo, p, grid, s);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_ns_gemm_tc_f32(int mode, const CUtensorMap* a, const CUtensorMap* b, const CUtensorMap* o,
                                  const NsGemmParams& p, int grid, cudaStream_t s) {
  if (p.num_tiles == 0) return cudaSuccess;
  switch (mode) {
    // symmetric outputs: first plane through map_xo, then map_xl, map_xh
    case MODE_F_SYRK: return launch_one<MODE_F_SYRK, 128, 3, 3>(a[0], a[1], b[0], b[1], o[2], o[1], o[0], p, grid, s, &a[2], &b[2]);
    case MODE_F_POLY: return launch_one<MODE_F_POLY, 128, 3, 3>(a[0], a[1], b[0], b[1], o[2], o[1], o[0], p, grid, s, &a[2], &b[2]);
    // the next X's planes through map_xh, map_xl, map_xo
    case MODE_F_UPDATE: return launch_one<MODE_F_UPDATE, 128, 3, 3>(a[0], a[1], b[0], b[1], o[0], o[1], o[2], p, grid, s, &a[2], &b[2]);
    case MODE_F_FINAL: return launch_one<MODE_F_FINAL, 128, 3, 3>(a[0], a[1], b[0], b[1], b[0], b[0], b[0], p, grid, s, &a[2], &b[2]);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_ns_gemm_tc_planes(int mode, int bn, const CUtensorMap& a0, const CUtensorMap& a1,
                                     const CUtensorMap& b0, const CUtensorMap& b1, const CUtensorMap& so,
                                     const CUtensorMap& so_lo, const NsGemmParams& p, int grid, cudaStream_t s) {
  if (p.num_tiles == 0) return cudaSuccess;
  if (bn == 128) {
    switch (mode) {
      case MODE_G_P: return launch_one<MODE_G_P, 128, 2, 2>(a0, a1, b0, b1, b0, so_lo, so, p, grid, s);
      case MODE_G_PROD: return launch_one<MODE_G_PROD, 128, 2, 2>(a0, a1, b0, b1, b0, so_lo, so, p, grid, s);
      case MODE_G_FINAL: return launch_one<MODE_G_FINAL, 128, 2, 1>(a0, a1, b0, b0, b0, b0, b0, p, grid, s);
      case MODE_G_FINAL_T: return launch_one<MODE_G_FINAL_T, 128, 2, 1>(a0, a1, b0, b0, b0, b0, b0, p, grid, s);
    }
  } else if (bn == 256) {
    switch (mode) {
      case MODE_G_P: return launch_one<MODE_G_P, 256, 2, 2>(a0, a1, b0, b1, b0, so_lo, so, p, grid, s);
      case MODE_G_PROD: return launch_one<MODE_G_PROD, 256, 2, 2>(a0, a1, b0, b1, b0, so_lo, so, p, grid, s);
      case MODE_G_FINAL: return launch_one<MODE_G_FINAL, 256, 2, 1>(a0, a1, b0, b0, b0, b0, b0, p, grid, s);
      case MODE_G_FINAL_T: return launch_one<MODE_G_FINAL_T, 256, 2, 1>(a0, a1, b0, b0, b0, b0, b0, p, grid, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace muon
