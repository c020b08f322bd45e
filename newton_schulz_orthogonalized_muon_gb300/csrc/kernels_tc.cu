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
// CTA layout (192 threads, 1 CTA per SM, persistent over output tiles):
//   warp 0  lane 0: TMA producer (64 x 64 bf16 boxes, 128-byte swizzle)
//   warp 1  lane 0: MMA issuer, tcgen05.mma.cta_group::1.kind::f16,
//                   M = 128, N = BN, K = 16, fp32 accumulator in TMEM
//   warps 2-5     : epilogue, one TMEM lane (= output row) per thread
// The accumulator is double buffered in TMEM (2 x BN columns), so the
// epilogue of one tile overlaps the main loop of the next.
//
// Every barrier wait is bounded (time limit): on expiry the kernel records
// ERRBIT_TIMEOUT, drains its own MMAs and TMA copies (again bounded), frees
// TMEM and returns.
#include "common.cuh"
#include "internal.h"

namespace muon {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;                    // bf16 elements in one 128-byte swizzle row
constexpr int EPI_WARPS = 8;                           // two per TMEM lane quadrant
constexpr int TC_THREADS = 64 + 32 * EPI_WARPS;        // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue
constexpr int BOX_BYTES = 64 * 64 * 2;    // one 64 x 64 bf16 TMA box
constexpr unsigned long long DRAIN_NS = 1000000000ull;

template <int BN, int AP, int BP>
struct Cfg {
  static constexpr int A_BYTES = BM * BK * 2;            // one plane of the A tile
  static constexpr int B_BYTES = BN * BK * 2;            // one plane of the B tile
  static constexpr int STAGE_BYTES = AP * A_BYTES + BP * B_BYTES;
  static constexpr int STAGES = (196608 / STAGE_BYTES) < 8 ? (196608 / STAGE_BYTES) : 8;
  static constexpr int TMEM_COLS = 2 * BN;
  // epilogue staging for transposed destinations: 16 columns x 128 rows fp32
  static constexpr int XPOSE_LD = BM + 4;
  static constexpr int XPOSE_BYTES = 2 * 16 * XPOSE_LD * 4 + 64;   // one 16 x 128 fp32 stage per column half
  static constexpr size_t SMEM = static_cast<size_t>(STAGES) * STAGE_BYTES + 1024 + 256 + XPOSE_BYTES;
};

// Named barriers of the epilogue: id 1 + half (the 128 threads of one column
// half), id 3 (all 256 epilogue threads).
__device__ __forceinline__ void epi_half_sync(int half) {
  asm volatile("bar.sync %0, 128;" ::"r"(1 + half) : "memory");
}
__device__ __forceinline__ void epi_all_sync() {
  asm volatile("bar.sync 3, 256;" ::: "memory");
}

template <int MODE>
struct ModeTraits {
  static constexpr bool kSym = (MODE == MODE_SYRK || MODE == MODE_POLY || MODE == MODE_G_R0 ||
                                MODE == MODE_G_P || MODE == MODE_G_PROD);
  static constexpr bool kMN = (MODE == MODE_UPDATE || MODE == MODE_FINAL || MODE == MODE_G_FINAL);
  static constexpr bool kKn = (MODE == MODE_SYRK || MODE == MODE_G_R0);   // K = n (else K = m)
  static constexpr bool kPlanesOut = (MODE == MODE_G_R0 || MODE == MODE_G_P || MODE == MODE_G_PROD);
};

// Warp-collective bounded wait: every lane polls, the warp leaves together.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort,
                                               uint64_t timeout_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    const bool ok = mbar_try_wait(a, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
    if ((it & 31u) == 31u) {
      const bool give_up = (*abort != 0) || (globaltimer_ns() - t0 > timeout_ns);
      if (__any_sync(0xffffffffu, give_up)) return false;
    }
  }
}

__device__ __forceinline__ void raise_timeout(volatile int* abort, unsigned* err) {
  *abort = 1;
  atomicOr(err, ERRBIT_TIMEOUT);
}

template <int MODE>
__device__ __forceinline__ void decode_tile(const NsGemmParams& p, int t, int& b, int& i, int& j) {
  b = t / p.tiles_per_mat;
  const int l = t - b * p.tiles_per_mat;
  if (ModeTraits<MODE>::kSym) {
    const int2 ij = p.tri[l];
    i = ij.x;
    j = ij.y;
  } else {
    j = l / p.mi;          // column-block major: neighbouring tiles share X's column block
    i = l - j * p.mi;
  }
}

// ------------------------------------------------------------ epilogues
// v[16]: accumulator values of row gr, columns gc0 .. gc0+15.
template <int MODE>
__device__ __forceinline__ void epilogue_sym(const NsGemmParams& p, int b, int gr, int gc0, float* v, float s) {
  const int m = p.m;
  if (gr >= m) return;
  const size_t mat = static_cast<size_t>(b) * m;
  if (MODE == MODE_SYRK || MODE == MODE_G_R0) {
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] *= s;
  } else if (MODE == MODE_POLY || MODE == MODE_G_P) {
    // v = b * A + c * acc (G_P: A = R = hi + lo planes, plus a on the diagonal)
    const __nv_bfloat16* ain = reinterpret_cast<const __nv_bfloat16*>(p.sym_in) + (mat + gr) * p.ldm;
    const __nv_bfloat16* alo =
        MODE == MODE_G_P ? reinterpret_cast<const __nv_bfloat16*>(p.sym_in_lo) + (mat + gr) * p.ldm : nullptr;
    float a[16];
    if (gc0 + 15 < m) {
      uint4 raw[2];
      raw[0] = *reinterpret_cast<const uint4*>(ain + gc0);
      raw[1] = *reinterpret_cast<const uint4*>(ain + gc0 + 8);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(raw);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float2 f = __bfloat1622float2(h[e]);
        a[2 * e] = f.x;
        a[2 * e + 1] = f.y;
      }
      if (MODE == MODE_G_P) {
        raw[0] = *reinterpret_cast<const uint4*>(alo + gc0);
        raw[1] = *reinterpret_cast<const uint4*>(alo + gc0 + 8);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 f = __bfloat1622float2(h[e]);
          a[2 * e] += f.x;
          a[2 * e + 1] += f.y;
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int gc = gc0 + e;
        a[e] = gc < m ? bf2f(ain[gc]) + (MODE == MODE_G_P ? bf2f(alo[gc]) : 0.f) : 0.f;
      }
    }
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      v[e] = fmaf(p.cb, a[e], p.cc * v[e]);
      if (gc0 + e == gr) {
        v[e] += p.ca;
        if (MODE == MODE_POLY) p.pdiag[mat + gr] = v[e];
      }
    }
  }
  constexpr bool kPlanes = ModeTraits<MODE>::kPlanesOut;
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.sym_out);
  __nv_bfloat16* outlo = kPlanes ? reinterpret_cast<__nv_bfloat16*>(p.sym_out_lo) : nullptr;
  float lo[16];
  if (kPlanes) {
#pragma unroll
    for (int e = 0; e < 16; ++e) lo[e] = v[e] - bf2f(f2bf(v[e]));
  }
  __nv_bfloat16* row = out + (mat + gr) * p.ldm;
  __nv_bfloat16* rowlo = kPlanes ? outlo + (mat + gr) * p.ldm : nullptr;
  if (gc0 >= gr && gc0 + 15 < m) {
    uint4 pk[2];
    uint32_t* w = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
    *reinterpret_cast<uint4*>(row + gc0) = pk[0];
    *reinterpret_cast<uint4*>(row + gc0 + 8) = pk[1];
    if (kPlanes) {
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(lo[2 * e], lo[2 * e + 1]);
      *reinterpret_cast<uint4*>(rowlo + gc0) = pk[0];
      *reinterpret_cast<uint4*>(rowlo + gc0 + 8) = pk[1];
    }
  } else {
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int gc = gc0 + e;
      if (gc >= gr && gc < m) {
        row[gc] = f2bf(v[e]);
        if (kPlanes) rowlo[gc] = f2bf(lo[e]);
      }
    }
  }
  // mirror below the diagonal: lanes hold consecutive rows, so each store
  // of the warp covers 32 consecutive elements of row gc.
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const int gc = gc0 + e;
    if (gc > gr && gc < m) {
      out[(mat + gc) * p.ldm + gr] = f2bf(v[e]);
      if (kPlanes) outlo[(mat + gc) * p.ldm + gr] = f2bf(lo[e]);
    }
  }
}

// Sixteen fp32-master values of row gr from column gc0 (0 beyond n).
__device__ __forceinline__ void load_x16(const NsGemmParams& p, const float* xrow, int gc0, float* x) {
  if (gc0 + 15 < p.n) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 x4 = *reinterpret_cast<const float4*>(xrow + gc0 + 4 * q);
      x[4 * q] = x4.x;
      x[4 * q + 1] = x4.y;
      x[4 * q + 2] = x4.z;
      x[4 * q + 3] = x4.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 16; ++e) x[e] = gc0 + e < p.n ? xrow[gc0 + e] : 0.f;
  }
}

// UPDATE / FINAL value (in place in v) from the accumulator and the fp32
// master x: s * (acc + P_rr x - P^_rr x^), x^ = bf16(x) being the operand copy
// whose diagonal term the accumulator holds.  G_FINAL: s * acc.
template <int MODE>
__device__ __forceinline__ void update_values(float* v, const float* x, float pd, float pdb, float s) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    if (MODE == MODE_G_FINAL)
      v[e] *= s;
    else
      v[e] = s * fmaf(pd, x[e], fmaf(-pdb, bf2f(f2bf(x[e])), v[e]));
  }
}

// Store of UPDATE (new fp32 master + bf16 operand copy) or of a FINAL /
// G_FINAL tile whose destination is not transposed.
template <int MODE>
__device__ __forceinline__ void update_store(const NsGemmParams& p, int b, int gr, int gc0, const float* v) {
  const int n = p.n;
  if (gr >= p.m) return;
  if (MODE == MODE_UPDATE) {
    const size_t rowoff = (static_cast<size_t>(b) * p.m + gr) * p.ldx;
    float* xrow = p.xf + rowoff;
    __nv_bfloat16* brow = p.xb_out + rowoff;
    if (gc0 + 15 < n) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<float4*>(xrow + gc0 + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      uint4 pk[2];
      uint32_t* w = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
      *reinterpret_cast<uint4*>(brow + gc0) = pk[0];
      *reinterpret_cast<uint4*>(brow + gc0 + 8) = pk[1];
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int gc = gc0 + e;
        if (gc < n) {
          xrow[gc] = v[e];
          brow[gc] = f2bf(v[e]);
        }
      }
    }
  } else {
    const OutEntry oe = p.out[b];
    if (gc0 + 15 < n) {
      store_out_16(oe, gr, gc0, v);
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e)
        if (gc0 + e < n) store_out_scalar(oe, gr, gc0 + e, v[e]);
    }
  }
}

// FINAL / G_FINAL tile into a transposed destination (out[c][r] = O[r][c]):
// the 128 epilogue threads of one column half stage 16 columns of the tile in shared memory
// and write them back as 16 destination rows of 128 contiguous elements, so
// every thread issues 16-byte vector accesses to one destination row.
__device__ __forceinline__ void store_transposed_chunk(const NsGemmParams& p, const OutEntry& oe, int i, int gc0,
                                                       int row_in_tile, const float* v, float* stage, int ld,
                                                       int half) {
#pragma unroll
  for (int e = 0; e < 16; ++e) stage[e * ld + row_in_tile] = v[e];
  epi_half_sync(half);
  const int tid = row_in_tile;            // 0..127 over the four epilogue warps
  const int wr = tid >> 3;                // destination row in this chunk (= NS column gc0 + wr)
  const int wc = (tid & 7) * 16;          // destination column offset (= NS row within the tile)
  const int gcol = gc0 + wr;
  const int grow0 = i * BM + wc;
  if (gcol < p.n && grow0 < p.m) {
    float o[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) o[k] = stage[wr * ld + wc + k];
    const OutEntry rowwise{oe.ptr, oe.ld, 0, oe.dtype, oe.alpha, oe.beta};
    if (grow0 + 15 < p.m) {
      store_out_16(rowwise, gcol, grow0, o);
    } else {
      for (int k = 0; k < 16 && grow0 + k < p.m; ++k) store_out_scalar(rowwise, gcol, grow0 + k, o[k]);
    }
  }
  epi_half_sync(half);
}

// --------------------------------------------------------------- kernel
template <int MODE, int BN, int AP, int BP>
__global__ void __launch_bounds__(TC_THREADS, 1)
    ns_gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a0, const __grid_constant__ CUtensorMap map_a1,
                      const __grid_constant__ CUtensorMap map_b0, const __grid_constant__ CUtensorMap map_b1,
                      const NsGemmParams p) {
  using C = Cfg<BN, AP, BP>;
  constexpr bool kUpd = ModeTraits<MODE>::kMN;
  constexpr bool kSym = ModeTraits<MODE>::kSym;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

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
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, C::TMEM_COLS);
  if (warp == 1 && lane == 0) {
    tma_prefetch_map(&map_a0);
    tma_prefetch_map(&map_b0);
    if (AP == 2) tma_prefetch_map(&map_a1);
    if (BP == 2) tma_prefetch_map(&map_b1);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
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
            const CUtensorMap* ma = pa == 0 ? &map_a0 : &map_a1;
            tma_load_3d(sa + pa * C::A_BYTES, ma, &full[s], kb * BK, i * BM, b);
            tma_load_3d(sa + pa * C::A_BYTES + BOX_BYTES, ma, &full[s], kb * BK, i * BM + 64, b);
          }
#pragma unroll
          for (int pb = 0; pb < BP; ++pb) {
            const CUtensorMap* mb = pb == 0 ? &map_b0 : &map_b1;
#pragma unroll
            for (int q = 0; q < BN / 64; ++q) {
              if (kUpd)
                tma_load_3d(sb + pb * C::B_BYTES + q * BOX_BYTES, mb, &full[s], j * BN + q * 64, kb * BK, b);
              else
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
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN);
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
            const uint32_t boff = kUpd ? kk * 2048 : kk * 32;
            const uint64_t b0 = kUpd ? sdesc_sw128(sb + boff, BOX_BYTES, 1024) : sdesc_sw128(sb + boff, 16, 1024);
            umma_bf16(d, a0, b0, idesc, (kb | kk) != 0 ? 1u : 0u);
            if (BP == 2) {   // hi(A) * lo(B)
              const uint32_t sb1 = sb + C::B_BYTES + boff;
              umma_bf16(d, a0, kUpd ? sdesc_sw128(sb1, BOX_BYTES, 1024) : sdesc_sw128(sb1, 16, 1024), idesc, 1u);
            }
            if (AP == 2) {   // lo(A) * hi(B)
              umma_bf16(d, sdesc_sw128(sa + C::A_BYTES + kk * 32, 16, 1024), b0, idesc, 1u);
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
  } else {
    // --------------------------------------------------------- epilogue
    // warps 2-9: TMEM lane quadrant = warp % 4 (hardware rule), column half =
    // (warp - 2) / 4; each thread owns one output row of its half.
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row_in_tile = quad * 32 + lane;
    const int ncols = kUpd ? p.n : p.m;
    constexpr bool kFinal = (MODE == MODE_FINAL || MODE == MODE_G_FINAL);
    constexpr bool kNeedX = (MODE == MODE_UPDATE || MODE == MODE_FINAL);
    // after the 256-byte barrier block; the extra 1024 bytes of the
    // allocation are the alignment slack of `smem`
    float* xstage = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE_BYTES + 256) + half * 16 * C::XPOSE_LD;
    volatile int* wait_ok =
        reinterpret_cast<volatile int*>(smem + C::STAGES * C::STAGE_BYTES + 256 + 2 * 16 * C::XPOSE_LD * 4);
    const int cbeg = half * (BN / 2), cend = cbeg + BN / 2;
    int acc = 0;
    uint32_t acc_ph = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      int b, i, j;
      decode_tile<MODE>(p, t, b, i, j);
      const bool staged = kFinal && p.out[b].transposed;   // uniform over the epilogue warps
      bool ok = mbar_wait_warp(&tfull[acc], acc_ph, abort, p.timeout_ns);
      if (staged) {
        // the staged store uses named barriers: all epilogue warps must agree to go on
        if (lane == 0) wait_ok[warp - 2] = ok ? 1 : 0;
        epi_all_sync();
        for (int w = 0; w < EPI_WARPS; ++w) ok = ok && wait_ok[w];
        epi_all_sync();
      }
      if (!ok) {
        if (lane == 0) raise_timeout(abort, p.err);
        break;
      }
      tc_fence_after();
      const int gr = i * BM + row_in_tile;
      const int warp_row0 = i * BM + quad * 32;
      float s = 1.f;
      if (p.scale != nullptr) {
        s = p.scale[b];
        if (ModeTraits<MODE>::kKn) s = s * s;
      }
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * BN);
      // UPDATE / FINAL: the fp32 master row and the diagonal of P for this row;
      // the master values of the next chunk are loaded before the current
      // chunk is processed, so their latency overlaps the current chunk.
      const bool rowok = gr < p.m;
      const float* xrow = kNeedX ? p.xf + (static_cast<size_t>(b) * p.m + (rowok ? gr : 0)) * p.ldx : nullptr;
      float pd = 0.f, pdb = 0.f;
      float xcur[16], xnext[16];
      if (kNeedX) {
        if (rowok) {
          pd = p.pdiag[static_cast<size_t>(b) * p.m + gr];
          pdb = bf2f(f2bf(pd));
        }
        const int g0 = j * BN + cbeg;
        if (rowok && g0 < ncols) load_x16(p, xrow, g0, xcur);
      }
#pragma unroll 1
      for (int c0 = cbeg; c0 < cend; c0 += 16) {
        const int gc0 = j * BN + c0;
        if (gc0 >= ncols) break;
        if (kSym && gc0 + 15 < warp_row0) continue;  // below the diagonal
        if (kNeedX && rowok && c0 + 16 < cend && gc0 + 16 < ncols) load_x16(p, xrow, gc0 + 16, xnext);
        float v[16];
        tmem_ld16(tbase + static_cast<uint32_t>(c0), v);
        if (kSym) {
          epilogue_sym<MODE>(p, b, gr, gc0, v, s);
        } else {
          update_values<MODE>(v, xcur, pd, pdb, s);
          if (staged)
            store_transposed_chunk(p, p.out[b], i, gc0, row_in_tile, v, xstage, C::XPOSE_LD, half);
          else
            update_store<MODE>(p, b, gr, gc0, v);
        }
        if (kNeedX) {
#pragma unroll
          for (int e = 0; e < 16; ++e) xcur[e] = xnext[e];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_ph ^= 1u;
    }
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
                       const NsGemmParams& p, int grid, cudaStream_t s) {
  auto kern = ns_gemm_tc_kernel<MODE, BN, AP, BP>;
  using C = Cfg<BN, AP, BP>;
  static bool configured = false;   // per instantiation; the attribute is per device function
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  kern<<<grid, TC_THREADS, C::SMEM, s>>>(a0, a1, b0, b1, p);
  return cudaGetLastError();
}

}  // namespace

size_t ns_gemm_tc_smem_bytes(int bn) { return bn == 256 ? Cfg<256, 1, 1>::SMEM : Cfg<128, 1, 1>::SMEM; }
int ns_gemm_tc_stages(int bn) { return bn == 256 ? Cfg<256, 1, 1>::STAGES : Cfg<128, 1, 1>::STAGES; }

cudaError_t launch_ns_gemm_tc(int mode, int bn, const CUtensorMap& ma, const CUtensorMap& mb,
                              const NsGemmParams& p, int grid, cudaStream_t s) {
  if (p.num_tiles == 0) return cudaSuccess;
  if (bn == 256) {
    switch (mode) {
      case MODE_SYRK: return launch_one<MODE_SYRK, 256, 1, 1>(ma, ma, mb, mb, p, grid, s);
      case MODE_POLY: return launch_one<MODE_POLY, 256, 1, 1>(ma, ma, mb, mb, p, grid, s);
      case MODE_UPDATE: return launch_one<MODE_UPDATE, 256, 1, 1>(ma, ma, mb, mb, p, grid, s);
      case MODE_FINAL: return launch_one<MODE_FINAL, 256, 1, 1>(ma, ma, mb, mb, p, grid, s);
      case MODE_G_R0: return launch_one<MODE_G_R0, 256, 1, 1>(ma, ma, mb, mb, p, grid, s);
    }
  } else if (bn == 128) {
    switch (mode) {
      case MODE_SYRK: return launch_one<MODE_SYRK, 128, 1, 1>(ma, ma, mb, mb, p, grid, s);
      case MODE_POLY: return launch_one<MODE_POLY, 128, 1, 1>(ma, ma, mb, mb, p, grid, s);
      case MODE_UPDATE: return launch_one<MODE_UPDATE, 128, 1, 1>(ma, ma, mb, mb, p, grid, s);
      case MODE_FINAL: return launch_one<MODE_FINAL, 128, 1, 1>(ma, ma, mb, mb, p, grid, s);
      case MODE_G_R0: return launch_one<MODE_G_R0, 128, 1, 1>(ma, ma, mb, mb, p, grid, s);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_ns_gemm_tc_planes(int mode, int bn, const CUtensorMap& a0, const CUtensorMap& a1,
                                     const CUtensorMap& b0, const CUtensorMap& b1, const NsGemmParams& p, int grid,
                                     cudaStream_t s) {
  if (p.num_tiles == 0) return cudaSuccess;
  if (bn == 128) {
    switch (mode) {
      case MODE_G_P: return launch_one<MODE_G_P, 128, 2, 2>(a0, a1, b0, b1, p, grid, s);
      case MODE_G_PROD: return launch_one<MODE_G_PROD, 128, 2, 2>(a0, a1, b0, b1, p, grid, s);
      case MODE_G_FINAL: return launch_one<MODE_G_FINAL, 128, 2, 1>(a0, a1, b0, b0, p, grid, s);
    }
  } else if (bn == 256) {
    switch (mode) {
      case MODE_G_P: return launch_one<MODE_G_P, 256, 2, 2>(a0, a1, b0, b1, p, grid, s);
      case MODE_G_PROD: return launch_one<MODE_G_PROD, 256, 2, 2>(a0, a1, b0, b1, p, grid, s);
      case MODE_G_FINAL: return launch_one<MODE_G_FINAL, 256, 2, 1>(a0, a1, b0, b0, p, grid, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace muon
