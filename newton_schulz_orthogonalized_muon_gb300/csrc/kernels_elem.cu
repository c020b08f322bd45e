// HBM-bound kernels of the Muon step.
//
//  * muon_prepare_kernel: momentum M <- mu*M + G, Nesterov U = G + mu*M
//    (else U = M), per-tile partial sums of U^2 for the Frobenius norm, and
//    the NS working copy of U (fp32 for the fp32 CUDA-core path; for the
//    bf16 tensor-core path the MMA operand hi = bf16(U) and the lo plane as
//    signed-byte codes of U - hi; for the fp32 tensor-core path three bf16
//    planes hi, bf16(U - hi), bf16(U - hi - lo)), transposed through shared
//    memory when the block has rows > cols.
//    ("迎接DeepSeek开源周…Muon优化器" (coreui.cn), §代码, Muon step;
//     "Muon Optimizer and the Distributed Implementation", §Newton-Schulz
//     Iteration, normalisation by the Frobenius norm.)
//  * norm_finalize_kernel: per-matrix 1 / (||U||_F + eps), summed in a fixed
//    order (deterministic), and a non-finite check.
//  * apply_kernel: the final update when no NS step runs (O = X0).
//  * adamw_kernel: the AdamW fallback of the same printed Muon class.
//  * wait_selftest_kernel: a bounded wait on a barrier nothing completes,
//    so the timeout path can be exercised without hanging a GPU.
#include <cstdlib>

#include "common.cuh"
#include "internal.h"
#include "launch_opts.h"

namespace muon {

constexpr int PT = 64;           // prepare tile: 64 x 64 elements

// bf16 pairs of hi = bf16(u) and lo = bf16(u - hi) for 2 * pairs values,
// and (l2w non-null) the third plane bf16(u - hi - lo)
__device__ __forceinline__ void split_hi_lo(const float* u, uint32_t* hw, uint32_t* lw, int pairs,
                                            uint32_t* l2w = nullptr) {
#pragma unroll
  for (int k = 0; k < pairs; ++k) {
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(u[2 * k], u[2 * k + 1]);
    const float2 hf = __bfloat1622float2(h2);
    hw[k] = *reinterpret_cast<const uint32_t*>(&h2);
    const float r0 = u[2 * k] - hf.x, r1 = u[2 * k + 1] - hf.y;
    const __nv_bfloat162 l2 = __floats2bfloat162_rn(r0, r1);
    lw[k] = *reinterpret_cast<const uint32_t*>(&l2);
    if (l2w != nullptr) {
      const float2 lf = __bfloat1622float2(l2);
      l2w[k] = pack_bf16x2(r0 - lf.x, r1 - lf.y);
    }
  }
}

// the lo code of one value, and a word of the codes of four
__device__ __forceinline__ int lo8_of(float u) {
  return lo8_code(__float_as_uint(u), __float_as_uint(bf2f(f2bf(u))));
}
__device__ __forceinline__ uint32_t lo8_word(const float* u) {
  return pack_lo8x4(lo8_of(u[0]), lo8_of(u[1]), lo8_of(u[2]), lo8_of(u[3]));
}

// the third plane of one value
__device__ __forceinline__ __nv_bfloat16 third_plane(float u) {
  const float r = u - bf2f(f2bf(u));
  return f2bf(r - bf2f(f2bf(r)));
}
constexpr int PREP_THREADS = 256;

// 16-byte asynchronous copy global -> shared (bypassing L1), and the waits
__device__ __forceinline__ void cp_async16(void* sdst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(sdst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// The NS working copy of 8 consecutive values u (16-byte aligned at xo)
// and of one value.  kHiLo8: the bf16 tensor-core path's hi plane and lo
// codes only (the planes of the other paths are neither computed nor
// stored there); otherwise every plane the parameters name.
template <bool kHiLo8>
__device__ __forceinline__ void write_x8(const PrepParams& p, long long xo, const float* u) {
  if constexpr (kHiLo8) {
    uint32_t hw[4];
    int q[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __nv_bfloat162 h2 = __floats2bfloat162_rn(u[2 * k], u[2 * k + 1]);
      hw[k] = *reinterpret_cast<const uint32_t*>(&h2);
      q[2 * k] = lo8_code(__float_as_uint(u[2 * k]), hw[k] << 16);
      q[2 * k + 1] = lo8_code(__float_as_uint(u[2 * k + 1]), hw[k] & 0xFFFF0000u);
    }
    *reinterpret_cast<uint4*>(p.xb + xo) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint2*>(p.xlo8 + xo) =
        make_uint2(pack_lo8x4(q[0], q[1], q[2], q[3]), pack_lo8x4(q[4], q[5], q[6], q[7]));
  } else {
    if (p.xf != nullptr) {
      *reinterpret_cast<float4*>(p.xf + xo) = make_float4(u[0], u[1], u[2], u[3]);
      *reinterpret_cast<float4*>(p.xf + xo + 4) = make_float4(u[4], u[5], u[6], u[7]);
    }
    if (p.xb != nullptr) {
      uint32_t hw[4], lw[4], l2w[4];
      split_hi_lo(u, hw, lw, 4, l2w);
      *reinterpret_cast<uint4*>(p.xb + xo) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      if (p.xlo8 != nullptr) *reinterpret_cast<uint2*>(p.xlo8 + xo) = make_uint2(lo8_word(u), lo8_word(u + 4));
      if (p.xlo != nullptr) *reinterpret_cast<uint4*>(p.xlo + xo) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      if (p.xlo2 != nullptr) *reinterpret_cast<uint4*>(p.xlo2 + xo) = make_uint4(l2w[0], l2w[1], l2w[2], l2w[3]);
    }
  }
}
// ... of 4 consecutive values (8-byte aligned at xo)
template <bool kHiLo8>
__device__ __forceinline__ void write_x4(const PrepParams& p, long long xo, const float* u) {
  if constexpr (kHiLo8) {
    uint32_t hw[2];
    int q[4];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const __nv_bfloat162 h2 = __floats2bfloat162_rn(u[2 * k], u[2 * k + 1]);
      hw[k] = *reinterpret_cast<const uint32_t*>(&h2);
      q[2 * k] = lo8_code(__float_as_uint(u[2 * k]), hw[k] << 16);
      q[2 * k + 1] = lo8_code(__float_as_uint(u[2 * k + 1]), hw[k] & 0xFFFF0000u);
    }
    *reinterpret_cast<uint2*>(p.xb + xo) = make_uint2(hw[0], hw[1]);
    *reinterpret_cast<uint32_t*>(p.xlo8 + xo) = pack_lo8x4(q[0], q[1], q[2], q[3]);
  } else {
    if (p.xf != nullptr) *reinterpret_cast<float4*>(p.xf + xo) = make_float4(u[0], u[1], u[2], u[3]);
    if (p.xb != nullptr) {
      uint32_t hw[2], lw[2], l2w[2];
      split_hi_lo(u, hw, lw, 2, l2w);
      *reinterpret_cast<uint2*>(p.xb + xo) = make_uint2(hw[0], hw[1]);
      if (p.xlo8 != nullptr) *reinterpret_cast<uint32_t*>(p.xlo8 + xo) = lo8_word(u);
      if (p.xlo != nullptr) *reinterpret_cast<uint2*>(p.xlo + xo) = make_uint2(lw[0], lw[1]);
      if (p.xlo2 != nullptr) *reinterpret_cast<uint2*>(p.xlo2 + xo) = make_uint2(l2w[0], l2w[1]);
    }
  }
}
template <bool kHiLo8>
__device__ __forceinline__ void write_x1(const PrepParams& p, long long xo, float u) {
  if (!kHiLo8 && p.xf != nullptr) p.xf[xo] = u;
  if (kHiLo8 || p.xb != nullptr) p.xb[xo] = f2bf(u);
  if (!kHiLo8 && p.xlo != nullptr) p.xlo[xo] = f2bf(u - bf2f(f2bf(u)));
  if (!kHiLo8 && p.xlo2 != nullptr) p.xlo2[xo] = third_plane(u);
  if (kHiLo8 || p.xlo8 != nullptr) p.xlo8[xo] = static_cast<int8_t>(lo8_of(u));
}

// Shared-memory placements of the prepare kernel (tile row rl, 8-column
// chunk ch, column lc): the staged G tile's 16-byte chunks swap halves on
// odd rows; the bf16 path's transpose tile orders a row's chunks by XOR
// with its 8-row band and with its parity (hi bits) or its second bit
// (codes).  The row pass's 8-byte reads and its 8- and 4-byte tile stores,
// and the column pass's reads of eight bands at once, then fall in
// distinct banks.
__device__ __forceinline__ int gst_col(int rl, int lc) { return (((lc >> 3) ^ ((rl & 1) << 2)) << 3) | (lc & 7); }
__device__ __forceinline__ int hi_chunk(int rl, int ch) { return ch ^ (rl >> 3) ^ ((rl & 1) << 2); }
__device__ __forceinline__ int lo_chunk(int rl, int ch) { return ch ^ (rl >> 3) ^ ((rl & 2) << 1); }

template <bool kHiLo8>
__global__ void __launch_bounds__(PREP_THREADS) muon_prepare_kernel(PrepParams p) {
  // transpose tile: fp32 U (padded rows) for the generic instance; for the
  // bf16 path the encoded hi bits (64 x 64 bf16) and lo codes (64 x 64
  // bytes), 12 KB, so six blocks fit on an SM; their chunks placed by
  // hi_chunk / lo_chunk.
  static_assert(PT == 64 && PREP_THREADS == 256, "eight 8-row bands, eight chunks, one warp per chunk");
  constexpr int TILE_BYTES = kHiLo8 ? PT * PT * 3 : PT * (PT + 1) * 4;
  __shared__ __align__(16) uint8_t tbuf[TILE_BYTES];
  float (*tile)[PT + 1] = reinterpret_cast<float (*)[PT + 1]>(tbuf);
  uint32_t* const thi = reinterpret_cast<uint32_t*>(tbuf);          // [PT][PT / 2] words
  uint8_t* const tlo = tbuf + PT * PT * 2;                           // [PT][PT] bytes
  __shared__ float red[PREP_THREADS / 32];
  // the block's bf16 G and fp32 M tiles, staged by cp.async: every load of
  // the block is in flight at once without holding registers (the kernel
  // waits on memory latency; with registers as the load targets its warps
  // kept the HBM ~70% busy)
  __shared__ __align__(16) __nv_bfloat16 gst[PT * PT];
  __shared__ __align__(16) float mst[PT * PT];
  // the workspace it writes is read by the previous group's kernels
  pdl_wait();
  pdl_launch_dependents();

  const int b = blockIdx.y;
  const SrcEntry e = p.src[b];
  const int tiles_x = (e.cols + PT - 1) / PT;
  const int r0 = (blockIdx.x / tiles_x) * PT;
  const int c0 = (blockIdx.x % tiles_x) * PT;
  const int tx = threadIdx.x & 7;   // column-group lane of a row
  const int ty = threadIdx.x >> 3;  // row within a 32-row pass
  const float mu = p.mu;
  const bool vec = ((e.cols & 7) == 0) && ((e.ld & 7) == 0) &&
                   ((reinterpret_cast<uintptr_t>(e.g) & 15) == 0) &&
                   (e.mom == nullptr || (reinterpret_cast<uintptr_t>(e.mom) & 15) == 0);
  const long long xbase = static_cast<long long>(b) * p.m * p.ldx;
  float ss = 0.f;
  const bool gstage = vec && e.gdtype == DT_BF16;
  const bool mstage = vec && e.mom != nullptr;
  if (gstage || mstage) {
    // chunks of 8 bf16 (G) and 4 fp32 (M) values; cols % 8 == 0 on this
    // path, so a chunk that starts inside the matrix ends inside it
    if (gstage) {
      for (int q = threadIdx.x; q < PT * 8; q += PREP_THREADS) {
        const int rl = q >> 3, c = c0 + (q & 7) * 8;
        if (r0 + rl < e.rows && c < e.cols)
          cp_async16(gst + rl * PT + gst_col(rl, (q & 7) * 8),
                     reinterpret_cast<const __nv_bfloat16*>(e.g) + static_cast<long long>(r0 + rl) * e.ld + c);
      }
    }
    if (mstage) {
      for (int q = threadIdx.x; q < PT * 16; q += PREP_THREADS) {
        const int rl = q >> 4, c = c0 + (q & 15) * 4;
        if (r0 + rl < e.rows && c < e.cols)
          cp_async16(mst + rl * PT + (q & 15) * 4, e.mom + static_cast<long long>(r0 + rl) * e.ld + c);
      }
    }
    cp_async_wait_all();
    __syncthreads();
  }

  // Row pass: thread (tx, ty) takes tile rows ty and ty + 32 and, in each,
  // the 4-column groups from 4tx and 32 + 4tx, so that the 8 lanes of a row
  // store contiguous segments (M 128 bytes, X hi 64, X codes 32) and every
  // 32-byte sector is written by one instruction.
#pragma unroll
  for (int pass = 0; pass < PT / 32; ++pass) {
    const int rl = ty + 32 * pass;
    const int r = r0 + rl;
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {
      const int lc = 32 * gi + 4 * tx;
      const int c = c0 + lc;
      float u[4] = {0.f, 0.f, 0.f, 0.f};
      if (r < e.rows) {
        const long long off = static_cast<long long>(r) * e.ld + c;
        if (vec) {
          if (c < e.cols) {   // cols % 8 == 0: a group that starts inside ends inside
            float g[4];
            if (e.gdtype == DT_BF16) {
              const uint2 raw = *reinterpret_cast<const uint2*>(gst + rl * PT + gst_col(rl, lc));
              const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
              const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
              g[0] = f0.x; g[1] = f0.y; g[2] = f1.x; g[3] = f1.y;
            } else {
              const float4 f = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(e.g) + off);
              g[0] = f.x; g[1] = f.y; g[2] = f.z; g[3] = f.w;
            }
            if (e.mom != nullptr) {
              const float4 m = *reinterpret_cast<const float4*>(mst + rl * PT + lc);
              const float mo[4] = {fmaf(mu, m.x, g[0]), fmaf(mu, m.y, g[1]), fmaf(mu, m.z, g[2]), fmaf(mu, m.w, g[3])};
              *reinterpret_cast<float4*>(e.mom + off) = make_float4(mo[0], mo[1], mo[2], mo[3]);
#pragma unroll
              for (int k = 0; k < 4; ++k) u[k] = p.nesterov ? fmaf(mu, mo[k], g[k]) : mo[k];
            } else {
#pragma unroll
              for (int k = 0; k < 4; ++k) u[k] = g[k];
            }
          }
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (c + k < e.cols) {
              const float gv = load_as_f32(e.g, off + k, e.gdtype);
              if (e.mom != nullptr) {
                const float mv = fmaf(mu, e.mom[off + k], gv);
                e.mom[off + k] = mv;
                u[k] = p.nesterov ? fmaf(mu, mv, gv) : mv;
              } else {
                u[k] = gv;
              }
            }
          }
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) ss = fmaf(u[k], u[k], ss);

      if (!e.transposed) {
        // NS orientation == parameter orientation: X[r][c]
        if (r < e.rows) {
          const long long xo = xbase + static_cast<long long>(r) * p.ldx + c;
          if (c + 3 < e.cols) {
            write_x4<kHiLo8>(p, xo, u);
          } else {
            for (int k = 0; k < 4 && c + k < e.cols; ++k) write_x1<kHiLo8>(p, xo + k, u[k]);
          }
        }
      } else if constexpr (kHiLo8) {
        uint32_t hw[2];
        int q[4];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(u[2 * k], u[2 * k + 1]);
          hw[k] = *reinterpret_cast<const uint32_t*>(&h2);
          q[2 * k] = lo8_code(__float_as_uint(u[2 * k]), hw[k] << 16);
          q[2 * k + 1] = lo8_code(__float_as_uint(u[2 * k + 1]), hw[k] & 0xFFFF0000u);
        }
        const int ch = lc >> 3, sub = tx & 1;     // the group is half `sub` of chunk ch
        *reinterpret_cast<uint2*>(thi + rl * (PT / 2) + hi_chunk(rl, ch) * 4 + sub * 2) = make_uint2(hw[0], hw[1]);
        *reinterpret_cast<uint32_t*>(tlo + rl * PT + lo_chunk(rl, ch) * 8 + sub * 4) = pack_lo8x4(q[0], q[1], q[2], q[3]);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) tile[rl][lc + k] = u[k];
      }
    }
  }

  if (e.transposed) __syncthreads();
  if (e.transposed) {
    const int wx = threadIdx.x & 7, wy = threadIdx.x >> 3;
    if constexpr (kHiLo8) {
      // X[c][r] = U[r][c]: warp w takes the tile's chunk w (columns 8w ..
      // 8w+7); lane (wx, j) reads rows 8wx .. 8wx+7 of its column pair
      // 8w+2j, 8w+2j+1 (one word of hi, two bytes of codes a row) and writes
      // both columns' X rows, 8 consecutive r each
      const int ch = threadIdx.x >> 5, j = wy & 3;
      uint32_t h[8], l[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int R = wx * 8 + k;
        h[k] = thi[R * (PT / 2) + hi_chunk(R, ch) * 4 + j];
        l[k] = *reinterpret_cast<const uint16_t*>(tlo + R * PT + lo_chunk(R, ch) * 8 + j * 2);
      }
      const int r = r0 + wx * 8;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int c = c0 + ch * 8 + j * 2 + half;
        if (c < e.cols) {
          const long long xo = xbase + static_cast<long long>(c) * p.ldx + r;
          const uint32_t hs = half ? 0x7632u : 0x5410u;   // the high or the low bf16 of each row's word
          const uint32_t ls = half ? 0x7531u : 0x6420u;   // the odd or the even byte of each row's pair
          const uint4 hv = make_uint4(__byte_perm(h[0], h[1], hs), __byte_perm(h[2], h[3], hs),
                                      __byte_perm(h[4], h[5], hs), __byte_perm(h[6], h[7], hs));
          const uint2 lv = make_uint2(__byte_perm(__byte_perm(l[0], l[1], 0x5410u), __byte_perm(l[2], l[3], 0x5410u), ls),
                                      __byte_perm(__byte_perm(l[4], l[5], 0x5410u), __byte_perm(l[6], l[7], 0x5410u), ls));
          if (r + 7 < e.rows) {
            *reinterpret_cast<uint4*>(p.xb + xo) = hv;
            *reinterpret_cast<uint2*>(p.xlo8 + xo) = lv;
          } else {
            const uint32_t hh[4] = {hv.x, hv.y, hv.z, hv.w}, ll[2] = {lv.x, lv.y};
            for (int k = 0; k < 8 && r + k < e.rows; ++k) {
              reinterpret_cast<uint16_t*>(p.xb)[xo + k] = static_cast<uint16_t>(hh[k >> 1] >> (16 * (k & 1)));
              reinterpret_cast<uint8_t*>(p.xlo8)[xo + k] = static_cast<uint8_t>(ll[k >> 2] >> (8 * (k & 3)));
            }
          }
        }
      }
    } else {
      // X[c][r] = U[r][c]: thread (wx, wy) writes X rows c0+wy+32*pass, 8 consecutive r
      // (16-byte hi stores; the column reads of the padded tile are free of bank conflicts)
#pragma unroll
      for (int pass = 0; pass < PT / 32; ++pass) {
        const int cl = wy + 32 * pass;
        const int c = c0 + cl;
        const int r = r0 + wx * 8;
        if (c < e.cols) {
          const long long xo = xbase + static_cast<long long>(c) * p.ldx + r;
          float u[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) u[k] = tile[wx * 8 + k][cl];
          if (r + 7 < e.rows) {
            write_x8<kHiLo8>(p, xo, u);
          } else {
            for (int k = 0; k < 8 && r + k < e.rows; ++k) write_x1<kHiLo8>(p, xo + k, u[k]);
          }
        }
      }
    }
  }

  // Block sum of U^2 in a fixed order.
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < PREP_THREADS / 32; ++w) t += red[w];
    p.partials[static_cast<long long>(b) * p.tiles_per_mat + blockIdx.x] = t;
  }
}

// One warp per matrix: scale[b] = 1 / (sqrt(sum of partials) + eps).
__global__ void norm_finalize_kernel(const float* partials, int tiles_per_mat, int batch, float eps, float* scale,
                                     unsigned* err) {
  pdl_wait();
  pdl_launch_dependents();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= batch) return;
  const float* pp = partials + static_cast<long long>(warp) * tiles_per_mat;
  double s = 0.0;
  for (int i = lane; i < tiles_per_mat; i += 32) s += static_cast<double>(pp[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) {
    if (!isfinite(s)) atomicOr(err, ERRBIT_NONFINITE);
    scale[warp] = static_cast<float>(1.0 / (sqrt(s) + static_cast<double>(eps)));
  }
}

// Final update with no Newton-Schulz step: O = X0 = scale * U (fp32 master).
__global__ void apply_kernel(ApplyParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.y;
  const OutEntry e = p.out[b];
  const float s = p.scale[b];
  const long long total = static_cast<long long>(p.m) * p.n;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / p.n), c = static_cast<int>(i % p.n);
    const float o = s * p.xf[(static_cast<long long>(b) * p.m + r) * p.ldx + c];
    store_out_scalar(e, r, c, o);
  }
}

// AdamW fallback, one chunk of one tensor per block (multi-tensor launch).
// Eight elements per thread and step: 16-byte loads/stores of the bf16
// parameter and gradient and two 16-byte accesses each for m and v; the
// ragged tail (or a misaligned tensor) goes element by element.
__device__ __forceinline__ void adamw_one(const AdamParams& p, const AdamTensor& t, long long i) {
  const float g = load_as_f32(t.g, i, t.gdtype);
  float m = t.m[i], v = t.v[i];
  m = fmaf(1.f - p.beta1, g - m, m);
  v = fmaf(1.f - p.beta2, fmaf(g, g, -v), v);
  t.m[i] = m;
  t.v[i] = v;
  const float u = m / (p.eps + sqrtf(v));
  store_from_f32(t.p, i, t.pdtype, fmaf(load_as_f32(t.p, i, t.pdtype), p.decay, -p.step_size * u));
}

__device__ __forceinline__ void load8(const void* base, long long i, int dtype, float* f) {
  if (dtype == DT_BF16) {
    const uint4 raw = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(base) + i);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 x = __bfloat1622float2(h[k]);
      f[2 * k] = x.x;
      f[2 * k + 1] = x.y;
    }
  } else {
    const float4 a = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + i);
    const float4 b = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + i + 4);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
}

__device__ __forceinline__ void store8(void* base, long long i, int dtype, const float* f) {
  if (dtype == DT_BF16) {
    uint4 raw;
    uint32_t* w = reinterpret_cast<uint32_t*>(&raw);
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = pack_bf16x2(f[2 * k], f[2 * k + 1]);
    *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(base) + i) = raw;
  } else {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + i) = make_float4(f[0], f[1], f[2], f[3]);
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + i + 4) = make_float4(f[4], f[5], f[6], f[7]);
  }
}

__global__ void __launch_bounds__(256) adamw_kernel(AdamParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const AdamChunk ch = p.chunks[blockIdx.x];
  const AdamTensor t = p.tensors[ch.tensor];
  const long long beg = ch.offset;
  const long long end = min(beg + static_cast<long long>(ADAM_CHUNK), t.numel);
  const bool vec = ((reinterpret_cast<uintptr_t>(t.p) | reinterpret_cast<uintptr_t>(t.g) |
                     reinterpret_cast<uintptr_t>(t.m) | reinterpret_cast<uintptr_t>(t.v)) & 15) == 0;
  const long long vend = vec ? beg + ((end - beg) / 8) * 8 : beg;
  const float omb1 = 1.f - p.beta1, omb2 = 1.f - p.beta2;
  for (long long i = beg + 8LL * threadIdx.x; i < vend; i += 8LL * blockDim.x) {
    float g[8], w[8], m[8], v[8];
    load8(t.g, i, t.gdtype, g);
    load8(t.p, i, t.pdtype, w);
    load8(t.m, i, DT_F32, m);
    load8(t.v, i, DT_F32, v);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      m[k] = fmaf(omb1, g[k] - m[k], m[k]);
      v[k] = fmaf(omb2, fmaf(g[k], g[k], -v[k]), v[k]);
      w[k] = fmaf(w[k], p.decay, -p.step_size * (m[k] / (p.eps + sqrtf(v[k]))));
    }
    store8(t.m, i, DT_F32, m);
    store8(t.v, i, DT_F32, v);
    store8(t.p, i, t.pdtype, w);
  }
  for (long long i = vend + threadIdx.x; i < end; i += blockDim.x) adamw_one(p, t, i);
}

// Bounded wait on a barrier that nothing completes: must give up within
// timeout_ns and report ERRBIT_TIMEOUT.
__global__ void wait_selftest_kernel(unsigned long long timeout_ns, unsigned* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait_bounded(&bar, 0, nullptr, timeout_ns)) atomicOr(err, ERRBIT_TIMEOUT);
  }
}

// Descriptor arena upload: 16-byte words from the pinned staging buffer
// (read through its device address) into the device descriptor buffer.
__global__ void desc_copy_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, size_t n16) {
  pdl_wait();               // earlier kernels may still read the descriptor buffer
  pdl_launch_dependents();
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n16;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    dst[i] = src[i];
}

// ------------------------------------------------------------- launchers
int pdl_level() {
  static const int level = [] {
    const char* v = std::getenv("MUON_PDL");
    if (v == nullptr) return 1;
    return v[0] == '0' ? 0 : v[0] == '2' ? 2 : 1;
  }();
  return level;
}

namespace {
thread_local bool g_elem_pdl = false;
}
void set_elementwise_pdl(bool on) { g_elem_pdl = on; }
bool elementwise_pdl() { return g_elem_pdl; }
// the element-wise kernels' launches: with PDL at level 2, or at level 1
// when the calling thread's current call asked for it
static bool elem_pdl() { return pdl_level() >= 2 || (pdl_level() == 1 && g_elem_pdl); }

cudaError_t launch_desc_copy(void* dst, const void* src, size_t bytes, cudaStream_t s) {
  const size_t n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  const int threads = 256;
  const int blocks = static_cast<int>(std::min<size_t>((n16 + threads - 1) / threads, 1024));
  return launch_k(elem_pdl(), desc_copy_kernel, dim3(blocks), dim3(threads), 0, s, static_cast<uint4*>(dst),
                  static_cast<const uint4*>(src), n16);
}
cudaError_t launch_prepare(const PrepParams& p, int batch, int tiles_per_mat, cudaStream_t s) {
  if (batch == 0 || tiles_per_mat == 0) return cudaSuccess;
  dim3 grid(tiles_per_mat, batch);
  const bool hilo8 = p.xb != nullptr && p.xlo8 != nullptr && p.xf == nullptr && p.xlo == nullptr && p.xlo2 == nullptr;
  if (hilo8) return launch_k(elem_pdl(), muon_prepare_kernel<true>, grid, dim3(PREP_THREADS), 0, s, p);
  return launch_k(elem_pdl(), muon_prepare_kernel<false>, grid, dim3(PREP_THREADS), 0, s, p);
}

cudaError_t launch_norm_finalize(const float* partials, int tiles_per_mat, int batch, float eps, float* scale,
                                 unsigned* err, cudaStream_t s) {
  if (batch == 0) return cudaSuccess;
  const int threads = 256;
  const int blocks = (batch * 32 + threads - 1) / threads;
  return launch_k(elem_pdl(), norm_finalize_kernel, dim3(blocks), dim3(threads), 0, s, partials, tiles_per_mat, batch, eps, scale,
                  err);
}

cudaError_t launch_apply(const ApplyParams& p, int batch, cudaStream_t s) {
  if (batch == 0) return cudaSuccess;
  const long long total = static_cast<long long>(p.m) * p.n;
  int bx = static_cast<int>((total + 255) / 256);
  if (bx > 1024) bx = 1024;
  if (bx < 1) bx = 1;
  return launch_k(elem_pdl(), apply_kernel, dim3(bx, batch), dim3(256), 0, s, p);
}

cudaError_t launch_adamw(const AdamParams& p, int n_chunks, cudaStream_t s) {
  if (n_chunks == 0) return cudaSuccess;
  return launch_k(elem_pdl(), adamw_kernel, dim3(n_chunks), dim3(256), 0, s, p);
}

cudaError_t launch_wait_selftest(unsigned long long timeout_ns, unsigned* err, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(timeout_ns, err);
  return cudaGetLastError();
}

}  // namespace muon
