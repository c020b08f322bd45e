// fp32 Newton-Schulz GEMMs on the CUDA cores (fp32 FMA, fp32 storage).
//
// Same modes as the tensor-core kernels (SYRK, POLY, UPDATE, FINAL and the
// Gram modes G_R0, G_P, G_PROD, G_FINAL; see kernels_tc.cu), for the fp32
// path whose accuracy bar (1e-4 relative) rules out bf16 operands.  The
// Gram iteration squares the condition number of X, so on this path its
// m x m matrices (and their products) are kept in fp64 (T = double); the
// standard iteration uses T = float.  X ping-pongs between two fp32 buffers
// because it is
// both an operand and the output of UPDATE.  64 x 64 output tiles, 256
// threads, 4 x 4 outputs per thread, K staged 16 at a time in shared memory.
#include "common.cuh"
#include "internal.h"

namespace muon {
namespace {

constexpr int ST = 64;   // output tile
constexpr int SK = 16;   // K step

template <int MODE, typename T>
__global__ void __launch_bounds__(256) ns_gemm_simt_kernel(NsGemmParams p) {
  __shared__ T As[SK][ST + 4];
  __shared__ T Bs[SK][ST + 4];
  constexpr bool kSym = (MODE == MODE_SYRK || MODE == MODE_POLY || MODE == MODE_G_R0 || MODE == MODE_G_P ||
                         MODE == MODE_G_PROD);
  constexpr bool kMN = (MODE == MODE_UPDATE || MODE == MODE_FINAL || MODE == MODE_G_FINAL);
  const int M = p.m;
  const int Ncols = kSym ? p.m : p.n;
  const int K = (MODE == MODE_SYRK || MODE == MODE_G_R0) ? p.n : p.m;
  const int i0 = blockIdx.y * ST;
  const int j0 = blockIdx.x * ST;
  if (kSym && j0 + ST - 1 < i0) return;   // tile strictly below the diagonal: mirrored by its partner
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;

  // operand A rows come from X (fp32) in SYRK / G_R0, else from an m x m T matrix;
  // operand B is X (fp32) in the MN-major modes and SYRK / G_R0, else T.
  constexpr bool kAx = (MODE == MODE_SYRK || MODE == MODE_G_R0);
  constexpr bool kBx = kAx || kMN;
  for (int b = blockIdx.z; b < p.batch; b += gridDim.z) {
    const float* ax = p.xf_in + static_cast<long long>(b) * M * p.ldx;
    const T* at = reinterpret_cast<const T*>(p.sym_in) + static_cast<long long>(b) * M * p.ldm;
    const T* bt = reinterpret_cast<const T*>(MODE == MODE_G_PROD ? p.op_b : p.sym_in) +
                  static_cast<long long>(b) * M * p.ldm;
    const long long lda = kAx ? p.ldx : p.ldm;
    const long long ldb = kBx ? p.ldx : p.ldm;
    auto aop = [&](long long i) -> T { return kAx ? static_cast<T>(ax[i]) : at[i]; };
    auto bop = [&](long long i) -> T { return kBx ? static_cast<T>(ax[i]) : bt[i]; };
    T acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += SK) {
      {  // A tile: rows i0.., k0..k0+15 -> As[k][row]
        const int r = threadIdx.x >> 2, kq = (threadIdx.x & 3) * 4;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int gr = i0 + r, gk = k0 + kq + e;
          As[kq + e][r] = (gr < M && gk < K) ? aop(static_cast<long long>(gr) * lda + gk) : T(0);
        }
      }
      if (kMN) {  // B operand X[k][c]
        const int kr = threadIdx.x >> 4, cq = (threadIdx.x & 15) * 4;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int gk = k0 + kr, gc = j0 + cq + e;
          Bs[kr][cq + e] = (gk < K && gc < Ncols) ? bop(static_cast<long long>(gk) * ldb + gc) : T(0);
        }
      } else {  // B operand rows j0.. (K-major): Bs[k][col] = op[col][k]
        const int r = threadIdx.x >> 2, kq = (threadIdx.x & 3) * 4;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int gc = j0 + r, gk = k0 + kq + e;
          Bs[kq + e][r] = (gc < Ncols && gk < K) ? bop(static_cast<long long>(gc) * ldb + gk) : T(0);
        }
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < SK; ++kk) {
        T av[4], bv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          av[e] = As[kk][ty * 4 + e];
          bv[e] = Bs[kk][tx * 4 + e];
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[r][c] = fma(av[r], bv[c], acc[r][c]);
      }
      __syncthreads();
    }

    T s = T(1);
    if (p.scale != nullptr) {
      s = static_cast<T>(p.scale[b]);
      if (MODE == MODE_SYRK || MODE == MODE_G_R0) s = s * s;
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int gr = i0 + ty * 4 + r;
      if (gr >= M) continue;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int gc = j0 + tx * 4 + c;
        if (gc >= Ncols) continue;
        T v = acc[r][c];
        if (kSym) {
          if (gc < gr) continue;
          T* out = reinterpret_cast<T*>(p.sym_out) + static_cast<long long>(b) * M * p.ldm;
          if (MODE == MODE_SYRK || MODE == MODE_G_R0) {
            v *= s;
          } else if (MODE == MODE_POLY || MODE == MODE_G_P) {
            v = fma(static_cast<T>(p.cb), at[static_cast<long long>(gr) * p.ldm + gc], static_cast<T>(p.cc) * v);
            if (MODE == MODE_G_P && gr == gc) v += static_cast<T>(p.ca);
          }
          out[static_cast<long long>(gr) * p.ldm + gc] = v;
          out[static_cast<long long>(gc) * p.ldm + gr] = v;
        } else {
          const long long xi = (static_cast<long long>(b) * M + gr) * p.ldx + gc;
          v = MODE == MODE_G_FINAL ? s * v : s * fma(static_cast<T>(p.ca), static_cast<T>(p.xf_in[xi]), v);
          if (MODE == MODE_UPDATE)
            p.xf_out[xi] = static_cast<float>(v);
          else
            store_out_scalar(p.out[b], gr, gc, static_cast<float>(v));
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_ns_gemm_simt(int mode, const NsGemmParams& p, cudaStream_t s, int wide) {
  if (p.batch == 0) return cudaSuccess;
  const bool sym = (mode == MODE_SYRK || mode == MODE_POLY || mode == MODE_G_R0 || mode == MODE_G_P ||
                    mode == MODE_G_PROD);
  const int ncols = sym ? p.m : p.n;
  dim3 grid((ncols + ST - 1) / ST, (p.m + ST - 1) / ST, p.batch < 65535 ? p.batch : 65535);
  if (!wide) {
    switch (mode) {
      case MODE_SYRK: ns_gemm_simt_kernel<MODE_SYRK, float><<<grid, 256, 0, s>>>(p); break;
      case MODE_POLY: ns_gemm_simt_kernel<MODE_POLY, float><<<grid, 256, 0, s>>>(p); break;
      case MODE_UPDATE: ns_gemm_simt_kernel<MODE_UPDATE, float><<<grid, 256, 0, s>>>(p); break;
      case MODE_FINAL: ns_gemm_simt_kernel<MODE_FINAL, float><<<grid, 256, 0, s>>>(p); break;
      default: return cudaErrorInvalidValue;
    }
  } else {
    switch (mode) {
      case MODE_G_R0: ns_gemm_simt_kernel<MODE_G_R0, double><<<grid, 256, 0, s>>>(p); break;
      case MODE_G_P: ns_gemm_simt_kernel<MODE_G_P, double><<<grid, 256, 0, s>>>(p); break;
      case MODE_G_PROD: ns_gemm_simt_kernel<MODE_G_PROD, double><<<grid, 256, 0, s>>>(p); break;
      case MODE_G_FINAL: ns_gemm_simt_kernel<MODE_G_FINAL, double><<<grid, 256, 0, s>>>(p); break;
      default: return cudaErrorInvalidValue;
    }
  }
  return cudaGetLastError();
}

}  // namespace muon
