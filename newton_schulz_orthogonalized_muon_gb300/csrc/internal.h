// Launch parameter blocks and launcher declarations shared by the kernel
// translation units and the host scheduler (muon_api.cu).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace muon {

// Programmatic dependent launch of the library's kernels, from the
// environment variable MUON_PDL (read once): 0 off; 1 (default) for the NS
// GEMM kernels, which cannot share an SM with the previous GEMM and so never
// wait beside a running kernel; 2 for every kernel.
int pdl_level();

// Launch `kern` on `s`, with programmatic stream serialization when `pdl`
// (the kernel must call pdl_wait() before touching memory an earlier kernel
// of the stream uses; common.cuh).
template <typename... Params, typename... Args>
cudaError_t launch_k(bool pdl, void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

struct SrcEntry;
struct OutEntry;

// ------------------------------------------------------------ prepare
struct PrepParams {
  const SrcEntry* src;     // [batch]
  float mu;
  int nesterov;
  int m;                   // NS rows (after the transpose rule)
  long long ldx;           // row stride of the NS workspace (elements)
  float* xf;               // fp32 copy [batch][m][ldx] or nullptr
  __nv_bfloat16* xb;       // bf16 operand copy = hi plane of the master, or nullptr (fp32 path)
  __nv_bfloat16* xlo;      // second bf16 plane bf16(U - bf16(U)) (fp32 tensor-core path), or nullptr
  int8_t* xlo8;            // lo plane of the bf16 path's master as signed-byte codes (lo8_code), or nullptr
  __nv_bfloat16* xlo2;     // third plane bf16(U - hi - lo) (fp32 tensor-core path), or nullptr
  float* partials;         // [batch][tiles_per_mat]
  int tiles_per_mat;
};

struct ApplyParams {
  const OutEntry* out;
  const float* scale;
  const float* xf;
  long long ldx;
  int m, n;
};

// --------------------------------------------------------------- AdamW
constexpr int ADAM_CHUNK = 16384;

struct AdamTensor {
  void* p;
  const void* g;
  float* m;
  float* v;
  long long numel;
  int pdtype, gdtype;
};

struct AdamChunk {
  int tensor;
  int pad;
  long long offset;
};

struct AdamParams {
  const AdamTensor* tensors;
  const AdamChunk* chunks;
  float beta1, beta2, eps;
  float decay;       // 1 - lr*wd
  float step_size;   // lr * sqrt(1 - beta2^t) / (1 - beta1^t)
};

// ------------------------------------------------ Newton-Schulz GEMMs
// Modes of the NS GEMM kernels (tensor-core path; P^ = bf16(P), X^ = bf16(X)):
//   SYRK   A = s^2 * X^ X^^T                 (symmetric, upper tiles, mirrored)
//   POLY   P = s*(a*I + b*A + c*A A)         (symmetric; fp32 diagonal kept aside;
//                                             s only in the first iteration)
//   UPDATE X' = P^ X^ + P_rr X - P^_rr X^    (master X = hi + lo, hi the bf16 operand)
//   FINAL  out = alpha*out + beta*X'         (parameter or caller matrix)
// The fp32 path (CUDA cores) evaluates the same iteration as
//   SYRK A = s^2 X X^T, POLY B = b*A + c*A A, UPDATE X' = s*(a*X + B X).
//
// Gram method (iterates on R = X X^T; every matrix below is m x m, symmetric,
// and stored as a pair of bf16 planes hi + lo, hi = bf16(v), lo = bf16(v - hi),
// so products of two such matrices are bf16x3: hi*hi + hi*lo + lo*hi):
//   G_R0    R = s^2 X X^T               (bf16 X operand, planes out)
//   G_P     P = a I + b R + c R R       (planes in/out)
//   G_PROD  C = A B                      (planes in/out; A, B commute)
//   G_FINAL out = alpha*out + beta*s*(Q X)  (Q planes, X bf16 MN-major)
//
// fp32 tensor-core path (fp32 parameters at the fp32 bar): every operand is
// held as three bf16 planes v = p0 + p1 + p2 (p0 = bf16(v), p1 = bf16(v - p0),
// p2 = bf16(v - p0 - p1): 24 mantissa bits), and a product of two such
// operands issues six MMAs per K step (p0q0 + p0q1 + p1q0 + p0q2 + p1q1 +
// p2q0) into one fp32 accumulator; the terms left out are below 2^-24 of the
// product.  The iteration is then the plain one, X' = P X:
//   F_SYRK   A = s^2 X X^T              (planes in, symmetric planes out)
//   F_POLY   P = a I + b A + c A A      (planes in and out)
//   F_UPDATE X' = s P X                  (planes in, planes out, no inputs read
//                                         in the epilogue)
//   F_FINAL  out = alpha*out + beta*s*(P X)   (element-wise destinations)
enum NsMode : int {
  MODE_SYRK = 0,
  MODE_POLY = 1,
  MODE_UPDATE = 2,
  MODE_FINAL = 3,
  MODE_G_R0 = 4,
  MODE_G_P = 5,
  MODE_G_PROD = 6,
  MODE_G_FINAL = 7,
  MODE_FINAL_T = 8,         // FINAL into bf16 destinations through per-matrix tensor maps
  MODE_G_FINAL_T = 9,       // G_FINAL likewise
  MODE_F_SYRK = 10,
  MODE_F_POLY = 11,
  MODE_F_UPDATE = 12,
  MODE_F_FINAL = 13
};

struct NsGemmParams {
  int m, n;                     // NS problem (m <= n)
  int batch;
  int tiles_per_mat;            // tiles of one matrix
  int num_tiles;                // batch * tiles_per_mat
  int mi;                       // row blocks of the output (UPDATE/FINAL)
  const int2* tri;              // (i, j) tile table of the symmetric modes
  const float* scale;           // per-matrix s = 1/||U||_F in the first iteration, or nullptr:
                                // SYRK writes s^2 X X^T, the bf16 path's POLY s P (its
                                // UPDATE / FINAL then apply none), the other updates s P X
  float ca, cb, cc;             // quintic coefficients
  // symmetric outputs (A or B matrix), row stride ldm
  void* sym_out;                // bf16 (tensor-core path) or fp32 (fp32 path)
  const void* sym_in;           // POLY: the A matrix for the b*A term (G_P: R hi plane)
  void* sym_out_lo;             // Gram modes: lo plane of the output
  int sym_n128;                 // CTA-pair symmetric products: tiles with at most 128 valid
                                // columns run N = 128 (B through a 64-row-box map)
  const void* sym_in_lo;        // G_P: R lo plane; F_POLY: A's second plane
  const void* sym_in_2;         // F_POLY: A's third plane
  const void* op_b;             // fp32 path, G_PROD: the second factor
  float* pdiag;                 // tensor-core path: fp32 diagonal of P [batch][m]
  long long ldm;
  // fp32 path: X operand / result, row stride ldx (the tensor-core path
  // reaches its master X through tensor maps)
  const float* xf_in;           // fp32 path: X operand (ping-pong partner of xf_out)
  float* xf_out;                // fp32 path: new X
  long long ldx;
  const OutEntry* out;          // FINAL destinations [batch]
  // FINAL_T / G_FINAL_T: one tensor map per destination [batch], 3-D {dest cols, dest
  // rows, 1}, bf16, 32 x 32 boxes with 64-byte swizzle (encode_box32), in
  // global memory (64-byte aligned)
  const CUtensorMap* wmap;
  unsigned* err;
  unsigned long long timeout_ns;
};

// tensor-core path (bf16 operands, fp32 accumulation in TMEM)
// BN: output tile width (128 or 256).  Maps are 3-D (x = column, y = row,
// z = matrix) bf16 maps with a 64 x 64 box and 128-byte swizzle.
// Operands with two planes (Gram modes) pass their lo-plane maps in a1 / b1.
// Symmetric products write their output through TMA: map_so is the output
// matrix (A or P), or for G_R0 / G_P / G_PROD its hi plane, and map_so_lo
// the lo plane (SYRK / POLY ignore it); bf16 with 32 x 32 boxes
// (encode_box32).
cudaError_t launch_ns_gemm_tc(int mode, int bn, const CUtensorMap& map_a, const CUtensorMap& map_b,
                              const CUtensorMap& map_so, const CUtensorMap& map_so_lo, const NsGemmParams& p,
                              int grid, cudaStream_t s);
// UPDATE / FINAL: the master X is hi + lo, hi being the bf16 operand copy.
// map_xh: hi plane of this iteration (= the B operand), map_xl: lo plane of
// signed-byte codes (updated in place), map_xo: hi plane of the next
// iteration (UPDATE); 32 x 32 boxes from encode_box32 (bf16 planes) and
// encode_lo8_box32 (the lo plane).
cudaError_t launch_ns_gemm_tc_update(int mode, int bn, const CUtensorMap& map_a, const CUtensorMap& map_b,
                                     const CUtensorMap& map_xh, const CUtensorMap& map_xl, const CUtensorMap& map_xo,
                                     const NsGemmParams& p, int grid, cudaStream_t s);
cudaError_t launch_ns_gemm_tc_planes(int mode, int bn, const CUtensorMap& map_a0, const CUtensorMap& map_a1,
                                     const CUtensorMap& map_b0, const CUtensorMap& map_b1, const CUtensorMap& map_so,
                                     const CUtensorMap& map_so_lo, const NsGemmParams& p, int grid, cudaStream_t s);
// fp32 tensor-core path (MODE_F_*; one CTA per SM, 128 x 128 tiles): a[3] and
// b[3] are the operands' three planes (64 x 128 boxes for K-major operands,
// 64 x 64 for the MN-major X of F_UPDATE / F_FINAL); o[3] are 32 x 32-box maps
// of the output's three planes (symmetric output of F_SYRK / F_POLY, the next
// X of F_UPDATE; unused by F_FINAL).
cudaError_t launch_ns_gemm_tc_f32(int mode, const CUtensorMap* a, const CUtensorMap* b, const CUtensorMap* o,
                                  const NsGemmParams& p, int grid, cudaStream_t s);
// CTA-pair variant (tcgen05 cta_group::2, 256 x 256 tiles): `pairs`
// clusters of two CTAs; tiles use 256-row blocks (p.tri / p.mi in 256-row
// units) and, for UPDATE / FINAL, 256-column blocks.
// map_b64 (SYRK / POLY, optional): the B operand again with 64-row boxes;
// given, tiles of a ragged last column block with at most 128 valid columns
// run N = 128 instead of 256.
cudaError_t launch_ns_gemm_pair(int mode, const CUtensorMap& map_a, const CUtensorMap& map_b,
                               const CUtensorMap& map_so, const CUtensorMap& map_so_lo, const NsGemmParams& p,
                               int pairs, cudaStream_t s, const CUtensorMap* map_b64 = nullptr);
// slots: epilogue input slots per warp of UPDATE (0: the default one; 2 for
// short K, where the epilogue bounds a tile)
cudaError_t launch_ns_gemm_pair_update(int mode, const CUtensorMap& map_a, const CUtensorMap& map_b,
                                      const CUtensorMap& map_xh, const CUtensorMap& map_xl, const CUtensorMap& map_xo,
                                      const NsGemmParams& p, int pairs, cudaStream_t s, int slots = 0);
// The Gram method's last product O = s Q X0 into bf16 destinations on CTA
// pairs (MODE_G_FINAL_T): a0 / a1 Q's hi and lo planes (128-row boxes), b X0
// read MN-major (64 x 64 boxes); 256 x 256 tiles as for UPDATE.
cudaError_t launch_ns_gemm_pair_gram_final(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b,
                                           const NsGemmParams& p, int pairs, cudaStream_t s);
cudaError_t launch_ns_gemm_pair_planes(int mode, const CUtensorMap& a0, const CUtensorMap& a1,
                                      const CUtensorMap& b0, const CUtensorMap& b1, const CUtensorMap& so,
                                      const CUtensorMap& so_lo, const NsGemmParams& p, int pairs, cudaStream_t s);
int ns_gemm_pair_max_pairs();

// Device copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from `src`, which may be mapped pinned host memory, to device memory.
cudaError_t launch_desc_copy(void* dst, const void* src, size_t bytes, cudaStream_t s);

// 3-D map {cols, rows, batch} (row stride ld elements, matrices rows * ld
// apart) with a 32 x 32 box: fp32 with 128-byte swizzle (32 floats = one
// 128-byte row) or bf16 with 64-byte swizzle: the epilogue's blocks of the
// master X's hi plane and of the destinations.
inline bool encode_box32(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, void* base, bool f32,
                         uint64_t cols, uint64_t rows, uint64_t batch, uint64_t ld) {
  const uint64_t es = f32 ? 4 : 2;
  cuuint64_t dims[3] = {cols, rows, batch};
  cuuint64_t strides[2] = {ld * es, rows * ld * es};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same 3-D map over the master X's lo plane of signed-byte codes (row
// stride ld bytes, a multiple of 16): 32 x 32 box, 32-byte swizzle.
inline bool encode_lo8_box32(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, void* base, uint64_t cols,
                             uint64_t rows, uint64_t batch, uint64_t ld) {
  cuuint64_t dims[3] = {cols, rows, batch};
  cuuint64_t strides[2] = {ld, rows * ld};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 SIMT path (CUDA cores).  wide = 0: fp32 m x m matrices; wide = 1:
// fp64 m x m matrices and accumulation (Gram modes of the fp32 path).
cudaError_t launch_ns_gemm_simt(int mode, const NsGemmParams& p, cudaStream_t s, int wide = 0);

// elementwise
cudaError_t launch_prepare(const PrepParams& p, int batch, int tiles_per_mat, cudaStream_t s);
cudaError_t launch_norm_finalize(const float* partials, int tiles_per_mat, int batch, float eps, float* scale,
                                 unsigned* err, cudaStream_t s);
cudaError_t launch_apply(const ApplyParams& p, int batch, cudaStream_t s);
cudaError_t launch_adamw(const AdamParams& p, int n_chunks, cudaStream_t s);
cudaError_t launch_wait_selftest(unsigned long long timeout_ns, unsigned* err, cudaStream_t s);

}  // namespace muon
