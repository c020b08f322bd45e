// Allocation-free Newton-Schulz orthogonalisation of one small matrix.
//
// Some callers cannot allocate device memory: code running inside a CUDA
// graph capture that forbids allocation, embedded runtimes with a fixed
// memory budget, or hosts where a custom allocator owns every byte.  The
// handle-based entry points allocate their workspace with cudaMalloc, so
// they cannot serve these callers.  muon_orthogonalize_noalloc runs the same
// kernels (prepare, norm, SYRK / POLY / UPDATE / FINAL) on one matrix, with
// every piece of scratch memory carved out of the file-scope device array
// below, whose size is fixed at build time.  Nothing here calls cudaMalloc,
// cudaFree or any allocating library routine.
//
// Device-side errors (a bounded wait that ran out, a non-finite Frobenius
// norm) are OR-ed into an error word at the start of the array.  The word
// starts at zero (cleared by the first call on each device), collects the
// errors of every later call, and is read and cleared by muon_noalloc_check.
#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "muon.h"

using namespace muon;

namespace {

// 24 MiB, held by every GPU that loads the library until the process exits.
constexpr size_t kScratchBytes = size_t(24) << 20;
// Largest problem: min(m, n) <= 1024 and m*n <= 2^20 elements.
constexpr int64_t kMaxSmallDim = 1024;
constexpr int64_t kMaxElements = int64_t(1) << 20;
constexpr int kMaxDevices = 64;
constexpr int kMaxTri = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct DeviceSetup {
  bool done = false;
  bool cleared = false;         // the error word has been zeroed on this device
  uint8_t* scratch = nullptr;   // device address of g_noalloc_scratch on this device
  int num_sms = 0;
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
};
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mu;
// time limit of every bounded device wait of these calls (process-wide)
std::atomic<unsigned long long> g_timeout_ns{4000000000ull};

// Descriptor block written into the scratch by a one-thread-block kernel,
// so that no host-to-device copy (and no staging buffer) is needed.
struct NoAllocDesc {
  SrcEntry src;
  OutEntry out;
  int ntri;
  int2 tri[kMaxTri];
};

__global__ void noalloc_setup_kernel(NoAllocDesc d, unsigned* err, int clear_err, SrcEntry* src, OutEntry* out,
                                     int2* tri) {
  if (threadIdx.x == 0) {
    if (clear_err) *err = 0u;   // first call on this device: the word starts at zero
    *src = d.src;
    *out = d.out;
  }
  for (int i = threadIdx.x; i < d.ntri; i += blockDim.x) tri[i] = d.tri[i];
}

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

bool encode_map(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, void* base, uint64_t cols, uint64_t rows,
                uint64_t ld, uint32_t box_rows = 128) {
  cuuint64_t dims[3] = {cols, rows, 1};
  cuuint64_t strides[2] = {ld * 2, rows * ld * 2};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Once per device, with that device current: resolve the scratch array's
// device address and the launch facts the kernels need.
muon_status_t setup_device(int dev, DeviceSetup** out) {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  DeviceSetup& s = g_setup[dev];
  if (!s.done) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return MUON_ERR_CUDA;
    if (!(prop.major == 10 && prop.minor == 3)) return MUON_ERR_UNSUPPORTED;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return MUON_ERR_CUDA;
    }
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return MUON_ERR_UNSUPPORTED;
    s.scratch = static_cast<uint8_t*>(ptr);
    s.num_sms = prop.multiProcessorCount;
    s.encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    s.done = true;
  }
  *out = &s;
  return MUON_OK;
}

}  // namespace

extern "C" muon_status_t muon_orthogonalize_noalloc(void* X, int32_t dtype, int64_t m, int64_t n, int32_t steps,
                                                    const float* coeffs, void* stream_arg) {
  if (dtype != MUON_F32 && dtype != MUON_BF16) return MUON_ERR_INVALID_ARG;
  if (m < 0 || n < 0 || steps < 0 || steps > 100) return MUON_ERR_INVALID_ARG;
  if (m == 0 || n == 0) return MUON_OK;
  if (X == nullptr) return MUON_ERR_INVALID_ARG;
  const int64_t mm = m < n ? m : n, nn = m < n ? n : m;
  if (mm > kMaxSmallDim || mm * nn > kMaxElements) return MUON_ERR_INVALID_ARG;   // beyond the static scratch
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MUON_ERR_CUDA;
  DeviceSetup* S = nullptr;
  muon_status_t st = setup_device(dev, &S);
  if (st != MUON_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_arg);
  const bool tc = (dtype == MUON_BF16);
  const float ca = coeffs ? coeffs[0] : 3.4445f, cb = coeffs ? coeffs[1] : -4.7750f, cc = coeffs ? coeffs[2] : 2.0315f;
  const int M = static_cast<int>(mm), N = static_cast<int>(nn);
  const long long ldx = (N + 15) / 16 * 16, ldm = (M + 7) / 8 * 8;
  const int prep_tiles = ((M + 63) / 64) * ((N + 63) / 64);
  const int bn_sym = M <= 128 ? 128 : 256, bn_upd = N <= 128 ? 128 : 256;

  // carve the scratch: descriptors first, then the same regions the
  // handle's workspace uses for one matrix
  uint8_t* base = S->scratch;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* p = base + off;
    off = up256(off + bytes);
    return p;
  };
  unsigned* err = reinterpret_cast<unsigned*>(take(sizeof(unsigned)));
  SrcEntry* src_d = reinterpret_cast<SrcEntry*>(take(sizeof(SrcEntry)));
  OutEntry* out_d = reinterpret_cast<OutEntry*>(take(sizeof(OutEntry)));
  int2* tri_d = reinterpret_cast<int2*>(take(sizeof(int2) * kMaxTri));
  const size_t xe = static_cast<size_t>(M) * ldx, se = static_cast<size_t>(M) * ldm;
  // fp32 copy of X0 (fp32 path, or no NS step); the tensor-core path's lo
  // plane of the master X = hi + lo (signed-byte codes) shares its space
  float* xf = reinterpret_cast<float*>(take(xe * 4));
  int8_t* xlo = (tc && steps > 0) ? reinterpret_cast<int8_t*>(xf) : nullptr;
  float* xf2 = tc ? nullptr : reinterpret_cast<float*>(take(xe * 4));
  __nv_bfloat16* xb0 = tc ? reinterpret_cast<__nv_bfloat16*>(take(xe * 2)) : nullptr;
  __nv_bfloat16* xb1 = tc ? reinterpret_cast<__nv_bfloat16*>(take(xe * 2)) : nullptr;
  void* symA = take(se * (tc ? 2 : 4));
  void* symB = take(se * (tc ? 2 : 4));
  float* pdiag = tc ? reinterpret_cast<float*>(take(static_cast<size_t>(M) * 4)) : nullptr;
  float* partials = reinterpret_cast<float*>(take(static_cast<size_t>(prep_tiles) * 4));
  float* scale = reinterpret_cast<float*>(take(4));
  if (off > kScratchBytes) return MUON_ERR_INVALID_ARG;

  NoAllocDesc d{};
  const int transposed = m > n ? 1 : 0;
  d.src = SrcEntry{X, nullptr, n, static_cast<int>(m), static_cast<int>(n), transposed, dtype};
  d.out = OutEntry{X, n, transposed, dtype, 0.f, 1.f};
  d.ntri = 0;
  const int mi_sym = (M + 127) / 128, nj_sym = (M + bn_sym - 1) / bn_sym;
  for (int i = 0; i < mi_sym; ++i)
    for (int j = 0; j < nj_sym; ++j)
      if ((j + 1) * bn_sym - 1 >= i * 128 && d.ntri < kMaxTri) d.tri[d.ntri++] = make_int2(i, j);
  bool clear_err;
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    clear_err = !S->cleared;
    S->cleared = true;
  }
  noalloc_setup_kernel<<<1, 64, 0, stream>>>(d, err, clear_err ? 1 : 0, src_d, out_d, tri_d);
  if (cudaGetLastError() != cudaSuccess) return MUON_ERR_CUDA;

  PrepParams pp{};
  pp.src = src_d;
  pp.m = M;
  pp.ldx = ldx;
  pp.xf = (tc && steps > 0) ? nullptr : xf;
  pp.xb = xb0;
  pp.xlo8 = xlo;
  pp.partials = partials;
  pp.tiles_per_mat = prep_tiles;
  if (launch_prepare(pp, 1, prep_tiles, stream) != cudaSuccess) return MUON_ERR_CUDA;
  if (launch_norm_finalize(partials, prep_tiles, 1, 1e-7f, scale, err, stream) != cudaSuccess) return MUON_ERR_CUDA;
  if (steps == 0) {
    ApplyParams ap{out_d, scale, xf, ldx, M, N};
    return launch_apply(ap, 1, stream) == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
  }
  CUtensorMap map_x[2], map_xmn[2], map_A, map_B, map_xh[2], map_xl, map_sa, map_sb;
  if (tc && !(encode_map(S->encode, &map_x[0], xb0, N, M, ldx) && encode_map(S->encode, &map_x[1], xb1, N, M, ldx) &&
              encode_map(S->encode, &map_xmn[0], xb0, N, M, ldx, 64) &&
              encode_map(S->encode, &map_xmn[1], xb1, N, M, ldx, 64) &&
              encode_map(S->encode, &map_A, symA, M, M, ldm) && encode_map(S->encode, &map_B, symB, M, M, ldm) &&
              encode_box32(S->encode, &map_xh[0], xb0, false, N, M, 1, ldx) &&
              encode_box32(S->encode, &map_xh[1], xb1, false, N, M, 1, ldx) &&
              encode_lo8_box32(S->encode, &map_xl, xlo, N, M, 1, ldx) &&
              encode_box32(S->encode, &map_sa, symA, false, M, M, 1, ldm) &&
              encode_box32(S->encode, &map_sb, symB, false, M, M, 1, ldm)))
    return MUON_ERR_CUDA;
  const int mi = (M + 127) / 128, nj = (N + bn_upd - 1) / bn_upd;
  for (int it = 0; it < steps; ++it) {
    const bool last = (it == steps - 1);
    NsGemmParams p{};
    p.m = M;
    p.n = N;
    p.batch = 1;
    p.scale = it == 0 ? scale : nullptr;
    p.ca = ca;
    p.cb = cb;
    p.cc = cc;
    p.ldm = ldm;
    p.ldx = ldx;
    p.out = out_d;
    p.err = err;
    p.timeout_ns = g_timeout_ns.load();
    p.pdiag = pdiag;
    cudaError_t e;
    if (tc) {
      NsGemmParams q = p;
      q.tiles_per_mat = d.ntri;
      q.num_tiles = d.ntri;
      q.tri = tri_d;
      q.sym_out = symA;
      const int gs = q.num_tiles < S->num_sms ? q.num_tiles : S->num_sms;
      e = launch_ns_gemm_tc(MODE_SYRK, bn_sym, map_x[it & 1], map_x[it & 1], map_sa, map_sa, q, gs, stream);
      if (e != cudaSuccess) return MUON_ERR_CUDA;
      // POLY keeps the scale: P' = s P in the first iteration
      q.sym_in = symA;
      q.sym_out = symB;
      e = launch_ns_gemm_tc(MODE_POLY, bn_sym, map_A, map_A, map_sb, map_sb, q, gs, stream);
      if (e != cudaSuccess) return MUON_ERR_CUDA;
      NsGemmParams u = p;
      u.mi = mi;
      u.tiles_per_mat = mi * nj;
      u.num_tiles = mi * nj;
      const int gu = u.num_tiles < S->num_sms ? u.num_tiles : S->num_sms;
      e = launch_ns_gemm_tc_update(last ? MODE_FINAL : MODE_UPDATE, bn_upd, map_B, map_xmn[it & 1], map_xh[it & 1],
                                   map_xl, map_xh[(it + 1) & 1], u, gu, stream);
    } else {
      float* xin = (it & 1) ? xf2 : xf;
      float* xout = (it & 1) ? xf : xf2;
      NsGemmParams q = p;
      q.xf_in = xin;
      q.sym_out = symA;
      e = launch_ns_gemm_simt(MODE_SYRK, q, stream);
      if (e != cudaSuccess) return MUON_ERR_CUDA;
      q.scale = nullptr;
      q.sym_in = symA;
      q.sym_out = symB;
      e = launch_ns_gemm_simt(MODE_POLY, q, stream);
      if (e != cudaSuccess) return MUON_ERR_CUDA;
      NsGemmParams u = p;
      u.sym_in = symB;
      u.xf_in = xin;
      u.xf_out = xout;
      e = launch_ns_gemm_simt(last ? MODE_FINAL : MODE_UPDATE, u, stream);
    }
    if (e != cudaSuccess) return MUON_ERR_CUDA;
  }
  return MUON_OK;
}

extern "C" muon_status_t muon_noalloc_check(void* stream_arg) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MUON_ERR_CUDA;
  DeviceSetup* S = nullptr;
  muon_status_t st = setup_device(dev, &S);
  if (st != MUON_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_arg);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MUON_ERR_CUDA;
  bool cleared;
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    cleared = S->cleared;
  }
  if (!cleared) return MUON_OK;     // no call has run on this device yet
  // the word sits at the start of the array; a plain copy into a host
  // variable and a memset on the caller's stream allocate nothing
  unsigned word = 0;
  if (cudaMemcpy(&word, S->scratch, sizeof(unsigned), cudaMemcpyDeviceToHost) != cudaSuccess) return MUON_ERR_CUDA;
  if (cudaMemsetAsync(S->scratch, 0, sizeof(unsigned), stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return MUON_ERR_CUDA;
  if (word & ERRBIT_TIMEOUT) return MUON_ERR_TIMEOUT;
  if (word & ERRBIT_NONFINITE) return MUON_ERR_NONFINITE;
  return MUON_OK;
}

extern "C" muon_status_t muon_noalloc_set_timeout_ns(uint64_t timeout_ns) {
  if (timeout_ns == 0) return MUON_ERR_INVALID_ARG;
  g_timeout_ns.store(timeout_ns);
  return MUON_OK;
}
