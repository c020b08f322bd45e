// C ABI and host scheduler of the Muon step (see include/muon.h).
//
// The scheduler turns a parameter list into same-shape groups of NS
// matrices: every parameter (or Muon-Split row block) becomes one m x n
// matrix with m <= n (transposed when it has more rows than columns), and all
// matrices of one (m, n) share one grouped launch per NS product.  A group
// larger than the workspace limit is processed in chunks.  Per chunk the
// launch sequence on the caller's stream is
//   prepare (momentum, Nesterov, U, partial norms) -> norm finalize ->
//   steps x [SYRK -> POLY -> UPDATE]  (the last UPDATE is FINAL and writes
//   the parameter) — or, with no NS step, one apply kernel.
// No host synchronisation happens inside a step.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <map>
#include <string>
#include <utility>
#include <vector>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "launch_opts.h"
#include "muon.h"

using namespace muon;

namespace {

constexpr float kDefaultCoeffs[3] = {3.4445f, -4.7750f, 2.0315f};
constexpr float kNormEps = 1e-7f;
constexpr int64_t kMaxDim = int64_t(1) << 30;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
size_t dtype_size(int dt) { return dt == DT_BF16 ? 2 : 4; }

struct Block {
  SrcEntry src;
  OutEntry out;
  int m, n;
};

}  // namespace

struct muon_handle_s {
  int device = 0;
  int num_sms = 0;
  size_t ws_limit = size_t(16) << 30;
  unsigned long long timeout_ns = 4000000000ull;
  void* ws = nullptr;
  size_t ws_cap = 0;
  void* desc = nullptr;
  size_t desc_cap = 0;
  // pinned staging buffers of the descriptor arena, used in turn, each with
  // the event after which the device has read it
  static constexpr int kStages = 3;
  void* hstage[kStages] = {};
  const void* hstage_dev[kStages] = {};   // the same memory as the device addresses it
  size_t hstage_cap[kStages] = {};
  cudaEvent_t stage_ev[kStages] = {};
  bool stage_pending[kStages] = {};
  int stage_next = 0;
  unsigned* err = nullptr;
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  std::string last;
  // per-launch event timing (muon_handle_set_profiling)
  struct ProfRec {
    cudaEvent_t a, b;
    int cls;
    int tag;
  };
  bool profiling = false;
  int prof_tag = -1;            // group index of the launches being issued
  std::vector<ProfRec> prof;
  size_t prof_used = 0;
  uint64_t launches = 0;
  bool use_pair = true;         // CTA-pair GEMMs for large groups (MUON_TC_PAIR=0 disables)
  bool pair_update = true;      // UPDATE / FINAL on pairs too (MUON_TC_PAIR=sym: symmetric products only)
  int pair_min_m = 1024;        // ragged m from here on runs its symmetric products on pairs too (MUON_TC_PAIR_MIN_M)
  int max_pairs = 0;
  bool final_tma = true;        // FINAL into bf16 destinations through tensor maps (MUON_FINAL_TMA=0 disables)
  bool f32_tc = true;           // fp32 standard method on the tensor cores, three bf16 planes (MUON_F32_TC=0:
                                // CUDA cores)
  int f32_tc_max_m = 2048;      // ... for groups up to this m (MUON_F32_TC_MAX_M); the products' fp32
                                // accumulation error grows with K = m (with two accumulators per tile:
                                // 2048 x 8192 5.7e-5, 4096 x 4096 7.5e-5, 4096 x 14336 1.0e-4 against
                                // the 1e-4 bar)
  // standard bf16 method: the next unit's preparation on a side stream while
  // the current unit's products run (MUON_OVERLAP=1)
  bool overlap = false;
  cudaStream_t side = nullptr;
  std::vector<cudaEvent_t> ovl_ev;
  // standard bf16 method on small sets: every same-shape group's chain on a
  // stream of its own, so small launches of different groups share the SMs
  // (MUON_CONCURRENT: 0 off, 1 whenever the groups fit the workspace limit
  // together; default: also only for sets of at most kConcMaxElements)
  int concurrent = -1;
  std::vector<cudaStream_t> conc;
  std::vector<cudaEvent_t> conc_ev;
};

namespace {

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

muon_status_t fail(muon_handle_t h, muon_status_t st, const std::string& msg) {
  if (h != nullptr) h->last = msg;
  return st;
}

muon_status_t cuda_fail(muon_handle_t h, cudaError_t e, const char* what) {
  return fail(h, MUON_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

#define MUON_CUDA_TRY(expr, what)                  \
  do {                                             \
    cudaError_t e_ = (expr);                       \
    if (e_ != cudaSuccess) return cuda_fail(h, e_, what); \
  } while (0)

constexpr size_t kMaxProfRecords = size_t(1) << 20;

int prof_start(muon_handle_t h, int cls, cudaStream_t s) {
  if (!h->profiling || h->prof_used >= kMaxProfRecords) return -1;
  if (h->prof_used == h->prof.size()) {
    muon_handle_s::ProfRec r{};
    if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) {
      cudaGetLastError();
      return -1;
    }
    h->prof.push_back(r);
  }
  const int slot = static_cast<int>(h->prof_used++);
  h->prof[slot].cls = cls;
  h->prof[slot].tag = h->prof_tag;
  cudaEventRecord(h->prof[slot].a, s);
  return slot;
}

void prof_stop(muon_handle_t h, int slot, cudaStream_t s) {
  if (slot >= 0) cudaEventRecord(h->prof[slot].b, s);
}

// Launch one kernel: optional event timing and the launch counter.
#define MUON_LAUNCH(cls, expr, what)                       \
  do {                                                     \
    const int slot_ = prof_start(h, (cls), stream);        \
    cudaError_t e_ = (expr);                               \
    if (e_ != cudaSuccess) return cuda_fail(h, e_, what);  \
    prof_stop(h, slot_, stream);                           \
    ++h->launches;                                         \
  } while (0)

muon_status_t ensure_ws(muon_handle_t h, size_t bytes) {
  if (bytes <= h->ws_cap) return MUON_OK;
  if (h->ws != nullptr) {
    cudaFree(h->ws);   // implicit device synchronisation: no launch still uses it
    h->ws = nullptr;
    h->ws_cap = 0;
  }
  const size_t cap = align_up(bytes, size_t(64) << 20);
  if (cudaMalloc(&h->ws, cap) != cudaSuccess) {
    cudaGetLastError();
    h->ws = nullptr;
    return fail(h, MUON_ERR_WORKSPACE, "workspace allocation of " + std::to_string(cap) + " bytes failed");
  }
  h->ws_cap = cap;
  return MUON_OK;
}

// The side stream and at least n events of the overlapped standard path,
// created on first use.
muon_status_t ensure_overlap_events(muon_handle_t h, size_t n) {
  if (h->side == nullptr && cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    h->side = nullptr;
    return fail(h, MUON_ERR_CUDA, "side stream creation failed");
  }
  while (h->ovl_ev.size() < n) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      return fail(h, MUON_ERR_CUDA, "event creation failed");
    }
    h->ovl_ev.push_back(e);
  }
  return MUON_OK;
}

// At least n streams and n + 1 events for concurrent groups, created on
// first use.
muon_status_t ensure_concurrent(muon_handle_t h, size_t n) {
  while (h->conc.size() < n) {
    cudaStream_t cs = nullptr;
    if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) {
      cudaGetLastError();
      return fail(h, MUON_ERR_CUDA, "stream creation failed");
    }
    h->conc.push_back(cs);
  }
  while (h->conc_ev.size() < n + 1) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      return fail(h, MUON_ERR_CUDA, "event creation failed");
    }
    h->conc_ev.push_back(e);
  }
  return MUON_OK;
}

// Copy a host descriptor arena to the handle's device descriptor buffer on
// `stream` through a pinned staging buffer (one of kStages, taken in turn).
// The copy is a kernel reading the pinned buffer through its device address,
// not a copy-engine transfer: a cudaMemcpyAsync here queues behind whatever
// host<->device copies the caller has in flight on other streams (a step's
// gradients, say), which held every call that overlapped them.
muon_status_t upload(muon_handle_t h, const std::vector<uint8_t>& arena, cudaStream_t stream, void** dev) {
  *dev = nullptr;
  if (arena.empty()) return MUON_OK;
  const int k = h->stage_next;
  h->stage_next = (k + 1) % muon_handle_s::kStages;
  if (h->stage_pending[k]) {
    MUON_CUDA_TRY(cudaEventSynchronize(h->stage_ev[k]), "descriptor staging wait");
    h->stage_pending[k] = false;
  }
  if (arena.size() > h->desc_cap) {
    if (h->desc != nullptr) cudaFree(h->desc);
    h->desc = nullptr;
    h->desc_cap = 0;
    const size_t cap = align_up(arena.size(), size_t(1) << 20);
    if (cudaMalloc(&h->desc, cap) != cudaSuccess) {
      cudaGetLastError();
      return fail(h, MUON_ERR_WORKSPACE, "descriptor buffer allocation failed");
    }
    h->desc_cap = cap;
  }
  if (arena.size() > h->hstage_cap[k]) {
    if (h->hstage[k] != nullptr) cudaFreeHost(h->hstage[k]);
    h->hstage[k] = nullptr;
    h->hstage_dev[k] = nullptr;
    h->hstage_cap[k] = 0;
    const size_t cap = align_up(arena.size(), size_t(1) << 20);
    void* dptr = nullptr;
    if (cudaHostAlloc(&h->hstage[k], cap, cudaHostAllocMapped) != cudaSuccess ||
        cudaHostGetDevicePointer(&dptr, h->hstage[k], 0) != cudaSuccess) {
      cudaGetLastError();
      if (h->hstage[k] != nullptr) cudaFreeHost(h->hstage[k]);
      h->hstage[k] = nullptr;
      return fail(h, MUON_ERR_WORKSPACE, "pinned staging allocation failed");
    }
    h->hstage_dev[k] = dptr;
    h->hstage_cap[k] = cap;
  }
  std::memcpy(h->hstage[k], arena.data(), arena.size());
  // both buffers are whole MiB, so the 16-byte rounding stays inside them
  MUON_CUDA_TRY(launch_desc_copy(h->desc, h->hstage_dev[k], align_up(arena.size(), 16), stream), "descriptor upload");
  ++h->launches;
  MUON_CUDA_TRY(cudaEventRecord(h->stage_ev[k], stream), "descriptor staging event");
  h->stage_pending[k] = true;
  *dev = h->desc;
  return MUON_OK;
}

template <typename T>
size_t arena_push(std::vector<uint8_t>& arena, const T* data, size_t count) {
  const size_t off = align_up(arena.size(), 256);
  arena.resize(off + sizeof(T) * count);
  if (count) std::memcpy(arena.data() + off, data, sizeof(T) * count);
  return off;
}

// Operand map: 64-column boxes with 128-byte swizzle, box_rows rows (128 for
// K-major operands, one box per 128-row block; 64 for the MN-major reads of
// X by the update product).
bool encode_map(muon_handle_t h, CUtensorMap* map, void* base, uint64_t cols, uint64_t rows, uint64_t batch,
                uint64_t ld, uint32_t box_rows = 128) {
  cuuint64_t dims[3] = {cols, rows, batch};
  cuuint64_t strides[2] = {ld * 2, rows * ld * 2};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = h->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tiles (i, j) of an m x m output that touch the upper triangle, for
// bm-row by bn-column tiles.
std::vector<int2> sym_tiles(int m, int bn, int bm = 128) {
  std::vector<int2> t;
  const int mi = static_cast<int>(ceil_div(m, bm)), nj = static_cast<int>(ceil_div(m, bn));
  for (int i = 0; i < mi; ++i)
    for (int j = 0; j < nj; ++j)
      if ((j + 1) * bn - 1 >= i * bm) t.push_back(make_int2(i, j));
  return t;
}

// Groups whose m fills 256-row pair tiles well run on the CTA-pair kernels:
// m a multiple of 256, or m >= pair_min_m (ragged last tile).
// CTA pairs from m = pair_min_m (1024 by default, MUON_TC_PAIR_MIN_M), and
// for m = 256 (one 256-row block, whose pair tiles halve the per-SM traffic
// of the wide X panels: 64 matrices 256 x 16384, 2.74 against 2.78 ms on
// one SM).  Between them the one-SM kernels won: GPT-2-small (m = 768)
// 1.515 -> 1.495 ms.
bool pair_group(int m, int pair_min_m) { return m >= 256 && (m >= pair_min_m || m == 256); }

struct GroupPlan {
  int m = 0, n = 0;
  long long ldx = 0, ldm = 0;
  int prep_tiles = 0;
  int bn_sym = 256, bn_upd = 256;
  size_t per_mat = 0;       // workspace bytes per matrix
  int chunk = 1;            // matrices per chunk
  std::vector<int> members; // block indices
  size_t tri_off = 0;
  int tri_count = 0;
  size_t tri128_off = 0;        // 128 x 128 symmetric tiles (Gram plane products)
  int tri128_count = 0;
  size_t tri256_off = 0;        // 256 x 256 symmetric tiles (CTA-pair kernels)
  int tri256_count = 0;
  bool pair = false;            // symmetric products on CTA pairs
  bool pair_upd = false;        // UPDATE / FINAL on CTA pairs
  std::vector<std::pair<size_t, size_t>> chunk_off;   // (src offset, out offset) per chunk
  std::vector<size_t> chunk_wmap;   // per chunk: offset of the destinations' tensor maps, or kNoMaps
};

constexpr size_t kNoMaps = ~size_t(0);

// UPDATE products with K = m up to this run the pair kernel with two epilogue
// input slots per warp: their main loop per tile is shorter than the latency
// chain of a one-slot epilogue.
constexpr int kShortK = 1024;

// One tensor map per destination of a chunk, for FINAL_T: possible when every
// destination is bf16 with a 16-byte aligned base and row stride (TMA's
// rules); the map covers the destination in its own orientation (n x m when
// the block was transposed).
bool encode_dest_maps(muon_handle_t h, const GroupPlan& g, const std::vector<OutEntry>& out,
                      std::vector<CUtensorMap>* maps) {
  maps->resize(out.size());
  for (size_t k = 0; k < out.size(); ++k) {
    const OutEntry& e = out[k];
    if (e.dtype != DT_BF16 || (reinterpret_cast<uintptr_t>(e.ptr) & 15) != 0 || ((e.ld * 2) & 15) != 0) return false;
    const uint64_t drows = e.transposed ? g.n : g.m, dcols = e.transposed ? g.m : g.n;
    if (!encode_box32(h->encode, &(*maps)[k], e.ptr, false, dcols, drows, 1, static_cast<uint64_t>(e.ld))) return false;
  }
  return true;
}

// Workspace region offsets for one chunk capacity `cap` (bytes from ws base).
//   standard, tensor cores: fp32 master X, two bf16 operand copies (ping-pong),
//                           bf16 A and P, fp32 diagonal of P
//   standard, fp32 path:    two fp32 X buffers (ping-pong), fp32 A and B
//   gram, tensor cores:     bf16 X0 (+ fp32 X0 when no NS step runs) and six
//                           m x m slots (R, T, P0, P1, Q0, Q1) of two bf16 planes
//   gram, fp32 path:        fp32 X0 and six fp64 m x m slots
//   standard, fp32 path on the tensor cores (f32tc): X as three bf16 planes
//                           in two ping-pong sets, A and P as three planes
//                           each (+ fp32 X0 when no NS step runs)
constexpr int kGramSlots = 6;
enum { SLOT_R = 0, SLOT_T = 1, SLOT_P0 = 2, SLOT_Q0 = 4 };

struct Regions {
  size_t xf, xf2, xlo, xb0, xb1, symA, symB, pdiag, partials, scale, total;
  size_t slot[kGramSlots], slot_lo[kGramSlots];
  size_t xp[2][3], ap[3], pp[3];   // f32tc planes
};

Regions regions(const GroupPlan& g, int cap, bool tc, bool gram, int steps, bool f32tc = false) {
  Regions r{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  const size_t xe = static_cast<size_t>(cap) * g.m * g.ldx;
  const size_t se = static_cast<size_t>(cap) * g.m * g.ldm;
  if (f32tc && !gram && !tc) {
    r.xf = (steps == 0) ? take(xe * 4) : 0;
    for (int q = 0; q < 2; ++q)
      for (int k = 0; k < 3; ++k) r.xp[q][k] = take(xe * 2);
    for (int k = 0; k < 3; ++k) r.ap[k] = take(se * 2);
    for (int k = 0; k < 3; ++k) r.pp[k] = take(se * 2);
  } else if (!gram) {
    if (tc) {
      // master X = hi + lo: hi is the operand copy (xb0 / xb1 ping-pong), lo
      // (one signed-byte code per element) in place; the fp32 copy only when
      // no NS step runs
      r.xf = (steps == 0) ? take(xe * 4) : 0;
      r.xlo = (steps == 0) ? 0 : take(xe);
      r.xb0 = take(xe * 2);
      r.xb1 = take(xe * 2);
      r.symA = take(se * 2);
      r.symB = take(se * 2);
      r.pdiag = take(static_cast<size_t>(cap) * g.m * 4);
    } else {
      r.xf = take(xe * 4);
      r.xf2 = take(xe * 4);
      r.symA = take(se * 4);
      r.symB = take(se * 4);
    }
  } else {
    if (tc) {
      r.xb0 = take(xe * 2);
      r.xf = (steps == 0) ? take(xe * 4) : 0;
      for (int k = 0; k < kGramSlots; ++k) {
        r.slot[k] = take(se * 2);
        r.slot_lo[k] = take(se * 2);
      }
    } else {
      r.xf = take(xe * 4);
      for (int k = 0; k < kGramSlots; ++k) r.slot[k] = take(se * 8);
    }
  }
  r.partials = take(static_cast<size_t>(cap) * g.prep_tiles * 4);
  r.scale = take(static_cast<size_t>(cap) * 4);
  r.total = off;
  return r;
}

// Gram method for one same-shape group ("DeepSpeed 集成 Muon 优化器实战",
// §核心算子: iterate on R = X X^T).  With P_k = aI + bR_k + cR_k^2:
//   R_0 = X0 X0^T;  Q_1 = P_0;  Q_{k+1} = P_k Q_k;  R_{k+1} = P_k R_k P_k;
//   O = Q X0,  X0 = s U (s = 1/||U||_F folded into the first and last products).
// All m x m iterates are polynomials in R_0, so they commute and are
// symmetric: every product is computed on its upper tiles and mirrored.
muon_status_t run_gram_group(muon_handle_t h, const GroupPlan& g, const Regions& R, uint8_t* ws, uint8_t* dbase,
                             int steps, const float* coeffs, int coeff_stride, bool tc, float mu, int nesterov,
                             cudaStream_t stream) {
  float* xf = reinterpret_cast<float*>(ws + R.xf);
  __nv_bfloat16* xb = tc ? reinterpret_cast<__nv_bfloat16*>(ws + R.xb0) : nullptr;
  float* partials = reinterpret_cast<float*>(ws + R.partials);
  float* scale = reinterpret_cast<float*>(ws + R.scale);
  void* hi[kGramSlots];
  void* lo[kGramSlots];
  for (int k = 0; k < kGramSlots; ++k) {
    hi[k] = ws + R.slot[k];
    lo[k] = tc ? static_cast<void*>(ws + R.slot_lo[k]) : nullptr;
  }
  // per slot: 64 x 64 operand maps of both planes, and 32 x 32 output maps
  CUtensorMap map_x, map_xmn, mhi[kGramSlots], mlo[kGramSlots], ohi[kGramSlots], olo[kGramSlots];
  if (tc) {
    bool ok = encode_map(h, &map_x, xb, g.n, g.m, g.chunk, g.ldx) &&
              encode_map(h, &map_xmn, xb, g.n, g.m, g.chunk, g.ldx, 64);
    for (int k = 0; k < kGramSlots && ok; ++k)
      ok = encode_map(h, &mhi[k], hi[k], g.m, g.m, g.chunk, g.ldm) &&
           encode_map(h, &mlo[k], lo[k], g.m, g.m, g.chunk, g.ldm) &&
           encode_box32(h->encode, &ohi[k], hi[k], false, g.m, g.m, g.chunk, g.ldm) &&
           encode_box32(h->encode, &olo[k], lo[k], false, g.m, g.m, g.chunk, g.ldm);
    if (!ok) return fail(h, MUON_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  }
  const int mi = static_cast<int>(ceil_div(g.m, 128));
  const int nj = static_cast<int>(ceil_div(g.n, g.bn_upd));
  for (size_t c = 0; c < g.chunk_off.size(); ++c) {
    const int cnt = static_cast<int>(std::min<size_t>(g.chunk, g.members.size() - c * g.chunk));
    const SrcEntry* src_d = reinterpret_cast<const SrcEntry*>(dbase + g.chunk_off[c].first);
    const OutEntry* out_d = reinterpret_cast<const OutEntry*>(dbase + g.chunk_off[c].second);
    const CUtensorMap* wmap_d =
        g.chunk_wmap[c] == kNoMaps ? nullptr : reinterpret_cast<const CUtensorMap*>(dbase + g.chunk_wmap[c]);
    PrepParams pp{};
    pp.src = src_d;
    pp.mu = mu;
    pp.nesterov = nesterov;
    pp.m = g.m;
    pp.ldx = g.ldx;
    pp.xf = (tc && steps > 0) ? nullptr : xf;
    pp.xb = xb;
    pp.partials = partials;
    pp.tiles_per_mat = g.prep_tiles;
    MUON_LAUNCH(MUON_K_PREPARE, launch_prepare(pp, cnt, g.prep_tiles, stream), "prepare launch");
    MUON_LAUNCH(MUON_K_NORM, launch_norm_finalize(partials, g.prep_tiles, cnt, kNormEps, scale, h->err, stream),
                "norm launch");
    if (steps == 0) {
      ApplyParams ap{out_d, scale, xf, g.ldx, g.m, g.n};
      MUON_LAUNCH(MUON_K_APPLY, launch_apply(ap, cnt, stream), "apply launch");
      continue;
    }
    NsGemmParams p{};
    p.m = g.m;
    p.n = g.n;
    p.batch = cnt;
    p.ldm = g.ldm;
    p.ldx = g.ldx;
    p.out = out_d;
    p.err = h->err;
    p.timeout_ns = h->timeout_ns;
    // symmetric products: tile table and grid
    NsGemmParams q = p;
    q.tiles_per_mat = tc ? g.tri128_count : 0;
    q.num_tiles = cnt * q.tiles_per_mat;
    q.tri = tc ? reinterpret_cast<const int2*>(dbase + g.tri128_off) : nullptr;
    const int grid_sym = std::max(1, std::min(q.num_tiles, h->num_sms));
    // R0 = s^2 X0 X0^T
    {
      NsGemmParams r0 = p;
      r0.scale = scale;
      r0.sym_out = hi[SLOT_R];
      r0.sym_out_lo = lo[SLOT_R];
      if (tc && g.pair) {
        r0.tiles_per_mat = g.tri256_count;
        r0.num_tiles = cnt * g.tri256_count;
        r0.tri = reinterpret_cast<const int2*>(dbase + g.tri256_off);
        const int pairs = std::min(r0.num_tiles, h->max_pairs);
        MUON_LAUNCH(MUON_K_SYRK, launch_ns_gemm_pair(MODE_G_R0, map_x, map_x, ohi[SLOT_R], olo[SLOT_R], r0, pairs, stream), "gram r0");
      } else if (tc) {
        r0.tiles_per_mat = g.tri_count;
        r0.num_tiles = cnt * g.tri_count;
        r0.tri = reinterpret_cast<const int2*>(dbase + g.tri_off);
        const int grid = std::min(r0.num_tiles, h->num_sms);
        MUON_LAUNCH(MUON_K_SYRK, launch_ns_gemm_tc(MODE_G_R0, g.bn_sym, map_x, map_x, ohi[SLOT_R], olo[SLOT_R], r0, grid, stream), "gram r0");
      } else {
        r0.xf_in = xf;
        MUON_LAUNCH(MUON_K_SYRK, launch_ns_gemm_simt(MODE_G_R0, r0, stream, 1), "gram r0");
      }
    }
    auto sym_product = [&](int mode, int a, int b, int out, int cls) -> muon_status_t {
      NsGemmParams t = q;
      t.sym_out = hi[out];
      t.sym_out_lo = lo[out];
      t.sym_in = hi[a];
      t.sym_in_lo = lo[a];
      t.op_b = hi[b];
      if (tc && g.pair) {
        t.tiles_per_mat = g.tri256_count;
        t.num_tiles = cnt * g.tri256_count;
        t.tri = reinterpret_cast<const int2*>(dbase + g.tri256_off);
        const int pairs = std::min(t.num_tiles, h->max_pairs);
        MUON_LAUNCH(cls, launch_ns_gemm_pair_planes(mode, mhi[a], mlo[a], mhi[b], mlo[b], ohi[out], olo[out], t, pairs, stream),
                    "gram product");
      } else if (tc) {
        MUON_LAUNCH(cls, launch_ns_gemm_tc_planes(mode, 128, mhi[a], mlo[a], mhi[b], mlo[b], ohi[out], olo[out], t, grid_sym,
                                                  stream),
                    "gram product");
      } else {
        MUON_LAUNCH(cls, launch_ns_gemm_simt(mode, t, stream, 1), "gram product");
      }
      return MUON_OK;
    };
    int qcur = -1, qnext = SLOT_Q0;
    for (int k = 0; k < steps; ++k) {
      const int pk = SLOT_P0 + (k & 1);
      q.ca = coeffs[k * coeff_stride];           // this step's (a, b, c)
      q.cb = coeffs[k * coeff_stride + 1];
      q.cc = coeffs[k * coeff_stride + 2];
      muon_status_t st = sym_product(MODE_G_P, SLOT_R, SLOT_R, pk, MUON_K_POLY);     // P = aI + bR + cR^2
      if (st != MUON_OK) return st;
      if (k == 0) {
        qcur = pk;
      } else {
        st = sym_product(MODE_G_PROD, pk, qcur, qnext, MUON_K_UPDATE);              // Q <- P Q
        if (st != MUON_OK) return st;
        qcur = qnext;
        qnext = (qnext == SLOT_Q0) ? SLOT_Q0 + 1 : SLOT_Q0;
      }
      if (k < steps - 1) {
        st = sym_product(MODE_G_PROD, pk, SLOT_R, SLOT_T, MUON_K_UPDATE);           // T = P R
        if (st != MUON_OK) return st;
        st = sym_product(MODE_G_PROD, SLOT_T, pk, SLOT_R, MUON_K_UPDATE);           // R <- T P
        if (st != MUON_OK) return st;
      }
    }
    // O = s Q X0 -> destination
    NsGemmParams f = p;
    f.scale = scale;
    f.sym_in = hi[qcur];
    f.wmap = wmap_d;
    if (tc && wmap_d != nullptr && g.pair_upd) {
      // on CTA pairs, 256 x 256 tiles, as the standard method's UPDATE
      const int mi2 = static_cast<int>(ceil_div(g.m, 256)), nj2 = static_cast<int>(ceil_div(g.n, 256));
      f.mi = mi2;
      f.tiles_per_mat = mi2 * nj2;
      f.num_tiles = cnt * mi2 * nj2;
      const int pairs = std::min(f.num_tiles, h->max_pairs);
      MUON_LAUNCH(MUON_K_FINAL, launch_ns_gemm_pair_gram_final(mhi[qcur], mlo[qcur], map_xmn, f, pairs, stream),
                  "gram final");
    } else if (tc) {
      f.mi = mi;
      f.tiles_per_mat = mi * nj;
      f.num_tiles = cnt * mi * nj;
      const int grid = std::min(f.num_tiles, h->num_sms);
      MUON_LAUNCH(MUON_K_FINAL,
                  launch_ns_gemm_tc_planes(wmap_d != nullptr ? MODE_G_FINAL_T : MODE_G_FINAL, g.bn_upd, mhi[qcur], mlo[qcur],
                                           map_xmn, map_xmn, map_xmn, map_xmn, f,
                                           grid, stream),
                  "gram final");
    } else {
      f.xf_in = xf;
      MUON_LAUNCH(MUON_K_FINAL, launch_ns_gemm_simt(MODE_G_FINAL, f, stream, 1), "gram final");
    }
  }
  return MUON_OK;
}

// Standard method of the fp32 path on the tensor cores for one same-shape
// group: X, A and P held as three bf16 planes (24 mantissa bits), every
// product six MMAs per K step with fp32 accumulation (internal.h, MODE_F_*):
//   prepare (X0 planes) -> norm -> steps x [F_SYRK -> F_POLY -> F_UPDATE]
// with the last F_UPDATE replaced by F_FINAL into the destinations.  The
// iteration is the pages' X <- (aI + bA + cA^2) X, A = X X^T ("Muon Optimizer
// and the Distributed Implementation", §Newton-Schulz Iteration).
muon_status_t run_f32tc_group(muon_handle_t h, const GroupPlan& g, const Regions& R, uint8_t* ws, uint8_t* dbase,
                              int steps, const float* coeffs, int coeff_stride, float mu, int nesterov,
                              cudaStream_t stream) {
  float* xf = reinterpret_cast<float*>(ws + R.xf);
  float* partials = reinterpret_cast<float*>(ws + R.partials);
  float* scale = reinterpret_cast<float*>(ws + R.scale);
  auto bf = [&](size_t off) { return reinterpret_cast<__nv_bfloat16*>(ws + off); };
  // per X set q and plane k: K-major (64 x 128 boxes), MN-major (64 x 64) and
  // 32 x 32 output maps; A and P planes: K-major operand and 32 x 32 output maps
  CUtensorMap xk[2][3], xmn[2][3], xo[2][3], ak[3], ao[3], pk[3], po[3];
  if (steps > 0) {
    bool ok = true;
    for (int q = 0; q < 2 && ok; ++q)
      for (int k = 0; k < 3 && ok; ++k)
        ok = encode_map(h, &xk[q][k], bf(R.xp[q][k]), g.n, g.m, g.chunk, g.ldx) &&
             encode_map(h, &xmn[q][k], bf(R.xp[q][k]), g.n, g.m, g.chunk, g.ldx, 64) &&
             encode_box32(h->encode, &xo[q][k], bf(R.xp[q][k]), false, g.n, g.m, g.chunk, g.ldx);
    for (int k = 0; k < 3 && ok; ++k)
      ok = encode_map(h, &ak[k], bf(R.ap[k]), g.m, g.m, g.chunk, g.ldm) &&
           encode_box32(h->encode, &ao[k], bf(R.ap[k]), false, g.m, g.m, g.chunk, g.ldm) &&
           encode_map(h, &pk[k], bf(R.pp[k]), g.m, g.m, g.chunk, g.ldm) &&
           encode_box32(h->encode, &po[k], bf(R.pp[k]), false, g.m, g.m, g.chunk, g.ldm);
    if (!ok) return fail(h, MUON_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  }
  const int mi = static_cast<int>(ceil_div(g.m, 128));
  const int nj = static_cast<int>(ceil_div(g.n, 128));
  for (size_t c = 0; c < g.chunk_off.size(); ++c) {
    const int cnt = static_cast<int>(std::min<size_t>(g.chunk, g.members.size() - c * g.chunk));
    const SrcEntry* src_d = reinterpret_cast<const SrcEntry*>(dbase + g.chunk_off[c].first);
    const OutEntry* out_d = reinterpret_cast<const OutEntry*>(dbase + g.chunk_off[c].second);
    PrepParams pp{};
    pp.src = src_d;
    pp.mu = mu;
    pp.nesterov = nesterov;
    pp.m = g.m;
    pp.ldx = g.ldx;
    pp.xf = steps > 0 ? nullptr : xf;
    pp.xb = steps > 0 ? bf(R.xp[0][0]) : nullptr;
    pp.xlo = steps > 0 ? bf(R.xp[0][1]) : nullptr;
    pp.xlo2 = steps > 0 ? bf(R.xp[0][2]) : nullptr;
    pp.partials = partials;
    pp.tiles_per_mat = g.prep_tiles;
    MUON_LAUNCH(MUON_K_PREPARE, launch_prepare(pp, cnt, g.prep_tiles, stream), "prepare launch");
    MUON_LAUNCH(MUON_K_NORM, launch_norm_finalize(partials, g.prep_tiles, cnt, kNormEps, scale, h->err, stream),
                "norm launch");
    if (steps == 0) {
      ApplyParams ap{out_d, scale, xf, g.ldx, g.m, g.n};
      MUON_LAUNCH(MUON_K_APPLY, launch_apply(ap, cnt, stream), "apply launch");
      continue;
    }
    for (int it = 0; it < steps; ++it) {
      const int cur = it & 1, nxt = cur ^ 1;
      const bool last = (it == steps - 1);
      NsGemmParams p{};
      p.m = g.m;
      p.n = g.n;
      p.batch = cnt;
      p.scale = it == 0 ? scale : nullptr;
      p.ca = coeffs[it * coeff_stride];
      p.cb = coeffs[it * coeff_stride + 1];
      p.cc = coeffs[it * coeff_stride + 2];
      p.ldm = g.ldm;
      p.ldx = g.ldx;
      p.out = out_d;
      p.err = h->err;
      p.timeout_ns = h->timeout_ns;
      NsGemmParams q = p;
      q.tiles_per_mat = g.tri128_count;
      q.num_tiles = cnt * g.tri128_count;
      q.tri = reinterpret_cast<const int2*>(dbase + g.tri128_off);
      const int grid_sym = std::max(1, std::min(q.num_tiles, h->num_sms));
      // A = s^2 X X^T
      MUON_LAUNCH(MUON_K_SYRK, launch_ns_gemm_tc_f32(MODE_F_SYRK, xk[cur], xk[cur], ao, q, grid_sym, stream),
                  "f32 syrk launch");
      // P = a I + b A + c A A
      q.scale = nullptr;
      q.sym_in = ws + R.ap[0];
      q.sym_in_lo = ws + R.ap[1];
      q.sym_in_2 = ws + R.ap[2];
      MUON_LAUNCH(MUON_K_POLY, launch_ns_gemm_tc_f32(MODE_F_POLY, ak, ak, po, q, grid_sym, stream), "f32 poly launch");
      // X' = s P X (planes), or the destination update
      NsGemmParams u = p;
      u.mi = mi;
      u.tiles_per_mat = mi * nj;
      u.num_tiles = cnt * mi * nj;
      const int grid = std::max(1, std::min(u.num_tiles, h->num_sms));
      MUON_LAUNCH(last ? MUON_K_FINAL : MUON_K_UPDATE,
                  launch_ns_gemm_tc_f32(last ? MODE_F_FINAL : MODE_F_UPDATE, pk, xmn[cur], xo[nxt], u, grid, stream),
                  "f32 update launch");
    }
  }
  return MUON_OK;
}

// Run prepare + Newton-Schulz + final write for every block.
// Strides, tile widths and the chunk (matrices per launch) of one same-shape
// group under the handle's workspace limit; returns the workspace bytes the
// group's chunk needs.
// The fp32 path's standard method runs on the tensor cores for this group.
bool f32tc_group(muon_handle_t h, const GroupPlan& g, bool tc, bool gram) {
  return !tc && !gram && h->f32_tc && g.m <= h->f32_tc_max_m;
}

size_t plan_group(muon_handle_t h, GroupPlan& g, bool tc, bool gram, int steps, size_t limit) {
  const bool f32tc = f32tc_group(h, g, tc, gram);
  g.ldx = static_cast<long long>(align_up(g.n, 16));   // 16: the lo plane's byte rows stay 16-byte aligned
  g.ldm = static_cast<long long>(align_up(g.m, 8));
  g.prep_tiles = static_cast<int>(ceil_div(g.m, 64) * ceil_div(g.n, 64));
  g.bn_sym = g.m <= 128 ? 128 : 256;
  g.bn_upd = g.n <= 128 ? 128 : 256;
  const size_t per1 = regions(g, 1, tc, gram, steps, f32tc).total;
  const size_t per2 = regions(g, 2, tc, gram, steps, f32tc).total;
  g.per_mat = per2 > per1 ? per2 - per1 : per1;
  const size_t fixed = per1 > g.per_mat ? per1 - g.per_mat : 0;
  size_t fit = limit > fixed ? (limit - fixed) / std::max<size_t>(g.per_mat, 1) : 1;
  fit = std::max<size_t>(fit, 1);
  fit = std::min<size_t>(fit, g.members.size());
  fit = std::min<size_t>(fit, 65535);
  const int tiles_upd = static_cast<int>(ceil_div(g.m, 128) * ceil_div(g.n, f32tc ? 128 : g.bn_upd));
  const int tiles_max = std::max({tiles_upd, g.prep_tiles, 1});
  fit = std::min<size_t>(fit, static_cast<size_t>((1u << 31) - 1) / static_cast<size_t>(tiles_max));
  g.chunk = static_cast<int>(fit);
  return regions(g, g.chunk, tc, gram, steps, f32tc).total;
}

constexpr size_t kConcMaxElements = size_t(1) << 28;

// Workspace bytes of the concurrent-groups layout (every group's regions
// side by side), or 0 when the call runs its groups one after another.
// Concurrent: the standard method on the bf16 path or the fp32 tensor-core
// path, two or more groups each in a single
// chunk, their regions within the workspace limit together, and (unless
// forced by MUON_CONCURRENT=1) at most kConcMaxElements NS elements in all:
// large groups fill the GPU with each launch on their own.
size_t concurrent_need(muon_handle_t h, const std::map<std::pair<int, int>, GroupPlan>& groups, bool tc, bool gram,
                       int steps, bool overlap) {
  if (gram || steps == 0 || overlap || h->concurrent == 0 || groups.size() < 2) return 0;
  size_t sum = 0, elems = 0;
  for (const auto& kv : groups) {
    const GroupPlan& g = kv.second;
    const bool f32tc = f32tc_group(h, g, tc, gram);
    if (!tc && !f32tc) return 0;                 // the fp32 CUDA-core path runs its groups in turn
    if (static_cast<size_t>(g.chunk) < g.members.size()) return 0;
    sum += align_up(regions(g, g.chunk, tc, gram, steps, f32tc).total, 256);
    elems += g.members.size() * static_cast<size_t>(g.m) * static_cast<size_t>(g.n);
  }
  if (sum > h->ws_limit) return 0;
  if (h->concurrent < 0 && elems > kConcMaxElements) return 0;
  return sum;
}

// coeffs: (a, b, c) of step k at coeffs[k * coeff_stride] (stride 0: one
// triple for every step, 3: a schedule of `steps` triples).
muon_status_t run_blocks(muon_handle_t h, const std::vector<Block>& blocks, float mu, int nesterov, int steps,
                         const float* coeffs, int coeff_stride, int ns_method, bool tc, cudaStream_t stream) {
  if (blocks.empty()) return MUON_OK;
  const bool gram = (ns_method == MUON_NS_GRAM);
  // small sets: the element-wise kernels chained by programmatic dependent
  // launch too (GPT-2-small 1.489 -> 1.451 ms); large sets keep it for the
  // GEMMs only
  size_t elems = 0;
  for (const Block& b : blocks) elems += static_cast<size_t>(b.m) * static_cast<size_t>(b.n);
  ElementwisePdlScope pdl_scope(elems <= kConcMaxElements);
  // unit preparation overlapped with the products (standard bf16 method):
  // two workspace halves, each planned under half the limit
  const bool overlap = h->overlap && tc && !gram && steps > 0;

  std::map<std::pair<int, int>, GroupPlan> groups;
  for (size_t i = 0; i < blocks.size(); ++i) {
    GroupPlan& g = groups[{blocks[i].m, blocks[i].n}];
    g.m = blocks[i].m;
    g.n = blocks[i].n;
    g.members.push_back(static_cast<int>(i));
  }

  std::vector<uint8_t> arena;
  size_t ws_need = 0;
  for (auto& kv : groups) {
    GroupPlan& g = kv.second;
    ws_need = std::max(ws_need, plan_group(h, g, tc, gram, steps, overlap ? h->ws_limit / 2 : h->ws_limit));
    if (f32tc_group(h, g, tc, gram)) {
      std::vector<int2> t128 = sym_tiles(g.m, 128);
      g.tri128_count = static_cast<int>(t128.size());
      g.tri128_off = arena_push(arena, t128.data(), t128.size());
    }
    if (tc) {
      std::vector<int2> tri = sym_tiles(g.m, g.bn_sym);
      g.tri_count = static_cast<int>(tri.size());
      g.tri_off = arena_push(arena, tri.data(), tri.size());
      if (gram) {
        std::vector<int2> t128 = sym_tiles(g.m, 128);
        g.tri128_count = static_cast<int>(t128.size());
        g.tri128_off = arena_push(arena, t128.data(), t128.size());
      }
      if (h->use_pair && h->max_pairs > 0 && pair_group(g.m, h->pair_min_m)) {
        std::vector<int2> t256 = sym_tiles(g.m, 256, 256);
        g.tri256_count = static_cast<int>(t256.size());
        g.tri256_off = arena_push(arena, t256.data(), t256.size());
        g.pair = true;
        // UPDATE / FINAL on pairs only without a ragged last row tile, or
        // from m = 2048 (a ragged tile costs them more than the symmetric
        // products)
        g.pair_upd = h->pair_update && (g.m % 256 == 0 || g.m >= 2048);
      }
    }
    for (size_t c0 = 0; c0 < g.members.size(); c0 += g.chunk) {
      const size_t cnt = std::min<size_t>(g.chunk, g.members.size() - c0);
      std::vector<SrcEntry> src(cnt);
      std::vector<OutEntry> out(cnt);
      for (size_t k = 0; k < cnt; ++k) {
        src[k] = blocks[g.members[c0 + k]].src;
        out[k] = blocks[g.members[c0 + k]].out;
      }
      const size_t so = arena_push(arena, src.data(), cnt);
      const size_t oo = arena_push(arena, out.data(), cnt);
      g.chunk_off.emplace_back(so, oo);
      std::vector<CUtensorMap> maps;
      const bool tma_out = tc && steps > 0 && h->final_tma && encode_dest_maps(h, g, out, &maps);
      g.chunk_wmap.push_back(tma_out ? arena_push(arena, maps.data(), maps.size()) : kNoMaps);
    }
  }

  const size_t conc_need = concurrent_need(h, groups, tc, gram, steps, overlap);
  if (conc_need > 0) ws_need = conc_need;
  const size_t half_bytes = align_up(ws_need, 256);
  muon_status_t st = ensure_ws(h, overlap ? 2 * half_bytes : ws_need);
  if (st != MUON_OK) return st;
  void* dev = nullptr;
  st = upload(h, arena, stream, &dev);
  if (st != MUON_OK) return st;
  uint8_t* dbase = static_cast<uint8_t*>(dev);
  uint8_t* ws = static_cast<uint8_t*>(h->ws);

  // The standard method's workspace regions of one same-shape group at
  // `base` (the workspace, or one of its halves when unit preparation
  // overlaps the products), and the tensor maps over them.
  struct StdSet {
    float *xf, *xf2, *pdiag, *partials, *scale;
    __nv_bfloat16* xb[2];
    int8_t* xlo;
    void *symA, *symB;
    bool n128;
    CUtensorMap map_x[2], map_xmn[2], map_A, map_A64, map_B, map_xh[2], map_xl, map_sa, map_sb;
  };
  auto make_set = [&](const GroupPlan& g, uint8_t* base, StdSet& S) -> muon_status_t {
    const Regions R = regions(g, g.chunk, tc, gram, steps, false);
    // pair symmetric products of a ragged m whose last 256-column block has
    // at most 128 valid columns: those tiles run N = 128 (64-row B boxes)
    S.n128 = tc && g.pair && g.m % 256 != 0 && g.m % 256 <= 128;
    S.xf = reinterpret_cast<float*>(base + R.xf);
    S.xf2 = tc ? nullptr : reinterpret_cast<float*>(base + R.xf2);
    S.xb[0] = tc ? reinterpret_cast<__nv_bfloat16*>(base + R.xb0) : nullptr;
    S.xb[1] = tc ? reinterpret_cast<__nv_bfloat16*>(base + R.xb1) : nullptr;
    S.symA = base + R.symA;
    S.symB = base + R.symB;
    S.pdiag = tc ? reinterpret_cast<float*>(base + R.pdiag) : nullptr;
    S.partials = reinterpret_cast<float*>(base + R.partials);
    S.scale = reinterpret_cast<float*>(base + R.scale);
    S.xlo = (tc && steps > 0) ? reinterpret_cast<int8_t*>(base + R.xlo) : nullptr;
    if (tc && steps > 0) {
      if (!encode_map(h, &S.map_x[0], S.xb[0], g.n, g.m, g.chunk, g.ldx) ||
          !encode_map(h, &S.map_x[1], S.xb[1], g.n, g.m, g.chunk, g.ldx) ||
          !encode_map(h, &S.map_xmn[0], S.xb[0], g.n, g.m, g.chunk, g.ldx, 64) ||
          !encode_map(h, &S.map_xmn[1], S.xb[1], g.n, g.m, g.chunk, g.ldx, 64) ||
          !encode_map(h, &S.map_A, S.symA, g.m, g.m, g.chunk, g.ldm) ||
          !encode_map(h, &S.map_A64, S.symA, g.m, g.m, g.chunk, g.ldm, 64) ||
          !encode_map(h, &S.map_B, S.symB, g.m, g.m, g.chunk, g.ldm) ||
          !encode_box32(h->encode, &S.map_xh[0], S.xb[0], false, g.n, g.m, g.chunk, g.ldx) ||
          !encode_box32(h->encode, &S.map_xh[1], S.xb[1], false, g.n, g.m, g.chunk, g.ldx) ||
          !encode_lo8_box32(h->encode, &S.map_xl, S.xlo, g.n, g.m, g.chunk, g.ldx) ||
          !encode_box32(h->encode, &S.map_sa, S.symA, false, g.m, g.m, g.chunk, g.ldm) ||
          !encode_box32(h->encode, &S.map_sb, S.symB, false, g.m, g.m, g.chunk, g.ldm))
        return fail(h, MUON_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    }
    return MUON_OK;
  };
  // chunk c: momentum, U, norm (and, with no NS step, the parameter write)
  auto prep = [&](const GroupPlan& g, StdSet& S, size_t c, cudaStream_t stream) -> muon_status_t {
    const int cnt = static_cast<int>(std::min<size_t>(g.chunk, g.members.size() - c * g.chunk));
    const SrcEntry* src_d = reinterpret_cast<const SrcEntry*>(dbase + g.chunk_off[c].first);
    const OutEntry* out_d = reinterpret_cast<const OutEntry*>(dbase + g.chunk_off[c].second);
    PrepParams pp{};
    pp.src = src_d;
    pp.mu = mu;
    pp.nesterov = nesterov;
    pp.m = g.m;
    pp.ldx = g.ldx;
    pp.xf = (tc && steps > 0) ? nullptr : S.xf;
    pp.xb = S.xb[0];
    pp.xlo8 = S.xlo;
    pp.partials = S.partials;
    pp.tiles_per_mat = g.prep_tiles;
    MUON_LAUNCH(MUON_K_PREPARE, launch_prepare(pp, cnt, g.prep_tiles, stream), "prepare launch");
    MUON_LAUNCH(MUON_K_NORM, launch_norm_finalize(S.partials, g.prep_tiles, cnt, kNormEps, S.scale, h->err, stream),
                "norm launch");

    if (steps == 0) {
      ApplyParams ap{out_d, S.scale, S.xf, g.ldx, g.m, g.n};
      MUON_LAUNCH(MUON_K_APPLY, launch_apply(ap, cnt, stream), "apply launch");
    }
    return MUON_OK;
  };
  // chunk c: the NS products, the last one writing the destinations
  auto products = [&](const GroupPlan& g, StdSet& S, size_t c, cudaStream_t stream) -> muon_status_t {
    if (steps == 0) return MUON_OK;
    const int mi = static_cast<int>(ceil_div(g.m, 128));
    const int nj = static_cast<int>(ceil_div(g.n, g.bn_upd));
    const int cnt = static_cast<int>(std::min<size_t>(g.chunk, g.members.size() - c * g.chunk));
    const OutEntry* out_d = reinterpret_cast<const OutEntry*>(dbase + g.chunk_off[c].second);
    const CUtensorMap* wmap_d =
        g.chunk_wmap[c] == kNoMaps ? nullptr : reinterpret_cast<const CUtensorMap*>(dbase + g.chunk_wmap[c]);
    // the last UPDATE writes the destinations: through their tensor maps
    // when the chunk has them
    const int final_mode = wmap_d != nullptr ? MODE_FINAL_T : MODE_FINAL;
    for (int it = 0; it < steps; ++it) {
      const bool last = (it == steps - 1);
      NsGemmParams p{};
      p.m = g.m;
      p.n = g.n;
      p.batch = cnt;
      p.scale = it == 0 ? S.scale : nullptr;
      p.ca = coeffs[it * coeff_stride];        // this iteration's (a, b, c)
      p.cb = coeffs[it * coeff_stride + 1];
      p.cc = coeffs[it * coeff_stride + 2];
      p.ldm = g.ldm;
      p.ldx = g.ldx;
      p.out = out_d;
      p.wmap = wmap_d;
      p.err = h->err;
      p.timeout_ns = h->timeout_ns;
      p.pdiag = S.pdiag;
      if (tc && g.pair) {
        // SYRK, POLY and (pair_upd) UPDATE / FINAL on CTA pairs, 256 x 256
        // tiles
        NsGemmParams q = p;
        q.tiles_per_mat = g.tri256_count;
        q.num_tiles = cnt * g.tri256_count;
        q.tri = reinterpret_cast<const int2*>(dbase + g.tri256_off);
        q.sym_out = S.symA;
        const int pairs = std::min(q.num_tiles, h->max_pairs);
        MUON_LAUNCH(MUON_K_SYRK,
                    launch_ns_gemm_pair(MODE_SYRK, S.map_x[it & 1], S.map_x[it & 1], S.map_sa, S.map_sa, q, pairs, stream,
                                        S.n128 ? &S.map_xmn[it & 1] : nullptr),
                    "syrk launch");
        q.scale = p.scale;                     // P' = s P in the first iteration
        q.sym_in = S.symA;
        q.sym_out = S.symB;
        MUON_LAUNCH(MUON_K_POLY,
                    launch_ns_gemm_pair(MODE_POLY, S.map_A, S.map_A, S.map_sb, S.map_sb, q, pairs, stream, S.n128 ? &S.map_A64 : nullptr),
                    "poly launch");
        NsGemmParams u = p;
        if (g.pair_upd) {
          const int mi2 = static_cast<int>(ceil_div(g.m, 256)), nj2 = static_cast<int>(ceil_div(g.n, 256));
          u.mi = mi2;
          u.tiles_per_mat = mi2 * nj2;
          u.num_tiles = cnt * mi2 * nj2;
          const int upairs = std::min(u.num_tiles, h->max_pairs);
          MUON_LAUNCH(last ? MUON_K_FINAL : MUON_K_UPDATE,
                      launch_ns_gemm_pair_update(last ? final_mode : MODE_UPDATE, S.map_B, S.map_xmn[it & 1],
                                                 S.map_xh[it & 1], S.map_xl, S.map_xh[(it + 1) & 1], u, upairs, stream,
                                                 g.m <= kShortK ? 2 : 0),
                      "update launch");
        } else {
          u.mi = mi;
          u.tiles_per_mat = mi * nj;
          u.num_tiles = cnt * mi * nj;
          const int grid = std::min(u.num_tiles, h->num_sms);
          MUON_LAUNCH(last ? MUON_K_FINAL : MUON_K_UPDATE,
                      launch_ns_gemm_tc_update(last ? final_mode : MODE_UPDATE, g.bn_upd, S.map_B, S.map_xmn[it & 1],
                                               S.map_xh[it & 1], S.map_xl, S.map_xh[(it + 1) & 1], u, grid, stream),
                      "update launch");
        }
      } else if (tc) {
        // SYRK: A = s^2 X X^T
        NsGemmParams q = p;
        q.tiles_per_mat = g.tri_count;
        q.num_tiles = cnt * g.tri_count;
        q.tri = reinterpret_cast<const int2*>(dbase + g.tri_off);
        q.sym_out = S.symA;
        int grid = std::min(q.num_tiles, h->num_sms);
        MUON_LAUNCH(MUON_K_SYRK, launch_ns_gemm_tc(MODE_SYRK, g.bn_sym, S.map_x[it & 1], S.map_x[it & 1], S.map_sa, S.map_sa, q, grid,
                                                       stream),
                    "syrk launch");
        // POLY: P = a I + b A + c A A, times s in the first iteration
        q.scale = p.scale;
        q.sym_in = S.symA;
        q.sym_out = S.symB;
        MUON_LAUNCH(MUON_K_POLY, launch_ns_gemm_tc(MODE_POLY, g.bn_sym, S.map_A, S.map_A, S.map_sb, S.map_sb, q, grid, stream), "poly launch");
        // UPDATE / FINAL: X = P^ X^ + P_rr X - P^_rr X^ (s inside P)
        NsGemmParams u = p;
        u.mi = mi;
        u.tiles_per_mat = mi * nj;
        u.num_tiles = cnt * mi * nj;
        grid = std::min(u.num_tiles, h->num_sms);
        MUON_LAUNCH(last ? MUON_K_FINAL : MUON_K_UPDATE,
                    launch_ns_gemm_tc_update(last ? final_mode : MODE_UPDATE, g.bn_upd, S.map_B, S.map_xmn[it & 1],
                                             S.map_xh[it & 1], S.map_xl, S.map_xh[(it + 1) & 1], u, grid, stream),
                    "update launch");
      } else {
        float* xin = (it & 1) ? S.xf2 : S.xf;
        float* xout = (it & 1) ? S.xf : S.xf2;
        NsGemmParams q = p;
        q.xf_in = xin;
        q.sym_out = S.symA;
        MUON_LAUNCH(MUON_K_SYRK, launch_ns_gemm_simt(MODE_SYRK, q, stream), "syrk launch");
        q.scale = nullptr;
        q.sym_in = S.symA;
        q.sym_out = S.symB;
        MUON_LAUNCH(MUON_K_POLY, launch_ns_gemm_simt(MODE_POLY, q, stream), "poly launch");
        NsGemmParams u = p;
        u.sym_in = S.symB;
        u.xf_in = xin;
        u.xf_out = xout;
        MUON_LAUNCH(last ? MUON_K_FINAL : MUON_K_UPDATE, launch_ns_gemm_simt(last ? MODE_FINAL : MODE_UPDATE, u, stream),
                    "update launch");
      }
    }
    return MUON_OK;
  };

  std::vector<GroupPlan*> order;              // ascending (m, n)
  for (auto& kv : groups) order.push_back(&kv.second);
  if (conc_need > 0) {
    // Concurrent groups: the group with the most work on the caller's
    // stream, every other on a stream of its own that first waits for
    // everything enqueued before (the descriptor upload included); the
    // caller's stream waits for each of them before the call returns.
    std::vector<GroupPlan*> by_work(order);
    std::stable_sort(by_work.begin(), by_work.end(), [](const GroupPlan* a, const GroupPlan* b) {
      const double wa = static_cast<double>(a->members.size()) * a->m * a->m * a->n;
      const double wb = static_cast<double>(b->members.size()) * b->m * b->m * b->n;
      return wa > wb;
    });
    std::map<const GroupPlan*, size_t> offset;   // the regions side by side, in (m, n) order
    size_t off = 0;
    for (GroupPlan* g : order) {
      offset[g] = off;
      off += align_up(regions(*g, g->chunk, tc, gram, steps, f32tc_group(h, *g, tc, gram)).total, 256);
    }
    const size_t nside = by_work.size() - 1;
    muon_status_t cst = ensure_concurrent(h, nside);
    if (cst != MUON_OK) return cst;
    MUON_CUDA_TRY(cudaEventRecord(h->conc_ev[0], stream), "concurrent start event");
    for (size_t k = 0; k < nside; ++k)
      MUON_CUDA_TRY(cudaStreamWaitEvent(h->conc[k], h->conc_ev[0], 0), "concurrent stream wait");
    for (size_t k = 0; k < by_work.size(); ++k) {
      GroupPlan& g = *by_work[k];
      cudaStream_t gs = k == 0 ? stream : h->conc[k - 1];
      h->prof_tag = static_cast<int>(std::find(order.begin(), order.end(), by_work[k]) - order.begin());
      if (f32tc_group(h, g, tc, gram)) {
        const Regions R = regions(g, g.chunk, tc, gram, steps, true);
        if ((cst = run_f32tc_group(h, g, R, ws + offset[&g], dbase, steps, coeffs, coeff_stride, mu, nesterov, gs)) !=
            MUON_OK)
          return cst;
        continue;
      }
      StdSet S;
      if ((cst = make_set(g, ws + offset[&g], S)) != MUON_OK) return cst;
      if ((cst = prep(g, S, 0, gs)) != MUON_OK) return cst;
      if ((cst = products(g, S, 0, gs)) != MUON_OK) return cst;
    }
    for (size_t k = 0; k < nside; ++k) {
      MUON_CUDA_TRY(cudaEventRecord(h->conc_ev[1 + k], h->conc[k]), "concurrent done event");
      MUON_CUDA_TRY(cudaStreamWaitEvent(stream, h->conc_ev[1 + k], 0), "concurrent join");
    }
    return MUON_OK;
  }
  if (!overlap) {
    for (size_t gi = 0; gi < order.size(); ++gi) {
      GroupPlan& g = *order[gi];
      h->prof_tag = static_cast<int>(gi);
      const bool f32tc = f32tc_group(h, g, tc, gram);
      const Regions R = regions(g, g.chunk, tc, gram, steps, f32tc);
      if (f32tc) {
        muon_status_t fst = run_f32tc_group(h, g, R, ws, dbase, steps, coeffs, coeff_stride, mu, nesterov, stream);
        if (fst != MUON_OK) return fst;
        continue;
      }
      if (gram) {
        muon_status_t gst = run_gram_group(h, g, R, ws, dbase, steps, coeffs, coeff_stride, tc, mu, nesterov, stream);
        if (gst != MUON_OK) return gst;
        continue;
      }
      StdSet S;
      muon_status_t sst = make_set(g, ws, S);
      if (sst != MUON_OK) return sst;
      for (size_t c = 0; c < g.chunk_off.size(); ++c) {
        sst = prep(g, S, c, stream);
        if (sst != MUON_OK) return sst;
        sst = products(g, S, c, stream);
        if (sst != MUON_OK) return sst;
      }
    }
    return MUON_OK;
  }

  // Overlapped: units (group, chunk) in launch order use the two workspace
  // halves in turn; unit u+1's preparation (an HBM-bound pass) runs on the
  // handle's side stream while unit u's products run on the caller's stream.
  // Events order it: the side stream starts after everything enqueued
  // before this call, prepares unit u+1 once unit u-1 (the last user of that
  // half) has finished, and the caller's stream waits for a unit's
  // preparation before its products, so every side-stream launch is joined
  // before the call's last products.
  struct Unit {
    int group;
    size_t chunk;
  };
  std::vector<Unit> units;
  for (size_t gi = 0; gi < order.size(); ++gi)
    for (size_t c = 0; c < order[gi]->chunk_off.size(); ++c) units.push_back(Unit{static_cast<int>(gi), c});
  std::vector<StdSet> sets(2 * order.size());
  std::vector<char> made(2 * order.size(), 0);
  auto set_of = [&](const Unit& u, int half, StdSet** out) -> muon_status_t {
    const size_t k = 2 * static_cast<size_t>(u.group) + static_cast<size_t>(half);
    if (!made[k]) {
      muon_status_t r = make_set(*order[u.group], ws + static_cast<size_t>(half) * half_bytes, sets[k]);
      if (r != MUON_OK) return r;
      made[k] = 1;
    }
    *out = &sets[k];
    return MUON_OK;
  };
  muon_status_t ost = ensure_overlap_events(h, 2 * units.size() + 1);
  if (ost != MUON_OK) return ost;
  cudaEvent_t ev_start = h->ovl_ev[0];
  auto ev_ready = [&](size_t u) { return h->ovl_ev[1 + 2 * u]; };
  auto ev_freed = [&](size_t u) { return h->ovl_ev[2 + 2 * u]; };
  MUON_CUDA_TRY(cudaEventRecord(ev_start, stream), "overlap start event");
  MUON_CUDA_TRY(cudaStreamWaitEvent(h->side, ev_start, 0), "side stream wait");
  {
    StdSet* S0 = nullptr;
    if ((ost = set_of(units[0], 0, &S0)) != MUON_OK) return ost;
    h->prof_tag = units[0].group;
    if ((ost = prep(*order[units[0].group], *S0, units[0].chunk, stream)) != MUON_OK) return ost;
  }
  for (size_t u = 0; u < units.size(); ++u) {
    if (u + 1 < units.size()) {
      const Unit& nx = units[u + 1];
      StdSet* Sn = nullptr;
      if ((ost = set_of(nx, static_cast<int>((u + 1) & 1), &Sn)) != MUON_OK) return ost;
      if (u >= 1) MUON_CUDA_TRY(cudaStreamWaitEvent(h->side, ev_freed(u - 1), 0), "side stream wait");
      h->prof_tag = nx.group;
      if ((ost = prep(*order[nx.group], *Sn, nx.chunk, h->side)) != MUON_OK) return ost;
      MUON_CUDA_TRY(cudaEventRecord(ev_ready(u + 1), h->side), "overlap ready event");
    }
    if (u >= 1) MUON_CUDA_TRY(cudaStreamWaitEvent(stream, ev_ready(u), 0), "stream wait");
    StdSet* S = nullptr;
    if ((ost = set_of(units[u], static_cast<int>(u & 1), &S)) != MUON_OK) return ost;
    h->prof_tag = units[u].group;
    if ((ost = products(*order[units[u].group], *S, units[u].chunk, stream)) != MUON_OK) return ost;
    MUON_CUDA_TRY(cudaEventRecord(ev_freed(u), stream), "overlap freed event");
  }
  return MUON_OK;
}

bool valid_dtype(int32_t d) { return d == MUON_F32 || d == MUON_BF16; }
bool valid_method(int32_t m) { return m == MUON_NS_STANDARD || m == MUON_NS_GRAM || m == MUON_NS_AUTO; }

// MUON_NS_AUTO: the Gram method for a same-shape group whose n is at least
// kAutoGramRatio times its m (bf16 path), where it measured faster than the
// standard method (64 bf16 matrices each: 1024 x 4096 1.02x, 2048 x 16384
// 1.43x, 256 x 4096 1.77x; 2048 x 4096 0.60x); the standard method otherwise.
constexpr int64_t kAutoGramRatio = 4;
bool auto_gram(const Block& b, bool tc) { return tc && static_cast<int64_t>(b.n) >= kAutoGramRatio * b.m; }

// run_blocks with MUON_NS_AUTO resolved: the standard groups, then the Gram
// groups, as two calls on the same stream (the workspace is reused in turn).
muon_status_t run_method(muon_handle_t h, const std::vector<Block>& blocks, float mu, int nesterov, int steps,
                         const float* coeffs, int coeff_stride, int ns_method, bool tc, cudaStream_t stream) {
  if (ns_method != MUON_NS_AUTO)
    return run_blocks(h, blocks, mu, nesterov, steps, coeffs, coeff_stride, ns_method, tc, stream);
  std::vector<Block> standard, gram;
  for (const Block& b : blocks) (auto_gram(b, tc) ? gram : standard).push_back(b);
  const muon_status_t st = run_blocks(h, standard, mu, nesterov, steps, coeffs, coeff_stride, MUON_NS_STANDARD, tc,
                                      stream);
  if (st != MUON_OK) return st;
  return run_blocks(h, gram, mu, nesterov, steps, coeffs, coeff_stride, MUON_NS_GRAM, tc, stream);
}

// Validate the parameter descriptors and expand them into NS blocks (one per
// Muon-Split head block, rows <= cols after the transpose rule) with their
// source / destination entries.  need_ptrs = false: shapes only (sizing).
muon_status_t build_blocks(muon_handle_t h, const muon_param_t* params, int32_t n_params,
                           const muon_step_options_t& o, bool need_ptrs, std::vector<Block>* out) {
  for (int32_t i = 0; i < n_params; ++i) {
    const muon_param_t& P = params[i];
    const std::string where = "param " + std::to_string(i) + ": ";
    if (!valid_dtype(P.param_dtype) || !valid_dtype(P.grad_dtype))
      return fail(h, MUON_ERR_INVALID_ARG, where + "bad dtype");
    if (P.rows < 0 || P.cols < 0 || P.rows > kMaxDim || P.cols > kMaxDim)
      return fail(h, MUON_ERR_INVALID_ARG, where + "negative or oversized shape");
    if (P.split_heads < 1 || (P.rows > 0 && P.rows % P.split_heads != 0))
      return fail(h, MUON_ERR_INVALID_ARG, where + "split_heads must be >= 1 and divide rows");
    if (P.reserved != 0 || P.scale_dim < 0) return fail(h, MUON_ERR_INVALID_ARG, where + "bad reserved/scale_dim");
    if (P.rows == 0 || P.cols == 0) continue;
    if (need_ptrs && (P.param == nullptr || P.grad == nullptr || P.momentum == nullptr))
      return fail(h, MUON_ERR_INVALID_ARG, where + "NULL pointer");
    const int64_t rb = P.rows / P.split_heads;
    // update scale: RMS matching update_rms * sqrt(max(A, B)) (or scale_dim),
    // or muP sqrt(d_out / d_in) of the stored (out x in) parameter
    double scale;
    if (o.scale_mode == MUON_SCALE_MUP) {
      scale = std::sqrt(static_cast<double>(P.rows) / static_cast<double>(P.cols));
    } else {
      const double sdim = static_cast<double>(P.scale_dim > 0 ? P.scale_dim : std::max(P.rows, P.cols));
      scale = static_cast<double>(o.update_rms) * std::sqrt(sdim);
    }
    const float beta = static_cast<float>(-static_cast<double>(o.lr) * o.extra_scale * scale);
    const float alpha = static_cast<float>(1.0 - static_cast<double>(o.lr) * o.wd);
    const size_t ge = dtype_size(P.grad_dtype), pe = dtype_size(P.param_dtype);
    for (int32_t hb = 0; hb < P.split_heads; ++hb) {
      const size_t off = static_cast<size_t>(hb) * rb * P.cols;
      Block bl;
      const int transposed = rb > P.cols ? 1 : 0;
      bl.src = SrcEntry{static_cast<const uint8_t*>(P.grad) + off * ge, P.momentum + off, P.cols,
                        static_cast<int>(rb), static_cast<int>(P.cols), transposed, P.grad_dtype};
      bl.out = OutEntry{static_cast<uint8_t*>(P.param) + off * pe, P.cols, transposed, P.param_dtype, alpha, beta};
      bl.m = static_cast<int>(std::min<int64_t>(rb, P.cols));
      bl.n = static_cast<int>(std::max<int64_t>(rb, P.cols));
      out->push_back(bl);
    }
  }
  return MUON_OK;
}

}  // namespace

extern "C" {

const char* muon_status_string(muon_status_t s) {
  switch (s) {
    case MUON_OK: return "ok";
    case MUON_ERR_INVALID_ARG: return "invalid argument";
    case MUON_ERR_UNSUPPORTED: return "unsupported";
    case MUON_ERR_WORKSPACE: return "workspace allocation failed";
    case MUON_ERR_CUDA: return "CUDA error";
    case MUON_ERR_NONFINITE: return "non-finite gradient norm";
    case MUON_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

const char* muon_last_error(muon_handle_t h) { return h == nullptr ? "null handle" : h->last.c_str(); }

int32_t muon_version(void) { return 10000; }

muon_status_t muon_handle_create(muon_handle_t* out, int device) {
  if (out == nullptr) return MUON_ERR_INVALID_ARG;
  *out = nullptr;
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || device < 0 || device >= count) {
    cudaGetLastError();
    return MUON_ERR_UNSUPPORTED;
  }
  DeviceGuard guard(device);
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return MUON_ERR_CUDA;
  if (!(prop.major == 10 && prop.minor == 3)) return MUON_ERR_UNSUPPORTED;   // built for sm_103a only
  muon_handle_t h = new (std::nothrow) muon_handle_s();
  if (h == nullptr) return MUON_ERR_WORKSPACE;
  h->device = device;
  h->num_sms = prop.multiProcessorCount;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr) {
    delete h;
    return MUON_ERR_UNSUPPORTED;
  }
  h->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  const char* pair_env = std::getenv("MUON_TC_PAIR");
  h->use_pair = !(pair_env != nullptr && pair_env[0] == '0');
  h->pair_update = h->use_pair && !(pair_env != nullptr && std::strcmp(pair_env, "sym") == 0);
  if (const char* mm = std::getenv("MUON_TC_PAIR_MIN_M")) {
    const long v = std::strtol(mm, nullptr, 10);
    if (v >= 256 && v <= (1L << 30)) h->pair_min_m = static_cast<int>(v);
  }
  h->max_pairs = h->use_pair ? ns_gemm_pair_max_pairs() : 0;
  if (const char* ft = std::getenv("MUON_FINAL_TMA")) h->final_tma = ft[0] != '0';
  if (const char* ft = std::getenv("MUON_F32_TC")) h->f32_tc = ft[0] != '0';
  if (const char* fm = std::getenv("MUON_F32_TC_MAX_M")) {
    const long v = std::strtol(fm, nullptr, 10);
    if (v >= 1 && v <= (1L << 30)) h->f32_tc_max_m = static_cast<int>(v);
  }
  if (const char* ov = std::getenv("MUON_OVERLAP")) h->overlap = ov[0] == '1';
  if (const char* cc = std::getenv("MUON_CONCURRENT")) h->concurrent = cc[0] == '0' ? 0 : cc[0] == '1' ? 1 : -1;
  bool ok = cudaMalloc(&h->err, sizeof(unsigned)) == cudaSuccess && cudaMemset(h->err, 0, sizeof(unsigned)) == cudaSuccess;
  for (int k = 0; ok && k < muon_handle_s::kStages; ++k)
    ok = cudaEventCreateWithFlags(&h->stage_ev[k], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    if (h->err) cudaFree(h->err);
    for (int k = 0; k < muon_handle_s::kStages; ++k)
      if (h->stage_ev[k]) cudaEventDestroy(h->stage_ev[k]);
    delete h;
    return MUON_ERR_WORKSPACE;
  }
  *out = h;
  return MUON_OK;
}

muon_status_t muon_handle_destroy(muon_handle_t h) {
  if (h == nullptr) return MUON_OK;
  DeviceGuard guard(h->device);
  cudaDeviceSynchronize();
  if (h->ws) cudaFree(h->ws);
  if (h->desc) cudaFree(h->desc);
  for (int k = 0; k < muon_handle_s::kStages; ++k) {
    if (h->hstage[k]) cudaFreeHost(h->hstage[k]);
    if (h->stage_ev[k]) cudaEventDestroy(h->stage_ev[k]);
  }
  if (h->err) cudaFree(h->err);
  for (cudaEvent_t e : h->ovl_ev) cudaEventDestroy(e);
  if (h->side) cudaStreamDestroy(h->side);
  for (cudaEvent_t e : h->conc_ev) cudaEventDestroy(e);
  for (cudaStream_t cs : h->conc) cudaStreamDestroy(cs);
  for (auto& r : h->prof) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  delete h;
  return MUON_OK;
}

muon_status_t muon_handle_set_workspace_limit(muon_handle_t h, size_t bytes) {
  if (h == nullptr || bytes == 0) return MUON_ERR_INVALID_ARG;
  h->ws_limit = bytes;
  return MUON_OK;
}

muon_status_t muon_handle_set_timeout_ns(muon_handle_t h, uint64_t timeout_ns) {
  if (h == nullptr || timeout_ns == 0) return MUON_ERR_INVALID_ARG;
  h->timeout_ns = timeout_ns;
  return MUON_OK;
}

muon_status_t muon_handle_check(muon_handle_t h, void* stream) {
  if (h == nullptr) return MUON_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MUON_CUDA_TRY(cudaStreamSynchronize(s), "stream synchronise");
  unsigned word = 0;
  MUON_CUDA_TRY(cudaMemcpy(&word, h->err, sizeof(unsigned), cudaMemcpyDeviceToHost), "error word read");
  MUON_CUDA_TRY(cudaMemset(h->err, 0, sizeof(unsigned)), "error word reset");
  if (word & ERRBIT_TIMEOUT) return fail(h, MUON_ERR_TIMEOUT, "a bounded device wait timed out");
  if (word & ERRBIT_NONFINITE) return fail(h, MUON_ERR_NONFINITE, "a Frobenius norm was not finite");
  return MUON_OK;
}

muon_status_t muon_orthogonalize(muon_handle_t h, void* X, int32_t dtype, int64_t batch, int64_t m, int64_t n,
                                 int32_t steps, const float* coeffs, int32_t ns_method, void* stream) {
  if (h == nullptr) return MUON_ERR_INVALID_ARG;
  if (!valid_dtype(dtype)) return fail(h, MUON_ERR_INVALID_ARG, "dtype must be MUON_F32 or MUON_BF16");
  if (batch < 0 || m < 0 || n < 0 || m > kMaxDim || n > kMaxDim || batch > kMaxDim)
    return fail(h, MUON_ERR_INVALID_ARG, "negative or oversized shape");
  if (steps < 0 || steps > 100) return fail(h, MUON_ERR_INVALID_ARG, "steps must be in [0, 100]");
  if (!valid_method(ns_method)) return fail(h, MUON_ERR_INVALID_ARG, "unknown ns_method");
  if (batch == 0 || m == 0 || n == 0) return MUON_OK;
  if (X == nullptr) return fail(h, MUON_ERR_INVALID_ARG, "X is NULL");
  DeviceGuard guard(h->device);
  const float* cf = coeffs ? coeffs : kDefaultCoeffs;
  const size_t es = dtype_size(dtype);
  std::vector<Block> blocks(static_cast<size_t>(batch));
  for (int64_t b = 0; b < batch; ++b) {
    uint8_t* base = static_cast<uint8_t*>(X) + static_cast<size_t>(b) * m * n * es;
    Block& bl = blocks[b];
    const int transposed = m > n ? 1 : 0;
    bl.src = SrcEntry{base, nullptr, n, static_cast<int>(m), static_cast<int>(n), transposed, dtype};
    bl.out = OutEntry{base, n, transposed, dtype, 0.f, 1.f};
    bl.m = static_cast<int>(std::min(m, n));
    bl.n = static_cast<int>(std::max(m, n));
  }
  return run_method(h, blocks, 0.f, 0, steps, cf, 0, ns_method, dtype == MUON_BF16, static_cast<cudaStream_t>(stream));
}

muon_status_t muon_workspace_size(muon_handle_t h, const muon_param_t* params, int32_t n_params, int32_t ns_method,
                                  int32_t ns_steps, int32_t ns_dtype, uint64_t* bytes) {
  if (h == nullptr) return MUON_ERR_INVALID_ARG;
  if (bytes == nullptr) return fail(h, MUON_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = 0;
  if (n_params < 0) return fail(h, MUON_ERR_INVALID_ARG, "n_params < 0");
  if (n_params > 0 && params == nullptr) return fail(h, MUON_ERR_INVALID_ARG, "params is NULL");
  if (!valid_dtype(ns_dtype)) return fail(h, MUON_ERR_INVALID_ARG, "ns_dtype must be MUON_F32 or MUON_BF16");
  if (!valid_method(ns_method)) return fail(h, MUON_ERR_INVALID_ARG, "unknown ns_method");
  if (ns_steps < 0 || ns_steps > 100) return fail(h, MUON_ERR_INVALID_ARG, "ns_steps must be in [0, 100]");
  muon_step_options_t o{};
  o.update_rms = 0.2f;
  o.extra_scale = 1.0f;
  std::vector<Block> blocks;
  const muon_status_t st = build_blocks(h, params, n_params, o, false, &blocks);
  if (st != MUON_OK) return st;
  // the same grouping and chunking muon_step plans (for MUON_NS_AUTO: the
  // larger of its two calls)
  const bool tc = ns_dtype == MUON_BF16;
  auto need_of = [&](const std::vector<Block>& bl, bool gram) {
    std::map<std::pair<int, int>, GroupPlan> groups;
    for (size_t i = 0; i < bl.size(); ++i) {
      GroupPlan& g = groups[{bl[i].m, bl[i].n}];
      g.m = bl[i].m;
      g.n = bl[i].n;
      g.members.push_back(static_cast<int>(i));
    }
    const bool overlap = h->overlap && tc && !gram && ns_steps > 0;
    size_t need = 0;
    for (auto& kv : groups)
      need = std::max(need, plan_group(h, kv.second, tc, gram, ns_steps, overlap ? h->ws_limit / 2 : h->ws_limit));
    const size_t conc_need = concurrent_need(h, groups, tc, gram, ns_steps, overlap);
    if (conc_need > 0) need = conc_need;
    return (overlap && need > 0) ? 2 * align_up(need, 256) : need;
  };
  if (ns_method == MUON_NS_AUTO) {
    std::vector<Block> standard, gram;
    for (const Block& b : blocks) (auto_gram(b, tc) ? gram : standard).push_back(b);
    *bytes = std::max(need_of(standard, false), need_of(gram, true));
  } else {
    *bytes = need_of(blocks, ns_method == MUON_NS_GRAM);
  }
  return MUON_OK;
}

muon_status_t muon_step_ex(muon_handle_t h, const muon_param_t* params, int32_t n_params,
                           const muon_step_options_t* opts, void* stream) {
  if (h == nullptr) return MUON_ERR_INVALID_ARG;
  if (opts == nullptr) return fail(h, MUON_ERR_INVALID_ARG, "opts is NULL");
  const muon_step_options_t o = *opts;
  if (n_params < 0) return fail(h, MUON_ERR_INVALID_ARG, "n_params < 0");
  if (n_params > 0 && params == nullptr) return fail(h, MUON_ERR_INVALID_ARG, "params is NULL");
  if (!valid_dtype(o.ns_dtype)) return fail(h, MUON_ERR_INVALID_ARG, "ns_dtype must be MUON_F32 or MUON_BF16");
  if (!valid_method(o.ns_method)) return fail(h, MUON_ERR_INVALID_ARG, "unknown ns_method");
  if (o.ns_steps < 0 || o.ns_steps > 100) return fail(h, MUON_ERR_INVALID_ARG, "ns_steps must be in [0, 100]");
  if (o.scale_mode != MUON_SCALE_RMS && o.scale_mode != MUON_SCALE_MUP)
    return fail(h, MUON_ERR_INVALID_ARG, "unknown scale_mode");
  if (o.coeffs_per_step != 0 && o.coeffs_per_step != 1)
    return fail(h, MUON_ERR_INVALID_ARG, "coeffs_per_step must be 0 or 1");
  if (o.coeffs_per_step && o.coeffs == nullptr && o.ns_steps > 0)
    return fail(h, MUON_ERR_INVALID_ARG, "a coefficient schedule needs coeffs");
  if (o.coeffs != nullptr) {
    const int nc = 3 * (o.coeffs_per_step ? o.ns_steps : 1);
    for (int k = 0; k < nc; ++k)
      if (!std::isfinite(o.coeffs[k])) return fail(h, MUON_ERR_INVALID_ARG, "non-finite coefficient");
  }
  if (!std::isfinite(o.lr) || !std::isfinite(o.wd) || !std::isfinite(o.mu) || !std::isfinite(o.update_rms) ||
      !std::isfinite(o.extra_scale))
    return fail(h, MUON_ERR_INVALID_ARG, "non-finite hyper-parameter");
  std::vector<Block> blocks;
  const muon_status_t bst = build_blocks(h, params, n_params, o, true, &blocks);
  if (bst != MUON_OK) return bst;
  if (blocks.empty()) return MUON_OK;
  DeviceGuard guard(h->device);
  const float* cf = o.coeffs ? o.coeffs : kDefaultCoeffs;
  return run_method(h, blocks, o.mu, o.nesterov ? 1 : 0, o.ns_steps, cf, o.coeffs_per_step ? 3 : 0, o.ns_method,
                    o.ns_dtype == MUON_BF16, static_cast<cudaStream_t>(stream));
}

muon_status_t muon_step(muon_handle_t h, const muon_param_t* params, int32_t n_params, float lr, float wd,
                        float mu, int32_t nesterov, int32_t ns_method, int32_t ns_steps, const float* coeffs,
                        float update_rms, int32_t ns_dtype, void* stream) {
  muon_step_options_t o{};
  o.lr = lr;
  o.wd = wd;
  o.mu = mu;
  o.nesterov = nesterov;
  o.ns_method = ns_method;
  o.ns_steps = ns_steps;
  o.coeffs = coeffs;
  o.ns_dtype = ns_dtype;
  o.scale_mode = MUON_SCALE_RMS;
  o.update_rms = update_rms;
  o.extra_scale = 1.0f;
  o.coeffs_per_step = 0;
  return muon_step_ex(h, params, n_params, &o, stream);
}

muon_status_t adamw_step(muon_handle_t h, void* const* params, const void* const* grads, float* const* exp_avg,
                         float* const* exp_avg_sq, const int64_t* numel, const int32_t* param_dtypes,
                         const int32_t* grad_dtypes, int32_t n, int64_t step, float lr, float beta1, float beta2,
                         float eps, float wd, void* stream_arg) {
  if (h == nullptr) return MUON_ERR_INVALID_ARG;
  if (n < 0) return fail(h, MUON_ERR_INVALID_ARG, "n < 0");
  if (n == 0) return MUON_OK;
  if (params == nullptr || grads == nullptr || exp_avg == nullptr || exp_avg_sq == nullptr || numel == nullptr ||
      param_dtypes == nullptr || grad_dtypes == nullptr)
    return fail(h, MUON_ERR_INVALID_ARG, "NULL array");
  if (step < 1) return fail(h, MUON_ERR_INVALID_ARG, "step counts from 1");
  if (!(beta1 >= 0.f && beta1 < 1.f && beta2 >= 0.f && beta2 < 1.f) || !std::isfinite(lr) || !std::isfinite(eps) ||
      !std::isfinite(wd))
    return fail(h, MUON_ERR_INVALID_ARG, "bad hyper-parameter");
  std::vector<AdamTensor> tensors;
  std::vector<AdamChunk> chunks;
  for (int32_t i = 0; i < n; ++i) {
    if (numel[i] < 0) return fail(h, MUON_ERR_INVALID_ARG, "negative numel");
    if (!valid_dtype(param_dtypes[i]) || !valid_dtype(grad_dtypes[i]))
      return fail(h, MUON_ERR_INVALID_ARG, "bad dtype");
    if (numel[i] == 0) continue;
    if (params[i] == nullptr || grads[i] == nullptr || exp_avg[i] == nullptr || exp_avg_sq[i] == nullptr)
      return fail(h, MUON_ERR_INVALID_ARG, "NULL tensor pointer");
    const int ti = static_cast<int>(tensors.size());
    tensors.push_back(AdamTensor{params[i], grads[i], exp_avg[i], exp_avg_sq[i], numel[i], param_dtypes[i],
                                 grad_dtypes[i]});
    for (int64_t off = 0; off < numel[i]; off += ADAM_CHUNK) chunks.push_back(AdamChunk{ti, 0, off});
  }
  if (chunks.empty()) return MUON_OK;
  DeviceGuard guard(h->device);
  std::vector<uint8_t> arena;
  const size_t to = arena_push(arena, tensors.data(), tensors.size());
  const size_t co = arena_push(arena, chunks.data(), chunks.size());
  void* dev = nullptr;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_arg);
  h->prof_tag = -1;
  muon_status_t st = upload(h, arena, stream, &dev);
  if (st != MUON_OK) return st;
  const double bc1 = 1.0 - std::pow(static_cast<double>(beta1), static_cast<double>(step));
  const double bc2 = 1.0 - std::pow(static_cast<double>(beta2), static_cast<double>(step));
  AdamParams p{};
  p.tensors = reinterpret_cast<const AdamTensor*>(static_cast<uint8_t*>(dev) + to);
  p.chunks = reinterpret_cast<const AdamChunk*>(static_cast<uint8_t*>(dev) + co);
  p.beta1 = beta1;
  p.beta2 = beta2;
  p.eps = eps;
  p.decay = static_cast<float>(1.0 - static_cast<double>(lr) * wd);
  p.step_size = static_cast<float>(static_cast<double>(lr) * std::sqrt(bc2) / bc1);
  MUON_LAUNCH(MUON_K_ADAMW, launch_adamw(p, static_cast<int>(chunks.size()), stream), "adamw launch");
  return MUON_OK;
}

muon_status_t muon_handle_set_profiling(muon_handle_t h, int32_t enable) {
  if (h == nullptr) return MUON_ERR_INVALID_ARG;
  h->profiling = enable != 0;
  h->prof_used = 0;
  return MUON_OK;
}

muon_status_t muon_handle_profile(muon_handle_t h, double* ms, int64_t* launches, int32_t n_classes) {
  if (h == nullptr || n_classes < 0 || n_classes > MUON_K_COUNT) return MUON_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  for (int32_t c = 0; c < n_classes; ++c) {
    if (ms) ms[c] = 0.0;
    if (launches) launches[c] = 0;
  }
  for (size_t i = 0; i < h->prof_used; ++i) {
    const auto& r = h->prof[i];
    MUON_CUDA_TRY(cudaEventSynchronize(r.b), "profile event wait");
    float t = 0.f;
    MUON_CUDA_TRY(cudaEventElapsedTime(&t, r.a, r.b), "profile elapsed time");
    if (r.cls < n_classes) {
      if (ms) ms[r.cls] += t;
      if (launches) launches[r.cls] += 1;
    }
  }
  h->prof_used = 0;
  return MUON_OK;
}

muon_status_t muon_handle_profile_records(muon_handle_t h, int32_t* cls, int32_t* tag, float* ms, int32_t capacity,
                                          int32_t* count) {
  if (h == nullptr || capacity < 0 || count == nullptr) return MUON_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  *count = static_cast<int32_t>(h->prof_used);
  for (size_t i = 0; i < h->prof_used; ++i) {
    const auto& r = h->prof[i];
    MUON_CUDA_TRY(cudaEventSynchronize(r.b), "profile event wait");
    float t = 0.f;
    MUON_CUDA_TRY(cudaEventElapsedTime(&t, r.a, r.b), "profile elapsed time");
    if (static_cast<int64_t>(i) < capacity) {
      if (cls) cls[i] = r.cls;
      if (tag) tag[i] = r.tag;
      if (ms) ms[i] = t;
    }
  }
  h->prof_used = 0;
  return MUON_OK;
}

muon_status_t muon_handle_launch_count(muon_handle_t h, uint64_t* count) {
  if (h == nullptr || count == nullptr) return MUON_ERR_INVALID_ARG;
  *count = h->launches;
  return MUON_OK;
}

muon_status_t muon_selftest_timeout(muon_handle_t h, uint64_t timeout_ns, void* stream) {
  if (h == nullptr || timeout_ns == 0 || timeout_ns > 10000000000ull) return MUON_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MUON_CUDA_TRY(launch_wait_selftest(timeout_ns, h->err, s), "selftest launch");
  return MUON_OK;
}

}  // extern "C"
