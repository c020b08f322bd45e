// Shared device-side helpers for the Muon kernels (sm_103a).
//
// PTX wrappers for mbarrier, TMA (cp.async.bulk.tensor), tcgen05 (MMA, TMEM
// alloc/ld/commit), a bounded barrier wait that gives up after a time limit
// and records an error instead of spinning forever, and the descriptor
// structs the host scheduler hands to the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace muon {

// ---------------------------------------------------------------- error word
// Bits OR-ed into the handle's device error word.
enum : unsigned {
  ERRBIT_TIMEOUT = 1u,     // a bounded wait ran out
  ERRBIT_NONFINITE = 2u,   // a Frobenius norm (hence an input) was NaN/Inf
};

enum DType : int { DT_F32 = 0, DT_BF16 = 1 };

// ------------------------------------------------------------ descriptors
// One matrix (or one Muon-Split row block) feeding the NS workspace.
struct SrcEntry {
  const void* g;     // gradient (or the matrix to orthogonalise), row-major
  float* mom;        // fp32 momentum buffer (same layout as g) or nullptr
  long long ld;      // row stride of g / mom in elements
  int rows, cols;    // block shape in the parameter's own orientation
  int transposed;    // 1: rows > cols, the NS works on the transpose
  int gdtype;        // DType of g
};

// Where the final Newton-Schulz result goes:
//   out = alpha * out_old + beta * O   (alpha == 0: out_old is not read)
struct OutEntry {
  void* ptr;         // parameter (or caller matrix) block, row-major
  long long ld;      // row stride in elements
  int transposed;    // 1: out[c][r] = O[r][c]
  int dtype;         // DType of ptr
  float alpha, beta;
};

// --------------------------------------------------------------- bf16 utils
__device__ __forceinline__ float bf2f(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ __nv_bfloat16 f2bf(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&t);
}

// ------------------------------------------------ lo plane as signed bytes
// The tensor-core path holds the master X as hi + lo.  x is kept to 24 bits
// (its fp32 pattern rounded at bit 8); hi = bf16(x), rounded to nearest, is
// the MMA operand, and the signed byte q = (bits(x) + 128 - (bits(hi) << 16))
// >> 8 carries the next 8 bits: (bits(hi) << 16) + (q << 8) is x's rounded
// pattern again, in integer arithmetic on the patterns (x and hi share
// their sign).  -128 <= q <= 128; q = 128 (x's 24-bit rounding falls on the
// midpoint between two bf16 values, about one value in 512) is stored as
// 127, one step short.  hi + lo keeps about 16 significant bits, as a bf16
// lo plane would, at 3 bytes per element.
// hi32 = bits(hi) << 16 (hi's fp32 pattern).
__device__ __forceinline__ int lo8_code(uint32_t xbits, uint32_t hi32) {
  const int d = static_cast<int>(xbits + 0x80u - hi32) >> 8;
  return d < 127 ? d : 127;
}
// byte k of w sign-extended and shifted left by 8 (prmt: byte 0 zero, byte
// 1 = byte k, bytes 2 and 3 replicate its sign)
__device__ __forceinline__ uint32_t lo8_shifted(uint32_t w, int k) {
  const uint32_t sel = 0x4u | (static_cast<uint32_t>(k) << 4) | ((static_cast<uint32_t>(k) | 8u) << 8) |
                       ((static_cast<uint32_t>(k) | 8u) << 12);
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(w), "r"(0u), "r"(sel));
  return d;
}
// x from hi's fp32 pattern and byte k of a word of codes
__device__ __forceinline__ float lo8_join(uint32_t hi32, uint32_t w, int k) {
  return __uint_as_float(hi32 + lo8_shifted(w, k));
}
// the low bytes of four codes into one word, code k in byte k
__device__ __forceinline__ uint32_t pack_lo8x4(int q0, int q1, int q2, int q3) {
  uint32_t t01, t23, w;
  asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(t01) : "r"(q0), "r"(q1));
  asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(t23) : "r"(q2), "r"(q3));
  asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(w) : "r"(t01), "r"(t23));
  return w;
}

__device__ __forceinline__ float load_as_f32(const void* base, long long idx, int dtype) {
  return dtype == DT_BF16 ? bf2f(reinterpret_cast<const __nv_bfloat16*>(base)[idx])
                          : reinterpret_cast<const float*>(base)[idx];
}

__device__ __forceinline__ void store_from_f32(void* base, long long idx, int dtype, float v) {
  if (dtype == DT_BF16)
    reinterpret_cast<__nv_bfloat16*>(base)[idx] = f2bf(v);
  else
    reinterpret_cast<float*>(base)[idx] = v;
}

// -------------------------------------------------------------- time / smem
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of parity `parity` of `bar` to complete.  Gives up and
// returns false when `*abort` becomes non-zero or after `timeout_ns`; the
// caller then records the error and unwinds.  Never spins unboundedly.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                  uint64_t timeout_ns) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(a, parity)) return true;
    if ((it & 31u) == 0u) {
      if (abort != nullptr && *abort) return false;
      if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
  }
}

// ------------------------------------------- programmatic dependent launch
// The library's kernels are launched with programmatic stream serialization
// (launch_k in internal.h): a kernel may be scheduled before the previous
// kernel of the stream has finished, so that its launch and prologue overlap
// that kernel's tail.  Every such kernel calls pdl_wait() before its first
// access to global memory that an earlier kernel of the stream reads or
// writes (the wait returns once the previous kernel has completed and its
// memory is visible; without the attribute it returns at once), and then
// pdl_launch_dependents(), which lets the next kernel be scheduled once every
// CTA of this grid has called it or exited.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// --------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load of one box into shared memory; completion is signalled as
// transaction bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// Makes a tensor map in global memory, written before this kernel, visible to
// this thread's later TMA operations that name it (the map is 128 bytes).
__device__ __forceinline__ void tensormap_acquire(const CUtensorMap* map) {
  asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(reinterpret_cast<uint64_t>(map))
               : "memory");
}

// Tiled bulk store shared -> global (3-D map; elements outside the tensor
// are not written), committed to this thread's bulk async-group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// every committed bulk store has finished reading its shared-memory source
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// every committed bulk store has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// orders this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses of the same memory
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ----------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem], bf16 inputs, fp32 accumulation, one CTA.
__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// Arrive once on `bar` when every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 16 consecutive fp32 columns of this warp's 32 TMEM lanes (one row per thread).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor (tcgen05 format, 128-byte swizzle).
//   start address, leading-dimension byte offset, stride-dimension byte offset
//   (all >> 4), descriptor version 1 at bit 46, swizzle mode 2 (128 B) at 61.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B, fp32 D, M x N tile.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format,
//   15 A major (0 = K), 16 B major (1 = MN), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(b_mn_major) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ------------------------------------------------------ clusters / CTA pairs
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster arrives and waits.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// shared::cluster address of the same shared-memory offset in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// TMEM allocation shared by the two CTAs of a pair: one warp of EACH CTA
// executes these collectively.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Pair MMA: A rows split 128 + 128 over the two CTAs, B's N split in halves,
// each CTA's TMEM receives its 128 rows x N.  Issued by the leader CTA only.
__device__ __forceinline__ void umma_bf16_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
// Arrive on the barrier at this offset in every CTA of `cta_mask` once the
// pair MMAs issued so far are complete.
__device__ __forceinline__ void umma_commit_pair_mc(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}
// TMA load into this CTA's shared memory whose completion is signalled on a
// barrier of the CTA pair (shared::cluster address, e.g. the leader's).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster, int x,
                                                 int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar_cluster)
      : "memory");
}

// --------------------------------------------------------------- epilogue
// Write one value of the final Newton-Schulz result to its destination:
//   dst = alpha * dst_old + beta * o   (row r, col c of the NS orientation).
__device__ __forceinline__ void store_out_scalar(const OutEntry& e, int r, int c, float o) {
  const long long idx = e.transposed ? static_cast<long long>(c) * e.ld + r : static_cast<long long>(r) * e.ld + c;
  float v = e.beta * o;
  if (e.alpha != 0.f) v = fmaf(e.alpha, load_as_f32(e.ptr, idx, e.dtype), v);
  store_from_f32(e.ptr, idx, e.dtype, v);
}

// Sixteen consecutive outputs o[0..15] of row r starting at column c0 (all
// in range).  Non-transposed destinations whose row segment is 16-byte
// aligned use vector loads and stores; everything else goes element by
// element (transposed writes are coalesced across the warp, whose lanes hold
// consecutive rows).
__device__ __forceinline__ void store_out_16(const OutEntry& e, int r, int c0, const float* o) {
  if (!e.transposed) {
    const long long idx = static_cast<long long>(r) * e.ld + c0;
    if (e.dtype == DT_BF16 && ((reinterpret_cast<uintptr_t>(reinterpret_cast<__nv_bfloat16*>(e.ptr) + idx) & 15) == 0)) {
      uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(e.ptr) + idx);
      uint4 w[2];
      if (e.alpha != 0.f) {
        w[0] = dst[0];
        w[1] = dst[1];
      }
      const __nv_bfloat162* old = reinterpret_cast<const __nv_bfloat162*>(w);
      uint4 res[2];
      uint32_t* rp = reinterpret_cast<uint32_t*>(res);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float v0 = e.beta * o[2 * k], v1 = e.beta * o[2 * k + 1];
        if (e.alpha != 0.f) {
          const float2 f = __bfloat1622float2(old[k]);
          v0 = fmaf(e.alpha, f.x, v0);
          v1 = fmaf(e.alpha, f.y, v1);
        }
        rp[k] = pack_bf16x2(v0, v1);
      }
      dst[0] = res[0];
      dst[1] = res[1];
      return;
    }
    if (e.dtype == DT_F32 && ((reinterpret_cast<uintptr_t>(reinterpret_cast<float*>(e.ptr) + idx) & 15) == 0)) {
      float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(e.ptr) + idx);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float4 v = make_float4(e.beta * o[4 * q], e.beta * o[4 * q + 1], e.beta * o[4 * q + 2], e.beta * o[4 * q + 3]);
        if (e.alpha != 0.f) {
          const float4 w = dst[q];
          v.x = fmaf(e.alpha, w.x, v.x);
          v.y = fmaf(e.alpha, w.y, v.y);
          v.z = fmaf(e.alpha, w.z, v.z);
          v.w = fmaf(e.alpha, w.w, v.w);
        }
        dst[q] = v;
      }
      return;
    }
  }
#pragma unroll
  for (int k = 0; k < 16; ++k) store_out_scalar(e, r, c0 + k, o[k]);
}

}  // namespace muon
