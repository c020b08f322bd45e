// Device code shared by the one-CTA (kernels_tc.cu) and CTA-pair
// (kernels_tc2.cu) tensor-core Newton-Schulz GEMMs: tile constants, bounded
// warp-wide waits, tile decoding and the epilogues of every mode.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace muon {
namespace tc {

constexpr int BM = 128;
constexpr int BK = 64;                    // bf16 elements in one 128-byte swizzle row
constexpr int EPI_WARPS = 8;                           // two per TMEM lane quadrant
constexpr int TC_THREADS = 64 + 32 * EPI_WARPS;        // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue
constexpr int BOX_BYTES = 64 * 64 * 2;    // one 64 x 64 bf16 TMA box
constexpr int MAX_DYN_SMEM = 232448;      // 227 KB opt-in dynamic shared memory per CTA
constexpr unsigned long long DRAIN_NS = 1000000000ull;


template <int MODE>
struct ModeTraits {
  static constexpr bool kSym = (MODE == MODE_SYRK || MODE == MODE_POLY || MODE == MODE_G_R0 ||
                                MODE == MODE_G_P || MODE == MODE_G_PROD || MODE == MODE_F_SYRK ||
                                MODE == MODE_F_POLY);
  static constexpr bool kMN =
      (MODE == MODE_UPDATE || MODE == MODE_FINAL || MODE == MODE_G_FINAL || MODE == MODE_FINAL_T ||
       MODE == MODE_G_FINAL_T || MODE == MODE_F_UPDATE || MODE == MODE_F_FINAL);
  static constexpr bool kTmaOut = (MODE == MODE_FINAL_T || MODE == MODE_G_FINAL_T);   // destinations by TMA
  static constexpr bool kKn = (MODE == MODE_SYRK || MODE == MODE_G_R0 || MODE == MODE_F_SYRK);   // K = n (else K = m)
  static constexpr bool kPlanesOut = (MODE == MODE_G_R0 || MODE == MODE_G_P || MODE == MODE_G_PROD);
  // bf16 planes each output value is stored as (symmetric products and F_UPDATE)
  static constexpr int kOutPlanes =
      kPlanesOut ? 2 : (MODE == MODE_F_SYRK || MODE == MODE_F_POLY || MODE == MODE_F_UPDATE) ? 3 : 1;
  static constexpr bool kF32 = (MODE == MODE_F_SYRK || MODE == MODE_F_POLY || MODE == MODE_F_UPDATE ||
                                MODE == MODE_F_FINAL);
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

// The fp32 tensor-core modes accumulate the even and the odd K steps of a
// tile in two TMEM accumulators, BN columns apart, and the epilogue adds
// them in fp32: the tensor core's fp32 accumulation loses accuracy along K
// (the fp32 path's error grew with K = m), and each half accumulates half
// the steps.  Every other mode keeps one accumulator per tile.
template <int MODE>
struct AccParts {
  static constexpr int v = ModeTraits<MODE>::kF32 ? 2 : 1;
};

// 16 columns of a tile's accumulator at `taddr`: the sum of its parts
// (`two`: the K loop had at least two steps, so the second part was written).
template <int MODE, int BN>
__device__ __forceinline__ void acc_ld16(uint32_t taddr, float* v, bool two) {
  tmem_ld16(taddr, v);
  if constexpr (AccParts<MODE>::v == 2) {
    if (two) {
      float w[16];
      tmem_ld16(taddr + static_cast<uint32_t>(BN), w);
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] += w[e];
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

// ------------------------------------------- UPDATE / FINAL / G_FINAL epilogue
// The master X of the tensor-core path is held as two planes, X = hi + lo:
// hi = bf16(X) is the MMA operand copy itself, lo a signed byte with the
// next 8 bits of X's pattern (lo8_code), about 16 significant bits in all at
// 3 bytes per element.  Each epilogue warp owns 32 rows (its TMEM
// lane quadrant) and half of the tile's columns, which it walks in 32 x 32
// blocks.  Per warp, in shared memory, SLOTS slots (3 KB for UPDATE, 4 KB
// for FINAL):
//   UPDATE / FINAL: [hi 32 x 32 bf16, 64-byte rows with 64-byte swizzle |
//   lo 32 x 32 codes, 32-byte rows with 32-byte swizzle], loaded by TMA up
//   to SLOTS blocks ahead (across tile boundaries) so the loads overlap the
//   main loop.  UPDATE writes the new hi and lo back in place and stores
//   both with TMA (hi to the other operand buffer, lo in place).
//   FINAL / G_FINAL: after the block's inputs are in registers the slot is
//   reused as 32 x 32 fp32 (128-byte rows, 128-byte swizzle) holding the
//   result in destination orientation (transposed when the destination is
//   out[c][r]), then written out as 16-byte row segments, eight lanes per
//   destination row.
//   FINAL_T (bf16 destinations with tensor maps): [hi | lo | W] (5 KB), W the
//   destination's 32 x 32 block in destination orientation, loaded by TMA
//   with hi and lo, updated in place and stored back by TMA; G_FINAL_T: [W].
//   F_UPDATE (fp32 tensor-core path): no inputs; the result's three bf16
//   planes leave by TMA through the slot, two 32 x 32 planes at a time.
//   F_FINAL: as G_FINAL.
// With the swizzles, one lane per row accessing 16-byte chunks of its row,
// and eight lanes covering one row, are free of bank conflicts.
template <int MODE, int XSLOTS = 2>
struct EpiLayout {
  static constexpr bool kMN = ModeTraits<MODE>::kMN;
  static constexpr bool kLoadX = (MODE == MODE_UPDATE || MODE == MODE_FINAL || MODE == MODE_FINAL_T);
  static constexpr bool kFill = kLoadX || ModeTraits<MODE>::kTmaOut;   // slots filled by TMA
  static constexpr int SLOTS = kFill ? XSLOTS : 1;         // input blocks in flight per warp
  static constexpr int X_BYTES = 3072;                // a block of the master: hi (2 KB) + lo codes (1 KB)
  static constexpr int SLOT_BYTES =
      MODE == MODE_FINAL_T ? 5120 : MODE == MODE_G_FINAL_T ? 2048 : MODE == MODE_UPDATE ? X_BYTES : 4096;
  static constexpr int LO_OFF = 2048;                 // lo codes (F_UPDATE: second plane) within a slot
  static constexpr int W_OFF = MODE == MODE_G_FINAL_T ? 0 : X_BYTES;   // destination block within a slot
  static constexpr int WARP_BYTES = SLOTS * SLOT_BYTES;   // a multiple of 1024
  static constexpr int BYTES = kMN ? EPI_WARPS * WARP_BYTES : 0;
};

// byte offset of 16-byte chunk q of row r: 128-byte rows, 128-byte swizzle
__device__ __forceinline__ uint32_t sw128_off(int r, int q) {
  return static_cast<uint32_t>(r * 128 + ((q ^ (r & 7)) << 4));
}
// byte offset of 16-byte chunk q of row r: 64-byte rows, 64-byte swizzle
__device__ __forceinline__ uint32_t sw64_off(int r, int q) {
  return static_cast<uint32_t>(r * 64 + ((q ^ ((r >> 1) & 3)) << 4));
}
// byte offset of 16-byte chunk q of row r: 32-byte rows, 32-byte swizzle
__device__ __forceinline__ uint32_t sw32_off(int r, int q) {
  return static_cast<uint32_t>(r * 32 + ((q ^ ((r >> 2) & 1)) << 4));
}
// hi patterns (fp32 bits) of 8 bf16 values, and the 8 values x = hi + lo
// joined with their codes, the elements 8 * (g & 1) .. + 7 of a 16-code chunk
__device__ __forceinline__ void lo8_unpack8(const uint4& hraw, const uint4& codes, int g, uint32_t* hi32, float* x) {
  const uint32_t hw[4] = {hraw.x, hraw.y, hraw.z, hraw.w};
  const uint32_t w0 = (g & 1) ? codes.z : codes.x;
  const uint32_t w1 = (g & 1) ? codes.w : codes.y;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    hi32[2 * e] = hw[e] << 16;
    hi32[2 * e + 1] = hw[e] & 0xFFFF0000u;
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    x[e] = lo8_join(hi32[e], w0, e);
    x[4 + e] = lo8_join(hi32[4 + e], w1, e);
  }
}
// byte offset of bf16 element (r, c) of a 32 x 32 block, 64-byte rows, 64-byte swizzle
__device__ __forceinline__ uint32_t sw64_elem(int r, int c) { return sw64_off(r, c >> 3) + 2u * (c & 7); }

__device__ __forceinline__ void unpack8(const uint4& raw, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 t = __bfloat1622float2(h[k]);
    f[2 * k] = t.x;
    f[2 * k + 1] = t.y;
  }
}

// out[r][c0 .. c0+3] = alpha * out + beta * o (not transposed, r < m, c0 < n)
__device__ __forceinline__ void store_out_4(const OutEntry& e, int r, int c0, int n, float4 o, float4 old) {
  const long long idx = static_cast<long long>(r) * e.ld + c0;
  const float ov[4] = {o.x, o.y, o.z, o.w};
  const float wv[4] = {old.x, old.y, old.z, old.w};
  float v[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) v[k] = fmaf(e.alpha, wv[k], e.beta * ov[k]);
  if (c0 + 3 < n) {
    if (e.dtype == DT_BF16) {
      __nv_bfloat16* q = reinterpret_cast<__nv_bfloat16*>(e.ptr) + idx;
      if ((reinterpret_cast<uintptr_t>(q) & 7) == 0) {
        *reinterpret_cast<uint2*>(q) = make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
        return;
      }
    } else {
      float* q = reinterpret_cast<float*>(e.ptr) + idx;
      if ((reinterpret_cast<uintptr_t>(q) & 15) == 0) {
        *reinterpret_cast<float4*>(q) = make_float4(v[0], v[1], v[2], v[3]);
        return;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (c0 + k < n) store_from_f32(e.ptr, idx + k, e.dtype, v[k]);
}

// The old destination values matching store_out_4, as raw bits so that the
// load can be issued well before its use: a 16-byte-aligned fp32 segment or
// an 8-byte-aligned bf16 segment is loaded whole (decode_out_4 converts it);
// anything else (ragged, misaligned) element by element, already as floats.
// Zeros when alpha == 0.
__device__ __forceinline__ bool out4_vec(const OutEntry& e, long long idx, int c0, int n) {
  if (c0 + 3 >= n) return false;
  const uintptr_t a = e.dtype == DT_BF16 ? reinterpret_cast<uintptr_t>(reinterpret_cast<const __nv_bfloat16*>(e.ptr) + idx)
                                         : reinterpret_cast<uintptr_t>(reinterpret_cast<const float*>(e.ptr) + idx);
  return (a & (e.dtype == DT_BF16 ? 7u : 15u)) == 0;
}

__device__ __forceinline__ uint4 load_out_4_raw(const OutEntry& e, int r, int c0, int n) {
  uint4 w = make_uint4(0u, 0u, 0u, 0u);
  if (e.alpha == 0.f) return w;
  const long long idx = static_cast<long long>(r) * e.ld + c0;
  if (out4_vec(e, idx, c0, n)) {
    if (e.dtype == DT_BF16) {
      const uint2 raw = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(e.ptr) + idx);
      w.x = raw.x;
      w.y = raw.y;
    } else {
      w = *reinterpret_cast<const uint4*>(reinterpret_cast<const float*>(e.ptr) + idx);
    }
    return w;
  }
  float t[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (c0 + k < n) t[k] = load_as_f32(e.ptr, idx + k, e.dtype);
  return make_uint4(__float_as_uint(t[0]), __float_as_uint(t[1]), __float_as_uint(t[2]), __float_as_uint(t[3]));
}

__device__ __forceinline__ float4 decode_out_4(const OutEntry& e, int r, int c0, int n, uint4 w) {
  if (e.alpha != 0.f && e.dtype == DT_BF16 && out4_vec(e, static_cast<long long>(r) * e.ld + c0, c0, n)) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
  return make_float4(__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z), __uint_as_float(w.w));
}

// One 32 x 32 destination block of a FINAL / G_FINAL warp: destination rows
// drow0 .. drow0+31 (< dlim), columns dcol0 .. dcol0+31 (< dcols); lane
// (rq = lane / 8, q = lane % 8) covers row 4 it + rq, columns 4q .. 4q+3.
struct OutBlock {
  OutEntry e;          // row-wise view of the destination (transposition folded into drow0 / dcol0)
  int drow0, dlim, dcol0, dcols;
};

__device__ __forceinline__ OutBlock out_block(const OutEntry& oe, int row0, int gcb, int m, int n) {
  const bool tr = oe.transposed != 0;
  OutBlock o;
  o.e = OutEntry{oe.ptr, oe.ld, 0, oe.dtype, oe.alpha, oe.beta};
  o.drow0 = tr ? gcb : row0;
  o.dlim = tr ? n : m;
  o.dcol0 = tr ? row0 : gcb;
  o.dcols = tr ? m : n;
  return o;
}

__device__ __forceinline__ void prefetch_out_block(const OutBlock& o, int lane, uint4* w) {
  const int rq = lane >> 3, q = lane & 7;
  const bool colok = o.dcol0 + 4 * q < o.dcols;
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int r = 4 * it + rq;
    w[it] = (o.drow0 + r < o.dlim && colok) ? load_out_4_raw(o.e, o.drow0 + r, o.dcol0 + 4 * q, o.dcols)
                                            : make_uint4(0u, 0u, 0u, 0u);
  }
}

// Where an epilogue warp's tiles are and whom it tells that the accumulator
// is free again: tiles t0, t0 + tstep, ...; tile row block i covers rows
// i * TROWS + row_off .. + 127 of this CTA; one-CTA kernel: the local
// "tmem empty" barrier; CTA pair: the leader's, at cluster addresses.
struct EpiTiles {
  int t0, tstep, row_off;
  bool remote;
  uint64_t* tempty;                 // local barriers (remote == false)
  uint32_t tempty_remote[2];        // leader's barriers (remote == true)
};

// The whole tile loop of one epilogue warp for the UPDATE / FINAL / G_FINAL
// modes.  wbuf: this warp's WARP_BYTES of shared memory (1024-aligned);
// xfull: this warp's SLOTS barriers.  Maps (3-D, 32 x 32 bf16 boxes, 64-byte
// swizzle): map_xh = hi plane read this iteration (the B operand), map_xl =
// lo plane (read and written in place), map_xo = hi plane written for the
// next iteration.  On return (also after a timeout, already recorded) the
// warp's loads have landed and its stores have completed.
template <int MODE, int BN, int TROWS, int XSLOTS>
__device__ __forceinline__ void mn_epilogue(const NsGemmParams& p, const CUtensorMap* map_xh,
                                            const CUtensorMap* map_xl, const CUtensorMap* map_xo, uint8_t* wbuf,
                                            uint64_t* xfull, uint64_t* tfull, const EpiTiles& et, volatile int* abort,
                                            uint32_t tmem_base, int warp, int lane) {
  using L = EpiLayout<MODE, XSLOTS>;
  constexpr int NB = BN / 64;                          // 32-column blocks per warp per tile
  const int quad = warp & 3;
  const int cbeg = ((warp - 2) >> 2) * (BN / 2);
  const uint32_t wsm = smem_u32(wbuf);
  const bool two_parts = ((ModeTraits<MODE>::kKn ? p.n : p.m) + BK - 1) / BK >= 2;

  // ---- input prefetch, in this warp's block order, at most SLOTS blocks ahead
  int pf_t = et.t0, pf_blk = 0;
  uint32_t issued = 0, done = 0;
  int wmap_b = -1;                 // FINAL_T: the last matrix whose tensor map lane 0 acquired
  auto issue_next = [&]() {
    while (pf_t < p.num_tiles) {
      int b, i, j;
      decode_tile<MODE>(p, pf_t, b, i, j);
      const int g0 = j * BN + cbeg;
      const int nb = g0 >= p.n ? 0 : min(NB, (p.n - g0 + 31) >> 5);
      if (pf_blk < nb) {
        if (lane == 0) {
          const int slot = static_cast<int>(issued % L::SLOTS);
          const uint32_t dst = wsm + slot * L::SLOT_BYTES;
          const int x = g0 + 32 * pf_blk, y = i * TROWS + et.row_off + quad * 32;
          if constexpr (ModeTraits<MODE>::kTmaOut) {
            // the destination block too (unless alpha = 0: nothing to read)
            const OutEntry& oe = p.out[b];
            const bool wread = oe.alpha != 0.f;
            if (b != wmap_b) {
              tensormap_acquire(&p.wmap[b]);
              wmap_b = b;
            }
            mbar_arrive_expect_tx(&xfull[slot], wread ? L::SLOT_BYTES : L::W_OFF);
            if (L::kLoadX) {
              tma_load_3d(dst, map_xh, &xfull[slot], x, y, b);
              tma_load_3d(dst + L::LO_OFF, map_xl, &xfull[slot], x, y, b);
            }
            if (wread) {
              const bool tr = oe.transposed != 0;
              tma_load_3d(dst + L::W_OFF, &p.wmap[b], &xfull[slot], tr ? y : x, tr ? x : y, 0);
            }
          } else {
            mbar_arrive_expect_tx(&xfull[slot], L::X_BYTES);
            tma_load_3d(dst, map_xh, &xfull[slot], x, y, b);
            tma_load_3d(dst + L::LO_OFF, map_xl, &xfull[slot], x, y, b);
          }
        }
        ++issued;
        ++pf_blk;
        return;
      }
      pf_t += et.tstep;
      pf_blk = 0;
    }
  };
  if (L::kFill) {
#pragma unroll
    for (int k = 0; k < L::SLOTS; ++k) issue_next();
  }

  bool ok = true;
  int acc = 0;
  uint32_t acc_ph = 0;
  uint4 wpre[8];                        // FINAL / G_FINAL: old destination values of the next block
  for (int t = et.t0; t < p.num_tiles; t += et.tstep) {
    int b, i, j;
    decode_tile<MODE>(p, t, b, i, j);
    if (MODE == MODE_FINAL || MODE == MODE_G_FINAL || MODE == MODE_F_FINAL) {
      // the tile's first block of old destination values, under the main loop
      const int g0p = j * BN + cbeg;
      if (g0p < p.n) prefetch_out_block(out_block(p.out[b], i * TROWS + et.row_off + quad * 32, g0p, p.m, p.n), lane, wpre);
    }
    if (!mbar_wait_warp(&tfull[acc], acc_ph, abort, p.timeout_ns)) {
      if (lane == 0) raise_timeout(abort, p.err);
      ok = false;
      break;
    }
    tc_fence_after();
    const int row0 = i * TROWS + et.row_off + quad * 32;
    const int gr = row0 + lane;
    // the first iteration's 1 / ||U||_F: UPDATE / FINAL / FINAL_T take it
    // folded into P (POLY wrote s P), the other modes apply it here
    constexpr bool kFolded = (MODE == MODE_UPDATE || MODE == MODE_FINAL || MODE == MODE_FINAL_T);
    const float s = (!kFolded && p.scale != nullptr) ? p.scale[b] : 1.f;
    // exact diagonal term: acc + P_rr x - P^_rr hi, hi being the operand copy
    // whose product with the rounded diagonal P^_rr the accumulator holds
    float pd = 0.f, pdb = 0.f;
    if (L::kLoadX && gr < p.m) {
      pd = p.pdiag[static_cast<size_t>(b) * p.m + gr];
      pdb = bf2f(f2bf(pd));
    }
    OutEntry oe{};
    if (MODE != MODE_UPDATE && MODE != MODE_F_UPDATE) oe = p.out[b];
    const uint32_t tb = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                        static_cast<uint32_t>(acc * BN * AccParts<MODE>::v + cbeg);
    const int g0 = j * BN + cbeg;
    const int nb = g0 >= p.n ? 0 : min(NB, (p.n - g0 + 31) >> 5);
#pragma unroll 1
    for (int k = 0; k < nb; ++k) {
      const int gcb = g0 + 32 * k;
      const int slot = L::kFill ? static_cast<int>(done % L::SLOTS) : 0;
      uint8_t* sbuf = wbuf + slot * L::SLOT_BYTES;
      if (L::kFill && !mbar_wait_warp(&xfull[slot], (done / L::SLOTS) & 1u, abort, p.timeout_ns)) {
        if (lane == 0) raise_timeout(abort, p.err);
        ok = false;
        break;
      }
      if constexpr (MODE == MODE_UPDATE) {
#pragma unroll
        for (int h = 0; h < 32; h += 16) {
          float v[16];
          acc_ld16<MODE, BN>(tb + static_cast<uint32_t>(32 * k + h), v, two_parts);
          uint4* pl = reinterpret_cast<uint4*>(sbuf + L::LO_OFF + sw32_off(lane, h >> 4));
          const uint4 codes = *pl;
          uint32_t nc[4];
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint4* ph = reinterpret_cast<uint4*>(sbuf + sw64_off(lane, (h >> 3) + q));
            uint32_t hi32[8];
            float x[8], o[8];
            lo8_unpack8(*ph, codes, q, hi32, x);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              o[e] = s * fmaf(pd, x[e], fmaf(-pdb, __uint_as_float(hi32[e]), v[8 * q + e]));
            uint4 nh;
            uint32_t* wh = reinterpret_cast<uint32_t*>(&nh);
            int qc[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(o[2 * e], o[2 * e + 1]);
              const uint32_t hw = *reinterpret_cast<const uint32_t*>(&h2);
              wh[e] = hw;
              qc[2 * e] = lo8_code(__float_as_uint(o[2 * e]), hw << 16);
              qc[2 * e + 1] = lo8_code(__float_as_uint(o[2 * e + 1]), hw & 0xFFFF0000u);
            }
            nc[2 * q] = pack_lo8x4(qc[0], qc[1], qc[2], qc[3]);
            nc[2 * q + 1] = pack_lo8x4(qc[4], qc[5], qc[6], qc[7]);
            *ph = nh;
          }
          *pl = make_uint4(nc[0], nc[1], nc[2], nc[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && row0 < p.m) {   // rows past m: nothing to store
          const uint32_t src = wsm + slot * L::SLOT_BYTES;
          tma_store_3d(map_xo, src, gcb, row0, b);
          tma_store_3d(map_xl, src + L::LO_OFF, gcb, row0, b);
          bulk_commit_group();
          bulk_wait_read_all();          // the slot may be refilled
        }
        __syncwarp();
      } else if constexpr (MODE == MODE_F_UPDATE) {
        // X' = s * acc as three bf16 planes p0 + p1 + p2, stored by TMA:
        // p0 and p1 through the slot's two halves, then p2 through the first
        float v[32];
        acc_ld16<MODE, BN>(tb + static_cast<uint32_t>(32 * k), v, two_parts);
        acc_ld16<MODE, BN>(tb + static_cast<uint32_t>(32 * k + 16), v + 16, two_parts);
        uint32_t w0[16], w1[16], w2[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float x0 = s * v[2 * e], x1 = s * v[2 * e + 1];
          const __nv_bfloat162 h0 = __floats2bfloat162_rn(x0, x1);
          const float2 f0 = __bfloat1622float2(h0);
          const float r0 = x0 - f0.x, r1 = x1 - f0.y;
          const __nv_bfloat162 h1 = __floats2bfloat162_rn(r0, r1);
          const float2 f1 = __bfloat1622float2(h1);
          w0[e] = *reinterpret_cast<const uint32_t*>(&h0);
          w1[e] = *reinterpret_cast<const uint32_t*>(&h1);
          w2[e] = pack_bf16x2(r0 - f1.x, r1 - f1.y);
        }
        const uint32_t src = wsm;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          *reinterpret_cast<uint4*>(sbuf + sw64_off(lane, q)) = make_uint4(w0[4 * q], w0[4 * q + 1], w0[4 * q + 2], w0[4 * q + 3]);
          *reinterpret_cast<uint4*>(sbuf + L::LO_OFF + sw64_off(lane, q)) =
              make_uint4(w1[4 * q], w1[4 * q + 1], w1[4 * q + 2], w1[4 * q + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && row0 < p.m) {
          tma_store_3d(map_xh, src, gcb, row0, b);
          tma_store_3d(map_xl, src + L::LO_OFF, gcb, row0, b);
          bulk_commit_group();
          bulk_wait_read_all();          // the first half may be rewritten
        }
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(sbuf + sw64_off(lane, q)) = make_uint4(w2[4 * q], w2[4 * q + 1], w2[4 * q + 2], w2[4 * q + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && row0 < p.m) {
          tma_store_3d(map_xo, src, gcb, row0, b);
          bulk_commit_group();
          bulk_wait_read_all();          // the slot is free for the next block
        }
        __syncwarp();
      } else if constexpr (ModeTraits<MODE>::kTmaOut) {
        // the block's correction terms (FINAL_T) into registers; the
        // destination block (destination orientation) is updated in place in
        // the slot: W = alpha W + beta O, rounded once to bf16, then stored
        // by TMA
        float corr[32];
        if constexpr (L::kLoadX) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t hi32[8];
            float x[8];
            lo8_unpack8(*reinterpret_cast<const uint4*>(sbuf + sw64_off(lane, q)),
                        *reinterpret_cast<const uint4*>(sbuf + L::LO_OFF + sw32_off(lane, q >> 1)), q, hi32, x);
#pragma unroll
            for (int e = 0; e < 8; ++e) corr[8 * q + e] = fmaf(pd, x[e], -pdb * __uint_as_float(hi32[e]));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) corr[e] = 0.f;
        }
        const bool tr = oe.transposed != 0;
        const bool wread = oe.alpha != 0.f;
        uint8_t* wsl = sbuf + L::W_OFF;
#pragma unroll
        for (int h = 0; h < 32; h += 16) {
          float v[16];
          acc_ld16<MODE, BN>(tb + static_cast<uint32_t>(32 * k + h), v, two_parts);
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = s * (v[e] + corr[h + e]);
          if (tr) {
            // destination row = block column c, column = block row (this lane)
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              unsigned short* wp = reinterpret_cast<unsigned short*>(wsl + sw64_elem(h + e, lane));
              const float old = wread ? bf2f(__ushort_as_bfloat16(*wp)) : 0.f;
              *wp = __bfloat16_as_ushort(f2bf(fmaf(oe.alpha, old, oe.beta * v[e])));
            }
          } else {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              uint4* wq = reinterpret_cast<uint4*>(wsl + sw64_off(lane, (h >> 3) + q));
              float old[8];
              if (wread) {
                unpack8(*wq, old);
              } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) old[e] = 0.f;
              }
              uint4 nw;
              uint32_t* w32 = reinterpret_cast<uint32_t*>(&nw);
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w32[e] = pack_bf16x2(fmaf(oe.alpha, old[2 * e], oe.beta * v[8 * q + 2 * e]),
                                     fmaf(oe.alpha, old[2 * e + 1], oe.beta * v[8 * q + 2 * e + 1]));
              *wq = nw;
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && row0 < p.m) {   // a block starting past the destination stores nothing
          tma_store_3d(&p.wmap[b], wsm + slot * L::SLOT_BYTES + L::W_OFF, tr ? row0 : gcb, tr ? gcb : row0, 0);
          bulk_commit_group();
          bulk_wait_read_all();          // the slot may be refilled
        }
        __syncwarp();
      } else {
        // FINAL / G_FINAL: the block's correction terms into registers, then
        // the slot holds the fp32 result in destination orientation
        float corr[32];
        if (MODE == MODE_FINAL) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t hi32[8];
            float x[8];
            lo8_unpack8(*reinterpret_cast<const uint4*>(sbuf + sw64_off(lane, q)),
                        *reinterpret_cast<const uint4*>(sbuf + L::LO_OFF + sw32_off(lane, q >> 1)), q, hi32, x);
#pragma unroll
            for (int e = 0; e < 8; ++e) corr[8 * q + e] = fmaf(pd, x[e], -pdb * __uint_as_float(hi32[e]));
          }
          __syncwarp();                  // every lane holds its row: the slot may be overwritten
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) corr[e] = 0.f;
        }
        const bool tr = oe.transposed != 0;
#pragma unroll
        for (int h = 0; h < 32; h += 16) {
          float v[16];
          acc_ld16<MODE, BN>(tb + static_cast<uint32_t>(32 * k + h), v, two_parts);
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = s * (v[e] + corr[h + e]);
          if (tr) {
            // slot row = block column c, position = block row (this lane)
#pragma unroll
            for (int e = 0; e < 16; ++e)
              *reinterpret_cast<float*>(sbuf + sw128_off(h + e, lane >> 2) + 4 * (lane & 3)) = v[e];
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<float4*>(sbuf + sw128_off(lane, (h >> 2) + q)) =
                  make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          }
        }
        __syncwarp();                    // the block's results are in the slot
        const OutBlock ob = out_block(oe, row0, gcb, p.m, p.n);
        const int rq = lane >> 3, q = lane & 7;
        const bool colok = ob.dcol0 + 4 * q < ob.dcols;
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int r = 4 * it + rq;
          if (ob.drow0 + r < ob.dlim && colok) {
            const float4 old = decode_out_4(ob.e, ob.drow0 + r, ob.dcol0 + 4 * q, ob.dcols, wpre[it]);
            store_out_4(ob.e, ob.drow0 + r, ob.dcol0 + 4 * q, ob.dcols,
                        *reinterpret_cast<const float4*>(sbuf + sw128_off(r, q)), old);
          }
        }
        // the next block's old destination values, one block ahead
        if (k + 1 < nb) prefetch_out_block(out_block(oe, row0, gcb + 32, p.m, p.n), lane, wpre);
        fence_proxy_async_smem();        // generic accesses of the slot before its next TMA fill
        __syncwarp();
      }
      ++done;
      if (L::kFill) issue_next();
    }
    if (!ok) break;
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if (et.remote)
        mbar_arrive_cluster(et.tempty_remote[acc]);
      else
        mbar_arrive(&et.tempty[acc]);
    }
    acc ^= 1;
    if (acc == 0) acc_ph ^= 1u;
  }
  // loads still in flight land before the CTA's shared memory goes away;
  // stores complete
  if (lane == 0) {
    for (uint32_t u = done; u < issued; ++u)
      mbar_wait_bounded(&xfull[u % L::SLOTS], (u / L::SLOTS) & 1u, nullptr, DRAIN_NS);
    if (MODE == MODE_UPDATE || MODE == MODE_F_UPDATE || ModeTraits<MODE>::kTmaOut) bulk_wait_all();
  }
  __syncwarp();
}

// ------------------------------------------- symmetric-product epilogue (TMA)
// Each epilogue warp owns 32 rows and half of the tile's columns and walks
// them in 32 x 32 blocks.  A block entirely below the diagonal is skipped
// (the block above writes it as its mirror).  Per warp, 4 KB of shared
// memory: [out | mirror], two 32 x 32 bf16 blocks with 64-byte rows and
// 64-byte swizzle.  An off-diagonal block goes out at (r, c) and, through
// the mirror buffer, transposed at (c, r); a diagonal block is assembled
// symmetric in the out buffer from its c >= r half (every element written
// once, so A and P are exactly symmetric).  Both leave by TMA bulk stores,
// clipped at the m x m edge.  POLY's b*A term (G_P's b*R) reads the block's
// rows of A (both planes of R) with 16-byte loads issued one block ahead.
// Gram-method outputs leave as two planes, hi then lo, through the same
// buffers.
constexpr int SYM_WARP_BYTES = 4096;

template <int MODE>
struct SymEpi {
  static constexpr bool kTma = ModeTraits<MODE>::kSym;
  static constexpr int BYTES = kTma ? EPI_WARPS * SYM_WARP_BYTES : 0;
};


// 32 bf16 of one row from column gc (zeros at and beyond column m), raw
__device__ __forceinline__ void load_row32_bf16(const __nv_bfloat16* rowp, int gc, int m, uint4* a) {
  if (gc + 31 < m) {
#pragma unroll
    for (int q = 0; q < 4; ++q) a[q] = *reinterpret_cast<const uint4*>(rowp + gc + 8 * q);
  } else {
    uint32_t w[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float lo = gc + 2 * e < m ? bf2f(rowp[gc + 2 * e]) : 0.f;
      const float hi = gc + 2 * e + 1 < m ? bf2f(rowp[gc + 2 * e + 1]) : 0.f;
      w[e] = pack_bf16x2(lo, hi);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) a[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  }
}

// The tile loop of one epilogue warp for the symmetric products.  map_so:
// the output (A, P, or the first plane of a Gram-method or fp32-path matrix;
// bf16 [batch][m][ldm]) with 32 x 32 boxes, 64-byte swizzle; map_so_lo and
// map_so_2: the further planes of a plane-split output (the residual of the
// planes before), written after the first through the same buffers.
template <int MODE, int BN, int TROWS>
__device__ __forceinline__ void sym_epilogue(const NsGemmParams& p, const CUtensorMap* map_so,
                                             const CUtensorMap* map_so_lo, const CUtensorMap* map_so_2, uint8_t* wbuf,
                                             uint64_t* tfull, const EpiTiles& et, volatile int* abort,
                                             uint32_t tmem_base, int warp, int lane) {
  constexpr int kNP = ModeTraits<MODE>::kOutPlanes;
  // the b * A term (b * R): A's planes read back
  constexpr bool kReadIn = (MODE == MODE_POLY || MODE == MODE_G_P || MODE == MODE_F_POLY);
  constexpr int kInPlanes = MODE == MODE_G_P ? 2 : MODE == MODE_F_POLY ? 3 : 1;
  constexpr int NB = BN / 64;                          // 32-column blocks per warp per tile
  const int quad = warp & 3;
  const int cbeg = ((warp - 2) >> 2) * (BN / 2);
  const int m = p.m;
  const bool two_parts = ((ModeTraits<MODE>::kKn ? p.n : p.m) + BK - 1) / BK >= 2;
  const uint32_t out_s = smem_u32(wbuf), mir_s = out_s + 2048;
  bool pending = false;                                // a bulk store may still read the buffers
  int acc = 0;
  uint32_t acc_ph = 0;
  uint4 apre[4];                                       // POLY / G_P / F_POLY: the next block's 32 values of A
  uint4 apre_lo[4];                                    // G_P, F_POLY: of its second plane
  uint4 apre_2[4];                                     // F_POLY: of its third plane
  for (int t = et.t0; t < p.num_tiles; t += et.tstep) {
    int b, i, j;
    decode_tile<MODE>(p, t, b, i, j);
    const int row0 = i * TROWS + et.row_off + quad * 32;
    const int gr = row0 + lane;
    const int g0 = j * BN + cbeg;
    // first block of this warp that is not below the diagonal
    int k0 = 0;
    while (k0 < NB && g0 + 32 * k0 + 31 < row0) ++k0;
    const __nv_bfloat16* arow = nullptr;
    const __nv_bfloat16* arow_lo = nullptr;
    const __nv_bfloat16* arow_2 = nullptr;
    if (kReadIn) {
      const size_t roff = (static_cast<size_t>(b) * m + (gr < m ? gr : 0)) * p.ldm;
      arow = reinterpret_cast<const __nv_bfloat16*>(p.sym_in) + roff;
      if (kInPlanes >= 2) arow_lo = reinterpret_cast<const __nv_bfloat16*>(p.sym_in_lo) + roff;
      if (kInPlanes >= 3) arow_2 = reinterpret_cast<const __nv_bfloat16*>(p.sym_in_2) + roff;
      if (k0 < NB && g0 + 32 * k0 < m && gr < m) {
        load_row32_bf16(arow, g0 + 32 * k0, m, apre);
        if (kInPlanes >= 2) load_row32_bf16(arow_lo, g0 + 32 * k0, m, apre_lo);
        if (kInPlanes >= 3) load_row32_bf16(arow_2, g0 + 32 * k0, m, apre_2);
      }
    }
    if (!mbar_wait_warp(&tfull[acc], acc_ph, abort, p.timeout_ns)) {
      if (lane == 0) raise_timeout(abort, p.err);
      break;
    }
    tc_fence_after();
    float s = 1.f, s1 = 1.f;
    if (p.scale != nullptr) {
      s1 = p.scale[b];
      s = s1 * s1;                                     // SYRK / G_R0 of the first iteration: s^2 X X^T
    }
    const uint32_t tb = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                        static_cast<uint32_t>(acc * BN * AccParts<MODE>::v + cbeg);
#pragma unroll 1
    for (int k = k0; k < NB; ++k) {
      const int gcb = g0 + 32 * k;
      if (gcb >= m) break;
      float v[32];
      acc_ld16<MODE, BN>(tb + static_cast<uint32_t>(32 * k), v, two_parts);
      acc_ld16<MODE, BN>(tb + static_cast<uint32_t>(32 * k + 16), v + 16, two_parts);
      const bool diag = (gcb == row0);
      if (MODE == MODE_SYRK || MODE == MODE_G_R0 || MODE == MODE_F_SYRK) {
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c] *= s;
      } else if (kReadIn) {
        float a[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) unpack8(apre[q], a + 8 * q);
        if (kInPlanes >= 2) {
          // planes added smallest first: a = p0 + (p1 + p2)
          float al[32];
#pragma unroll
          for (int q = 0; q < 4; ++q) unpack8(apre_lo[q], al + 8 * q);
          if (kInPlanes >= 3) {
            float a2[32];
#pragma unroll
            for (int q = 0; q < 4; ++q) unpack8(apre_2[q], a2 + 8 * q);
#pragma unroll
            for (int c = 0; c < 32; ++c) al[c] += a2[c];
          }
#pragma unroll
          for (int c = 0; c < 32; ++c) a[c] += al[c];
        }
        // the next block's A, under this block's stores
        if (k + 1 < NB && gcb + 32 < m && gr < m) {
          load_row32_bf16(arow, gcb + 32, m, apre);
          if (kInPlanes >= 2) load_row32_bf16(arow_lo, gcb + 32, m, apre_lo);
          if (kInPlanes >= 3) load_row32_bf16(arow_2, gcb + 32, m, apre_2);
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c] = fmaf(p.cb, a[c], p.cc * v[c]);
        if (diag && gr < m) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c == lane) v[c] += p.ca;
        }
        if (MODE == MODE_POLY) {
          // the first iteration's s folded into P: the update reads s P
          if (p.scale != nullptr) {
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] *= s1;
          }
          if (diag && gr < m) {
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (c == lane) p.pdiag[static_cast<size_t>(b) * m + gr] = v[c];
          }
        }
      }
#pragma unroll 1
      for (int pl = 0; pl < kNP; ++pl) {
      if (pl >= 1) {
        // next plane: the rounding residual of the plane just written
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c] -= bf2f(f2bf(v[c]));
      }
      // the buffers are free once the previous bulk stores have read them
      if (lane == 0 && pending) bulk_wait_read_all();
      __syncwarp();
      if (!diag) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 pk = make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                                      pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(out_s + sw64_off(lane, q)), "r"(pk.x),
                       "r"(pk.y), "r"(pk.z), "r"(pk.w)
                       : "memory");
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const __nv_bfloat16 h = f2bf(v[c]);
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(mir_s + sw64_elem(c, lane)),
                       "h"(*reinterpret_cast<const unsigned short*>(&h))
                       : "memory");
        }
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (c >= lane) {
            const __nv_bfloat16 h = f2bf(v[c]);
            const unsigned short hb = *reinterpret_cast<const unsigned short*>(&h);
            asm volatile("st.shared.u16 [%0], %1;" ::"r"(out_s + sw64_elem(lane, c)), "h"(hb) : "memory");
            if (c > lane) asm volatile("st.shared.u16 [%0], %1;" ::"r"(out_s + sw64_elem(c, lane)), "h"(hb) : "memory");
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && row0 < m) {
        const CUtensorMap* mo = pl == 0 ? map_so : pl == 1 ? map_so_lo : map_so_2;
        tma_store_3d(mo, out_s, gcb, row0, b);
        if (!diag) tma_store_3d(mo, mir_s, row0, gcb, b);
        bulk_commit_group();
        pending = true;
      }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if (et.remote)
        mbar_arrive_cluster(et.tempty_remote[acc]);
      else
        mbar_arrive(&et.tempty[acc]);
    }
    acc ^= 1;
    if (acc == 0) acc_ph ^= 1u;
  }
  if (lane == 0) bulk_wait_all();
  __syncwarp();
}

}  // namespace tc
}  // namespace muon
