// Device code of the selected-token log-probability kernels: the arithmetic
// contract (tile partials, the fixed-order merge, the gradient formula), the
// streaming forward, the merge, the small-batch cluster forward and the
// backward.  Everything is in an anonymous namespace: each translation unit
// that includes this header instantiates what it launches (the library is
// built without relocatable device code), and has its own watchdog word.
#pragma once

#include "../../include/bil.h"
#include "device_common.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {


// ---------------------------------------------------------------------------
// The arithmetic contract.
// ---------------------------------------------------------------------------

constexpr int kGroup = 8;  // elements a lane takes at a time: 16 bytes of bf16/fp16

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Butterfly sum: every lane ends with the same value, because a + b == b + a
// bitwise at every level.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

template <int DT>
struct Elem;

template <>
struct Elem<BIL_BF16> {
  static constexpr int kBytes = 2;
  static constexpr uint32_t kNegInf = 0xff80u;  // -inf bit pattern
  __device__ static __forceinline__ float one(const unsigned char* p) {
    return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(p)) << 16);
  }
  // the two elements of a packed word, low half first (exact widening)
  __device__ static __forceinline__ void pair(uint32_t w, float& lo, float& hi) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
  }
  __device__ static __forceinline__ uint32_t max2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
  }
};

template <>
struct Elem<BIL_F16> {
  static constexpr int kBytes = 2;
  static constexpr uint32_t kNegInf = 0xfc00u;
  __device__ static __forceinline__ float one(const unsigned char* p) {
    return __half2float(*reinterpret_cast<const __half*>(p));
  }
  __device__ static __forceinline__ void pair(uint32_t w, float& lo, float& hi) {
    __half2 h = *reinterpret_cast<const __half2*>(&w);
    const float2 f = __half22float2(h);
    lo = f.x;
    hi = f.y;
  }
  __device__ static __forceinline__ uint32_t max2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
  }
};

template <>
struct Elem<BIL_F32> {
  static constexpr int kBytes = 4;
  static constexpr uint32_t kNegInf = 0xff800000u;
  __device__ static __forceinline__ float one(const unsigned char* p) {
    return *reinterpret_cast<const float*>(p);
  }
};

// contract_exp on both halves of a pair of exponents
__device__ __forceinline__ uint64_t exp2_pair(uint64_t d) {
  const uint64_t a = mul2(d, pk(kLog2e, kLog2e));
  return pk(ex2_approx(lo_of(a)), ex2_approx(hi_of(a)));
}

// Temperature: the softmax sees z = x * rcp, rcp = 1/temperature rounded to
// float32 on the host.  rcp = 1 leaves every value (and so every bit) as it is.
//
// Per-group building blocks of the tile reduction.  A group is 8 consecutive
// elements = kW 32-bit words (4 for 16-bit types, 8 for float32).
template <int DT>
struct Group {
  static constexpr int EB = Elem<DT>::kBytes;
  static constexpr int kW = EB * kGroup / 4;
  static constexpr int kVec = kW / 4;  // 16-byte vectors per group

  __device__ static __forceinline__ void load(const unsigned char* p, uint32_t (&w)[kW]) {
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      const uint4 q = *reinterpret_cast<const uint4*>(p + 16 * v);
      w[4 * v] = q.x;
      w[4 * v + 1] = q.y;
      w[4 * v + 2] = q.z;
      w[4 * v + 3] = q.w;
    }
  }
  // The group whose first element sits `off` bytes past the 16-byte aligned
  // address p (0 <= off < 16, a multiple of the element size): the kVec + 1
  // aligned vectors from p are read whole and the group's words taken out of
  // them, WOFF = off / 4 words in and then sh = 8 * (off % 4) bits down.
  // The words are those `load` reads from a 16-byte aligned copy of the group.
  // Only the first nvec vectors are read (the rest count as zero): a partial
  // group in global memory reads only the vectors that hold its elements.
  template <int WOFF>
  __device__ static __forceinline__ void load_shifted(const unsigned char* p, unsigned sh, uint32_t (&w)[kW],
                                                      int nvec = kVec + 1) {
    uint32_t v[4 * (kVec + 1)];
#pragma unroll
    for (int q = 0; q <= kVec; ++q) {
      const uint4 x = q < nvec ? *reinterpret_cast<const uint4*>(p + 16 * q) : make_uint4(0u, 0u, 0u, 0u);
      v[4 * q] = x.x;
      v[4 * q + 1] = x.y;
      v[4 * q + 2] = x.z;
      v[4 * q + 3] = x.w;
    }
#pragma unroll
    for (int j = 0; j < kW; ++j) w[j] = __funnelshift_r(v[j + WOFF], v[j + WOFF + 1], sh);
  }
  // elements j >= rem (past the vocabulary) become -inf: they cannot win the
  // max and add exp(-inf) = +0 to the sums, i.e. leave them unchanged
  __device__ static __forceinline__ void mask_tail(uint32_t (&w)[kW], int rem) {
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      if (j >= rem) {
        if (EB == 4) {
          w[j] = Elem<DT>::kNegInf;
        } else if (j & 1) {
          w[j / 2] = (w[j / 2] & 0x0000ffffu) | (Elem<DT>::kNegInf << 16);
        } else {
          w[j / 2] = (w[j / 2] & 0xffff0000u) | Elem<DT>::kNegInf;
        }
      }
    }
  }
  // running max of the stored values: packed pairs for 16-bit types, one
  // float per slot for float32
  __device__ static __forceinline__ void max_init(uint32_t (&mx)[kW]) {
#pragma unroll
    for (int i = 0; i < kW; ++i) mx[i] = EB == 4 ? Elem<DT>::kNegInf : (Elem<DT>::kNegInf * 0x10001u);
  }
  __device__ static __forceinline__ void max_acc(uint32_t (&mx)[kW], const uint32_t (&w)[kW]) {
#pragma unroll
    for (int i = 0; i < kW; ++i) {
      if constexpr (EB == 4) {
        mx[i] = __float_as_uint(fmaxf(__uint_as_float(mx[i]), __uint_as_float(w[i])));
      } else {
        mx[i] = Elem<DT>::max2(mx[i], w[i]);
      }
    }
  }
  __device__ static __forceinline__ float max_fin(const uint32_t (&mx)[kW]) {
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kW; ++i) {
      if constexpr (EB == 4) {
        m = fmaxf(m, __uint_as_float(mx[i]));
      } else {
        float lo, hi;
        Elem<DT>::pair(mx[i], lo, hi);
        m = fmaxf(m, fmaxf(lo, hi));
      }
    }
    return m;
  }
  // the pair of stored values at slots (2k, 2k+1), widened exactly
  __device__ static __forceinline__ uint64_t xpair(const uint32_t (&w)[kW], int k) {
    if constexpr (EB == 4) {
      return static_cast<uint64_t>(w[2 * k]) | (static_cast<uint64_t>(w[2 * k + 1]) << 32);
    } else {
      float lo, hi;
      Elem<DT>::pair(w[k], lo, hi);
      return pk(lo, hi);
    }
  }
  // a[k] holds the slot accumulators (a_2k, a_2k+1) of e = 2^t for the tile
  // term t = (x - shift) * c, c = rcp * log2e rounded once (rcp = 1: c =
  // log2e, so t is the exponent exp(x - shift) of the contract takes); with
  // ENT, u[k] those of e * t.  The multiply comes last: no packed multiply
  // here ever feeds an add, so the code generator has nothing to contract
  // into a fused multiply-add.
  //
  // p log p -> 0 as p -> 0: an element with z = -inf (or one masked past the
  // vocabulary, or whose t overflows) has e = 0 and t = -inf, and its entropy
  // term must be 0, not 0 * inf.  CLAMP takes max(t, -FLT_MAX) for the term,
  // which leaves every finite t as it is; without CLAMP such an element makes
  // the sum NaN, and the caller then sums the entropy terms again with it (a
  // NaN logit makes the sum NaN either way).  The bits are the same.
  template <bool ENT, bool CLAMP>
  __device__ static __forceinline__ void sum_acc(uint64_t (&a)[4], uint64_t (&u)[4], const uint32_t (&w)[kW],
                                                 uint64_t shift2, uint64_t c2) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint64_t t = mul2(sub2(xpair(w, k), shift2), c2);
      const uint64_t e = pk(ex2_approx(lo_of(t)), ex2_approx(hi_of(t)));
      a[k] = add2(a[k], e);
      if (ENT) u[k] = fma2(e, CLAMP ? pk(fmaxf(lo_of(t), kNegMax), fmaxf(hi_of(t), kNegMax)) : t, u[k]);
    }
  }
};

// Groups lane `lane` holds of a tile of `valid` elements: g = lane + 32 i.
__device__ __forceinline__ int lane_groups(int valid, int lane) {
  const int groups = (valid + kGroup - 1) / kGroup;
  return groups > lane ? (groups - lane + kLanes - 1) / kLanes : 0;
}

// One tile's float32 partial, computed by one warp: the max m of z, the sum
// s of exp(z - m) and, when asked, the entropy sum u of exp(z - m) * (z - m).
// The reduction order is fixed by the element positions alone:
//   * element p of the tile (global column t*tile_v + p) sits in group
//     g = p / 8 at slot j = p % 8; lane l takes groups l, l+32, l+64, ... in
//     increasing order; `valid` elements exist (the rest are past the
//     vocabulary and do not take part);
//   * max: exact, so its order does not matter (NaN never wins); it is taken
//     on the stored values, m_x, and the partial's max is m = m_x * rcp
//     (the max of the scaled values, since x -> x * rcp (rcp > 0) rounds
//     monotonically);
//   * sums: t = (x - m_x) * c with c = rcp * log2e, each operation rounded
//     (t = (z - m) log2 e in real arithmetic); lane accumulator a_j (slot j)
//     adds e = 2^t (ex2.approx) for its groups in increasing order; the
//     lane's sum is ((a0+a1)+(a2+a3))+((a4+a5)+(a6+a7)); the warp's sum is
//     the butterfly over lanes (xor 16, 8, 4, 2, 1); the entropy sum follows
//     the same tree with u_j = fma(e, t, u_j), and u is that sum times ln 2
//     (rounded once), i.e. sum e (z - m) in real arithmetic;
//   * a tile whose max is -inf shifts by 0 instead, so it sums to 0 (or NaN
//     if it holds a NaN) and its max stays -inf.
// Nothing here depends on the row, the kernel or the launch geometry.  Two
// implementations follow, one reading a register copy of the lane's groups
// (tiles of up to TileRegs::kMaxTile elements) and one reading shared memory
// twice (larger tiles); they perform the same operations in the same order.
struct TilePartial {
  float m, s, u;
};

__device__ __forceinline__ float tree8(const uint64_t (&a)[4]) {
  return __fadd_rn(__fadd_rn(__fadd_rn(lo_of(a[0]), hi_of(a[0])), __fadd_rn(lo_of(a[1]), hi_of(a[1]))),
                   __fadd_rn(__fadd_rn(lo_of(a[2]), hi_of(a[2])), __fadd_rn(lo_of(a[3]), hi_of(a[3]))));
}

template <bool ENT>
__device__ __forceinline__ TilePartial finish_tile(float m, const uint64_t (&a)[4], const uint64_t (&u)[4]) {
  TilePartial r;
  r.m = m;
  r.s = warp_sum(tree8(a));
  r.u = ENT ? __fmul_rn(warp_sum(tree8(u)), kLn2) : 0.0f;
  return r;
}

template <int DT>
struct TileRegs {
  static constexpr int kW = Group<DT>::kW;
  static constexpr int kMaxGroups = 64 / kW;                     // 64 registers of tile data per lane
  static constexpr int kMaxTile = kMaxGroups * kLanes * kGroup;  // 4096 (16-bit) / 2048 (float32)
  uint32_t w[kMaxGroups][kW];
};

// Group g of a tile held in memory from `tile` on.  WOFF < 0: the tile starts
// at `tile`, which is 16-byte aligned.  WOFF >= 0: `tile` is the 16-byte
// boundary below the tile's first element, which sits off = 4 * WOFF + sh / 8
// bytes past it (the memory from `tile` up to the 16-byte boundary after the
// group must be readable; bytes outside the tile only reach masked slots).
// nvec: as for Group::load_shifted (WOFF >= 0 only).
template <int DT, int WOFF>
__device__ __forceinline__ void load_group(const unsigned char* tile, int g, unsigned sh,
                                           uint32_t (&w)[Group<DT>::kW], int nvec = Group<DT>::kVec + 1) {
  const unsigned char* p = tile + static_cast<size_t>(g) * kGroup * Elem<DT>::kBytes;
  if constexpr (WOFF < 0) {
    Group<DT>::load(p, w);
  } else {
    Group<DT>::template load_shifted<WOFF>(p, sh, w, nvec);
  }
}

// FULL: the tile holds exactly TileRegs::kMaxTile valid elements, so every
// lane has kMaxGroups whole groups and no test is needed per group.  WOFF, sh:
// as for load_group.  EXACT (WOFF >= 0): a partial last group reads only the
// 16-byte vectors that hold its elements (for tiles in global memory, where
// the next vector may lie past the row's storage).
template <int DT, bool FULL, int WOFF = -1, bool EXACT = false>
__device__ __forceinline__ void tile_load_regs_t(const unsigned char* tile, int valid, int lane, TileRegs<DT>& r,
                                                 unsigned sh = 0) {
  const int ng = FULL ? TileRegs<DT>::kMaxGroups : lane_groups(valid, lane);
  const int rem = valid % kGroup;
  const int last = (valid - 1) / kGroup;  // index of the last group
#pragma unroll
  for (int i = 0; i < TileRegs<DT>::kMaxGroups; ++i) {
    if (FULL || i < ng) {
      const int g = lane + kLanes * i;
      int nvec = Group<DT>::kVec + 1;
      if (EXACT && WOFF >= 0 && !FULL && rem != 0 && g == last) {
        const int off = 4 * (WOFF < 0 ? 0 : WOFF) + static_cast<int>(sh / 8);
        nvec = (off + rem * Elem<DT>::kBytes + 15) / 16;
      }
      load_group<DT, WOFF>(tile, g, sh, r.w[i], nvec);
      if (!FULL && rem != 0 && g == last) Group<DT>::mask_tail(r.w[i], rem);
    }
  }
}

template <int DT, bool FULL, bool ENT, bool CLAMP>
__device__ __forceinline__ TilePartial tile_reduce_regs_t(const TileRegs<DT>& r, int valid, int lane, float rcp) {
  const int ng = FULL ? TileRegs<DT>::kMaxGroups : lane_groups(valid, lane);
  uint32_t mx[Group<DT>::kW];
  Group<DT>::max_init(mx);
#pragma unroll
  for (int i = 0; i < TileRegs<DT>::kMaxGroups; ++i)
    if (FULL || i < ng) Group<DT>::max_acc(mx, r.w[i]);
  const float mx_all = warp_max(Group<DT>::max_fin(mx));
  const float m = rcp == 1.0f ? mx_all : __fmul_rn(mx_all, rcp);
  const float shift = (mx_all == -INFINITY) ? 0.0f : mx_all;  // in stored units
  const float c = __fmul_rn(rcp, kLog2e);                     // rcp = 1: log2e exactly
  const uint64_t shift2 = pk(shift, shift), c2 = pk(c, c);
  uint64_t a[4] = {0, 0, 0, 0}, u[4] = {0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < TileRegs<DT>::kMaxGroups; ++i)
    if (FULL || i < ng) Group<DT>::template sum_acc<ENT, CLAMP>(a, u, r.w[i], shift2, c2);
  return finish_tile<ENT>(m, a, u);
}

template <int DT, int WOFF, bool EXACT>
__device__ __forceinline__ void tile_load_regs_w(const unsigned char* tile, int valid, int lane, TileRegs<DT>& r,
                                                 unsigned sh) {
  if (valid == TileRegs<DT>::kMaxTile) {
    tile_load_regs_t<DT, true, WOFF, EXACT>(tile, valid, lane, r, sh);
  } else {
    tile_load_regs_t<DT, false, WOFF, EXACT>(tile, valid, lane, r, sh);
  }
}

// The lane's groups of a tile whose first element sits `off` bytes past the
// 16-byte aligned address `tile` (SHIFTED = false: off is 0).  EXACT: as for
// tile_load_regs_t.
template <int DT, bool SHIFTED = false, bool EXACT = false>
__device__ __forceinline__ void tile_load_regs(const unsigned char* tile, int valid, int lane, TileRegs<DT>& r,
                                               unsigned off = 0) {
  const unsigned sh = 8u * (off & 3u);
  if (!SHIFTED || off == 0) return tile_load_regs_w<DT, -1, EXACT>(tile, valid, lane, r, 0);
  switch (off >> 2) {
    case 0: return tile_load_regs_w<DT, 0, EXACT>(tile, valid, lane, r, sh);
    case 1: return tile_load_regs_w<DT, 1, EXACT>(tile, valid, lane, r, sh);
    case 2: return tile_load_regs_w<DT, 2, EXACT>(tile, valid, lane, r, sh);
    default: return tile_load_regs_w<DT, 3, EXACT>(tile, valid, lane, r, sh);
  }
}

// CLAMP: as for Group::sum_acc.  With ENT and CLAMP = false the entropy sum
// comes out NaN when the tile holds an element whose term needs the clamp;
// the caller then reloads the tile and takes its u from a CLAMP = true pass
// (same m and s; the same u bits a clamped pass gives in one go).
template <int DT, bool ENT, bool CLAMP = !ENT>
__device__ __forceinline__ TilePartial tile_reduce_regs(const TileRegs<DT>& r, int valid, int lane, float rcp) {
  return valid == TileRegs<DT>::kMaxTile ? tile_reduce_regs_t<DT, true, ENT, CLAMP>(r, valid, lane, rcp)
                                         : tile_reduce_regs_t<DT, false, ENT, CLAMP>(r, valid, lane, rcp);
}

template <int DT, bool ENT, int WOFF>
__device__ __forceinline__ TilePartial tile_reduce_smem_t(const unsigned char* tile, int valid, int lane, float rcp,
                                                          unsigned sh) {
  const int groups = (valid + kGroup - 1) / kGroup;
  const int rem = valid % kGroup;
  uint32_t mx[Group<DT>::kW];
  Group<DT>::max_init(mx);
  for (int g = lane; g < groups; g += kLanes) {
    uint32_t w[Group<DT>::kW];
    load_group<DT, WOFF>(tile, g, sh, w);
    if (rem != 0 && g == groups - 1) Group<DT>::mask_tail(w, rem);
    Group<DT>::max_acc(mx, w);
  }
  const float mx_all = warp_max(Group<DT>::max_fin(mx));
  const float m = rcp == 1.0f ? mx_all : __fmul_rn(mx_all, rcp);
  const float shift = (mx_all == -INFINITY) ? 0.0f : mx_all;  // in stored units
  const float c = __fmul_rn(rcp, kLog2e);                     // rcp = 1: log2e exactly
  const uint64_t shift2 = pk(shift, shift), c2 = pk(c, c);
  uint64_t a[4] = {0, 0, 0, 0}, u[4] = {0, 0, 0, 0};
  for (int g = lane; g < groups; g += kLanes) {
    uint32_t w[Group<DT>::kW];
    load_group<DT, WOFF>(tile, g, sh, w);
    if (rem != 0 && g == groups - 1) Group<DT>::mask_tail(w, rem);
    Group<DT>::template sum_acc<ENT, false>(a, u, w, shift2, c2);
  }
  TilePartial tp = finish_tile<ENT>(m, a, u);
  if (ENT && tp.u != tp.u) {  // NaN (warp-uniform): the entropy terms again, with the clamp
    uint64_t a2[4] = {0, 0, 0, 0}, u2[4] = {0, 0, 0, 0};
    for (int g = lane; g < groups; g += kLanes) {
      uint32_t w[Group<DT>::kW];
      load_group<DT, WOFF>(tile, g, sh, w);
      if (rem != 0 && g == groups - 1) Group<DT>::mask_tail(w, rem);
      Group<DT>::template sum_acc<ENT, true>(a2, u2, w, shift2, c2);
    }
    tp.u = finish_tile<ENT>(m, a2, u2).u;
  }
  return tp;
}

// off, SHIFTED: as for tile_load_regs.
template <int DT, bool ENT, bool SHIFTED = false>
__device__ __forceinline__ TilePartial tile_reduce_smem(const unsigned char* tile, int valid, int lane, float rcp,
                                                        unsigned off = 0) {
  const unsigned sh = 8u * (off & 3u);
  if (!SHIFTED || off == 0) return tile_reduce_smem_t<DT, ENT, -1>(tile, valid, lane, rcp, 0);
  switch (off >> 2) {
    case 0: return tile_reduce_smem_t<DT, ENT, 0>(tile, valid, lane, rcp, sh);
    case 1: return tile_reduce_smem_t<DT, ENT, 1>(tile, valid, lane, rcp, sh);
    case 2: return tile_reduce_smem_t<DT, ENT, 2>(tile, valid, lane, rcp, sh);
    default: return tile_reduce_smem_t<DT, ENT, 3>(tile, valid, lane, rcp, sh);
  }
}

// The fixed-order merge of one row's T tile partials, by one warp (all lanes
// return the same values):
//   M = max_t m_t;  w_t = exp(m_t - M);  S = fma(s_t, w_t, S) for t = 0, 1,
//   ..., T-1 (one rounding per step, from S = 0);  LSE = M + log(S) (log:
//   CUDA logf).
// With ENT, also the entropy from the partial sums u_t (an exact rewrite of
// -sum p log p, since log p = (z - m_t) + (m_t - M) - log S in tile t):
//   v_t = fma(m_t - M, s_t, u_t);  U = fma(v_t, w_t, U) in the same order;
//   H = log(S) - U / S.
// M = -inf (no finite logit in the row) gives LSE = -inf, or NaN if a partial
// sum is NaN, and H = NaN.  The exponentials are computed in parallel across
// lanes; the chains of fused multiply-adds are the same sequential chains in
// every lane.
// Floats of shared scratch one warp's merge_lse uses (SCRATCH): four batch
// columns of 32.
constexpr int kMergeScratch = 4 * kLanes;
// bil_logp_merge gives each row a block (merge_block_kernel) from this many tiles on, for batches of
// at most one row per SM: the warp merge pays a load's latency per batch of 32 tiles.
constexpr int kMergeBlockMinTiles = 128;

// SCRATCH selects how the sequential chain is fed; both perform the same
// operations in the same order.  SCRATCH = true: the batch after the current
// one is loaded while the current one is chained, the batch's terms go through
// the warp's shared `scratch`, and the 32 steps are unrolled with no test
// (latency: a one-row merge of 594 tiles takes 7 us instead of 18).  SCRATCH =
// false: a compact loop with shuffles and no scratch, for the streaming
// forward, whose consumer code it keeps small (the unrolled forms cost that
// kernel 1.5-4% with the entropy).
template <bool ENT, bool SCRATCH>
__device__ __forceinline__ float merge_lse(const float* m, const float* s, const float* u, int T, int lane,
                                           float* entropy, float* scratch) {
  float M = -INFINITY;  // exact: any order
  if (SCRATCH) {
#pragma unroll 4
    for (int t = lane; t < T; t += kLanes) M = fmaxf(M, m[t]);
  } else {
    for (int t = lane; t < T; t += kLanes) M = fmaxf(M, m[t]);
  }
  M = warp_max(M);
  if (M == -INFINITY) {
    bool nan = false;
    for (int t = lane; t < T; t += kLanes) nan |= isnan(s[t]);
    if (ENT) *entropy = __int_as_float(0x7fc00000);
    return __any_sync(0xffffffffu, nan) ? __int_as_float(0x7fc00000) : -INFINITY;
  }
  float S = 0.0f, U = 0.0f;
  if (!SCRATCH) {
    // S = fma(s_t, e_t, S) for t = 0, 1, ..., T-1, one rounding per step, and U alike
    for (int t0 = 0; t0 < T; t0 += kLanes) {
      const int t = t0 + lane;
      float e = 0.0f, st = 0.0f, dm = 0.0f, ut = 0.0f;
      if (t < T) {
        dm = __fsub_rn(m[t], M);
        e = contract_exp(dm);
        st = s[t];
        if (ENT) {
          ut = u[t];
          dm = fmaxf(dm, kNegMax);  // a tile of -inf (s_t = 0) then adds 0, not -inf * 0
        }
      }
      const int n = min(kLanes, T - t0);
      for (int j = 0; j < n; ++j) {
        const float ej = __shfl_sync(0xffffffffu, e, j);
        const float sj = __shfl_sync(0xffffffffu, st, j);
        S = __fmaf_rn(sj, ej, S);
        if (ENT) {
          const float dmj = __shfl_sync(0xffffffffu, dm, j);
          const float uj = __shfl_sync(0xffffffffu, ut, j);
          U = __fmaf_rn(__fmaf_rn(dmj, sj, uj), ej, U);
        }
      }
    }
  } else {
    // S = fma(s_t, e_t, S) for t = 0, 1, ..., T-1, one rounding per step, and U
    // alike.  Lane l holds batch entries t0 + l; the batch after the current one
    // is loaded while the current one is chained, so the loads' latency is paid
    // once, not once per batch.
    float mc = -INFINITY, sc = 0.0f, uc = 0.0f;  // this batch's (m_t, s_t, u_t) of the lane
    if (lane < T) {
      mc = m[lane];
      sc = s[lane];
      if (ENT) uc = u[lane];
    }
    for (int t0 = 0; t0 < T; t0 += kLanes) {
      const int tn = t0 + kLanes + lane;
      float mn = -INFINITY, sn = 0.0f, un = 0.0f;  // the next batch, in flight during this one
      if (tn < T) {
        mn = m[tn];
        sn = s[tn];
        if (ENT) un = u[tn];
      }
      float e = 0.0f, st = 0.0f, dm = 0.0f, ut = 0.0f;
      if (t0 + lane < T) {
        dm = __fsub_rn(mc, M);
        e = contract_exp(dm);
        st = sc;
        if (ENT) {
          ut = uc;
          dm = fmaxf(dm, kNegMax);  // a tile of -inf (s_t = 0) then adds 0, not -inf * 0
        }
      }
      // Every batch takes 32 steps with no test: a lane past the last tile holds
      // e = s = d = u = 0, and fma(0, 0, S) is S exactly (S starts at +0, adds
      // only terms >= 0 and so is never -0; U adds only terms <= 0 and is never
      // -0 either).  The batch's terms go through the warp's shared scratch, and
      // every lane runs the chain from broadcast reads, which do not depend on
      // S and so issue ahead of the fused multiply-adds.
      __syncwarp();  // the previous batch's reads of the scratch are done
      scratch[lane] = e;
      scratch[kLanes + lane] = st;
      if (ENT) {
        scratch[2 * kLanes + lane] = dm;
        scratch[3 * kLanes + lane] = ut;
      }
      __syncwarp();
#pragma unroll
      for (int j = 0; j < kLanes; ++j) {
        const float ej = scratch[j];
        const float sj = scratch[kLanes + j];
        S = __fmaf_rn(sj, ej, S);
        if (ENT) U = __fmaf_rn(__fmaf_rn(scratch[2 * kLanes + j], sj, scratch[3 * kLanes + j]), ej, U);
      }
      mc = mn;
      sc = sn;
      uc = un;
    }
  }
  const float logS = logf(S);
  if (ENT) *entropy = __fsub_rn(logS, __fdiv_rn(U, S));
  return __fadd_rn(M, logS);
}

// ---------------------------------------------------------------------------
// Bounded waits.  Every wait polls a bounded number of times; one that runs
// out records a bit in g_watchdog and reports failure so that the kernel can
// stop instead of hanging.
// ---------------------------------------------------------------------------

__device__ unsigned int g_watchdog;

constexpr unsigned kWatchFull = 1u;      // consumer waited too long for a tile
constexpr unsigned kWatchEmpty = 2u;     // producer waited too long for a free stage
constexpr unsigned kWatchRowSlot = 4u;   // producer waited too long for a free row slot
constexpr unsigned kWatchDrain = 8u;     // producer waited too long for its own copies
constexpr unsigned kWatchProtocol = 16u; // a consumer met a unit outside the launch's ranges
constexpr unsigned kWatchSelfTest = 512u; // the self-test's wait on a barrier nothing arrives at

__device__ __forceinline__ bool warp_wait(uint64_t* bar, unsigned parity, volatile int* abort,
                                          unsigned code) {
  return warp_wait_watch(bar, parity, abort, code, &g_watchdog);
}

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.  Both
// addresses 16-byte aligned, bytes a multiple of 16.  The logits are read
// once, so the copy asks L2 to evict them first.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------
// The streaming forward (fused) and tile-partials kernel.
// ---------------------------------------------------------------------------

// Blocks of one producer and up to seven consumer warps, two blocks per SM:
// 16 warps at no more than 128 registers each fill an SM's register file.
#ifndef BIL_STREAM_MAX_CONSUMERS
#define BIL_STREAM_MAX_CONSUMERS 7
#endif
constexpr int kStreamThreads = 256;
constexpr int kMaxConsumers = BIL_STREAM_MAX_CONSUMERS < kStreamThreads / 32 - 1 ? BIL_STREAM_MAX_CONSUMERS
                                                                                  : kStreamThreads / 32 - 1;

struct StreamParams {
  const unsigned char* logits;  // column 0 = global column tile_begin * tile_v
  int64_t n_rows, vocab, ld;    // ld in elements
  int tile_v, tile_begin, tile_end, num_tiles;
  const int64_t* targets;
  int64_t ignore_index;
  float rcp;  // 1 / temperature, rounded to float32 on the host
  // fused outputs
  float* logp;
  float* lse;
  float* entropy;  // with ENT
  // partials outputs
  float* part_max;
  float* part_sum;
  float* part_ent;  // with ENT
  int64_t ld_part;
  float* target_logit;
  // pipeline shape
  int stages, consumers, row_slots;
  unsigned stage_bytes;
};

struct UnitDesc {
  int64_t row;   // -1: no more units for this consumer
  int32_t tile;  // global tile index
  int32_t slot;  // fused: row slot
};

struct RowSlot {
  int64_t row;
  int64_t target;
  float target_logit;
  int done;  // tiles reduced so far
};

// Shared-memory layout (dynamic):
//   [stages * stage_bytes]      tile ring, 128-byte aligned stages
//   [stages] uint64 full, [stages] uint64 empty, [row_slots] uint64 row_free
//   [stages] UnitDesc
//   [row_slots] RowSlot, then [row_slots][num_tiles] float m, [row_slots][num_tiles] float s
//   int abort
struct Smem {
  unsigned char* ring;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* row_free;
  UnitDesc* desc;
  RowSlot* slots;
  float* slot_m;
  float* slot_s;
  float* slot_u;
  int* abort;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline size_t stream_smem_bytes(int stages, unsigned stage_bytes, int row_slots,
                                                    int num_tiles, bool fused, bool ent, Smem* out,
                                                    unsigned char* base) {
  const size_t slot_floats = fused ? static_cast<size_t>(row_slots) * num_tiles : 0;
  size_t off = 0;
  const size_t ring = off;
  off += static_cast<size_t>(stages) * stage_bytes;
  off = align_up(off, 8);
  const size_t full = off;
  off += sizeof(uint64_t) * stages;
  const size_t empty = off;
  off += sizeof(uint64_t) * stages;
  const size_t row_free = off;
  off += sizeof(uint64_t) * (fused ? row_slots : 0);
  const size_t desc = off;
  off += sizeof(UnitDesc) * stages;
  const size_t slots = off;
  off += sizeof(RowSlot) * (fused ? row_slots : 0);
  const size_t sm = off;
  off += sizeof(float) * slot_floats;
  const size_t ss = off;
  off += sizeof(float) * slot_floats;
  const size_t su = off;
  off += sizeof(float) * (ent ? slot_floats : 0);
  const size_t ab = off;
  off += sizeof(int);
  if (out != nullptr) {
    out->ring = base + ring;
    out->full = reinterpret_cast<uint64_t*>(base + full);
    out->empty = reinterpret_cast<uint64_t*>(base + empty);
    out->row_free = reinterpret_cast<uint64_t*>(base + row_free);
    out->desc = reinterpret_cast<UnitDesc*>(base + desc);
    out->slots = reinterpret_cast<RowSlot*>(base + slots);
    out->slot_m = reinterpret_cast<float*>(base + sm);
    out->slot_s = reinterpret_cast<float*>(base + ss);
    out->slot_u = reinterpret_cast<float*>(base + su);
    out->abort = reinterpret_cast<int*>(base + ab);
  }
  return off;
}

// ENT: also the entropy partials (partials) or the entropy (fused).
template <int DT, bool FUSED, bool ALIGNED, bool ENT>
__global__ void __launch_bounds__(kStreamThreads, 2) stream_kernel(const StreamParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  constexpr int EB = Elem<DT>::kBytes;
  Smem sm;
  stream_smem_bytes(p.stages, p.stage_bytes, p.row_slots, p.num_tiles, FUSED, ENT, &sm, smem_raw);
  const int warp = threadIdx.x / kLanes;
  const int lane = threadIdx.x % kLanes;
  const int S = p.stages;
  const int W = p.consumers;
  volatile int* abort = sm.abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    if (FUSED) {
      for (int r = 0; r < p.row_slots; ++r) mbar_init(&sm.row_free[r], 1);
    }
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  griddep_wait();  // the barriers above are shared memory; from here on global memory is read
  griddep_launch_dependents();

  const int tiles_here = p.tile_end - p.tile_begin;

  if (warp == 0) {
    // ---------------- producer warp ----------------
    const uint64_t policy = evict_first_policy();
    // The block's share of the work: whole rows (fused) or a contiguous range
    // of (row, tile) units (partials).  Positions advance incrementally: no
    // 64-bit division inside the loop.
    int64_t u0, u1;
    if (FUSED) {
      u0 = p.n_rows * blockIdx.x / gridDim.x * tiles_here;
      u1 = p.n_rows * (blockIdx.x + 1) / gridDim.x * tiles_here;
    } else {
      const int64_t total = p.n_rows * tiles_here;
      u0 = total * blockIdx.x / gridDim.x;
      u1 = total * (blockIdx.x + 1) / gridDim.x;
    }
    int64_t row = u0 / tiles_here;
    int ti = static_cast<int>(u0 - row * tiles_here);  // tile within the range
    int64_t left = u1 - u0;
    int64_t k = 0;                 // units put in the ring
    int stage = 0;                 // ring cursor: stage of unit k and its fill parity
    unsigned phase = 0;
    int slot = 0;                  // fused: row-slot cursor and its use parity
    unsigned slot_phase = 0;
    bool ok = true;
    while (left > 0 && ok) {
      const int64_t target = p.targets[row];
      const int n = static_cast<int>(min(static_cast<int64_t>(tiles_here - ti), left));  // this row's units
      if (target == p.ignore_index) {
        // Inactive row: its logits are never read.
        if (FUSED) {
          if (lane == 0) {
            p.logp[row] = 0.0f;
            if (p.lse != nullptr) p.lse[row] = 0.0f;
            if (ENT) p.entropy[row] = 0.0f;
          }
        } else {
          for (int i = lane; i < n; i += kLanes) {
            p.part_max[row * p.ld_part + p.tile_begin + ti + i] = -INFINITY;
            p.part_sum[row * p.ld_part + p.tile_begin + ti + i] = 0.0f;
            if (ENT) p.part_ent[row * p.ld_part + p.tile_begin + ti + i] = 0.0f;
          }
        }
      } else {
        if (FUSED) {
          ok = warp_wait(&sm.row_free[slot], slot_phase ^ 1u, abort, kWatchRowSlot);
          if (!ok) break;
          if (lane == 0) {
            RowSlot& rs = sm.slots[slot];
            rs.row = row;
            rs.target = target;
            rs.target_logit = __int_as_float(0x7fc00000);
            rs.done = 0;
          }
        }
        const unsigned char* row_src = p.logits + row * p.ld * EB;
        for (int i = 0; i < n; ++i) {
          const int tile = p.tile_begin + ti + i;
          ok = warp_wait(&sm.empty[stage], phase ^ 1u, abort, kWatchEmpty);
          if (!ok) break;
          const int64_t col0 = static_cast<int64_t>(tile) * p.tile_v;  // global column
          const int valid = static_cast<int>(min(static_cast<int64_t>(p.tile_v), p.vocab - col0));
          const unsigned char* src = row_src + static_cast<int64_t>(ti + i) * p.tile_v * EB;
          const unsigned off = ALIGNED ? 0u : static_cast<unsigned>(reinterpret_cast<uintptr_t>(src) & 15u);
          unsigned char* dst = sm.ring + static_cast<size_t>(stage) * p.stage_bytes;
          if (lane == 0) {
            UnitDesc d;
            d.row = row;
            d.tile = tile;
            d.slot = slot;
            sm.desc[stage] = d;
          }
          // One bulk copy of the 16-byte aligned span that covers the tile: it
          // starts off bytes before the tile's first element (rows that are
          // not 16-byte aligned) and every 16 bytes of it hold an element of
          // the tile, so it reads no page the tile does not touch.  The stage
          // holds tile_v elements plus 128 bytes when rows are not aligned.
          if (lane == 0) {
            const unsigned bytes = static_cast<unsigned>(align_up(off + static_cast<size_t>(valid) * EB, 16));
            mbar_arrive_expect_tx(&sm.full[stage], bytes);
            bulk_g2s(dst, src - off, bytes, &sm.full[stage], policy);
          }
          __syncwarp();
          ++k;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (FUSED && ++slot == p.row_slots) {
          slot = 0;
          slot_phase ^= 1u;
        }
      }
      left -= n;
      ++row;
      ti = 0;
    }
    // One end marker per consumer warp: units k, k+1, ..., k+W-1 map to
    // consumers k % W, ..., so each consumer sees exactly one.
    for (int w = 0; w < W && ok; ++w) {
      ok = warp_wait(&sm.empty[stage], phase ^ 1u, abort, kWatchEmpty);
      if (!ok) break;
      if (lane == 0) {
        UnitDesc d;
        d.row = -1;
        d.tile = 0;
        d.slot = 0;
        sm.desc[stage] = d;
        mbar_arrive(&sm.full[stage]);
      }
      __syncwarp();
      ++k;
      if (++stage == S) {
        stage = 0;
        phase ^= 1u;
      }
    }
    // Drain: no bulk copy of ours may still be landing in shared memory when
    // the block exits (consumers that gave up leave fills unconsumed).  The
    // latest fill of every used stage must have completed; normally they all
    // have and this costs one poll per stage.
    if (lane == 0) {
      for (int s = 0; s < S && s < k; ++s) {
        const int64_t last = ((k - 1 - s) / S) * S + s;  // latest unit issued into stage s
        const unsigned fill = static_cast<unsigned>(last / S);
        const long long start = global_ns();
        while (!mbar_try_wait(&sm.full[s], fill & 1u)) {
          if (global_ns() - start > kWaitLimitNs) {
            atomicOr(&g_watchdog, kWatchDrain);
            break;
          }
        }
      }
    }
    return;
  }

  // ---------------- consumer warps ----------------
  // Consumer cw takes units cw, cw+W, cw+2W, ...: with S a multiple of W
  // these sit in its own stages cw, cw+W, ... in fill order, and each step
  // wraps the ring at most once.
  const int cw = warp - 1;
  int stage = cw;
  unsigned phase = 0;
  for (;; stage += W) {
    if (stage >= S) {
      stage -= S;
      phase ^= 1u;
    }
    if (!warp_wait(&sm.full[stage], phase, abort, kWatchFull)) break;
    const UnitDesc d = sm.desc[stage];
    if (d.row < 0) break;
    // A unit outside this launch's ranges can only come from a broken
    // pipeline protocol: record it and stop rather than touch memory with it.
    if (d.row >= p.n_rows || d.tile < p.tile_begin || d.tile >= p.tile_end ||
        (FUSED && (d.slot < 0 || d.slot >= p.row_slots))) {
      if (lane == 0) {
        atomicOr(&g_watchdog, kWatchProtocol);
        *abort = 1;
      }
      break;
    }
    const unsigned char* tile = sm.ring + static_cast<size_t>(stage) * p.stage_bytes;
    const int64_t col0 = static_cast<int64_t>(d.tile) * p.tile_v;
    const int valid = static_cast<int>(min(static_cast<int64_t>(p.tile_v), p.vocab - col0));
    // where the producer's copy put the tile's first element (its source address mod 16)
    const unsigned off =
        ALIGNED ? 0u
                : static_cast<unsigned>((reinterpret_cast<uintptr_t>(p.logits) +
                                         static_cast<uint64_t>(d.row) * p.ld * EB +
                                         static_cast<uint64_t>(d.tile - p.tile_begin) * p.tile_v * EB) & 15u);
    // The target logit is copied from the tile that owns it, never summed
    // (scaled by the temperature exactly as the tile's values are).
    const int64_t target = FUSED ? sm.slots[d.slot].target : p.targets[d.row];
    const bool owner = target >= col0 && target < col0 + valid;
    float tl = 0.0f;
    if (owner) {
      tl = Elem<DT>::one(tile + off + static_cast<size_t>(target - col0) * EB);
      if (p.rcp != 1.0f) tl = __fmul_rn(tl, p.rcp);
    }
    TilePartial tp;
    if (p.tile_v <= TileRegs<DT>::kMaxTile) {
      // Copy the lane's groups to registers and hand the stage back to the
      // producer at once, so that its next fill overlaps this reduction.
      TileRegs<DT> regs;
      tile_load_regs<DT, !ALIGNED>(tile, valid, lane, regs, off);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[stage]);
      tp = tile_reduce_regs<DT, ENT, false>(regs, valid, lane, p.rcp);
      if (ENT && tp.u != tp.u) {
        // The entropy terms need the clamp (a -inf logit or a masked column)
        // or a logit is NaN: take u from a clamped pass over the tile, read
        // again from global memory (the stage has been handed back).
        const unsigned char* g = p.logits + d.row * p.ld * EB + static_cast<int64_t>(d.tile - p.tile_begin) * p.tile_v * EB;
        if (ALIGNED) {
          tile_load_regs<DT>(g, valid, lane, regs);
        } else {
          tile_load_regs<DT, true, true>(g - off, valid, lane, regs, off);
        }
        tp.u = tile_reduce_regs<DT, ENT, true>(regs, valid, lane, p.rcp).u;
      }
    } else {
      tp = tile_reduce_smem<DT, ENT, !ALIGNED>(tile, valid, lane, p.rcp, off);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[stage]);  // the stage may be refilled now
    }

    if (!FUSED) {
      if (lane == 0) {
        p.part_max[d.row * p.ld_part + d.tile] = tp.m;
        p.part_sum[d.row * p.ld_part + d.tile] = tp.s;
        if (ENT) p.part_ent[d.row * p.ld_part + d.tile] = tp.u;
        if (owner) p.target_logit[d.row] = tl;
      }
      continue;
    }
    RowSlot& rs = sm.slots[d.slot];
    float* sm_m = sm.slot_m + static_cast<size_t>(d.slot) * p.num_tiles;
    float* sm_s = sm.slot_s + static_cast<size_t>(d.slot) * p.num_tiles;
    float* sm_u = sm.slot_u + static_cast<size_t>(d.slot) * p.num_tiles;
    int before = 0;
    if (lane == 0) {
      sm_m[d.tile] = tp.m;
      sm_s[d.tile] = tp.s;
      if (ENT) sm_u[d.tile] = tp.u;
      if (owner) rs.target_logit = tl;
      __threadfence_block();
      before = atomicAdd(&rs.done, 1);
    }
    before = __shfl_sync(0xffffffffu, before, 0);
    if (before != p.num_tiles - 1) continue;
    // This warp reduced the row's last tile: merge the row.
    __threadfence_block();
    __syncwarp();
    float H = 0.0f;
    const float L = merge_lse<ENT, false>(sm_m, sm_s, sm_u, p.num_tiles, lane, &H, nullptr);
    if (lane == 0) {
      const int64_t row = rs.row;
      const bool valid_target = rs.target >= 0 && rs.target < p.vocab;
      p.logp[row] = valid_target ? __fsub_rn(rs.target_logit, L) : __int_as_float(0x7fc00000);
      if (p.lse != nullptr) p.lse[row] = L;
      if (ENT) p.entropy[row] = H;
      __threadfence_block();
      mbar_arrive(&sm.row_free[d.slot]);
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// Small-batch forward: one row per thread-block cluster.
//
// With a handful of rows the streaming forward has one block per row, and one
// SM streams the whole row.  Here a cluster of kSplitCtas blocks (on as many
// SMs) shares each row: warp w of cluster rank c takes tiles c*kSplitWarps + w,
// then + kSplitCtas*kSplitWarps, ...; each reduces its tile straight from
// global memory with tile_load_regs / tile_reduce_regs (the same functions,
// and so the same bits, as the streaming forward) and writes the partial into
// the cluster's rank-0 block through distributed shared memory.  After one
// cluster barrier the rank-0 block merges the row with merge_lse.  The bits
// are those of the streaming forward; only the work split differs.  Used for
// 16-bit types with tiles of at most TileRegs::kMaxTile elements.  ALIGNED
// (rows start on 16-byte boundaries): a group of 8 elements is one 16-byte
// unit inside the row.  Otherwise a group is read as the two 16-byte units
// that hold it and shifted into place, and a partial last group reads only the
// units that hold its elements: no read leaves the 16-byte units that hold
// the row's elements.
// ---------------------------------------------------------------------------

constexpr int kSplitCtas = 8;   // blocks per cluster (the portable maximum)
constexpr int kSplitWarps = 5;  // 40 warps per row: a 151936-column row in 4096-column tiles is 38 tiles

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The shared::cluster address of `p` (a shared variable of this block) in the
// block of cluster rank `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Every thread of every block of the cluster arrives; the release / acquire
// pair makes the distributed shared-memory stores before it visible after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int DT, bool ENT, bool ALIGNED>
__global__ void __launch_bounds__(kSplitWarps * kLanes) split_row_kernel(const StreamParams p) {
  constexpr int EB = Elem<DT>::kBytes;
  __shared__ float sm_m[BIL_MAX_FUSED_TILES];
  __shared__ float sm_s[BIL_MAX_FUSED_TILES];
  __shared__ float sm_u[ENT ? BIL_MAX_FUSED_TILES : 1];
  __shared__ float sm_tl;
  griddep_wait();
  griddep_launch_dependents();
  const uint32_t rank = cluster_ctarank();
  const int64_t row = static_cast<int64_t>(blockIdx.x) / kSplitCtas;  // a cluster is kSplitCtas consecutive blocks
  const int warp = threadIdx.x / kLanes;
  const int lane = threadIdx.x % kLanes;
  const int64_t target = row < p.n_rows ? p.targets[row] : p.ignore_index;
  const bool active = row < p.n_rows && target != p.ignore_index;
  if (rank == 0 && threadIdx.x == 0) sm_tl = __int_as_float(0x7fc00000);
  cluster_sync_all();  // rank 0's initial value is in place before any block writes into it
  if (active) {
    const unsigned char* row_src = p.logits + row * p.ld * EB;
    for (int t = static_cast<int>(rank) * kSplitWarps + warp; t < p.num_tiles; t += kSplitCtas * kSplitWarps) {
      const int64_t col0 = static_cast<int64_t>(t) * p.tile_v;
      const int valid = static_cast<int>(min(static_cast<int64_t>(p.tile_v), p.vocab - col0));
      const unsigned char* tile = row_src + col0 * EB;
      TileRegs<DT> regs;
      if (ALIGNED) {
        tile_load_regs<DT>(tile, valid, lane, regs);
      } else {
        // 16-byte loads from the boundary below the tile, shifted into place;
        // every load holds an element of the tile
        const unsigned off = static_cast<unsigned>(reinterpret_cast<uintptr_t>(tile) & 15u);
        tile_load_regs<DT, true, true>(tile - off, valid, lane, regs, off);
      }
      TilePartial tp = tile_reduce_regs<DT, ENT, false>(regs, valid, lane, p.rcp);
      if (ENT && tp.u != tp.u) {  // as in stream_kernel: u from a clamped pass
        if (ALIGNED) {
          tile_load_regs<DT>(tile, valid, lane, regs);
        } else {
          const unsigned off = static_cast<unsigned>(reinterpret_cast<uintptr_t>(tile) & 15u);
          tile_load_regs<DT, true, true>(tile - off, valid, lane, regs, off);
        }
        tp.u = tile_reduce_regs<DT, ENT, true>(regs, valid, lane, p.rcp).u;
      }
      if (lane == 0) {
        st_cluster(cluster_addr(&sm_m[t], 0), tp.m);
        st_cluster(cluster_addr(&sm_s[t], 0), tp.s);
        if (ENT) st_cluster(cluster_addr(&sm_u[t], 0), tp.u);
        if (target >= col0 && target < col0 + valid) {
          float tl = Elem<DT>::one(tile + (target - col0) * EB);
          if (p.rcp != 1.0f) tl = __fmul_rn(tl, p.rcp);
          st_cluster(cluster_addr(&sm_tl, 0), tl);
        }
      }
    }
  }
  cluster_sync_all();
  if (rank != 0 || warp != 0 || row >= p.n_rows) return;
  if (!active) {
    if (lane == 0) {
      p.logp[row] = 0.0f;
      if (p.lse != nullptr) p.lse[row] = 0.0f;
      if (ENT) p.entropy[row] = 0.0f;
    }
    return;
  }
  float H = 0.0f;
  __shared__ float sm_scratch[kMergeScratch];
  const float L = merge_lse<ENT, true>(sm_m, sm_s, sm_u, p.num_tiles, lane, &H, sm_scratch);
  if (lane == 0) {
    const bool valid_target = target >= 0 && target < p.vocab;
    p.logp[row] = valid_target ? __fsub_rn(sm_tl, L) : __int_as_float(0x7fc00000);
    if (p.lse != nullptr) p.lse[row] = L;
    if (ENT) p.entropy[row] = H;
  }
}

// One warp waits, with the kernels' own bounded wait, on an mbarrier that no
// thread and no copy ever arrives at.  The wait runs out after its limit, sets
// kWatchSelfTest in the watchdog word and returns; nothing faults or hangs.
__global__ void __launch_bounds__(kLanes) watchdog_selftest_kernel() {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort = 0;
  }
  __syncthreads();
  warp_wait(&bar, 0u, &abort, kWatchSelfTest);
}

// ---------------------------------------------------------------------------
// Merge kernel: one warp per row, the same merge_lse as the fused forward.
// ---------------------------------------------------------------------------

template <bool ENT>
__global__ void __launch_bounds__(256) merge_kernel(const float* __restrict__ part_max,
                                                    const float* __restrict__ part_sum,
                                                    const float* __restrict__ part_ent, int64_t n_rows,
                                                    int num_tiles, int64_t ld_part,
                                                    const float* __restrict__ target_logit,
                                                    const int64_t* __restrict__ targets,
                                                    int64_t ignore_index, int64_t vocab, float* logp,
                                                    float* lse, float* entropy) {
  __shared__ float sm_scratch[256 / kLanes][kMergeScratch];  // one per warp of the (256-thread) block
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x % kLanes;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / kLanes);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / kLanes) + threadIdx.x / kLanes;
       row < n_rows; row += warps) {
    const int64_t t = targets[row];
    if (t == ignore_index) {
      if (lane == 0) {
        logp[row] = 0.0f;
        if (lse != nullptr) lse[row] = 0.0f;
        if (ENT) entropy[row] = 0.0f;
      }
      continue;
    }
    float H = 0.0f;
    const float L = merge_lse<ENT, true>(part_max + row * ld_part, part_sum + row * ld_part,
                                   ENT ? part_ent + row * ld_part : nullptr, num_tiles, lane, &H,
                                   sm_scratch[threadIdx.x / kLanes]);
    if (lane == 0) {
      const bool valid = t >= 0 && t < vocab;
      logp[row] = valid ? __fsub_rn(target_logit[row], L) : __int_as_float(0x7fc00000);
      if (lse != nullptr) lse[row] = L;
      if (ENT) entropy[row] = H;
    }
  }
}

// The same merge with one block per row, for a few rows of many tiles (the
// fused LM-head's decode-sized batches: 594 tiles of 256).  The block loads
// the row's partials and takes their exponentials in parallel into shared
// memory (`sm`: T floats each of e_t and s_t, with ENT also of the clamped
// m_t - M and of u_t), and one thread runs merge_lse's chains over them in the
// same order with the same operations, so the bits are the warp merge's; the
// loads' latency is paid once instead of once per batch of 32 tiles.
template <bool ENT>
__global__ void __launch_bounds__(256) merge_block_kernel(const float* __restrict__ part_max,
                                                          const float* __restrict__ part_sum,
                                                          const float* __restrict__ part_ent, int64_t n_rows,
                                                          int num_tiles, int64_t ld_part,
                                                          const float* __restrict__ target_logit,
                                                          const int64_t* __restrict__ targets,
                                                          int64_t ignore_index, int64_t vocab, float* logp,
                                                          float* lse, float* entropy) {
  extern __shared__ float sm[];
  __shared__ float red[256 / kLanes];
  __shared__ int red_nan[256 / kLanes];
  griddep_wait();
  griddep_launch_dependents();
  const int T = num_tiles;
  const int lane = threadIdx.x % kLanes, warp = threadIdx.x / kLanes, nwarps = blockDim.x / kLanes;
  float* se = sm;
  float* ss = sm + T;
  float* sd = sm + 2 * T;
  float* su = sm + 3 * T;
  for (int64_t row = blockIdx.x; row < n_rows; row += gridDim.x) {
    const int64_t t = targets[row];
    if (t == ignore_index) {
      if (threadIdx.x == 0) {
        logp[row] = 0.0f;
        if (lse != nullptr) lse[row] = 0.0f;
        if (ENT) entropy[row] = 0.0f;
      }
      continue;
    }
    const float* m = part_max + row * ld_part;
    const float* s = part_sum + row * ld_part;
    float mx = -INFINITY;  // exact: any order
    for (int i = threadIdx.x; i < T; i += blockDim.x) mx = fmaxf(mx, m[i]);
    mx = warp_max(mx);
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    float M = red[0];
    for (int w = 1; w < nwarps; ++w) M = fmaxf(M, red[w]);
    float L, H = 0.0f;
    if (M == -INFINITY) {  // no finite logit: as merge_lse
      bool nan = false;
      for (int i = threadIdx.x; i < T; i += blockDim.x) nan |= isnan(s[i]);
      nan = __any_sync(0xffffffffu, nan);
      if (lane == 0) red_nan[warp] = nan ? 1 : 0;
      __syncthreads();
      int any = 0;
      for (int w = 0; w < nwarps; ++w) any |= red_nan[w];
      L = any ? __int_as_float(0x7fc00000) : -INFINITY;
      H = __int_as_float(0x7fc00000);
    } else {
      for (int i = threadIdx.x; i < T; i += blockDim.x) {
        const float dm = __fsub_rn(m[i], M);
        se[i] = contract_exp(dm);
        ss[i] = s[i];
        if (ENT) {
          sd[i] = fmaxf(dm, kNegMax);  // a tile of -inf (s_t = 0) then adds 0, not -inf * 0
          su[i] = part_ent[row * ld_part + i];
        }
      }
      __syncthreads();
      L = 0.0f;
      if (threadIdx.x == 0) {
        float S = 0.0f, U = 0.0f;
#pragma unroll 8
        for (int i = 0; i < T; ++i) {
          S = __fmaf_rn(ss[i], se[i], S);
          if (ENT) U = __fmaf_rn(__fmaf_rn(sd[i], ss[i], su[i]), se[i], U);
        }
        const float logS = logf(S);
        if (ENT) H = __fsub_rn(logS, __fdiv_rn(U, S));
        L = __fadd_rn(M, logS);
      }
    }
    if (threadIdx.x == 0) {
      const bool valid = t >= 0 && t < vocab;
      logp[row] = valid ? __fsub_rn(target_logit[row], L) : __int_as_float(0x7fc00000);
      if (lse != nullptr) lse[row] = L;
      if (ENT) entropy[row] = H;
    }
    __syncthreads();  // the shared arrays and `red` are free for the next row
  }
}

// ---------------------------------------------------------------------------
// Backward: dlogits[r, c] = g[r] * ([c == t_r] - exp(x[r, c] - lse[r])).// ---------------------------------------------------------------------------
// Backward: dlogits[r, c] = g[r] * ([c == t_r] - exp(x[r, c] - lse[r])).
// Work unit: (row, chunk of kBwdChunk columns), spread over a persistent grid.
// Purely elementwise given lse and g, so the bits cannot depend on the unit
// size, the grid, or whether a row is read in 16-byte vectors or one element
// at a time.
// ---------------------------------------------------------------------------

#ifndef BIL_BWD_GROUPS
#define BIL_BWD_GROUPS 4
#endif
constexpr int kBwdThreads = 256;
constexpr int kBwdGroupsPerThread = BIL_BWD_GROUPS;  // 16-byte loads a thread has in flight per unit
constexpr int kBwdChunk = kBwdThreads * kBwdGroupsPerThread * kGroup;  // 8192 columns per work unit

template <int OT>
struct Out;
template <>
struct Out<BIL_F32> {
  static constexpr int kBytes = 4;
  __device__ static __forceinline__ void store8(unsigned char* p, const float (&v)[kGroup]) {
    float4* q = reinterpret_cast<float4*>(p);
    __stcs(q, make_float4(v[0], v[1], v[2], v[3]));
    __stcs(q + 1, make_float4(v[4], v[5], v[6], v[7]));
  }
  __device__ static __forceinline__ void store1(unsigned char* p, float v) {
    *reinterpret_cast<float*>(p) = v;
  }
};
template <>
struct Out<BIL_BF16> {
  static constexpr int kBytes = 2;
  __device__ static __forceinline__ void store8(unsigned char* p, const float (&v)[kGroup]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    __stcs(reinterpret_cast<uint4*>(p), make_uint4(w[0], w[1], w[2], w[3]));
  }
  __device__ static __forceinline__ void store1(unsigned char* p, float v) {
    *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(v);
  }
};
template <>
struct Out<BIL_F16> {
  static constexpr int kBytes = 2;
  __device__ static __forceinline__ void store8(unsigned char* p, const float (&v)[kGroup]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    __stcs(reinterpret_cast<uint4*>(p), make_uint4(w[0], w[1], w[2], w[3]));
  }
  __device__ static __forceinline__ void store1(unsigned char* p, float v) {
    *reinterpret_cast<__half*>(p) = __float2half_rn(v);
  }
};

// A group of 8 gradient elements from its stored logits, none of them the
// row's target column, with the same operations as grad_elem in packed pairs.
template <int DT>
__device__ __forceinline__ void grad_group(const uint32_t (&w)[Group<DT>::kW], const RowMeta& m, float rcp, bool ent,
                                           float (&y)[kGroup]) {
  const bool scaled = rcp != 1.0f;
  const uint64_t L2 = pk(m.lse, m.lse), nL2 = pk(-m.lse, -m.lse), g2 = pk(m.g, m.g), rcp2 = pk(rcp, rcp);
  const uint64_t ngh2 = pk(-m.gh, -m.gh), H2 = pk(m.H, m.H);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint64_t x = Group<DT>::xpair(w, k);
    const uint64_t a = scaled ? fma2(x, rcp2, nL2) : sub2(x, L2);
    const uint64_t p = exp2_pair(a);                  // (p_2k, p_2k+1)
    uint64_t d;
    if (ent) {
      const uint64_t ac = pk(fmaxf(lo_of(a), kNegMax), fmaxf(hi_of(a), kNegMax));
      // -t3 = (-gh) * (p * (a + H)) is exactly -(gh * (p * (a + H))): rounding
      // to nearest is symmetric in the sign
      const uint64_t nt3 = mul2(ngh2, mul2(p, add2(ac, H2)));
      d = fma2(g2, sub2(0, p), nt3);                  // g * (0 - p) - t3, one rounding
    } else {
      d = mul2(g2, sub2(0, p));                       // g * (0 - p)
    }
    if (scaled) d = mul2(d, rcp2);
    y[2 * k] = lo_of(d);
    y[2 * k + 1] = hi_of(d);
  }
}

template <int DT>
__device__ __forceinline__ void load_group_stream(const unsigned char* p, uint32_t (&w)[Group<DT>::kW]) {
#pragma unroll
  for (int v = 0; v < Group<DT>::kVec; ++v) {
    const uint4 q = __ldcs(reinterpret_cast<const uint4*>(p) + v);
    w[4 * v] = q.x;
    w[4 * v + 1] = q.y;
    w[4 * v + 2] = q.z;
    w[4 * v + 3] = q.w;
  }
}

struct BwdParams {
  const unsigned char* logits;
  int64_t n_rows, vocab, ld;
  const int64_t* targets;
  int64_t ignore_index;
  const float* lse;
  const float* grad;
  const float* entropy;       // with an entropy gradient: the forward's entropy
  const float* grad_entropy;  // NULL: no entropy term
  float rcp;
  unsigned char* dlogits;
  int64_t ld_out, out_cols;
};

__device__ __forceinline__ RowMeta row_meta(const BwdParams& bp, int64_t row) {
  RowMeta m{0, 0.0f, 0.0f, 0.0f, 0.0f};
  if (row < bp.n_rows) {
    m.target = bp.targets[row];
    m.lse = bp.lse[row];
    m.g = bp.grad[row];
    if (bp.grad_entropy != nullptr) {
      m.H = bp.entropy[row];
      m.gh = bp.grad_entropy[row];
    }
  }
  return m;
}

// How the backward reads and writes its rows.
enum BwdRows {
  kBwdAligned = 0,        // every input and output row starts on a 16-byte boundary
  kBwdSharedOffsets = 1,  // input and output rows share their offset from one: groups from the first
                          // column where both are aligned, the few columns around them one by one
  kBwdScalar = 2,         // element by element
};

template <int DT, int OT, int ROWS>
__global__ void __launch_bounds__(kBwdThreads) bwd_kernel(const BwdParams bp) {
  const unsigned char* __restrict__ logits = bp.logits;
  const int64_t n_rows = bp.n_rows, vocab = bp.vocab, ld = bp.ld, ignore_index = bp.ignore_index;
  unsigned char* __restrict__ dlogits = bp.dlogits;
  const int64_t ld_out = bp.ld_out, out_cols = bp.out_cols;
  const float rcp = bp.rcp;
  const bool ent = bp.grad_entropy != nullptr;
  constexpr int EB = Elem<DT>::kBytes;
  constexpr int OB = Out<OT>::kBytes;
  // Work unit u = row * chunks + chunk, units strided by the grid; (row,
  // chunk) advance by a precomputed quotient and remainder.
  const int64_t chunks = (out_cols + kBwdChunk - 1) / kBwdChunk;
  const int64_t d_row = gridDim.x / chunks, d_chunk = gridDim.x % chunks;
  int64_t row = blockIdx.x / chunks, chunk = blockIdx.x % chunks;
  RowMeta meta = row_meta(bp, row);
  while (row < n_rows) {
    int64_t next_row = row + d_row, next_chunk = chunk + d_chunk;
    if (next_chunk >= chunks) {
      next_chunk -= chunks;
      ++next_row;
    }
    const RowMeta next = row_meta(bp, next_row);  // in flight during this unit

    const int64_t c0 = chunk * kBwdChunk;
    const int64_t c1 = min(c0 + kBwdChunk, out_cols);
    const int64_t t = meta.target;
    unsigned char* out = dlogits + row * ld_out * OB;
    const bool active = t != ignore_index;
    const bool valid_target = t >= 0 && t < vocab;
    const int64_t v1 = min(c1, vocab);  // [c0, v1): gradient; [max(c0, vocab), c1): pad
    if (!active || !valid_target) {
      const float fill = active ? __int_as_float(0x7fc00000) : 0.0f;
      for (int64_t c = c0 + threadIdx.x; c < v1; c += kBwdThreads) Out<OT>::store1(out + c * OB, fill);
    } else if (ROWS == kBwdScalar) {
      const unsigned char* in = logits + row * ld * EB;
      for (int64_t c = c0 + threadIdx.x; c < v1; c += kBwdThreads)
        Out<OT>::store1(out + c * OB, grad_elem(Elem<DT>::one(in + c * EB), meta, c == t, rcp, ent));
    } else {
      // Groups of 8 columns go by 16-byte vectors from the first column cg at
      // which the input and the output are both 16-byte aligned: c0 itself
      // when every row is aligned; otherwise the first such column of
      // [c0, c0 + 8), if there is one (the rows of a contiguous [N, V] input
      // and output share their offsets, whatever V).  All of a thread's loads
      // are issued before any arithmetic.  The columns before cg and after the
      // last whole group go one by one, with the same operations.
      const unsigned char* in = logits + row * ld * EB;
      int64_t cg = c0;
      if (ROWS == kBwdSharedOffsets) {
        cg = v1;
        for (int k = 0; k < kGroup; ++k) {
          const int64_t c = c0 + k;
          const uintptr_t a = reinterpret_cast<uintptr_t>(in + c * EB) | reinterpret_cast<uintptr_t>(out + c * OB);
          if (c < v1 && (a & 15u) == 0) {
            cg = c;
            break;
          }
        }
      }
      const int64_t gend = cg + ((v1 - cg) / kGroup) * kGroup;
      // With shared offsets fewer than 8 columns precede cg and fewer than 8
      // follow gend in every unit, so a thread has at most one of each; they
      // are read with the groups rather than after them, so that no warp waits
      // for memory twice more per unit.  (Aligned rows have a tail only at the
      // end of a row whose length is not a multiple of 8.)
      const int64_t ch = c0 + threadIdx.x, ct = gend + threadIdx.x;
      const bool head = ROWS == kBwdSharedOffsets && ch < cg, tail = ROWS == kBwdSharedOffsets && ct < v1;
      const float xh = head ? Elem<DT>::one(in + ch * EB) : 0.0f;
      const float xt = tail ? Elem<DT>::one(in + ct * EB) : 0.0f;
      uint32_t w[kBwdGroupsPerThread][Group<DT>::kW];
#pragma unroll
      for (int i = 0; i < kBwdGroupsPerThread; ++i) {
        const int64_t c = cg + (static_cast<int64_t>(i) * kBwdThreads + threadIdx.x) * kGroup;
        if (c < gend) load_group_stream<DT>(in + c * EB, w[i]);
      }
#pragma unroll
      for (int i = 0; i < kBwdGroupsPerThread; ++i) {
        const int64_t c = cg + (static_cast<int64_t>(i) * kBwdThreads + threadIdx.x) * kGroup;
        if (c < gend) {
          float y[kGroup];
          grad_group<DT>(w[i], meta, rcp, ent, y);
          Out<OT>::store8(out + c * OB, y);
          // The row's target column, if it is in this group: g * (1 - p) and
          // the rest, stored over the group's value (same thread, same address:
          // this store lands last).
          if (static_cast<uint64_t>(t - c) < static_cast<uint64_t>(kGroup))
            Out<OT>::store1(out + t * OB, grad_elem(Elem<DT>::one(in + t * EB), meta, true, rcp, ent));
        }
      }
      if (head) Out<OT>::store1(out + ch * OB, grad_elem(xh, meta, ch == t, rcp, ent));
      if (tail) Out<OT>::store1(out + ct * OB, grad_elem(xt, meta, ct == t, rcp, ent));
      if (ROWS == kBwdAligned) {
        for (int64_t c = gend + threadIdx.x; c < v1; c += kBwdThreads)
          Out<OT>::store1(out + c * OB, grad_elem(Elem<DT>::one(in + c * EB), meta, c == t, rcp, ent));
      }
    }
    for (int64_t c = max(c0, vocab) + threadIdx.x; c < c1; c += kBwdThreads) Out<OT>::store1(out + c * OB, 0.0f);
    row = next_row;
    chunk = next_chunk;
    meta = next;
  }
}

}  // namespace
