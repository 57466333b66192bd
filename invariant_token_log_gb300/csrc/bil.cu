// Batch-invariant selected-token log-probability for sm_103a (GB300).
//
// Operator: "Batch-Invariant LogP" operator page, sections "Reference
// Semantics" (what is computed), "Tensor Parallel" steps 1-6 (the fixed-tile
// (max, sumexp) partials and their fixed-order merge) and "Batch-Invariance"
// (one row's result depends on that row only; the backward recomputes the
// softmax from the saved per-row LSE).  The C ABI is declared in include/bil.h.
//
// Kernels
//   stream_kernel<FUSED=true>   forward: every tile of a row -> shared-memory
//                               partials -> fixed-order merge -> logp, lse.
//   stream_kernel<FUSED=false>  partials of a tile range -> [N, ld_part] buffers.
//   merge_kernel                fixed-order merge of [N, T] partials -> logp, lse.
//   bwd_kernel                  dlogits = g * (onehot - exp(x - lse)).
//
// The forward streams each row exactly once.  A producer warp moves whole
// tiles HBM -> shared memory with 1-D bulk asynchronous copies
// (cp.async.bulk, completion counted on an mbarrier) into a ring of stages;
// consumer warps reduce one tile each.  Nothing on this path is a contraction,
// so no tensor cores are used: the forward is bound by HBM bandwidth, with
// the exponential unit second.
//
// The arithmetic contract (what makes the bits reproducible) lives in
// tile_reduce() and merge_lse() and nowhere else: every kernel that produces
// a tile partial or an LSE calls them, so the fused and the split paths give
// identical bits by construction.  All floating-point operations that matter
// are written with explicit round-to-nearest intrinsics, and the file is
// compiled with contraction off, so inlining cannot change them.

#include "../../include/bil.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>

namespace {

// ---------------------------------------------------------------------------
// The arithmetic contract.
// ---------------------------------------------------------------------------

constexpr int kLanes = 32;
constexpr int kGroup = 8;  // elements a lane takes at a time: 16 bytes of bf16/fp16

// log2(e) rounded to float32: exp(a) is evaluated as 2^(a * log2(e)).
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2_approx(float a) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
  return r;
}

// exp(a) of the contract: one rounded multiply, then the hardware base-2
// exponential (flushes results below 2^-126 to zero).
__device__ __forceinline__ float contract_exp(float a) { return ex2_approx(__fmul_rn(a, kLog2e)); }

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
  __device__ static __forceinline__ void group(const unsigned char* p, float (&x)[kGroup]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static __forceinline__ float one(const unsigned char* p) {
    return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(p)) << 16);
  }
};

template <>
struct Elem<BIL_F16> {
  static constexpr int kBytes = 2;
  __device__ static __forceinline__ void group(const unsigned char* p, float (&x)[kGroup]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      float2 f = __half22float2(h);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  }
  __device__ static __forceinline__ float one(const unsigned char* p) {
    return __half2float(*reinterpret_cast<const __half*>(p));
  }
};

template <>
struct Elem<BIL_F32> {
  static constexpr int kBytes = 4;
  __device__ static __forceinline__ void group(const unsigned char* p, float (&x)[kGroup]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 16);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
  __device__ static __forceinline__ float one(const unsigned char* p) {
    return *reinterpret_cast<const float*>(p);
  }
};

// One tile's float32 (max, sum-exp) partial, computed by one warp from the
// tile's elements in shared memory.  The reduction order is fixed by the
// element positions alone:
//   * element p of the tile (global column t*tile_v + p) sits in group
//     g = p / 8 at slot j = p % 8; lane l takes groups l, l+32, l+64, ... in
//     increasing order; `valid` elements exist (the rest are past the
//     vocabulary and do not take part);
//   * max: exact, so its order does not matter (NaN never wins);
//   * sum: lane accumulator a_j (slot j) adds exp(x - m) for its groups in
//     increasing order; the lane's sum is ((a0+a1)+(a2+a3))+((a4+a5)+(a6+a7));
//     the warp's sum is the butterfly over lanes (xor 16, 8, 4, 2, 1);
//   * a tile whose max is -inf shifts by 0 instead, so it sums to 0 (or NaN
//     if it holds a NaN) and its max stays -inf.
// Nothing here depends on the row, the kernel or the launch geometry.
template <int DT>
__device__ __forceinline__ void tile_reduce(const unsigned char* tile, int valid, int lane,
                                            float& m_out, float& s_out) {
  constexpr int EB = Elem<DT>::kBytes;
  const int full_groups = valid / kGroup;
  const int rem = valid - full_groups * kGroup;  // elements in the ragged last group
  float m = -INFINITY;
  int g = lane;
#pragma unroll 4
  for (; g < full_groups; g += kLanes) {
    float x[kGroup];
    Elem<DT>::group(tile + static_cast<size_t>(g) * kGroup * EB, x);
#pragma unroll
    for (int j = 0; j < kGroup; ++j) m = fmaxf(m, x[j]);
  }
  if (rem != 0 && g == full_groups) {
#pragma unroll
    for (int j = 0; j < kGroup; ++j)
      if (j < rem) m = fmaxf(m, Elem<DT>::one(tile + (static_cast<size_t>(g) * kGroup + j) * EB));
  }
  m = warp_max(m);
  const float shift = (m == -INFINITY) ? 0.0f : m;

  float a[kGroup];
#pragma unroll
  for (int j = 0; j < kGroup; ++j) a[j] = 0.0f;
  g = lane;
#pragma unroll 4
  for (; g < full_groups; g += kLanes) {
    float x[kGroup];
    Elem<DT>::group(tile + static_cast<size_t>(g) * kGroup * EB, x);
#pragma unroll
    for (int j = 0; j < kGroup; ++j) a[j] = __fadd_rn(a[j], contract_exp(__fsub_rn(x[j], shift)));
  }
  if (rem != 0 && g == full_groups) {
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      if (j < rem) {
        const float x = Elem<DT>::one(tile + (static_cast<size_t>(g) * kGroup + j) * EB);
        a[j] = __fadd_rn(a[j], contract_exp(__fsub_rn(x, shift)));
      }
    }
  }
  float s = __fadd_rn(__fadd_rn(__fadd_rn(a[0], a[1]), __fadd_rn(a[2], a[3])),
                      __fadd_rn(__fadd_rn(a[4], a[5]), __fadd_rn(a[6], a[7])));
  s = warp_sum(s);
  m_out = m;
  s_out = s;
}

// The fixed-order merge of one row's T tile partials, by one warp (all lanes
// return the same value):
//   M = max_t m_t;  S = fma(s_t, exp(m_t - M), S) for t = 0, 1, ..., T-1
//   (one rounding per step, from S = 0);  LSE = M + log(S) (log: CUDA logf).
// M = -inf (no finite logit in the row) gives LSE = -inf, or NaN if a partial
// sum is NaN.  The exponentials are computed in parallel across lanes; the
// chain of fused multiply-adds is the same sequential chain in every lane.
__device__ __forceinline__ float merge_lse(const float* m, const float* s, int T, int lane) {
  float M = -INFINITY;
  for (int t = lane; t < T; t += kLanes) M = fmaxf(M, m[t]);
  M = warp_max(M);
  if (M == -INFINITY) {
    bool nan = false;
    for (int t = lane; t < T; t += kLanes) nan |= isnan(s[t]);
    return __any_sync(0xffffffffu, nan) ? __int_as_float(0x7fc00000) : -INFINITY;
  }
  float S = 0.0f;
  for (int t0 = 0; t0 < T; t0 += kLanes) {
    const int t = t0 + lane;
    float e = 0.0f, st = 0.0f;
    if (t < T) {
      e = contract_exp(__fsub_rn(m[t], M));
      st = s[t];
    }
    const int n = min(kLanes, T - t0);
    for (int j = 0; j < n; ++j) {
      const float ej = __shfl_sync(0xffffffffu, e, j);
      const float sj = __shfl_sync(0xffffffffu, st, j);
      S = __fmaf_rn(sj, ej, S);
    }
  }
  return __fadd_rn(M, logf(S));
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
constexpr long long kWaitLimitNs = 2000000000LL;  // 2 s per wait

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ long long global_ns() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Warp-wide wait until the phase with parity `parity` has completed.  Every
// lane polls (so every lane gets the barrier's acquire ordering) and the warp
// leaves together.  Returns false if the wait ran out, or if another warp of
// the block gave up (*abort set); the caller then stops.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, unsigned parity, volatile int* abort,
                                          unsigned code) {
  long long start = 0;
  for (unsigned spin = 0;; ++spin) {
    const bool done = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    if ((spin & 255u) == 255u) {
      int stop = 0;
      if ((threadIdx.x % kLanes) == 0) {
        const long long now = global_ns();
        if (start == 0) {
          start = now;
        } else if (*abort) {
          stop = 1;
        } else if (now - start > kWaitLimitNs) {
          atomicOr(&g_watchdog, code);
          *abort = 1;
          stop = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
  }
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
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

struct StreamParams {
  const unsigned char* logits;  // column 0 = global column tile_begin * tile_v
  int64_t n_rows, vocab, ld;    // ld in elements
  int tile_v, tile_begin, tile_end, num_tiles;
  const int64_t* targets;
  int64_t ignore_index;
  // fused outputs
  float* logp;
  float* lse;
  // partials outputs
  float* part_max;
  float* part_sum;
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
  int* abort;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline size_t stream_smem_bytes(int stages, unsigned stage_bytes, int row_slots,
                                                    int num_tiles, bool fused, Smem* out,
                                                    unsigned char* base) {
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
  off += sizeof(float) * (fused ? static_cast<size_t>(row_slots) * num_tiles : 0);
  const size_t ss = off;
  off += sizeof(float) * (fused ? static_cast<size_t>(row_slots) * num_tiles : 0);
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
    out->abort = reinterpret_cast<int*>(base + ab);
  }
  return off;
}

template <int DT, bool FUSED, bool BULK>
__global__ void __launch_bounds__(32 * 9) stream_kernel(const StreamParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  constexpr int EB = Elem<DT>::kBytes;
  Smem sm;
  stream_smem_bytes(p.stages, p.stage_bytes, p.row_slots, p.num_tiles, FUSED, &sm, smem_raw);
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

  const int tiles_here = p.tile_end - p.tile_begin;

  if (warp == 0) {
    // ---------------- producer warp ----------------
    const uint64_t policy = evict_first_policy();
    int64_t k = 0;      // units issued
    int64_t rows = 0;   // rows started (fused: row-slot uses)
    // The block's share of the work: whole rows (fused) or a contiguous range
    // of (row, tile) units (partials).
    int64_t u0, u1;
    if (FUSED) {
      u0 = p.n_rows * blockIdx.x / gridDim.x * tiles_here;
      u1 = p.n_rows * (blockIdx.x + 1) / gridDim.x * tiles_here;
    } else {
      const int64_t total = p.n_rows * tiles_here;
      u0 = total * blockIdx.x / gridDim.x;
      u1 = total * (blockIdx.x + 1) / gridDim.x;
    }
    bool ok = true;
    int64_t cur_row = -1, cur_target = 0;
    int cur_slot = 0;
    for (int64_t u = u0; u < u1 && ok; ++u) {
      const int64_t row = u / tiles_here;
      const int tile = p.tile_begin + static_cast<int>(u - row * tiles_here);
      if (row != cur_row) {
        cur_row = row;
        cur_target = p.targets[row];
        if (cur_target == p.ignore_index) {
          // Inactive row: its logits are never read.
          if (FUSED) {
            if (lane == 0) {
              p.logp[row] = 0.0f;
              if (p.lse != nullptr) p.lse[row] = 0.0f;
            }
          } else {
            // this block's units of the row: tiles [tile, tile + n)
            const int64_t n = min((row + 1) * tiles_here, u1) - u;
            for (int64_t i = lane; i < n; i += kLanes) {
              p.part_max[row * p.ld_part + tile + i] = -INFINITY;
              p.part_sum[row * p.ld_part + tile + i] = 0.0f;
            }
          }
          u = (row + 1) * tiles_here - 1;  // skip the row's remaining units
          continue;
        }
        if (FUSED) {
          cur_slot = static_cast<int>(rows % p.row_slots);
          const unsigned use = static_cast<unsigned>(rows / p.row_slots);
          ok = warp_wait(&sm.row_free[cur_slot], (use & 1u) ^ 1u, abort, kWatchRowSlot);
          if (!ok) break;
          if (lane == 0) {
            RowSlot& rs = sm.slots[cur_slot];
            rs.row = row;
            rs.target = cur_target;
            rs.target_logit = __int_as_float(0x7fc00000);
            rs.done = 0;
          }
          ++rows;
        }
      }
      const int stage = static_cast<int>(k % S);
      const unsigned fill = static_cast<unsigned>(k / S);
      ok = warp_wait(&sm.empty[stage], (fill & 1u) ^ 1u, abort, kWatchEmpty);
      if (!ok) break;
      const int64_t col0 = static_cast<int64_t>(tile) * p.tile_v;  // global column
      const int valid = static_cast<int>(min(static_cast<int64_t>(p.tile_v), p.vocab - col0));
      const unsigned char* src =
          p.logits + (row * p.ld + (col0 - static_cast<int64_t>(p.tile_begin) * p.tile_v)) * EB;
      unsigned char* dst = sm.ring + static_cast<size_t>(stage) * p.stage_bytes;
      if (lane == 0) {
        UnitDesc d;
        d.row = row;
        d.tile = tile;
        d.slot = cur_slot;
        sm.desc[stage] = d;
      }
      if (BULK) {
        if (lane == 0) {
          const unsigned bytes = static_cast<unsigned>(align_up(static_cast<size_t>(valid) * EB, 16));
          mbar_arrive_expect_tx(&sm.full[stage], bytes);
          bulk_g2s(dst, src, bytes, &sm.full[stage], policy);
        }
      } else {
        // Rows that are not 16-byte aligned: the producer warp copies the
        // tile element by element into the same shared-memory layout.
        for (int i = lane; i < valid; i += kLanes) {
          if (EB == 2) {
            reinterpret_cast<uint16_t*>(dst)[i] = reinterpret_cast<const uint16_t*>(src)[i];
          } else {
            reinterpret_cast<uint32_t*>(dst)[i] = reinterpret_cast<const uint32_t*>(src)[i];
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.full[stage]);
      }
      __syncwarp();
      ++k;
    }
    // One end marker per consumer warp: units k, k+1, ..., k+W-1 map to
    // consumers k % W, ..., so each consumer sees exactly one.
    for (int w = 0; w < W && ok; ++w, ++k) {
      const int stage = static_cast<int>(k % S);
      const unsigned fill = static_cast<unsigned>(k / S);
      ok = warp_wait(&sm.empty[stage], (fill & 1u) ^ 1u, abort, kWatchEmpty);
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
    }
    // Drain: no bulk copy of ours may still be landing in shared memory when
    // the block exits (consumers that gave up leave fills unconsumed).  The
    // latest fill of every used stage must have completed; normally they all
    // have and this costs one poll per stage.
    if (BULK && lane == 0) {
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
  const int cw = warp - 1;
  for (int64_t k = cw;; k += W) {
    const int stage = static_cast<int>(k % S);
    const unsigned fill = static_cast<unsigned>(k / S);
    if (!warp_wait(&sm.full[stage], fill & 1u, abort, kWatchFull)) break;
    const UnitDesc d = sm.desc[stage];
    if (d.row < 0) break;
    const unsigned char* tile = sm.ring + static_cast<size_t>(stage) * p.stage_bytes;
    const int64_t col0 = static_cast<int64_t>(d.tile) * p.tile_v;
    const int valid = static_cast<int>(min(static_cast<int64_t>(p.tile_v), p.vocab - col0));
    float m, s;
    tile_reduce<DT>(tile, valid, lane, m, s);
    // The target logit is copied from the tile that owns it, never summed.
    const int64_t target = FUSED ? sm.slots[d.slot].target : p.targets[d.row];
    const bool owner = target >= col0 && target < col0 + valid;
    float tl = 0.0f;
    if (owner) tl = Elem<DT>::one(tile + static_cast<size_t>(target - col0) * EB);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[stage]);  // the stage may be refilled now

    if (!FUSED) {
      if (lane == 0) {
        p.part_max[d.row * p.ld_part + d.tile] = m;
        p.part_sum[d.row * p.ld_part + d.tile] = s;
        if (owner) p.target_logit[d.row] = tl;
      }
      continue;
    }
    RowSlot& rs = sm.slots[d.slot];
    float* sm_m = sm.slot_m + static_cast<size_t>(d.slot) * p.num_tiles;
    float* sm_s = sm.slot_s + static_cast<size_t>(d.slot) * p.num_tiles;
    int before = 0;
    if (lane == 0) {
      sm_m[d.tile] = m;
      sm_s[d.tile] = s;
      if (owner) rs.target_logit = tl;
      __threadfence_block();
      before = atomicAdd(&rs.done, 1);
    }
    before = __shfl_sync(0xffffffffu, before, 0);
    if (before != p.num_tiles - 1) continue;
    // This warp reduced the row's last tile: merge the row.
    __threadfence_block();
    __syncwarp();
    const float L = merge_lse(sm_m, sm_s, p.num_tiles, lane);
    if (lane == 0) {
      const int64_t row = rs.row;
      const bool valid_target = rs.target >= 0 && rs.target < p.vocab;
      p.logp[row] = valid_target ? __fsub_rn(rs.target_logit, L) : __int_as_float(0x7fc00000);
      if (p.lse != nullptr) p.lse[row] = L;
      __threadfence_block();
      mbar_arrive(&sm.row_free[d.slot]);
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// Merge kernel: one warp per row, the same merge_lse as the fused forward.
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(256) merge_kernel(const float* __restrict__ part_max,
                                                    const float* __restrict__ part_sum, int64_t n_rows,
                                                    int num_tiles, int64_t ld_part,
                                                    const float* __restrict__ target_logit,
                                                    const int64_t* __restrict__ targets,
                                                    int64_t ignore_index, int64_t vocab, float* logp,
                                                    float* lse) {
  const int lane = threadIdx.x % kLanes;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / kLanes);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / kLanes) + threadIdx.x / kLanes;
       row < n_rows; row += warps) {
    const int64_t t = targets[row];
    if (t == ignore_index) {
      if (lane == 0) {
        logp[row] = 0.0f;
        if (lse != nullptr) lse[row] = 0.0f;
      }
      continue;
    }
    const float L = merge_lse(part_max + row * ld_part, part_sum + row * ld_part, num_tiles, lane);
    if (lane == 0) {
      const bool valid = t >= 0 && t < vocab;
      logp[row] = valid ? __fsub_rn(target_logit[row], L) : __int_as_float(0x7fc00000);
      if (lse != nullptr) lse[row] = L;
    }
  }
}

// ---------------------------------------------------------------------------
// Backward: dlogits[r, c] = g[r] * ([c == t_r] - exp(x[r, c] - lse[r])).
// Work unit: (row, chunk of kBwdChunk columns), spread over a persistent grid.
// Purely elementwise given lse and g, so the bits cannot depend on the unit
// size, the grid, or whether a row is read in 16-byte vectors or one element
// at a time.
// ---------------------------------------------------------------------------

constexpr int kBwdThreads = 256;
constexpr int kBwdGroupsPerThread = 4;
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

// One element of the gradient, exactly as the formula reads.
__device__ __forceinline__ float grad_elem(float x, float L, float g, bool is_target) {
  const float p = contract_exp(__fsub_rn(x, L));
  return __fmul_rn(g, __fsub_rn(is_target ? 1.0f : 0.0f, p));
}

template <int DT>
__device__ __forceinline__ void load_group_global(const unsigned char* p, float (&x)[kGroup]) {
  if (Elem<DT>::kBytes == 2) {
    const uint4 v = __ldcs(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (DT == BIL_BF16) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
      } else {
        __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
        float2 f = __half22float2(h);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
      }
    }
  } else {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
    const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}

template <int DT, int OT, bool VEC>
__global__ void __launch_bounds__(kBwdThreads) bwd_kernel(
    const unsigned char* __restrict__ logits, int64_t n_rows, int64_t vocab, int64_t ld,
    const int64_t* __restrict__ targets, int64_t ignore_index, const float* __restrict__ lse,
    const float* __restrict__ grad, unsigned char* __restrict__ dlogits, int64_t ld_out,
    int64_t out_cols) {
  constexpr int EB = Elem<DT>::kBytes;
  constexpr int OB = Out<OT>::kBytes;
  const int64_t chunks = (out_cols + kBwdChunk - 1) / kBwdChunk;
  const int64_t units = n_rows * chunks;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int64_t row = u / chunks;
    const int64_t c0 = (u - row * chunks) * kBwdChunk;
    const int64_t c1 = min(c0 + kBwdChunk, out_cols);
    const int64_t t = targets[row];
    unsigned char* out = dlogits + row * ld_out * OB;
    const bool active = t != ignore_index;
    const bool valid_target = t >= 0 && t < vocab;
    const float L = active ? lse[row] : 0.0f;
    const float g = active ? grad[row] : 0.0f;
    // columns [c0, min(c1, vocab)) hold gradient, [max(c0, vocab), c1) are pad
    const int64_t v1 = min(c1, vocab);
    if (!active || !valid_target) {
      const float fill = active ? __int_as_float(0x7fc00000) : 0.0f;
      for (int64_t c = c0 + threadIdx.x; c < v1; c += kBwdThreads) Out<OT>::store1(out + c * OB, fill);
    } else if (VEC) {
      // c0 is a multiple of 8; groups fully inside [c0, v1) go by 16-byte
      // vectors, all of a thread's loads issued before any arithmetic.
      const unsigned char* in = logits + row * ld * EB;
      const int64_t gend = c0 + ((v1 - c0) / kGroup) * kGroup;
      float x[kBwdGroupsPerThread][kGroup];
#pragma unroll
      for (int i = 0; i < kBwdGroupsPerThread; ++i) {
        const int64_t c = c0 + (static_cast<int64_t>(i) * kBwdThreads + threadIdx.x) * kGroup;
        if (c < gend) load_group_global<DT>(in + c * EB, x[i]);
      }
#pragma unroll
      for (int i = 0; i < kBwdGroupsPerThread; ++i) {
        const int64_t c = c0 + (static_cast<int64_t>(i) * kBwdThreads + threadIdx.x) * kGroup;
        if (c < gend) {
          float y[kGroup];
#pragma unroll
          for (int j = 0; j < kGroup; ++j) y[j] = grad_elem(x[i][j], L, g, c + j == t);
          Out<OT>::store8(out + c * OB, y);
        }
      }
      for (int64_t c = gend + threadIdx.x; c < v1; c += kBwdThreads)
        Out<OT>::store1(out + c * OB, grad_elem(Elem<DT>::one(in + c * EB), L, g, c == t));
    } else {
      const unsigned char* in = logits + row * ld * EB;
      for (int64_t c = c0 + threadIdx.x; c < v1; c += kBwdThreads)
        Out<OT>::store1(out + c * OB, grad_elem(Elem<DT>::one(in + c * EB), L, g, c == t));
    }
    for (int64_t c = max(c0, vocab) + threadIdx.x; c < c1; c += kBwdThreads) Out<OT>::store1(out + c * OB, 0.0f);
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------

int elem_bytes(int dtype) {
  switch (dtype) {
    case BIL_F32: return 4;
    case BIL_BF16: return 2;
    case BIL_F16: return 2;
    default: return 0;
  }
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct DeviceInfo {
  int sms = 0;
  int max_smem_optin = 0;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];

int device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BIL_E_CUDA;
  DeviceInfo& d = g_devices[dev];
  if (d.sms == 0) {
    int sms = 0, smem = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return BIL_E_CUDA;
    if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return BIL_E_CUDA;
    d.max_smem_optin = smem;
    d.sms = sms;  // written last: a non-zero sms marks the entry complete
  }
  *out = d;
  return BIL_OK;
}

// Check active targets on the host (validate=1).  Copies the targets in
// chunks through a stack buffer; synchronises the stream.
int check_targets_host(const int64_t* targets, int64_t n, int64_t ignore_index, int64_t vocab,
                       cudaStream_t stream) {
  constexpr int64_t kChunk = 2048;
  int64_t buf[kChunk];
  for (int64_t i = 0; i < n; i += kChunk) {
    const int64_t m = std::min(kChunk, n - i);
    if (cudaMemcpyAsync(buf, targets + i, m * sizeof(int64_t), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
      return BIL_E_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return BIL_E_CUDA;
    for (int64_t j = 0; j < m; ++j) {
      const int64_t t = buf[j];
      if (t != ignore_index && (t < 0 || t >= vocab)) return BIL_E_TARGET_RANGE;
    }
  }
  return BIL_OK;
}

// Pipeline shape for a stage size: about 96 KB of ring per block so that two
// blocks share an SM, at least two stages, one consumer warp per two stages.
struct StreamShape {
  int stages, consumers, row_slots;
  size_t smem;
};

StreamShape stream_shape(unsigned stage_bytes, int num_tiles, bool fused) {
  StreamShape s;
  s.stages = static_cast<int>(std::max<size_t>(2, std::min<size_t>(32, (96u * 1024u) / stage_bytes)));
  s.consumers = std::max(1, std::min(8, s.stages / 2));
  s.row_slots = fused ? 4 : 0;
  s.smem = stream_smem_bytes(s.stages, stage_bytes, s.row_slots, num_tiles, fused, nullptr, nullptr);
  return s;
}

template <int DT, bool FUSED, bool BULK>
int launch_stream_t(const StreamParams& p0, cudaStream_t stream) {
  DeviceInfo dev;
  if (int st = device_info(&dev)) return st;
  StreamParams p = p0;
  StreamShape shape = stream_shape(p.stage_bytes, p.num_tiles, FUSED);
  if (shape.smem > static_cast<size_t>(dev.max_smem_optin)) return BIL_E_UNSUPPORTED;
  p.stages = shape.stages;
  p.consumers = shape.consumers;
  p.row_slots = shape.row_slots;
  auto kernel = stream_kernel<DT, FUSED, BULK>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(shape.smem)) != cudaSuccess)
    return BIL_E_CUDA;
  const int threads = kLanes * (1 + shape.consumers);
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, shape.smem) != cudaSuccess)
    return BIL_E_CUDA;
  per_sm = std::max(1, per_sm);
  const int64_t tiles_here = p.tile_end - p.tile_begin;
  const int64_t work = FUSED ? p.n_rows : p.n_rows * tiles_here;
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(work, static_cast<int64_t>(dev.sms) * per_sm));
  kernel<<<static_cast<unsigned>(grid), threads, shape.smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? BIL_OK : BIL_E_CUDA;
}

template <bool FUSED>
int launch_stream(int dtype, const StreamParams& p, cudaStream_t stream) {
  const int eb = elem_bytes(dtype);
  const bool bulk = aligned(p.logits, 16) && (p.ld * eb) % 16 == 0;
  switch (dtype) {
    case BIL_BF16:
      return bulk ? launch_stream_t<BIL_BF16, FUSED, true>(p, stream) : launch_stream_t<BIL_BF16, FUSED, false>(p, stream);
    case BIL_F16:
      return bulk ? launch_stream_t<BIL_F16, FUSED, true>(p, stream) : launch_stream_t<BIL_F16, FUSED, false>(p, stream);
    case BIL_F32:
      return bulk ? launch_stream_t<BIL_F32, FUSED, true>(p, stream) : launch_stream_t<BIL_F32, FUSED, false>(p, stream);
    default:
      return BIL_E_DTYPE;
  }
}

int check_tile(int dtype, int64_t vocab, int32_t tile_v, int64_t* num_tiles) {
  const int eb = elem_bytes(dtype);
  if (eb == 0) return BIL_E_DTYPE;
  if (tile_v <= 0 || tile_v % kGroup != 0) return BIL_E_INVALID_ARG;
  if (static_cast<int64_t>(tile_v) * eb > BIL_MAX_TILE_BYTES) return BIL_E_UNSUPPORTED;
  *num_tiles = (vocab + tile_v - 1) / tile_v;
  if (*num_tiles > INT32_MAX) return BIL_E_UNSUPPORTED;
  return BIL_OK;
}

template <int DT, int OT>
int launch_bwd_t(bool vec, const unsigned char* logits, int64_t n_rows, int64_t vocab, int64_t ld,
                 const int64_t* targets, int64_t ignore_index, const float* lse, const float* grad,
                 unsigned char* dlogits, int64_t ld_out, int64_t out_cols, cudaStream_t stream) {
  DeviceInfo dev;
  if (int st = device_info(&dev)) return st;
  auto kernel = vec ? bwd_kernel<DT, OT, true> : bwd_kernel<DT, OT, false>;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kBwdThreads, 0) != cudaSuccess)
    return BIL_E_CUDA;
  per_sm = std::max(1, per_sm);
  const int64_t units = n_rows * ((out_cols + kBwdChunk - 1) / kBwdChunk);
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(units, static_cast<int64_t>(dev.sms) * per_sm));
  kernel<<<static_cast<unsigned>(grid), kBwdThreads, 0, stream>>>(logits, n_rows, vocab, ld, targets, ignore_index,
                                                                  lse, grad, dlogits, ld_out, out_cols);
  return cudaGetLastError() == cudaSuccess ? BIL_OK : BIL_E_CUDA;
}

template <int DT>
int launch_bwd_dt(int out_dtype, bool vec, const unsigned char* logits, int64_t n_rows, int64_t vocab,
                  int64_t ld, const int64_t* targets, int64_t ignore_index, const float* lse,
                  const float* grad, unsigned char* dlogits, int64_t ld_out, int64_t out_cols,
                  cudaStream_t stream) {
  switch (out_dtype) {
    case BIL_F32:
      return launch_bwd_t<DT, BIL_F32>(vec, logits, n_rows, vocab, ld, targets, ignore_index, lse, grad, dlogits,
                                       ld_out, out_cols, stream);
    case BIL_BF16:
      return launch_bwd_t<DT, BIL_BF16>(vec, logits, n_rows, vocab, ld, targets, ignore_index, lse, grad,
                                        dlogits, ld_out, out_cols, stream);
    case BIL_F16:
      return launch_bwd_t<DT, BIL_F16>(vec, logits, n_rows, vocab, ld, targets, ignore_index, lse, grad, dlogits,
                                       ld_out, out_cols, stream);
    default:
      return BIL_E_DTYPE;
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------

extern "C" {

const char* bil_contract_id(void) {
  return "bil.v1"
         ";tile=fixed tile_v columns, valid columns < vocab"
         ";lanes=32x8: lane l takes 8-element groups l, l+32, ... in order"
         ";max=exact"
         ";exp(a)=ex2.approx.ftz.f32(a*rn log2e), a=x-rn m"
         ";lane_sum=8 slot accumulators, ((a0+a1)+(a2+a3))+((a4+a5)+(a6+a7))"
         ";warp_sum=butterfly xor 16,8,4,2,1"
         ";merge=M=max m_t; S=fma(s_t,exp(m_t-M),S) t=0..T-1; LSE=M+rn logf(S)"
         ";logp=x_t-rn LSE"
         ";bwd=g*rn(onehot-rn exp(x-rn lse)), store rn";
}

const char* bil_status_string(int status) {
  switch (status) {
    case BIL_OK: return "ok";
    case BIL_E_INVALID_ARG: return "invalid argument";
    case BIL_E_DTYPE: return "unsupported element type";
    case BIL_E_ALIGN: return "pointer not aligned to its element size";
    case BIL_E_TARGET_RANGE: return "active target outside [0, vocab)";
    case BIL_E_CUDA: return "CUDA runtime error";
    case BIL_E_UNSUPPORTED: return "beyond this build's limits";
    default: return "unknown status";
  }
}

int bil_logp_fwd(const void* logits, int dtype, int64_t n_rows, int64_t vocab, int64_t ld,
                 const int64_t* target_ids, int64_t ignore_index, int32_t tile_v, float* logp, float* lse,
                 int validate, bil_stream_t stream) {
  if (n_rows < 0 || vocab < 1 || ld < vocab) return BIL_E_INVALID_ARG;
  int64_t num_tiles = 0;
  if (int st = check_tile(dtype, vocab, tile_v, &num_tiles)) return st;
  if (n_rows == 0) return BIL_OK;
  if (logits == nullptr || target_ids == nullptr || logp == nullptr) return BIL_E_INVALID_ARG;
  const int eb = elem_bytes(dtype);
  if (!aligned(logits, eb) || !aligned(target_ids, 8) || !aligned(logp, 4) || (lse && !aligned(lse, 4)))
    return BIL_E_ALIGN;
  if (num_tiles > BIL_MAX_FUSED_TILES) return BIL_E_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (validate) {
    if (int st = check_targets_host(target_ids, n_rows, ignore_index, vocab, s)) return st;
  }
  StreamParams p{};
  p.logits = static_cast<const unsigned char*>(logits);
  p.n_rows = n_rows;
  p.vocab = vocab;
  p.ld = ld;
  p.tile_v = tile_v;
  p.tile_begin = 0;
  p.tile_end = static_cast<int>(num_tiles);
  p.num_tiles = static_cast<int>(num_tiles);
  p.targets = target_ids;
  p.ignore_index = ignore_index;
  p.logp = logp;
  p.lse = lse;
  p.stage_bytes = static_cast<unsigned>(static_cast<size_t>(tile_v) * eb);
  return launch_stream<true>(dtype, p, s);
}

int bil_logp_tile_partials(const void* logits, int dtype, int64_t n_rows, int64_t vocab, int64_t ld,
                           int32_t tile_v, int32_t tile_begin, int32_t tile_end, const int64_t* target_ids,
                           int64_t ignore_index, float* part_max, float* part_sum, int64_t ld_part,
                           float* target_logit, bil_stream_t stream) {
  if (n_rows < 0 || vocab < 1) return BIL_E_INVALID_ARG;
  int64_t num_tiles = 0;
  if (int st = check_tile(dtype, vocab, tile_v, &num_tiles)) return st;
  if (tile_begin < 0 || tile_end <= tile_begin || tile_end > num_tiles) return BIL_E_INVALID_ARG;
  if (ld_part < num_tiles) return BIL_E_INVALID_ARG;
  // The shard holds global columns [tile_begin*tile_v, min(tile_end*tile_v, vocab)).
  const int64_t shard_cols = std::min<int64_t>(static_cast<int64_t>(tile_end) * tile_v, vocab) -
                             static_cast<int64_t>(tile_begin) * tile_v;
  if (ld < shard_cols) return BIL_E_INVALID_ARG;
  if (n_rows == 0) return BIL_OK;
  if (logits == nullptr || target_ids == nullptr || part_max == nullptr || part_sum == nullptr ||
      target_logit == nullptr)
    return BIL_E_INVALID_ARG;
  const int eb = elem_bytes(dtype);
  if (!aligned(logits, eb) || !aligned(target_ids, 8) || !aligned(part_max, 4) || !aligned(part_sum, 4) ||
      !aligned(target_logit, 4))
    return BIL_E_ALIGN;
  StreamParams p{};
  p.logits = static_cast<const unsigned char*>(logits);
  p.n_rows = n_rows;
  p.vocab = vocab;
  p.ld = ld;
  p.tile_v = tile_v;
  p.tile_begin = tile_begin;
  p.tile_end = tile_end;
  p.num_tiles = static_cast<int>(num_tiles);
  p.targets = target_ids;
  p.ignore_index = ignore_index;
  p.part_max = part_max;
  p.part_sum = part_sum;
  p.ld_part = ld_part;
  p.target_logit = target_logit;
  p.stage_bytes = static_cast<unsigned>(static_cast<size_t>(tile_v) * eb);
  return launch_stream<false>(dtype, p, reinterpret_cast<cudaStream_t>(stream));
}

int bil_logp_merge(const float* part_max, const float* part_sum, int64_t n_rows, int32_t num_tiles,
                   int64_t ld_part, const float* target_logit, const int64_t* target_ids, int64_t ignore_index,
                   int64_t vocab, float* logp, float* lse, int validate, bil_stream_t stream) {
  if (n_rows < 0 || num_tiles < 1 || ld_part < num_tiles || vocab < 1) return BIL_E_INVALID_ARG;
  if (n_rows == 0) return BIL_OK;
  if (part_max == nullptr || part_sum == nullptr || target_logit == nullptr || target_ids == nullptr ||
      logp == nullptr)
    return BIL_E_INVALID_ARG;
  if (!aligned(part_max, 4) || !aligned(part_sum, 4) || !aligned(target_logit, 4) || !aligned(target_ids, 8) ||
      !aligned(logp, 4) || (lse && !aligned(lse, 4)))
    return BIL_E_ALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (validate) {
    if (int st = check_targets_host(target_ids, n_rows, ignore_index, vocab, s)) return st;
  }
  DeviceInfo dev;
  if (int st = device_info(&dev)) return st;
  const int threads = 256;
  const int64_t rows_per_block = threads / kLanes;
  const int64_t grid = std::max<int64_t>(
      1, std::min<int64_t>((n_rows + rows_per_block - 1) / rows_per_block, static_cast<int64_t>(dev.sms) * 8));
  merge_kernel<<<static_cast<unsigned>(grid), threads, 0, s>>>(part_max, part_sum, n_rows, num_tiles, ld_part,
                                                                target_logit, target_ids, ignore_index, vocab,
                                                                logp, lse);
  return cudaGetLastError() == cudaSuccess ? BIL_OK : BIL_E_CUDA;
}

int bil_logp_bwd(const void* logits, int dtype, int64_t n_rows, int64_t vocab, int64_t ld,
                 const int64_t* target_ids, int64_t ignore_index, const float* lse, const float* grad_logp,
                 void* dlogits, int dlogits_dtype, int64_t ld_out, int64_t out_cols, bil_stream_t stream) {
  const int eb = elem_bytes(dtype);
  const int ob = elem_bytes(dlogits_dtype);
  if (eb == 0 || ob == 0) return BIL_E_DTYPE;
  if (n_rows < 0 || vocab < 1 || ld < vocab || out_cols < vocab || ld_out < out_cols) return BIL_E_INVALID_ARG;
  if (n_rows == 0) return BIL_OK;
  if (logits == nullptr || target_ids == nullptr || lse == nullptr || grad_logp == nullptr || dlogits == nullptr)
    return BIL_E_INVALID_ARG;
  if (!aligned(logits, eb) || !aligned(target_ids, 8) || !aligned(lse, 4) || !aligned(grad_logp, 4) ||
      !aligned(dlogits, ob))
    return BIL_E_ALIGN;
  const bool vec = aligned(logits, 16) && (ld * eb) % 16 == 0 && aligned(dlogits, 16) && (ld_out * ob) % 16 == 0;
  const unsigned char* in = static_cast<const unsigned char*>(logits);
  unsigned char* out = static_cast<unsigned char*>(dlogits);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (dtype) {
    case BIL_BF16:
      return launch_bwd_dt<BIL_BF16>(dlogits_dtype, vec, in, n_rows, vocab, ld, target_ids, ignore_index, lse,
                                     grad_logp, out, ld_out, out_cols, s);
    case BIL_F16:
      return launch_bwd_dt<BIL_F16>(dlogits_dtype, vec, in, n_rows, vocab, ld, target_ids, ignore_index, lse,
                                    grad_logp, out, ld_out, out_cols, s);
    case BIL_F32:
      return launch_bwd_dt<BIL_F32>(dlogits_dtype, vec, in, n_rows, vocab, ld, target_ids, ignore_index, lse,
                                    grad_logp, out, ld_out, out_cols, s);
    default:
      return BIL_E_DTYPE;
  }
}

int bil_watchdog_status(unsigned int* flags, int clear) {
  if (flags == nullptr) return BIL_E_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return BIL_E_CUDA;
  if (cudaMemcpyFromSymbol(flags, g_watchdog, sizeof(unsigned int)) != cudaSuccess) return BIL_E_CUDA;
  if (clear) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_watchdog, &zero, sizeof(unsigned int)) != cudaSuccess) return BIL_E_CUDA;
  }
  return BIL_OK;
}

}  // extern "C"
