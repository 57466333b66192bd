// Fused LM-head + selected-token log-probability ("linear logp") for sm_103a.
//
// Operator: "[RFC][ROCm] End-to-end optimization of bitwise VIME R/R beyond
// native P/P", section "Workstream 3: fused ROCm LM-head and linear logp":
// the LM-head projection z = hidden . weight^T and the vocabulary statistics
// of the "Batch-Invariant LogP" operator ("Tensor Parallel", steps 1-6) are
// one operation.  Each vocabulary tile's (max, sum-exp[, entropy statistic],
// target logit) is produced from the projection's accumulator, without
// storing the [rows, vocabulary] logits unless the caller asks for them, and
// the tiles are then merged in the operator's one fixed order (the library's
// merge kernel).  The C ABI is declared in include/bil.h.
//
// One GEMM body C = A . B^T (16-bit operands), persistent, one block per SM,
// warp-specialised:
//   warp 0      TMA producer: 128-row A tile and 256-row B tile per 64-element
//               K block, 128-byte swizzled, into a 4-stage ring;
//   warp 1      MMA issuer: one thread issues tcgen05.mma (bf16/fp16 in, fp32
//               accumulate in tensor memory), K blocks in increasing order,
//               four K=16 steps each; two accumulator buffers of 256 columns;
//   warps 2-5   epilogue: thread i of the warp reading lanes [32q, 32q+32)
//               owns row 32q+i of the tile and reads its 256 columns from
//               tensor memory; a large output (dZ, the optional logits) goes
//               out 32 rows x 64 bytes at a time through two staging boxes
//               of the warp's own and TMA stores;
//   warp 6      the store GEMMs' lockstep service (see lockstep_service).
// The accumulator of one tile is read while the next tile's MMAs run.  Three
// epilogues make three kernels:
//   linear_partials_kernel   forward: A = hidden, B = weight; the tile's
//                            partial of the operator (and, optionally, the
//                            logits);
//   linear_grad_kernel       backward: the same projection recomputed; dZ by
//                            the logits path's gradient formula, stored as
//                            [rows, vocab];
//   linear_store_kernel      backward: dhidden = dZ . W and dweight =
//                            dZ^T . hidden, stored as they are.  Each operand
//                            is read where it lies, K-major ([rows, K]) or
//                            MN-major ([K, rows], copied in 64 x 64 boxes);
//                            from 256 rows on the work unit is two 128-row A
//                            tiles sharing one B tile (a 3-stage ring of
//                            64 KB stages, both accumulators in tensor memory
//                            at once).
//
// What fixes the bits of z[r, c] is the K order (K blocks in order, four
// K=16 steps each, from a zeroed accumulator), the same for every row and
// every tile, and what fixes the partial is the per-thread reduction order
// below; neither depends on the number of rows, the row's position, the
// launch geometry or the vocabulary split, so the result is batch-invariant
// and split-invariant like the logits path.

#include "../../include/bil.h"
#include "device_common.cuh"
#include "internal.h"

#include <cuda.h>  // CUtensorMap and its enums (types only; the encoder is fetched at run time)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>

namespace {

__device__ unsigned int g_watchdog_linear;

constexpr unsigned kWatchAccFull = 32u;    // epilogue waited too long for an accumulator
constexpr unsigned kWatchStageFree = 64u;  // producer waited too long for a free stage
constexpr unsigned kWatchMma = 128u;       // MMA issuer waited too long for a stage or an accumulator
constexpr unsigned kWatchOwnDrain = 256u;  // producer or MMA issuer waited too long for its own work

constexpr int kBM = 128;      // rows per tile: one tensor-memory lane per row
constexpr int kBN = 256;      // vocabulary columns per tile = the operator's tile width here
constexpr int kBK = 64;       // K per stage: 64 x 16 bits = one 128-byte swizzle row
constexpr int kUmmaK = 16;    // K of one tcgen05.mma kind::f16
constexpr int kStages = 4;
constexpr unsigned kStageABytes = kBM * kBK * 2;  // 16 KB
constexpr unsigned kStageBBytes = kBN * kBK * 2;  // 32 KB
constexpr unsigned kStageBytes = kStageABytes + kStageBBytes;
constexpr int kAccCols = kBN;            // one 32-bit tensor-memory column per output column
constexpr uint32_t kTmemCols = 2 * kAccCols;  // two accumulator buffers: 512 columns
constexpr int kEpiWarps = 4;
constexpr int kSyncWarp = 2 + kEpiWarps;  // the store GEMMs' lockstep (see lockstep_service)
constexpr int kThreads = 32 * (kSyncWarp + 1);
constexpr int kChunk = 32;               // columns per tensor-memory load
constexpr int kMGroup = 32;              // row tiles per raster group (L2 reuse of the weight tiles)

static_assert(BIL_LINEAR_TILE_V == kBN, "the C ABI's tile width is the kernel's N tile");

struct alignas(8) LinearSmem {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
  // lockstep of the store GEMMs: the copy thread's position (K blocks issued),
  // the position it may issue up to, and whether it has issued everything
  uint32_t sync_pos;
  uint32_t sync_allowed;
  int sync_done;
};

// The epilogues that store a large output (the gradient pass's dZ, the
// forward's optional logits) hand it to TMA through per-warp staging boxes in
// shared memory (1), or store it with per-thread vector stores (0).
#ifndef BIL_EPILOGUE_TMA_STORE
#define BIL_EPILOGUE_TMA_STORE 1
#endif
constexpr int kStoreBox = 32;  // rows and columns of one dZ store box: a warp's rows, one TMEM chunk
constexpr uint32_t kStoreBoxBytes = kStoreBox * kStoreBox * 2;           // 2 KB of 16-bit elements
constexpr size_t kStagingBytes = BIL_EPILOGUE_TMA_STORE ? 4 * 2 * kStoreBoxBytes : 0;  // 4 warps x 2 buffers
constexpr size_t kSmemBytes = 1024 /* alignment slack */ + kStages * size_t(kStageBytes) + sizeof(LinearSmem) +
                              (BIL_EPILOGUE_TMA_STORE ? 1024 + kStagingBytes : 0);

// What the epilogue warps do with a finished accumulator tile.
enum EpilogueMode {
  kModePartials = 0,  // the operator's tile partials (and, optionally, the logits)
  kModeGrad = 1,      // dZ = d(g logp + gh H)/dz, stored as 16-bit in [rows, vocab] and [vocab, rows]
  kModeStore = 2,     // C = A . B^T stored as it is (float32, or rounded to 16 bits)
};

struct LinearParams {
  int64_t n_rows;       // rows of A (valid output rows)
  int64_t shard_cols;   // rows of B (valid output columns): weight rows of the shard in the forward
  int tile_begin;       // global tile index of the shard's first column
  int num_n;            // tiles of the shard
  int num_m;            // row tiles
  int k_blocks;         // ceil(hidden / kBK)
  const int64_t* targets;
  int64_t ignore_index;
  float rcp;
  float* part_max;
  float* part_sum;
  float* part_ent;
  int64_t ld_part;
  float* target_logit;
  unsigned char* logits;  // NULL: not stored
  int logits_dtype;
  int64_t ld_logits;
  uint32_t idesc;
  unsigned a_box_bytes;  // bytes one A copy brings: its box's rows (kBM, or fewer for a batch of
                         // fewer rows) x kBK 16-bit columns
  int m_group;          // row tiles per raster group
  // kModeGrad
  const float* lse;
  const float* grad_logp;
  const float* entropy;        // with grad_entropy: the forward's entropy
  const float* grad_entropy;   // NULL: no entropy term
  int64_t vocab;               // targets outside [0, vocab) give NaN rows
  unsigned char* dz;           // [n_rows, ld_dz] 16-bit
  int64_t ld_dz;
  // kModeStore
  unsigned char* out;          // [n_rows, ld_out]
  int out_dtype;
  int64_t ld_out;
  unsigned sync_tag;           // non-zero: the copy threads keep in step (see lockstep_service)
  int a_mn, b_mn;              // 1: the operand is stored [K, rows] (rows contiguous), else [rows, K]
};

// ---------------------------------------------------------------------------
// tcgen05 / TMA wrappers.
// ---------------------------------------------------------------------------

// Instruction descriptor of tcgen05.mma kind::f16: D float32 (bits 4-5 = 1),
// A and B bf16 (bits 7-9, 10-12 = 1) or fp16 (0), A and B K-major (bits 15,
// 16 = 0) or MN-major (1), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t make_idesc(bool bf16, bool a_mn = false, bool b_mn = false) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(kBN >> 3) << 17) |
         (static_cast<uint32_t>(kBM >> 4) << 24);
}

// Shared-memory matrix descriptor of a K-major operand stored the way a TMA
// load with 128-byte swizzle writes it: rows of 128 bytes (64 elements of K),
// 8-row groups 1024 bytes apart (stride byte offset), start address >> 4 in
// bits 0-13, leading byte offset (unused for this layout) 16 bytes, the fixed
// 0b001 in bits 46-48, swizzle mode 2 (128 bytes) in bits 61-63.  The 8-row
// groups start on 1024-byte boundaries, so the base offset is 0; a K step
// within the 128-byte row advances the start address by 32 bytes.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(16 >> 4) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// The same for an MN-major operand (rows contiguous in memory), as TMA loads
// with 128-byte swizzle write it in boxes of 64 rows x 64 K: each K index is
// one 128-byte line of 64 consecutive rows, 8 K indices make a 1024-byte
// swizzle atom (stride byte offset between the atoms along K), and the next
// 64 rows are the next box, kMnBoxBytes further on (leading byte offset).  A
// K step of 16 advances the start address by 16 lines = 2048 bytes, two whole
// atoms.
constexpr int kMnBox = 64;                                // rows (and K) per box of an MN-major operand
constexpr uint32_t kMnBoxBytes = kMnBox * kBK * 2;        // 8 KB
__device__ __forceinline__ uint64_t smem_desc_mn(uint32_t addr) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(kMnBoxBytes >> 4) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// One box from shared memory to global memory (the tensor map's box; parts
// past the matrix are not written), in this thread's current bulk group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int c0, int c1, const void* src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Until at most one of this thread's bulk groups still reads shared memory.
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// Until all of this thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D (tensor memory) = A . B^T (+ D when accumulate != 0), one thread.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 consecutive 32-bit columns of this thread's tensor-memory lane, waited
// for in the same statement (so no use of the registers can be scheduled
// before the data has arrived).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[kChunk]) {
  __syncwarp();  // the load is warp-wide (.sync.aligned): the warp must be converged
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Row tile m and column tile n of work unit u: groups of `group` row tiles;
// within a group the row tile varies fastest, so the blocks working at one
// time share a few B tiles (and their A tiles) through L2.
__device__ __forceinline__ void unit_coords(int64_t u, int num_m, int num_n, int group, int& m, int& n) {
  const int64_t per_group = static_cast<int64_t>(group) * num_n;
  const int g = static_cast<int>(u / per_group);
  const int r = static_cast<int>(u - g * per_group);
  const int m0 = g * group;
  const int gm = min(group, num_m - m0);
  n = r / gm;
  m = m0 + (r - n * gm);
}

// A warp hands one 2 KB box (32 rows of 64 bytes: 32 16-bit or 16 float32
// values per row) to TMA: each lane writes its row's four 16-byte words into
// the warp's next staging buffer (two, used in turn), and lane 0 stores the
// box at (column x, row y) of `map` once the store that used the buffer before
// has read it.  `issued` counts the warp's boxes.
__device__ __forceinline__ void store_box(unsigned char* staging, const CUtensorMap* map, int x, int y, int lane,
                                          uint32_t& issued, const uint32_t (&w)[16]) {
  unsigned char* box = staging + (issued & 1u) * kStoreBoxBytes;
  if (lane == 0) bulk_wait_read_1();
  __syncwarp();
  uint4* dst = reinterpret_cast<uint4*>(box + lane * 64);
#pragma unroll
  for (int j = 0; j < 4; ++j) dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  fence_proxy_async_smem();  // the writes above, before the bulk copy reads them
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, x, y, box);
    bulk_commit();
  }
  ++issued;
}

// ---------------------------------------------------------------------------
// The epilogue of one row of one tile: the tile partial of the operator, over
// the tile's valid columns [0, vcols), from the float32 accumulator acc.
//
//   m_acc = max over valid c of acc_c (exact);  m = m_acc *rn rcp
//   t_c = (acc_c -rn m_acc) *rn c, c = rcp *rn log2e (m_acc = -inf: shift 0),
//   e_c = 2^t_c (ex2.approx), as the logits path's tile terms; the target
//   logit is acc_t *rn rcp
//   slot accumulators a_j, j = 0..7, take e_c for c = 8g + j, g = 0, 1, ...,
//   31 in order; s = ((a0+a1)+(a2+a3))+((a4+a5)+(a6+a7)); the entropy sum
//   u = ln2 *rn (sum e_c * max(t_c, -FLT_MAX) in the same slots and tree, one
//   fma per column).
//
// This is one lane of the logits path's in-tile order with 32 groups and no
// warp butterfly: a tile here is one thread's row.
// ---------------------------------------------------------------------------

// With `box_map` (the logits' store map), the logits go out through the warp's
// staging boxes with TMA (all 32 lanes of the warp call this together; `store`
// and out_row are then unused, and rows or columns past the matrix are not
// written); else `store` rows write them with vector stores.
template <bool ENT>
__device__ __forceinline__ void row_partial(uint32_t taddr, int vcols, float rcp, int64_t tloc, bool store,
                                            unsigned char* out_row, int out_dtype, float& m_out, float& s_out,
                                            float& u_out, float& tl_out, const CUtensorMap* box_map = nullptr,
                                            unsigned char* staging = nullptr, int box_x = 0, int box_y = 0,
                                            int lane = 0, uint32_t* issued = nullptr) {
  uint32_t r[kChunk];
  float mx = -INFINITY;  // max of the unscaled accumulator
  float tl = 0.0f;
#pragma unroll 1
  for (int c0 = 0; c0 < kBN; c0 += kChunk) {
    tmem_ld32(taddr + c0, r);
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      const float acc = __uint_as_float(r[j]);
      if (c0 + j < vcols) mx = fmaxf(mx, acc);
      if (c0 + j == tloc) tl = __fmul_rn(acc, rcp);
    }
    if (box_map != nullptr && c0 < vcols) {
      if (out_dtype == BIL_F32) {  // two boxes of 16 columns
        uint32_t w0[16], w1[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          w0[j] = r[j];
          w1[j] = r[16 + j];
        }
        store_box(staging, box_map, box_x + c0, box_y, lane, *issued, w0);
        store_box(staging, box_map, box_x + c0 + 16, box_y, lane, *issued, w1);
      } else {
        uint32_t pk16[kChunk / 2];
#pragma unroll
        for (int j = 0; j < kChunk; j += 2) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
          pk16[j / 2] = *reinterpret_cast<const uint32_t*>(&h);
        }
        store_box(staging, box_map, box_x + c0, box_y, lane, *issued, pk16);
      }
    } else if (store && c0 < vcols) {
      if (out_dtype == BIL_F32) {
        float* o = reinterpret_cast<float*>(out_row) + c0;
        if (c0 + kChunk <= vcols) {
#pragma unroll
          for (int j = 0; j < kChunk; j += 4)
            *reinterpret_cast<uint4*>(o + j) = make_uint4(r[j], r[j + 1], r[j + 2], r[j + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < kChunk; ++j)
            if (c0 + j < vcols) o[j] = __uint_as_float(r[j]);
        }
      } else {
        __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out_row) + c0;
        uint32_t pk[kChunk / 2];
#pragma unroll
        for (int j = 0; j < kChunk; j += 2) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
          pk[j / 2] = *reinterpret_cast<const uint32_t*>(&h);
        }
        if (c0 + kChunk <= vcols) {
#pragma unroll
          for (int j = 0; j < kChunk / 2; j += 4)
            *reinterpret_cast<uint4*>(o + 2 * j) = make_uint4(pk[j], pk[j + 1], pk[j + 2], pk[j + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < kChunk; ++j)
            if (c0 + j < vcols) o[j] = __float2bfloat16_rn(__uint_as_float(r[j]));
        }
      }
    }
  }
  const float m = __fmul_rn(mx, rcp);
  const float shift = (mx == -INFINITY) ? 0.0f : mx;
  const float c = __fmul_rn(rcp, kLog2e);  // rcp = 1: log2e
  float a[8], u[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    a[j] = 0.0f;
    u[j] = 0.0f;
  }
  if constexpr (ENT) {
    // The entropy variant runs this pass on packed float32 pairs (faster there;
    // the plain variant is as fast in the scalar form): slot pair q holds slots
    // (2q, 2q + 1), and columns c0 + 2k, c0 + 2k + 1 go to pair k % 4 in column
    // order, so each slot's operations are the scalar form's, in its order.
    uint64_t a2[4] = {0, 0, 0, 0}, u2[4] = {0, 0, 0, 0};
    const uint64_t shift2 = pk(shift, shift), c2 = pk(c, c);
#pragma unroll 1
    for (int c0 = 0; c0 < kBN; c0 += kChunk) {
      tmem_ld32(taddr + c0, r);
#pragma unroll
      for (int k = 0; k < kChunk / 2; ++k) {
        const uint64_t x = static_cast<uint64_t>(r[2 * k]) | (static_cast<uint64_t>(r[2 * k + 1]) << 32);
        const uint64_t t = mul2(sub2(x, shift2), c2);
        float e0 = ex2_approx(lo_of(t)), e1 = ex2_approx(hi_of(t));
        if (c0 + 2 * k >= vcols) e0 = 0.0f;  // columns past the vocabulary add nothing
        if (c0 + 2 * k + 1 >= vcols) e1 = 0.0f;
        const uint64_t e = pk(e0, e1);
        a2[k % 4] = add2(a2[k % 4], e);
        u2[k % 4] = fma2(e, pk(fmaxf(lo_of(t), kNegMax), fmaxf(hi_of(t), kNegMax)), u2[k % 4]);
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      a[2 * q] = lo_of(a2[q]);
      a[2 * q + 1] = hi_of(a2[q]);
      u[2 * q] = lo_of(u2[q]);
      u[2 * q + 1] = hi_of(u2[q]);
    }
  } else {
#pragma unroll 1
    for (int c0 = 0; c0 < kBN; c0 += kChunk) {
      tmem_ld32(taddr + c0, r);
#pragma unroll
      for (int j = 0; j < kChunk; ++j) {
        const float t = __fmul_rn(__fsub_rn(__uint_as_float(r[j]), shift), c);
        float e = ex2_approx(t);
        if (c0 + j >= vcols) e = 0.0f;  // columns past the vocabulary add nothing
        a[j % 8] = __fadd_rn(a[j % 8], e);
      }
    }
  }
  s_out = __fadd_rn(__fadd_rn(__fadd_rn(a[0], a[1]), __fadd_rn(a[2], a[3])),
                    __fadd_rn(__fadd_rn(a[4], a[5]), __fadd_rn(a[6], a[7])));
  if (ENT)
    u_out = __fmul_rn(__fadd_rn(__fadd_rn(__fadd_rn(u[0], u[1]), __fadd_rn(u[2], u[3])),
                                __fadd_rn(__fadd_rn(u[4], u[5]), __fadd_rn(u[6], u[7]))),
                      kLn2);
  m_out = m;
  tl_out = tl;
}

// float -> 16-bit storage, round to nearest even.
template <int DT>
__device__ __forceinline__ uint16_t to16(float v) {
  if (DT == BIL_BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  return __half_as_ushort(__float2half_rn(v));
}

// 32 consecutive values of one row -> 16-bit elements at o[0..n), n <= 32:
// four 16-byte stores when all 32 are in range.
template <int DT>
__device__ __forceinline__ void store_row16(uint16_t* o, const float (&v)[kChunk], int n) {
  if (n >= kChunk) {
    uint32_t pk[kChunk / 2];
#pragma unroll
    for (int j = 0; j < kChunk; j += 2)
      pk[j / 2] = static_cast<uint32_t>(to16<DT>(v[j])) | (static_cast<uint32_t>(to16<DT>(v[j + 1])) << 16);
#pragma unroll
    for (int j = 0; j < kChunk / 2; j += 4)
      *reinterpret_cast<uint4*>(o + 2 * j) = make_uint4(pk[j], pk[j + 1], pk[j + 2], pk[j + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < kChunk; ++j)
      if (j < n) o[j] = to16<DT>(v[j]);
  }
}

// The gradient tile of one row: dZ[row, c] for the tile's columns, by the
// library's backward formula (grad_elem) from the float32 accumulator, stored
// rounded to 16 bits into dz (row-major).  Inactive rows are +0.0; an active
// row whose target is outside [0, vocab) is NaN.
template <bool ENT, int DT>
__device__ __forceinline__ void row_grad(uint32_t taddr, int vcols, float rcp, int64_t tloc, bool valid, bool active,
                                         bool bad_target, const RowMeta& meta, uint16_t* dz_row) {
  uint32_t r[kChunk];
  float d[kChunk];
#pragma unroll 1
  for (int c0 = 0; c0 < kBN; c0 += kChunk) {
    tmem_ld32(taddr + c0, r);
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      float v = 0.0f;
      if (active) v = grad_elem(__uint_as_float(r[j]), meta, c0 + j == tloc, rcp, ENT);
      if (bad_target) v = __int_as_float(0x7fc00000);
      d[j] = v;
    }
    if (valid && c0 < vcols) store_row16<DT>(dz_row + c0, d, vcols - c0);
  }
}

// The same gradient tile through shared memory: chunk by chunk (32 columns),
// the warp's 32 rows go into one of its two 2 KB staging boxes (row-major,
// lane i's row at 64 i bytes), and lane 0 stores the box to dz with TMA at
// (column x0 + chunk, row y0); rows and columns past the matrix are not
// written.  `issued` counts the warp's boxes (it picks the buffer).
template <bool ENT, int DT>
__device__ __forceinline__ void row_grad_tma(uint32_t taddr, int vcols, float rcp, int64_t tloc, bool active,
                                             bool bad_target, const RowMeta& meta, unsigned char* staging,
                                             const CUtensorMap* map, int x0, int y0, int lane, uint32_t& issued) {
  uint32_t r[kChunk];
  float d[kChunk];
  const int nchunks = (vcols + kChunk - 1) / kChunk;  // chunks past the vocabulary hold no column
#pragma unroll 1
  for (int c0 = 0; c0 < kBN; c0 += kChunk) {
    tmem_ld32(taddr + c0, r);
    if (c0 / kChunk >= nchunks) continue;
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      float v = 0.0f;
      if (active) v = grad_elem(__uint_as_float(r[j]), meta, c0 + j == tloc, rcp, ENT);
      if (bad_target) v = __int_as_float(0x7fc00000);
      d[j] = v;
    }
    uint32_t pk16[kChunk / 2];
#pragma unroll
    for (int j = 0; j < kChunk; j += 2)
      pk16[j / 2] = static_cast<uint32_t>(to16<DT>(d[j])) | (static_cast<uint32_t>(to16<DT>(d[j + 1])) << 16);
    store_box(staging, map, x0 + c0, y0, lane, issued, pk16);
  }
}

// One row of C = A . B^T as it is: float32, or rounded to 16 bits.
template <int OT>
__device__ __forceinline__ void row_store(uint32_t taddr, int vcols, bool valid, unsigned char* out_row) {
  uint32_t r[kChunk];
  float v[kChunk];
#pragma unroll 1
  for (int c0 = 0; c0 < kBN; c0 += kChunk) {
    tmem_ld32(taddr + c0, r);
    if (valid && c0 < vcols) {
      if (OT == BIL_F32) {
        float* o = reinterpret_cast<float*>(out_row) + c0;
        if (c0 + kChunk <= vcols) {
#pragma unroll
          for (int j = 0; j < kChunk; j += 4)
            *reinterpret_cast<uint4*>(o + j) = make_uint4(r[j], r[j + 1], r[j + 2], r[j + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < kChunk; ++j)
            if (c0 + j < vcols) o[j] = __uint_as_float(r[j]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < kChunk; ++j) v[j] = __uint_as_float(r[j]);
        store_row16<OT>(reinterpret_cast<uint16_t*>(out_row) + c0, v, vcols - c0);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Soft lockstep of the store GEMMs' copy threads.  Their K is long (the
// vocabulary for dhidden), and the blocks of one wave read the same A and B
// tiles at the same K position: when they drift apart by more K blocks than
// L2 holds for the wave, the tiles they share come from DRAM again for every
// block that reads them late (with one-half units at 16384 x 151936 x 4096:
// 46 GB of DRAM reads for dhidden's 5 GB of dZ and 1.2 GB of weight, against
// 27 GB in step).
//
// A service warp per block (kSyncWarp) publishes, every few microseconds,
// how many K blocks its copy thread has issued (in a 128-byte line of its
// own), reads every block's position, and tells its copy thread in shared
// memory how far it may go: kSyncLead K blocks past the slowest block of
// the same launch.  The copy thread only
// reads that bound, so the polling stays off its path.  Positions are tagged
// with a per-launch number, so stale entries of other launches count for
// nothing; a block that has issued all its copies publishes the largest
// position.  Every wait is bounded: the copy thread waits at most kSyncWaitNs
// for the bound to move and otherwise stops keeping step for the rest of the
// launch; the service warp stops when its copy thread is done or has not
// moved for the wait limit.  None of this touches what is computed: a tile's
// copies, MMAs and K order do not depend on it.
// ---------------------------------------------------------------------------

#ifndef BIL_STORE_LOCKSTEP
#define BIL_STORE_LOCKSTEP 1
#endif

// Work units of the store GEMMs: 2 (two 128-row halves, from 256 rows on) or 1.
#ifndef BIL_STORE_HALVES
#define BIL_STORE_HALVES 2
#endif

#ifndef BIL_STORE_SYNC_LEAD
#define BIL_STORE_SYNC_LEAD 64
#endif
#ifndef BIL_STORE_SYNC_MIN_KBLOCKS
#define BIL_STORE_SYNC_MIN_KBLOCKS 1024
#endif
constexpr int kSyncLead = BIL_STORE_SYNC_LEAD;                // K blocks a copy thread may run ahead
constexpr int kSyncMinKBlocks = BIL_STORE_SYNC_MIN_KBLOCKS;   // the shortest K (in blocks of kBK) that keeps step
constexpr int kSyncMaxBlocks = 1024;
constexpr long long kSyncWaitNs = 50000;   // 50 us
constexpr unsigned kSyncPollNs = 4000;     // the service warp's pause between two updates
constexpr uint32_t kSyncDone = 0xffffffffu;
constexpr int kSyncSlotWords = 16;         // one 128-byte line per block: no two blocks write one line

__device__ unsigned long long g_sync_pos[kSyncMaxBlocks * kSyncSlotWords];

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* a, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(a), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* a) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
  return v;
}

__device__ __forceinline__ void lockstep_publish(unsigned tag, uint32_t pos) {
  st_relaxed_u64(&g_sync_pos[blockIdx.x * kSyncSlotWords], (static_cast<unsigned long long>(tag) << 32) | pos);
}

// The service warp's loop (all 32 lanes).
__device__ __forceinline__ void lockstep_service(unsigned tag, LinearSmem& sm, volatile int* abort, int lane) {
  volatile uint32_t* pos_p = &sm.sync_pos;
  volatile uint32_t* allowed_p = &sm.sync_allowed;
  volatile int* done_p = &sm.sync_done;
  uint32_t last = kSyncDone;
  long long last_move = 0;
  for (;;) {
    const uint32_t pos = __shfl_sync(0xffffffffu, *pos_p, 0);
    const int stop = __shfl_sync(0xffffffffu, (*done_p != 0 || *abort != 0) ? 1 : 0, 0);
    if (stop) break;
    if (lane == 0) lockstep_publish(tag, pos);
    uint32_t slowest = kSyncDone;
    for (int b = lane; b < static_cast<int>(gridDim.x); b += kLanes) {
      const unsigned long long v = ld_relaxed_u64(&g_sync_pos[b * kSyncSlotWords]);
      if (static_cast<unsigned>(v >> 32) == tag) slowest = min(slowest, static_cast<uint32_t>(v));
    }
    slowest = __reduce_min_sync(0xffffffffu, slowest);
    if (lane == 0) *allowed_p = slowest == kSyncDone ? kSyncDone : slowest + static_cast<uint32_t>(kSyncLead);
    const long long now = __shfl_sync(0xffffffffu, global_ns(), 0);
    if (pos != last) {
      last = pos;
      last_move = now;
    } else if (now - last_move > kWaitLimitNs) {
      break;  // the copy thread has stopped moving: leave it unbounded
    }
    __nanosleep(kSyncPollNs);
  }
  if (lane == 0) {
    *allowed_p = kSyncDone;
    lockstep_publish(tag, kSyncDone);  // never wait for this block again
  }
}

// The copy thread's side: publish the position, and wait (at most
// kSyncWaitNs) until it is within the bound.  Returns false when the wait ran
// out (the caller then stops keeping step).
__device__ __forceinline__ bool lockstep_gate(LinearSmem& sm, uint32_t pos) {
  volatile uint32_t* allowed_p = &sm.sync_allowed;
  *reinterpret_cast<volatile uint32_t*>(&sm.sync_pos) = pos;
  if (pos <= *allowed_p) return true;
  const long long start = global_ns();
  while (pos > *allowed_p) {
    if (global_ns() - start > kSyncWaitNs) return false;
    __nanosleep(200);
  }
  return true;
}

// The GEMM C = A . B^T (A [rows, K], B [cols, K], both K-major 16-bit) with
// one of the epilogues above.  See the file's head for the block structure.
//
// HALVES = 2 (the store epilogue only): a work unit is 2 x kBM rows.  A stage
// holds both 128-row A tiles and the B tile, and the two MMAs of a K step (one
// per A tile, each into its own 256 accumulator columns) share the B tile, so
// a block copies 32 KB per 128 x 256 x 64 of MMA work instead of 48 KB, and a
// wave of blocks covers twice the rows (each B tile is read from DRAM half as
// often).  The two accumulators fill tensor memory: one buffer, so the
// epilogue of a unit does not overlap the next unit's MMAs, which costs little
// when K is long.  Each output element still sums its K blocks in order, four
// K=16 steps each: the same bits as with HALVES = 1.
template <int MODE, bool ENT, int DT, int HALVES = 1>
__device__ __forceinline__ void gemm_body(const CUtensorMap& tmap_hidden, const CUtensorMap& tmap_weight,
                                          const CUtensorMap& tmap_out, const LinearParams& p) {
  static_assert(HALVES == 1 || (HALVES == 2 && MODE == kModeStore), "two-half units are for the store epilogue");
  constexpr unsigned kStageBytesH = HALVES * kStageABytes + kStageBBytes;
  constexpr int kStagesH = static_cast<int>(kStages * size_t(kStageBytes) / kStageBytesH);  // 4, or 3 of 64 KB
  static_assert(kStagesH >= 3 && kStagesH <= kStages, "the stage ring fits the shared memory of the 1-half layout");
  constexpr int kAccBufs = HALVES == 1 ? 2 : 1;
  constexpr int kRowsPerUnit = HALVES * kBM;
  extern __shared__ unsigned char smem_raw[];
  // Stage buffers start on a 1024-byte boundary (the 128-byte swizzle pattern
  // repeats every 8 rows = 1024 bytes).
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  LinearSmem& sm = *reinterpret_cast<LinearSmem*>(base + kStages * size_t(kStageBytes));
  volatile int* abort = &sm.abort;
  const int warp = threadIdx.x / kLanes;
  const int lane = threadIdx.x % kLanes;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.acc_full[b], 1);
      mbar_init(&sm.acc_empty[b], kEpiWarps);
    }
    mbar_init(&sm.mma_done, 1);
    sm.abort = 0;
    sm.sync_pos = 0;
    sm.sync_allowed = kSyncLead;
    sm.sync_done = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sm.tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sm.tmem_base;

  const int64_t total = static_cast<int64_t>(p.num_m) * p.num_n;

  const bool lockstep = MODE == kModeStore && p.sync_tag != 0u;
  if (warp == 0) {
    if (lane == 0) {
      // ---- producer ----
      bool sync_on = lockstep;
      int64_t it = 0;
      bool ok = true;
      for (int64_t u = blockIdx.x; u < total && ok; u += gridDim.x) {
        int m, n;
        unit_coords(u, p.num_m, p.num_n, p.m_group, m, n);
        for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
          if (sync_on) sync_on = lockstep_gate(sm, static_cast<uint32_t>(it));
          const int s = static_cast<int>(it % kStagesH);
          const unsigned ph = static_cast<unsigned>((it / kStagesH) & 1);
          if (!thread_wait_watch(&sm.empty[s], ph ^ 1u, abort, kWatchStageFree, &g_watchdog_linear, true)) {
            ok = false;
            break;
          }
          unsigned char* a_dst = base + s * size_t(kStageBytesH);
          unsigned char* b_dst = a_dst + HALVES * kStageABytes;
          mbar_arrive_expect_tx(&sm.full[s], HALVES * p.a_box_bytes + kStageBBytes);
          // Boxes past the last row (or K) read zeros.  A K-major operand comes
          // in one box of 128 (A) or 256 (B) rows by 64 K, an MN-major one in
          // boxes of 64 rows by 64 K (their coordinates: row, then K).
          if (MODE == kModeStore && p.a_mn) {
#pragma unroll
            for (int j = 0; j < HALVES * kBM / kMnBox; ++j)
              tma_load_2d(a_dst + j * kMnBoxBytes, &tmap_hidden, m * HALVES * kBM + j * kMnBox, kb * kBK, &sm.full[s]);
          } else {
#pragma unroll
            for (int h = 0; h < HALVES; ++h)
              tma_load_2d(a_dst + h * kStageABytes, &tmap_hidden, kb * kBK, (m * HALVES + h) * kBM, &sm.full[s]);
          }
          if (MODE == kModeStore && p.b_mn) {
#pragma unroll
            for (int j = 0; j < kBN / kMnBox; ++j)
              tma_load_2d(b_dst + j * kMnBoxBytes, &tmap_weight, n * kBN + j * kMnBox, kb * kBK, &sm.full[s]);
          } else {
            tma_load_2d(b_dst, &tmap_weight, kb * kBK, n * kBN, &sm.full[s]);
          }
        }
      }
      if (lockstep) *reinterpret_cast<volatile int*>(&sm.sync_done) = 1;
      // Wait (bounded, whatever happened) for the copies still in flight: the
      // last min(it, kStagesH) fills, one per stage.
      for (int64_t i = it > kStagesH ? it - kStagesH : 0; i < it; ++i) {
        const int s = static_cast<int>(i % kStagesH);
        if (!thread_wait_watch(&sm.full[s], static_cast<unsigned>((i / kStagesH) & 1), abort, kWatchOwnDrain,
                               &g_watchdog_linear, false))
          break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer ----
      int64_t it = 0;
      int local = 0;
      bool ok = true;
      for (int64_t u = blockIdx.x; u < total && ok; u += gridDim.x, ++local) {
        const int b = local % kAccBufs;
        const unsigned use = static_cast<unsigned>(local / kAccBufs);
        if (!thread_wait_watch(&sm.acc_empty[b], (use & 1u) ^ 1u, abort, kWatchMma, &g_watchdog_linear, true)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * kAccCols);
        for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
          const int s = static_cast<int>(it % kStagesH);
          const unsigned ph = static_cast<unsigned>((it / kStagesH) & 1);
          if (!thread_wait_watch(&sm.full[s], ph, abort, kWatchMma, &g_watchdog_linear, true)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(base + s * size_t(kStageBytesH));
          const uint32_t b_addr = a_addr + HALVES * kStageABytes;
          const bool a_mn = MODE == kModeStore && p.a_mn, b_mn = MODE == kModeStore && p.b_mn;
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k) {
            // a K step: 32 bytes along a K-major line, 16 lines of an MN-major box
            const uint64_t bdesc = b_mn ? smem_desc_mn(b_addr + k * kUmmaK * 128) : smem_desc(b_addr + k * kUmmaK * 2);
#pragma unroll
            for (int h = 0; h < HALVES; ++h) {
              const uint32_t ah = a_addr + h * kStageABytes;  // an MN-major half is two boxes: the same 16 KB
              const uint64_t adesc = a_mn ? smem_desc_mn(ah + k * kUmmaK * 128) : smem_desc(ah + k * kUmmaK * 2);
              umma_f16(d_tmem + static_cast<uint32_t>(h * kAccCols), adesc, bdesc, p.idesc, (kb | k) != 0 ? 1u : 0u);
            }
          }
          umma_commit(&sm.empty[s]);  // the stage is free once these MMAs have read it
        }
        if (!ok) break;
        umma_commit(&sm.acc_full[b]);
      }
      // Every MMA this thread issued completes before the block frees tensor memory.
      umma_commit(&sm.mma_done);
      thread_wait_watch(&sm.mma_done, 0u, abort, kWatchOwnDrain, &g_watchdog_linear, false);
    }
  } else if (warp == kSyncWarp) {
    if (lockstep) lockstep_service(p.sync_tag, sm, abort, lane);
  } else {
    // ---- epilogue ----
    const int q = warp & 3;  // this warp reads tensor-memory lanes [32q, 32q + 32)
    const int row_in_tile = q * 32 + lane;
    int local = 0;
    uint32_t store_boxes = 0;  // dZ boxes this warp has handed to TMA
    for (int64_t u = blockIdx.x; u < total; u += gridDim.x, ++local) {
      int m, n;
      unit_coords(u, p.num_m, p.num_n, p.m_group, m, n);
      const int b = local % kAccBufs;
      const unsigned use = static_cast<unsigned>(local / kAccBufs);
      const int64_t row = static_cast<int64_t>(m) * kRowsPerUnit + row_in_tile;
      const bool valid = row < p.n_rows;
      const int64_t col0 = static_cast<int64_t>(n) * kBN;  // shard-local column of the tile's column 0
      const int vcols = static_cast<int>(p.shard_cols - col0 < kBN ? p.shard_cols - col0 : kBN);
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * kAccCols);
      if constexpr (MODE == kModePartials) {
        const int64_t t = valid ? p.targets[row] : p.ignore_index;
        const bool active = valid && t != p.ignore_index;
        const int64_t gcol0 = static_cast<int64_t>(p.tile_begin + n) * kBN;
        const int64_t tloc = active ? t - gcol0 : -1;
        if (!warp_wait_watch(&sm.acc_full[b], use & 1u, abort, kWatchAccFull, &g_watchdog_linear)) break;
        tc_fence_after();
        float mt, st, ut = 0.0f, tl;
#if BIL_EPILOGUE_TMA_STORE
        if (p.logits != nullptr) {  // the logits through the warp's staging boxes with TMA
          unsigned char* staging = reinterpret_cast<unsigned char*>(
                                       (reinterpret_cast<uintptr_t>(&sm + 1) + 1023) & ~static_cast<uintptr_t>(1023)) +
                                   q * 2 * kStoreBoxBytes;
          row_partial<ENT>(taddr, vcols, p.rcp, tloc, false, nullptr, p.logits_dtype, mt, st, ut, tl, &tmap_out,
                           staging, static_cast<int>(col0), static_cast<int>(m * kBM + q * 32), lane, &store_boxes);
        } else {
          row_partial<ENT>(taddr, vcols, p.rcp, tloc, false, nullptr, p.logits_dtype, mt, st, ut, tl);
        }
#else
        const bool store = valid && p.logits != nullptr;
        unsigned char* out_row =
            store ? p.logits + (row * p.ld_logits + col0) * (p.logits_dtype == BIL_F32 ? 4 : 2) : nullptr;
        row_partial<ENT>(taddr, vcols, p.rcp, tloc, store, out_row, p.logits_dtype, mt, st, ut, tl);
#endif
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_empty[b]);
        if (valid) {
          const int64_t at = row * p.ld_part + p.tile_begin + n;
          p.part_max[at] = active ? mt : -INFINITY;
          p.part_sum[at] = active ? st : 0.0f;
          if (ENT) p.part_ent[at] = active ? ut : 0.0f;
          if (tloc >= 0 && tloc < vcols) p.target_logit[row] = tl;
        }
      } else if constexpr (MODE == kModeGrad) {
        RowMeta meta{p.ignore_index, 0.0f, 0.0f, 0.0f, 0.0f};
        if (valid) {
          meta.target = p.targets[row];
          meta.lse = p.lse[row];
          meta.g = p.grad_logp[row];
          if (ENT) {
            meta.H = p.entropy[row];
            meta.gh = p.grad_entropy[row];
          }
        }
        const bool active = valid && meta.target != p.ignore_index;
        const bool bad_target = active && (meta.target < 0 || meta.target >= p.vocab);
        const int64_t gcol0 = static_cast<int64_t>(p.tile_begin + n) * kBN;
        const int64_t tloc = active ? meta.target - gcol0 : -1;
        if (!warp_wait_watch(&sm.acc_full[b], use & 1u, abort, kWatchAccFull, &g_watchdog_linear)) break;
        tc_fence_after();
#if BIL_EPILOGUE_TMA_STORE
        unsigned char* staging = reinterpret_cast<unsigned char*>(
                                     (reinterpret_cast<uintptr_t>(&sm + 1) + 1023) & ~static_cast<uintptr_t>(1023)) +
                                 q * 2 * kStoreBoxBytes;
        row_grad_tma<ENT, DT>(taddr, vcols, p.rcp, tloc, active, bad_target, meta, staging, &tmap_out,
                              static_cast<int>(col0), static_cast<int>(m * kBM + q * 32), lane, store_boxes);
#else
        uint16_t* dz_row = valid ? reinterpret_cast<uint16_t*>(p.dz) + row * p.ld_dz + col0 : nullptr;
        row_grad<ENT, DT>(taddr, vcols, p.rcp, tloc, valid, active, bad_target, meta, dz_row);
#endif
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_empty[b]);
      } else {
        if (!warp_wait_watch(&sm.acc_full[b], use & 1u, abort, kWatchAccFull, &g_watchdog_linear)) break;
        tc_fence_after();
        const int eb = DT == BIL_F32 ? 4 : 2;
#pragma unroll 1
        for (int h = 0; h < HALVES; ++h) {  // half h: rows [h kBM, (h + 1) kBM) of the unit
          const int64_t row_h = row + h * kBM;
          const bool valid_h = row_h < p.n_rows;
          unsigned char* out_row = valid_h ? p.out + (row_h * p.ld_out + col0) * eb : nullptr;
          row_store<DT>(taddr + static_cast<uint32_t>(h * kAccCols), vcols, valid_h, out_row);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_empty[b]);
      }
    }
    // the staging boxes stay in use until their stores have completed
    if (BIL_EPILOGUE_TMA_STORE && lane == 0 && store_boxes != 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                 : "memory");
  }
}

// Forward: the tile partials of hidden . weight^T.
template <bool ENT>
__global__ void __launch_bounds__(kThreads, 1)
    linear_partials_kernel(const __grid_constant__ CUtensorMap tmap_hidden,
                           const __grid_constant__ CUtensorMap tmap_weight,
                           const __grid_constant__ CUtensorMap tmap_out, const LinearParams p) {
  gemm_body<kModePartials, ENT, 0>(tmap_hidden, tmap_weight, tmap_out, p);
}

// Backward, first pass: hidden . weight^T recomputed, dZ stored (16-bit DT).
template <bool ENT, int DT>
__global__ void __launch_bounds__(kThreads, 1)
    linear_grad_kernel(const __grid_constant__ CUtensorMap tmap_hidden, const __grid_constant__ CUtensorMap tmap_weight,
                       const __grid_constant__ CUtensorMap tmap_dz, const LinearParams p) {
  gemm_body<kModeGrad, ENT, DT>(tmap_hidden, tmap_weight, tmap_dz, p);
}

// Backward, the two contractions of dZ: C = A . B^T stored as OT, in work
// units of HALVES x 128 rows.
template <int OT, int HALVES>
__global__ void __launch_bounds__(kThreads, 1)
    linear_store_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                        const __grid_constant__ CUtensorMap tmap_out, const LinearParams p) {
  gemm_body<kModeStore, false, OT, HALVES>(tmap_a, tmap_b, tmap_out, p);
}

// dst[i] = ((src_0[i] + src_1[i]) + src_2[i]) + ... , sources in order.
constexpr int kMaxSumSources = 16;
struct SumSources {
  const float* src[kMaxSumSources];
};

__global__ void __launch_bounds__(256) sum_f32_kernel(SumSources s, int count, int64_t n, float* __restrict__ dst) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float acc = s.src[0][i];
    for (int k = 1; k < count; ++k) acc = __fadd_rn(acc, s.src[k][i]);
    dst[i] = acc;
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------

// cuTensorMapEncodeTiled, fetched from the driver at run time (no link-time
// dependency on the driver library).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// A 2-D tensor map over a row-major [rows, cols] matrix of 16-bit elements
// (row stride ld elements), box = box_rows x 64 elements, 128-byte swizzle;
// reads past the matrix fill zeros.
int make_map(CUtensorMap* map, const void* ptr, int dtype, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return BIL_E_CUDA;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      dtype == BIL_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUresult r = fn(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BIL_OK : BIL_E_CUDA;
}

// The tensor map an epilogue stores a [rows, cols] output (row stride ld
// elements) through from the warps' staging boxes: 32 rows of 64 bytes, i.e.
// 32 columns of a 16-bit type or 16 of float32, no swizzle (a box in shared
// memory is row-major).
int make_store_map(CUtensorMap* map, void* ptr, int dtype, int64_t rows, int64_t cols, int64_t ld) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return BIL_E_CUDA;
  const int eb = dtype == BIL_F32 ? 4 : 2;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * eb};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(64 / eb), static_cast<cuuint32_t>(kStoreBox)};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = dtype == BIL_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : dtype == BIL_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUresult r = fn(map, dt, 2, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BIL_OK : BIL_E_CUDA;
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

typedef void (*GemmKernel)(CUtensorMap, CUtensorMap, CUtensorMap, LinearParams);

// One persistent block per SM (at most one per work unit).
// mo: the output's tensor map for an epilogue that stores with TMA (the
// gradient pass's dZ), else any valid map (unused).
int launch_gemm(GemmKernel kernel, const CUtensorMap& mh, const CUtensorMap& mw, const CUtensorMap& mo,
                const LinearParams& p, cudaStream_t stream) {
  int sms = 0, smem_optin = 0;
  if (int st = bil_internal::device_limits(&sms, &smem_optin)) return st;
  if (static_cast<size_t>(smem_optin) < kSmemBytes) return BIL_E_UNSUPPORTED;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes)) !=
      cudaSuccess)
    return BIL_E_CUDA;
  const int64_t total = static_cast<int64_t>(p.num_m) * p.num_n;
  const int grid = static_cast<int>(std::min<int64_t>(total, sms));
  kernel<<<grid, kThreads, kSmemBytes, stream>>>(mh, mw, mo, p);
  return cudaGetLastError() == cudaSuccess ? BIL_OK : BIL_E_CUDA;
}

// Raster group for the store GEMMs: enough row tiles that one wave of blocks
// covers every column tile of them (each A tile is then read from DRAM once).
int store_group(int num_n) {
  int sms = 0, smem = 0;
  if (bil_internal::device_limits(&sms, &smem) != BIL_OK || sms <= 0) sms = 148;
  return std::max(1, sms / std::max(1, num_n));
}

// A 16-byte aligned base and a row stride of a multiple of 16 bytes (what TMA
// and the epilogues' vector stores need).
bool rows16(const void* p, int64_t ld, int64_t elem_bytes) {
  return aligned_to(p, 16) && (ld * elem_bytes) % 16 == 0;
}

// Workspace layout of bil_linear_logp_fwd: part_max, part_sum[, part_ent]
// ([n_rows, num_tiles] float32 each), target_logit [n_rows], each block
// starting on a 256-byte boundary.
size_t round256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

struct Workspace {
  size_t part, tl, total;
};

Workspace workspace_layout(int64_t n_rows, int64_t num_tiles, bool ent) {
  Workspace w;
  w.part = round256(static_cast<size_t>(n_rows) * static_cast<size_t>(num_tiles) * sizeof(float));
  w.tl = round256(static_cast<size_t>(n_rows) * sizeof(float));
  w.total = w.part * (ent ? 3 : 2) + w.tl;
  return w;
}

// The vocabulary and the [n_rows, num_tiles] partials within the extent limit,
// so that workspace_layout's sizes cannot overflow.
bool workspace_fits(int64_t n_rows, int64_t vocab) {
  return vocab <= BIL_MAX_EXTENT_BYTES && bil_internal::extent_ok(n_rows, (vocab + kBN - 1) / kBN, 4);
}

// Device scratch of bil_linear_logp_fwd_static: one array per device image,
// never allocated or freed at run time.
static __device__ __align__(256) unsigned char g_linear_static_scratch[BIL_LINEAR_STATIC_SCRATCH_BYTES];

constexpr int kMaxStaticDevices = 64;
struct StaticScratch {
  CUcontext ctx;  // the context the address was looked up in
  void* ptr;
};
StaticScratch g_static_scratch[kMaxStaticDevices];
std::mutex g_static_scratch_mutex;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// cuCtxGetCurrent, fetched from the driver at run time like the encoder.
CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// The array's device address on the current device.  It is looked up (with
// that device current) on the first call in each context and cached with the
// context it belongs to: the address is a property of the module as loaded
// into one context, so after a device reset, or under another context made
// current on the same device, the next call looks it up again rather than
// reuse an address that no longer maps the array.
int static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxStaticDevices) return BIL_E_CUDA;
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  if (get_ctx == nullptr) return BIL_E_CUDA;
  CUcontext ctx = nullptr;  // stays null on a thread where the runtime has made no context current yet
  if (get_ctx(&ctx) != CUDA_SUCCESS) return BIL_E_CUDA;
  std::lock_guard<std::mutex> lock(g_static_scratch_mutex);
  StaticScratch& e = g_static_scratch[dev];
  if (ctx == nullptr || e.ptr == nullptr || e.ctx != ctx) {
    void* ptr = nullptr;  // the lookup also makes the device's primary context current if none is
    if (cudaGetSymbolAddress(&ptr, g_linear_static_scratch) != cudaSuccess || ptr == nullptr) return BIL_E_CUDA;
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return BIL_E_CUDA;
    e.ctx = ctx;
    e.ptr = ptr;
  }
  *out = e.ptr;
  return BIL_OK;
}

// The next per-launch tag of the store GEMMs' lockstep (never 0).
unsigned next_sync_tag() {
  static std::atomic<unsigned> counter{0};
  unsigned t = 0;
  while (t == 0) t = counter.fetch_add(1u, std::memory_order_relaxed) + 1u;
  return t;
}

// C [a_rows, n_cols] = A . B^T over K = k with the store epilogue, in units of
// two 128-row halves from 256 rows on (one otherwise), rastered in groups of
// row units that one wave covers with every column tile, the copy threads in
// lockstep when every block's position fits the tag's 32 bits.
int launch_store(const CUtensorMap& ma, const CUtensorMap& mb, int64_t a_rows, int64_t n_cols, int64_t k, bool bf16,
                 bool a_mn, bool b_mn, void* out, int out_dtype, int64_t ld_out, cudaStream_t s) {
  const int halves = BIL_STORE_HALVES == 2 && a_rows >= 2 * kBM ? 2 : 1;
  LinearParams p{};
  p.n_rows = a_rows;
  p.shard_cols = n_cols;
  p.num_n = static_cast<int>((n_cols + kBN - 1) / kBN);
  p.num_m = static_cast<int>((a_rows + halves * kBM - 1) / (halves * kBM));
  p.k_blocks = static_cast<int>((k + kBK - 1) / kBK);
  p.idesc = make_idesc(bf16, a_mn, b_mn);
  p.a_box_bytes = kStageABytes;  // kBM-row boxes (K-major), or two of 64 rows (MN-major)
  p.a_mn = a_mn ? 1 : 0;
  p.b_mn = b_mn ? 1 : 0;
  p.m_group = store_group(p.num_n);
  p.out = static_cast<unsigned char*>(out);
  p.out_dtype = out_dtype;
  p.ld_out = ld_out;
  int sms = 0, smem = 0;
  if (int st = bil_internal::device_limits(&sms, &smem)) return st;
  const int64_t total = static_cast<int64_t>(p.num_m) * p.num_n;
  const int64_t grid = std::min<int64_t>(total, sms);
  const int64_t iters = (total + grid - 1) / grid * p.k_blocks;  // K blocks one block issues
  // Only units of a long K drift apart far enough to matter (measured on 16384 x 151936 x 4096 with
  // one-half units: dhidden, K = 151936, read 46 GB of DRAM alone and 27 GB in step, 5% faster; dweight,
  // K = 16384, read 26 GB either way and was 1% slower in step; with two-half units dweight in step
  // read the same 17.8 GB in the same time).
  p.sync_tag = BIL_STORE_LOCKSTEP && p.k_blocks >= kSyncMinKBlocks && grid <= kSyncMaxBlocks &&
                       iters + kSyncLead < INT32_MAX
                   ? next_sync_tag()
                   : 0u;
  GemmKernel kern;
  if (halves == 2)
    kern = out_dtype == BIL_F32    ? linear_store_kernel<BIL_F32, 2>
           : out_dtype == BIL_BF16 ? linear_store_kernel<BIL_BF16, 2>
                                   : linear_store_kernel<BIL_F16, 2>;
  else
    kern = out_dtype == BIL_F32    ? linear_store_kernel<BIL_F32, 1>
           : out_dtype == BIL_BF16 ? linear_store_kernel<BIL_BF16, 1>
                                   : linear_store_kernel<BIL_F16, 1>;
  return launch_gemm(kern, ma, mb, mb, p, s);
}

// A store GEMM operand with `rows` rows (M or N) over K = k: stored [rows, k]
// (K-major) and copied in boxes of box_rows x 64 K, or stored [k, rows] (mn:
// MN-major) and copied in boxes of 64 rows x 64 K.
int operand_map(CUtensorMap* map, const void* ptr, int dtype, int64_t rows, int64_t k, int64_t ld, bool mn,
                int box_rows) {
  return mn ? make_map(map, ptr, dtype, k, rows, ld, kMnBox) : make_map(map, ptr, dtype, rows, k, ld, box_rows);
}

// dZ of the shard's columns from the recomputed projection (maps: hidden with
// kBM-row boxes, weight with kBN-row boxes), stored as dz.
int launch_grad(const CUtensorMap& mh, const CUtensorMap& mw, int dtype, int64_t n_rows, int64_t hidden_size,
                int64_t cols, int32_t tile_begin, int32_t tile_end, float rcp, const int64_t* targets,
                int64_t ignore_index, const float* lse, const float* grad_logp, const float* entropy,
                const float* grad_entropy, int64_t vocab, void* dz, int64_t ld_dz, cudaStream_t s) {
  LinearParams p{};
  p.n_rows = n_rows;
  p.shard_cols = cols;
  p.tile_begin = tile_begin;
  p.num_n = tile_end - tile_begin;
  p.num_m = static_cast<int>((n_rows + kBM - 1) / kBM);
  p.k_blocks = static_cast<int>((hidden_size + kBK - 1) / kBK);
  p.targets = targets;
  p.ignore_index = ignore_index;
  p.rcp = rcp;
  p.idesc = make_idesc(dtype == BIL_BF16);
  p.a_box_bytes = kStageABytes;
  p.m_group = kMGroup;
  p.lse = lse;
  p.grad_logp = grad_logp;
  p.entropy = entropy;
  p.grad_entropy = grad_entropy;
  p.vocab = vocab;
  p.dz = static_cast<unsigned char*>(dz);
  p.ld_dz = ld_dz;
  const bool ent = entropy != nullptr;
  GemmKernel k = dtype == BIL_BF16 ? (ent ? linear_grad_kernel<true, BIL_BF16> : linear_grad_kernel<false, BIL_BF16>)
                                   : (ent ? linear_grad_kernel<true, BIL_F16> : linear_grad_kernel<false, BIL_F16>);
  CUtensorMap mdz = mw;
  if (BIL_EPILOGUE_TMA_STORE) {
    if (int st = make_store_map(&mdz, dz, dtype, n_rows, cols, ld_dz)) return st;
  }
  return launch_gemm(k, mh, mw, mdz, p, s);
}

// Host-side checks of the gradient pass's arguments (those bil_linear_logp_bwd
// and bil_linear_logp_grad share); *cols = the shard's vocabulary columns.
int check_grad_args(const void* hidden, const void* weight, int64_t n_rows, int64_t hidden_size, int64_t ld_hidden,
                    int64_t vocab, int64_t ld_weight, int32_t tile_begin, int32_t tile_end, const int64_t* targets,
                    const float* lse, const float* grad_logp, const float* entropy, const float* grad_entropy,
                    const void* dz, int64_t ld_dz, int64_t* cols_out) {
  if (vocab < 1) return BIL_E_INVALID_ARG;
  if (vocab > BIL_MAX_EXTENT_BYTES) return BIL_E_UNSUPPORTED;
  const int64_t num_tiles = (vocab + kBN - 1) / kBN;
  if (num_tiles > INT32_MAX / 2) return BIL_E_UNSUPPORTED;
  if (tile_begin < 0 || tile_begin >= tile_end || tile_end > num_tiles) return BIL_E_INVALID_ARG;
  // the shard: global vocabulary columns [tile_begin * 256, min(tile_end * 256, vocab))
  const int64_t cols = std::min<int64_t>(static_cast<int64_t>(tile_end) * kBN, vocab) -
                       static_cast<int64_t>(tile_begin) * kBN;
  if (n_rows < 0 || hidden_size < 1 || ld_hidden < hidden_size || ld_weight < hidden_size || ld_dz < cols)
    return BIL_E_INVALID_ARG;
  if ((entropy == nullptr) != (grad_entropy == nullptr)) return BIL_E_INVALID_ARG;
  {
    using bil_internal::extent_ok;
    if (!extent_ok(n_rows, ld_hidden, 2) || !extent_ok(cols, ld_weight, 2) || !extent_ok(n_rows, ld_dz, 2))
      return BIL_E_UNSUPPORTED;
  }
  if (weight == nullptr) return BIL_E_INVALID_ARG;
  if (!rows16(weight, ld_weight, 2)) return BIL_E_ALIGN;
  *cols_out = cols;
  if (n_rows == 0) return BIL_OK;
  if (hidden == nullptr || targets == nullptr || lse == nullptr || grad_logp == nullptr || dz == nullptr)
    return BIL_E_INVALID_ARG;
  if (!rows16(hidden, ld_hidden, 2) || !rows16(dz, ld_dz, 2)) return BIL_E_ALIGN;
  if (!aligned_to(targets, 8) || !aligned_to(lse, 4) || !aligned_to(grad_logp, 4) ||
      (entropy && (!aligned_to(entropy, 4) || !aligned_to(grad_entropy, 4))))
    return BIL_E_ALIGN;
  if (n_rows > INT32_MAX - kBM || cols > INT32_MAX - kBN || hidden_size > INT32_MAX - kBN) return BIL_E_UNSUPPORTED;
  return BIL_OK;
}

}  // namespace

namespace bil_internal {

int linear_watchdog(unsigned int* flags, int clear) {
  if (cudaMemcpyFromSymbol(flags, g_watchdog_linear, sizeof(unsigned int)) != cudaSuccess) return BIL_E_CUDA;
  if (clear) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_watchdog_linear, &zero, sizeof(unsigned int)) != cudaSuccess) return BIL_E_CUDA;
  }
  return BIL_OK;
}

}  // namespace bil_internal

extern "C" {

int bil_linear_logp_partials(const void* hidden, const void* weight, int dtype, int64_t n_rows,
                             int64_t hidden_size, int64_t ld_hidden, int64_t vocab, int64_t ld_weight,
                             int32_t tile_begin, int32_t tile_end, float temperature, const int64_t* target_ids,
                             int64_t ignore_index, float* part_max, float* part_sum, float* part_ent,
                             int64_t ld_part, float* target_logit, void* logits, int logits_dtype,
                             int64_t ld_logits, bil_stream_t stream) {
  bil_internal::NvtxRange nvtx_range("bil_linear_logp_partials");
  if (dtype != BIL_BF16 && dtype != BIL_F16) return BIL_E_DTYPE;
  if (n_rows < 0 || hidden_size < 1 || vocab < 1 || ld_hidden < hidden_size || ld_weight < hidden_size)
    return BIL_E_INVALID_ARG;
  if (vocab > BIL_MAX_EXTENT_BYTES) return BIL_E_UNSUPPORTED;
  const int64_t num_tiles = (vocab + kBN - 1) / kBN;
  if (num_tiles > INT32_MAX / 2) return BIL_E_UNSUPPORTED;
  if (tile_begin < 0 || tile_begin >= tile_end || tile_end > num_tiles || ld_part < num_tiles)
    return BIL_E_INVALID_ARG;
  const int64_t shard_cols = std::min<int64_t>(static_cast<int64_t>(tile_end) * kBN, vocab) -
                             static_cast<int64_t>(tile_begin) * kBN;
  if (logits != nullptr) {
    if (logits_dtype != BIL_F32 && logits_dtype != BIL_BF16) return BIL_E_DTYPE;
    if (ld_logits < shard_cols) return BIL_E_INVALID_ARG;
  }
  if (!bil_internal::extent_ok(n_rows, ld_hidden, 2) || !bil_internal::extent_ok(shard_cols, ld_weight, 2) ||
      !bil_internal::extent_ok(n_rows, ld_part, 4) ||
      (logits != nullptr && !bil_internal::extent_ok(n_rows, ld_logits, logits_dtype == BIL_F32 ? 4 : 2)))
    return BIL_E_UNSUPPORTED;
  float rcp = 1.0f;
  if (int st = bil_internal::temperature_rcp(temperature, &rcp)) return st;
  if (n_rows == 0) return BIL_OK;
  if (hidden == nullptr || weight == nullptr || target_ids == nullptr || part_max == nullptr ||
      part_sum == nullptr || target_logit == nullptr)
    return BIL_E_INVALID_ARG;
  // TMA: 16-byte aligned bases and row strides.
  if (!aligned_to(hidden, 16) || !aligned_to(weight, 16) || (ld_hidden * 2) % 16 != 0 || (ld_weight * 2) % 16 != 0)
    return BIL_E_ALIGN;
  if (!aligned_to(target_ids, 8) || !aligned_to(part_max, 4) || !aligned_to(part_sum, 4) ||
      (part_ent && !aligned_to(part_ent, 4)) || !aligned_to(target_logit, 4))
    return BIL_E_ALIGN;
  if (logits != nullptr) {
    const int64_t eb = logits_dtype == BIL_F32 ? 4 : 2;
    if (!aligned_to(logits, 16) || (ld_logits * eb) % 16 != 0) return BIL_E_ALIGN;
  }
  if (n_rows > (static_cast<int64_t>(INT32_MAX) - kBM) || shard_cols > INT32_MAX - kBN) return BIL_E_UNSUPPORTED;

  // A batch of fewer than kBM rows is copied with a box of exactly its rows:
  // no part of the box lies outside the hidden states (measured: copies of a
  // 128-row box mostly past the end slowed the weight stream by up to 35% at
  // 1-12 rows).  The stage's other rows keep stale bytes; the tensor cores
  // turn them into accumulator rows of their own, which no thread stores.
  const int a_rows = static_cast<int>(n_rows < kBM ? n_rows : kBM);
  CUtensorMap mh, mw;
  if (int st = make_map(&mh, hidden, dtype, n_rows, hidden_size, ld_hidden, a_rows)) return st;
  if (int st = make_map(&mw, weight, dtype, shard_cols, hidden_size, ld_weight, kBN)) return st;

  LinearParams p{};
  p.n_rows = n_rows;
  p.shard_cols = shard_cols;
  p.tile_begin = tile_begin;
  p.num_n = tile_end - tile_begin;
  p.num_m = static_cast<int>((n_rows + kBM - 1) / kBM);
  p.k_blocks = static_cast<int>((hidden_size + kBK - 1) / kBK);
  p.targets = target_ids;
  p.ignore_index = ignore_index;
  p.rcp = rcp;
  p.part_max = part_max;
  p.part_sum = part_sum;
  p.part_ent = part_ent;
  p.ld_part = ld_part;
  p.target_logit = target_logit;
  p.logits = static_cast<unsigned char*>(logits);
  p.logits_dtype = logits_dtype;
  p.ld_logits = ld_logits;
  p.idesc = make_idesc(dtype == BIL_BF16);
  p.a_box_bytes = static_cast<unsigned>(a_rows) * kBK * 2;
  p.m_group = kMGroup;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  CUtensorMap mo = mw;
  if (BIL_EPILOGUE_TMA_STORE && logits != nullptr) {
    if (int st = make_store_map(&mo, logits, logits_dtype, n_rows, shard_cols, ld_logits)) return st;
  }
  return launch_gemm(part_ent != nullptr ? linear_partials_kernel<true> : linear_partials_kernel<false>, mh, mw, mo,
                     p, s);
}

int bil_linear_logp_workspace_bytes(int64_t n_rows, int64_t vocab, int entropy, int64_t* bytes) {
  if (n_rows < 0 || vocab < 1 || bytes == nullptr) return BIL_E_INVALID_ARG;
  if (!workspace_fits(n_rows, vocab)) return BIL_E_UNSUPPORTED;
  const int64_t num_tiles = (vocab + kBN - 1) / kBN;
  *bytes = static_cast<int64_t>(workspace_layout(n_rows, num_tiles, entropy != 0).total);
  return BIL_OK;
}

int bil_linear_logp_fwd(const void* hidden, const void* weight, int dtype, int64_t n_rows, int64_t hidden_size,
                        int64_t ld_hidden, int64_t vocab, int64_t ld_weight, float temperature,
                        const int64_t* target_ids, int64_t ignore_index, float* logp, float* lse, float* entropy,
                        void* logits, int logits_dtype, int64_t ld_logits, void* workspace,
                        int64_t workspace_bytes, int validate, bil_stream_t stream) {
  bil_internal::NvtxRange nvtx_range("bil_linear_logp_fwd");
  if (n_rows < 0 || vocab < 1) return BIL_E_INVALID_ARG;
  if (!workspace_fits(n_rows, vocab)) return BIL_E_UNSUPPORTED;
  const int64_t num_tiles = (vocab + kBN - 1) / kBN;
  const Workspace w = workspace_layout(n_rows, num_tiles, entropy != nullptr);
  if (n_rows == 0) return BIL_OK;
  if (logp == nullptr || workspace == nullptr) return BIL_E_INVALID_ARG;
  if (workspace_bytes < static_cast<int64_t>(w.total)) return BIL_E_INVALID_ARG;
  if (!aligned_to(workspace, 256)) return BIL_E_ALIGN;
  if (!aligned_to(logp, 4) || (lse && !aligned_to(lse, 4)) || (entropy && !aligned_to(entropy, 4)))
    return BIL_E_ALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (validate && target_ids != nullptr) {
    if (int st = bil_internal::check_targets_host(target_ids, n_rows, ignore_index, vocab, s)) return st;
  }
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  float* pm = reinterpret_cast<float*>(ws);
  float* ps = reinterpret_cast<float*>(ws + w.part);
  float* pe = entropy != nullptr ? reinterpret_cast<float*>(ws + 2 * w.part) : nullptr;
  float* tl = reinterpret_cast<float*>(ws + w.part * (entropy != nullptr ? 3 : 2));
  if (int st = bil_linear_logp_partials(hidden, weight, dtype, n_rows, hidden_size, ld_hidden, vocab, ld_weight, 0,
                                        static_cast<int32_t>(num_tiles), temperature, target_ids, ignore_index, pm,
                                        ps, pe, num_tiles, tl, logits, logits_dtype, ld_logits, stream))
    return st;
  return bil_logp_merge(pm, ps, pe, n_rows, static_cast<int32_t>(num_tiles), num_tiles, tl, target_ids,
                        ignore_index, vocab, logp, lse, entropy, 0, stream);
}

int bil_sum_f32(const float* const* srcs, int count, int64_t n, float* dst, bil_stream_t stream) {
  bil_internal::NvtxRange nvtx_range("bil_sum_f32");
  if (srcs == nullptr || count < 1 || count > kMaxSumSources || n < 0 || dst == nullptr) return BIL_E_INVALID_ARG;
  SumSources s{};
  for (int k = 0; k < count; ++k) {
    if (srcs[k] == nullptr) return BIL_E_INVALID_ARG;
    if (!aligned_to(srcs[k], 4)) return BIL_E_ALIGN;
    s.src[k] = srcs[k];
  }
  if (!aligned_to(dst, 4)) return BIL_E_ALIGN;
  if (n == 0) return BIL_OK;
  int sms = 0, smem = 0;
  if (int st = bil_internal::device_limits(&sms, &smem)) return st;
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, static_cast<int64_t>(sms) * 8));
  sum_f32_kernel<<<static_cast<unsigned>(grid), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(s, count, n, dst);
  return cudaGetLastError() == cudaSuccess ? BIL_OK : BIL_E_CUDA;
}

int bil_linear_logp_bwd(const void* hidden, const void* weight, int dtype, int64_t n_rows, int64_t hidden_size,
                        int64_t ld_hidden, int64_t vocab, int64_t ld_weight, int32_t tile_begin, int32_t tile_end,
                        float temperature, const int64_t* target_ids, int64_t ignore_index, const float* lse,
                        const float* grad_logp, const float* entropy, const float* grad_entropy, void* dz,
                        int64_t ld_dz, void* dhidden, int dhidden_dtype, int64_t ld_dhidden, void* dweight,
                        int dweight_dtype, int64_t ld_dweight, bil_stream_t stream) {
  bil_internal::NvtxRange nvtx_range("bil_linear_logp_bwd");
  if (dtype != BIL_BF16 && dtype != BIL_F16) return BIL_E_DTYPE;
  for (int ot : {dhidden_dtype, dweight_dtype})
    if (ot != BIL_F32 && ot != dtype) return BIL_E_DTYPE;
  int64_t cols = 0;
  if (int st = check_grad_args(hidden, weight, n_rows, hidden_size, ld_hidden, vocab, ld_weight, tile_begin, tile_end,
                               target_ids, lse, grad_logp, entropy, grad_entropy, dz, ld_dz, &cols))
    return st;
  if (ld_dhidden < hidden_size || ld_dweight < hidden_size) return BIL_E_INVALID_ARG;
  const int64_t eo_h = dhidden_dtype == BIL_F32 ? 4 : 2, eo_w = dweight_dtype == BIL_F32 ? 4 : 2;
  if (!bil_internal::extent_ok(n_rows, ld_dhidden, eo_h) || !bil_internal::extent_ok(cols, ld_dweight, eo_w))
    return BIL_E_UNSUPPORTED;
  float rcp = 1.0f;
  if (int st = bil_internal::temperature_rcp(temperature, &rcp)) return st;
  if (dweight == nullptr) return BIL_E_INVALID_ARG;
  if (!rows16(dweight, ld_dweight, eo_w)) return BIL_E_ALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (n_rows == 0) {  // dweight is a sum over no rows
    return cudaMemset2DAsync(dweight, static_cast<size_t>(ld_dweight * eo_w), 0,
                             static_cast<size_t>(hidden_size * eo_w), static_cast<size_t>(cols), s) == cudaSuccess
               ? BIL_OK
               : BIL_E_CUDA;
  }
  if (dhidden == nullptr) return BIL_E_INVALID_ARG;
  if (!rows16(dhidden, ld_dhidden, eo_h)) return BIL_E_ALIGN;

  // Every tensor map is encoded before anything is queued.  The store GEMMs
  // read dz, weight and hidden where they lie, as MN-major operands where
  // their rows run along K:
  //   grad:     A = hidden [n, H],            B = weight [V, H]             (K = H)
  //   dhidden:  A = dz [n, V],                B = weight [V, H] as [K, H]   (K = V)
  //   dweight:  A = dz [n, V] as [K, V],      B = hidden [n, H] as [K, H]   (K = n)
  CUtensorMap maps[6];
  {
    int st = make_map(&maps[0], hidden, dtype, n_rows, hidden_size, ld_hidden, kBM);
    if (!st) st = make_map(&maps[1], weight, dtype, cols, hidden_size, ld_weight, kBN);
    if (!st) st = operand_map(&maps[2], dz, dtype, n_rows, cols, ld_dz, false, kBM);
    if (!st) st = operand_map(&maps[3], weight, dtype, hidden_size, cols, ld_weight, true, kBN);
    if (!st) st = operand_map(&maps[4], dz, dtype, cols, n_rows, ld_dz, true, kBM);
    if (!st) st = operand_map(&maps[5], hidden, dtype, hidden_size, n_rows, ld_hidden, true, kBN);
    if (st) return st;
  }
  const bool bf16 = dtype == BIL_BF16;
  // 1. dZ from the recomputed projection, stored as dz [n, V]
  if (int st = launch_grad(maps[0], maps[1], dtype, n_rows, hidden_size, cols, tile_begin, tile_end, rcp, target_ids,
                           ignore_index, lse, grad_logp, entropy, grad_entropy, vocab, dz, ld_dz, s))
    return st;
  // 2. dhidden = dZ . weight
  if (int st = launch_store(maps[2], maps[3], n_rows, hidden_size, cols, bf16, false, true, dhidden, dhidden_dtype,
                            ld_dhidden, s))
    return st;
  // 3. dweight = dZ^T . hidden
  return launch_store(maps[4], maps[5], cols, hidden_size, n_rows, bf16, true, true, dweight, dweight_dtype,
                      ld_dweight, s);
}

int bil_linear_logp_grad(const void* hidden, const void* weight, int dtype, int64_t n_rows, int64_t hidden_size,
                         int64_t ld_hidden, int64_t vocab, int64_t ld_weight, int32_t tile_begin, int32_t tile_end,
                         float temperature, const int64_t* target_ids, int64_t ignore_index, const float* lse,
                         const float* grad_logp, const float* entropy, const float* grad_entropy, void* dz,
                         int64_t ld_dz, bil_stream_t stream) {
  bil_internal::NvtxRange nvtx_range("bil_linear_logp_grad");
  if (dtype != BIL_BF16 && dtype != BIL_F16) return BIL_E_DTYPE;
  int64_t cols = 0;
  if (int st = check_grad_args(hidden, weight, n_rows, hidden_size, ld_hidden, vocab, ld_weight, tile_begin, tile_end,
                               target_ids, lse, grad_logp, entropy, grad_entropy, dz, ld_dz, &cols))
    return st;
  float rcp = 1.0f;
  if (int st = bil_internal::temperature_rcp(temperature, &rcp)) return st;
  if (n_rows == 0) return BIL_OK;
  CUtensorMap mh, mw;
  if (int st = make_map(&mh, hidden, dtype, n_rows, hidden_size, ld_hidden, kBM)) return st;
  if (int st = make_map(&mw, weight, dtype, cols, hidden_size, ld_weight, kBN)) return st;
  return launch_grad(mh, mw, dtype, n_rows, hidden_size, cols, tile_begin, tile_end, rcp, target_ids, ignore_index, lse,
                     grad_logp, entropy, grad_entropy, vocab, dz, ld_dz, reinterpret_cast<cudaStream_t>(stream));
}

int bil_linear_gemm(const void* a, int a_layout, const void* b, int b_layout, int dtype, int64_t m, int64_t n,
                    int64_t k, int64_t lda, int64_t ldb, void* c, int c_dtype, int64_t ldc, bil_stream_t stream) {
  bil_internal::NvtxRange nvtx_range("bil_linear_gemm");
  if (dtype != BIL_BF16 && dtype != BIL_F16) return BIL_E_DTYPE;
  if (c_dtype != BIL_F32 && c_dtype != dtype) return BIL_E_DTYPE;
  for (int layout : {a_layout, b_layout})
    if (layout != BIL_LAYOUT_K_MAJOR && layout != BIL_LAYOUT_MN_MAJOR) return BIL_E_INVALID_ARG;
  const bool a_mn = a_layout == BIL_LAYOUT_MN_MAJOR, b_mn = b_layout == BIL_LAYOUT_MN_MAJOR;
  // stored shapes: A [m, k] or [k, m], B [n, k] or [k, n]
  const int64_t a_srows = a_mn ? k : m, a_scols = a_mn ? m : k;
  const int64_t b_srows = b_mn ? k : n, b_scols = b_mn ? n : k;
  if (m < 0 || n < 0 || k < 1 || lda < a_scols || ldb < b_scols || ldc < n) return BIL_E_INVALID_ARG;
  const int64_t ec = c_dtype == BIL_F32 ? 4 : 2;
  if (!bil_internal::extent_ok(a_srows, lda, 2) || !bil_internal::extent_ok(b_srows, ldb, 2) ||
      !bil_internal::extent_ok(m, ldc, ec))
    return BIL_E_UNSUPPORTED;
  if (m == 0 || n == 0) return BIL_OK;
  if (a == nullptr || b == nullptr || c == nullptr) return BIL_E_INVALID_ARG;
  if (!rows16(a, lda, 2) || !rows16(b, ldb, 2) || !rows16(c, ldc, ec)) return BIL_E_ALIGN;
  if (m > INT32_MAX - kBN || n > INT32_MAX - kBN || k > INT32_MAX - kBK) return BIL_E_UNSUPPORTED;
  CUtensorMap ma, mb;
  if (int st = operand_map(&ma, a, dtype, m, k, lda, a_mn, kBM)) return st;
  if (int st = operand_map(&mb, b, dtype, n, k, ldb, b_mn, kBN)) return st;
  return launch_store(ma, mb, m, n, k, dtype == BIL_BF16, a_mn, b_mn, c, c_dtype, ldc,
                      reinterpret_cast<cudaStream_t>(stream));
}

int bil_linear_logp_fwd_static(const void* hidden, const void* weight, int dtype, int64_t n_rows,
                               int64_t hidden_size, int64_t ld_hidden, int64_t vocab, int64_t ld_weight,
                               float temperature, const int64_t* target_ids, int64_t ignore_index, float* logp,
                               float* lse, float* entropy, int validate, bil_stream_t stream) {
  bil_internal::NvtxRange nvtx_range("bil_linear_logp_fwd_static");
  if (n_rows < 0 || vocab < 1) return BIL_E_INVALID_ARG;
  if (!workspace_fits(n_rows, vocab)) return BIL_E_UNSUPPORTED;
  const int64_t num_tiles = (vocab + kBN - 1) / kBN;
  const Workspace w = workspace_layout(n_rows, num_tiles, entropy != nullptr);
  if (w.total > BIL_LINEAR_STATIC_SCRATCH_BYTES) return BIL_E_UNSUPPORTED;
  if (n_rows == 0) return BIL_OK;
  void* scratch = nullptr;
  if (int st = static_scratch(&scratch)) return st;
  return bil_linear_logp_fwd(hidden, weight, dtype, n_rows, hidden_size, ld_hidden, vocab, ld_weight, temperature,
                             target_ids, ignore_index, logp, lse, entropy, nullptr, BIL_F32, 0, scratch,
                             static_cast<int64_t>(BIL_LINEAR_STATIC_SCRATCH_BYTES), validate, stream);
}

}  // extern "C"
