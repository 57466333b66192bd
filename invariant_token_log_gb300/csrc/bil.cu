// Batch-invariant selected-token log-probability for sm_103a (GB300): host side
// of the logits path and its kernels' launches.
//
// Operator: "Batch-Invariant LogP" operator page, sections "Reference
// Semantics" (what is computed), "Tensor Parallel" steps 1-6 (the fixed-tile
// (max, sumexp) partials and their fixed-order merge) and "Batch-Invariance"
// (one row's result depends on that row only; the backward recomputes the
// softmax from the saved per-row LSE).  The C ABI is declared in include/bil.h.
//
// Kernels (device code in logp_device.cuh)
//   stream_kernel<FUSED=true>   forward: every tile of a row -> shared-memory
//                               partials -> fixed-order merge -> logp, lse.
//   stream_kernel<FUSED=false>  partials of a tile range -> [N, ld_part] buffers.
//   split_row_kernel            forward of up to 128 rows (16 off 16-byte
//                               boundaries), one row per cluster.
//   merge_kernel                fixed-order merge of [N, T] partials -> logp, lse.
//   bwd_kernel                  dlogits = g * (onehot - exp(x - lse)); rows aligned,
//                               at offsets shared by input and output, or scalar.
// The fused LM-head is in linear.cu.
//
// The forward streams each row exactly once.  A producer warp moves whole
// tiles HBM -> shared memory with 1-D bulk asynchronous copies
// (cp.async.bulk, completion counted on an mbarrier) into a ring of stages;
// consumer warps reduce one tile each.  Rows that do not start on a 16-byte
// boundary are copied from the boundary below each tile, and the consumers
// shift the tile's words back into place as they read them.  Nothing on this
// path is a contraction, so no tensor cores are used: the forward is bound by
// HBM bandwidth, with the exponential unit second.
//
// The arithmetic contract (what makes the bits reproducible) lives in the
// tile reduction, merge_lse and the gradient formula of logp_device.cuh and
// nowhere else: every kernel that produces a tile partial, an LSE or a
// gradient calls them, so all paths give identical bits by construction.
// All floating-point operations that matter are written with explicit
// round-to-nearest or fused intrinsics, and the files are compiled with
// contraction off.

#include "../../include/bil.h"
#include "device_common.cuh"
#include "internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <utility>

#include "logp_device.cuh"

namespace {
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

// Whether every one of n_rows rows of ld elements of elem_bytes bytes from p
// starts on a 16-byte boundary (a single row's stride is never used).
bool rows_aligned16(const void* p, int64_t n_rows, int64_t ld, int elem_bytes) {
  return aligned(p, 16) && (n_rows <= 1 || (ld * elem_bytes) % 16 == 0);
}

struct DeviceInfo {
  int sms = 0;
  int max_smem_optin = 0;
};

// Per-device attributes, queried once per device and shared by every host
// thread: the shared-memory limit is stored first and the SM count published
// after it with release order, so a thread that reads a non-zero SM count
// (acquire) also sees the limit.  Threads that race to fill an entry store the
// same values.
constexpr int kMaxDevices = 64;
std::atomic<int> g_device_sms[kMaxDevices];
std::atomic<int> g_device_smem[kMaxDevices];

int device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BIL_E_CUDA;
  int sms = g_device_sms[dev].load(std::memory_order_acquire);
  if (sms == 0) {
    int smem = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return BIL_E_CUDA;
    if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return BIL_E_CUDA;
    g_device_smem[dev].store(smem, std::memory_order_relaxed);
    g_device_sms[dev].store(sms, std::memory_order_release);
  }
  out->sms = sms;
  out->max_smem_optin = g_device_smem[dev].load(std::memory_order_relaxed);
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

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel in the stream finishes (its launch latency hides
// behind that kernel's tail).  Only kernels that wait for their predecessor
// with griddep_wait() before touching global memory are launched this way:
// the forward's stream, cluster and merge kernels.  (The backward is not: the
// wait made its element-by-element loads twice as slow.)  cluster > 1:
// thread-block clusters of that many blocks along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), int64_t grid, int block, size_t smem, cudaStream_t stream,
                       int cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(block), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Pipeline shape for a stage size: a ring of about BIL_STREAM_RING_BYTES per
// block (two blocks share an SM), at least two stages, up to
// kMaxConsumers consumer warps, and a stage count that is a multiple of the
// consumer count.  The last rule is what keeps the barrier protocol sound:
// consumer c then owns stages c, c+W, c+2W, ... and meets them in fill
// order, so it can never wait on a stage two fills ahead of the copy that is
// landing in it (a wait only tells the parity of a stage's fill count apart).
#ifndef BIL_STREAM_RING_BYTES
#define BIL_STREAM_RING_BYTES (96 * 1024)
#endif
struct StreamShape {
  int stages, consumers, row_slots;
  size_t smem;
};

StreamShape stream_shape(unsigned stage_bytes, int num_tiles, bool fused, bool ent) {
  StreamShape s;
  const int most = static_cast<int>(std::max<size_t>(2, std::min<size_t>(32, BIL_STREAM_RING_BYTES / stage_bytes)));
  s.consumers = std::min(kMaxConsumers, most);
  s.stages = (most / s.consumers) * s.consumers;
  s.row_slots = fused ? 4 : 0;
  s.smem = stream_smem_bytes(s.stages, stage_bytes, s.row_slots, num_tiles, fused, ent, nullptr, nullptr);
  return s;
}

template <int DT, bool FUSED, bool ALIGNED, bool ENT>
int launch_stream_t(const StreamParams& p0, cudaStream_t stream) {
  DeviceInfo dev;
  if (int st = device_info(&dev)) return st;
  StreamParams p = p0;
  StreamShape shape = stream_shape(p.stage_bytes, p.num_tiles, FUSED, ENT);
  if (shape.smem > static_cast<size_t>(dev.max_smem_optin)) return BIL_E_UNSUPPORTED;
  if (shape.consumers < 1 || shape.stages % shape.consumers != 0) return BIL_E_UNSUPPORTED;
  p.stages = shape.stages;
  p.consumers = shape.consumers;
  p.row_slots = shape.row_slots;
  auto kernel = stream_kernel<DT, FUSED, ALIGNED, ENT>;
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
  if (launch_pdl(kernel, grid, threads, shape.smem, stream, 1, p) != cudaSuccess) return BIL_E_CUDA;
  return cudaGetLastError() == cudaSuccess ? BIL_OK : BIL_E_CUDA;
}

template <int DT, bool FUSED>
int launch_stream_dt(bool aligned_rows, bool ent, const StreamParams& p, cudaStream_t stream) {
  if (ent)
    return aligned_rows ? launch_stream_t<DT, FUSED, true, true>(p, stream)
                        : launch_stream_t<DT, FUSED, false, true>(p, stream);
  return aligned_rows ? launch_stream_t<DT, FUSED, true, false>(p, stream)
                      : launch_stream_t<DT, FUSED, false, false>(p, stream);
}

template <bool FUSED>
int launch_stream(int dtype, bool ent, const StreamParams& p0, cudaStream_t stream) {
  const int eb = elem_bytes(dtype);
  // Every tile starts 16-byte aligned, or the copies start up to 15 bytes
  // early and a stage holds 128 bytes more than the tile.
  const bool aligned_rows = rows_aligned16(p0.logits, p0.n_rows, p0.ld, eb);
  StreamParams p = p0;
  p.stage_bytes = static_cast<unsigned>(static_cast<size_t>(p.tile_v) * eb + (aligned_rows ? 0 : 128));
  switch (dtype) {
    case BIL_BF16: return launch_stream_dt<BIL_BF16, FUSED>(aligned_rows, ent, p, stream);
    case BIL_F16: return launch_stream_dt<BIL_F16, FUSED>(aligned_rows, ent, p, stream);
    case BIL_F32: return launch_stream_dt<BIL_F32, FUSED>(aligned_rows, ent, p, stream);
    default: return BIL_E_DTYPE;
  }
}

// Rows at or below which the forward takes the cluster path (one row per
// cluster of kSplitCtas blocks) when it applies.  Rows off 16-byte
// boundaries cost the cluster path two 16-byte loads per group, and it beats
// the streaming path only for fewer rows (measured on 50257- and
// 151935-column rows: the crossover lies between 7 and 64 rows for the first).
#ifndef BIL_SPLIT_MAX_ROWS
#define BIL_SPLIT_MAX_ROWS 128
#endif
#ifndef BIL_SPLIT_MAX_ROWS_UNALIGNED
#define BIL_SPLIT_MAX_ROWS_UNALIGNED 16
#endif

template <int DT, bool ENT, bool ALIGNED>
int launch_split_t(const StreamParams& p, cudaStream_t stream) {
  if (launch_pdl(split_row_kernel<DT, ENT, ALIGNED>, p.n_rows * kSplitCtas, kSplitWarps * kLanes, 0, stream,
                 kSplitCtas, p) != cudaSuccess)
    return BIL_E_CUDA;
  return cudaGetLastError() == cudaSuccess ? BIL_OK : BIL_E_CUDA;
}

// Whether the fused forward of these rows takes the cluster path.
bool use_split(int dtype, const StreamParams& p) {
  const int eb = elem_bytes(dtype);
  const int64_t most = rows_aligned16(p.logits, p.n_rows, p.ld, eb) ? BIL_SPLIT_MAX_ROWS : BIL_SPLIT_MAX_ROWS_UNALIGNED;
  return eb == 2 && p.n_rows >= 1 && p.n_rows <= most && p.tile_v <= 4096 && p.num_tiles <= BIL_MAX_FUSED_TILES;
}

template <int DT, bool ENT>
int launch_split_dt(const StreamParams& p, cudaStream_t stream) {
  return rows_aligned16(p.logits, p.n_rows, p.ld, elem_bytes(DT)) ? launch_split_t<DT, ENT, true>(p, stream)
                                                                   : launch_split_t<DT, ENT, false>(p, stream);
}

int launch_split(int dtype, bool ent, const StreamParams& p, cudaStream_t stream) {
  switch (dtype) {
    case BIL_BF16: return ent ? launch_split_dt<BIL_BF16, true>(p, stream) : launch_split_dt<BIL_BF16, false>(p, stream);
    case BIL_F16: return ent ? launch_split_dt<BIL_F16, true>(p, stream) : launch_split_dt<BIL_F16, false>(p, stream);
    default: return BIL_E_DTYPE;
  }
}

// rows x pitch x eb <= BIL_MAX_EXTENT_BYTES, without forming the product.
bool extent_ok(int64_t rows, int64_t pitch, int64_t eb) {
  return rows <= 0 || pitch <= BIL_MAX_EXTENT_BYTES / eb / rows;
}

int check_tile(int dtype, int64_t vocab, int32_t tile_v, int64_t* num_tiles) {
  const int eb = elem_bytes(dtype);
  if (eb == 0) return BIL_E_DTYPE;
  if (tile_v <= 0 || tile_v % kGroup != 0) return BIL_E_INVALID_ARG;
  if (static_cast<int64_t>(tile_v) * eb > BIL_MAX_TILE_BYTES) return BIL_E_UNSUPPORTED;
  if (vocab > BIL_MAX_EXTENT_BYTES) return BIL_E_UNSUPPORTED;
  *num_tiles = (vocab + tile_v - 1) / tile_v;
  if (*num_tiles > INT32_MAX) return BIL_E_UNSUPPORTED;
  return BIL_OK;
}

// The temperature's reciprocal as the kernels use it: 1/T computed in double
// and rounded once to float32.  T must be finite and > 0.
int temperature_rcp(float temperature, float* rcp) {
  if (!(temperature > 0.0f) || !std::isfinite(temperature)) return BIL_E_INVALID_ARG;
  const double r = 1.0 / static_cast<double>(temperature);
  if (!(r < 3.0e38)) return BIL_E_INVALID_ARG;
  *rcp = static_cast<float>(r);
  return BIL_OK;
}

// Resident warps per SM for the vectorised backward without the entropy
// term.  Its loop is a bare stream (load, a few operations, store), and more
// resident warps than this oversubscribe the memory system: on GB300 the
// 16-bit training backward (16384 x 151936) took 1.61 ms with the 40 warps
// that fit and 1.52 ms with 32; 24 warps took 1.68 ms.  The entropy term's
// extra arithmetic per element wants every warp that fits (1.55 ms with 40,
// 1.60 ms with 32), and so does the element-by-element path for rows off
// 16-byte boundaries (its scalar loads need the warps to keep bytes in
// flight).
#ifndef BIL_BWD_PLAIN_WARPS_PER_SM
#define BIL_BWD_PLAIN_WARPS_PER_SM 32
#endif

// rows: a BwdRows value.  The rows that go by 16-byte vectors (aligned, or
// input and output at shared offsets) take the warp cap below.
template <int DT, int OT>
int launch_bwd_t(int rows, const BwdParams& bp, cudaStream_t stream) {
  DeviceInfo dev;
  if (int st = device_info(&dev)) return st;
  auto kernel = rows == kBwdAligned         ? bwd_kernel<DT, OT, kBwdAligned>
                : rows == kBwdSharedOffsets ? bwd_kernel<DT, OT, kBwdSharedOffsets>
                                            : bwd_kernel<DT, OT, kBwdScalar>;
  const bool streamed = rows != kBwdScalar;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kBwdThreads, 0) != cudaSuccess)
    return BIL_E_CUDA;
  if (streamed && bp.grad_entropy == nullptr)
    per_sm = std::min(per_sm, BIL_BWD_PLAIN_WARPS_PER_SM / (kBwdThreads / kLanes));
  per_sm = std::max(1, per_sm);
  const int64_t units = bp.n_rows * ((bp.out_cols + kBwdChunk - 1) / kBwdChunk);
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(units, static_cast<int64_t>(dev.sms) * per_sm));
  kernel<<<static_cast<unsigned>(grid), kBwdThreads, 0, stream>>>(bp);
  return cudaGetLastError() == cudaSuccess ? BIL_OK : BIL_E_CUDA;
}

template <int DT>
int launch_bwd_dt(int out_dtype, int rows, const BwdParams& bp, cudaStream_t stream) {
  switch (out_dtype) {
    case BIL_F32: return launch_bwd_t<DT, BIL_F32>(rows, bp, stream);
    case BIL_BF16: return launch_bwd_t<DT, BIL_BF16>(rows, bp, stream);
    case BIL_F16: return launch_bwd_t<DT, BIL_F16>(rows, bp, stream);
    default: return BIL_E_DTYPE;
  }
}

// ---------------------------------------------------------------------------
// Measurement: the throughput of the exponential unit, the logits path's
// second bound after HBM (one ex2.approx per element in every pass).  Each
// thread runs 8 independent chains x <- 2^(-x) of the contract's ex2.approx
// (x stays in [0.5, 1]); thread 0 of each block records the block's SM and
// that SM's cycle counter before and after the loop.
// ---------------------------------------------------------------------------

constexpr int kExpRateThreads = 256;
constexpr int kExpRateChains = 8;

__global__ void __launch_bounds__(kExpRateThreads) exp_rate_kernel(int iters, float* sink, long long* rec) {
  float x[kExpRateChains];
#pragma unroll
  for (int j = 0; j < kExpRateChains; ++j) x[j] = 0.5f + 0.0625f * j + 1e-7f * threadIdx.x;
  __syncthreads();
  const long long t0 = clock64();
#pragma unroll 1
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < kExpRateChains; ++j) x[j] = ex2_approx(-x[j]);
  }
  __syncthreads();
  const long long t1 = clock64();
  float s = 0.0f;
#pragma unroll
  for (int j = 0; j < kExpRateChains; ++j) s += x[j];
  if (s < 0.0f) sink[0] = s;  // never true (every x is positive): keeps the chains live
  if (threadIdx.x == 0) {
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    rec[3 * blockIdx.x] = smid;
    rec[3 * blockIdx.x + 1] = t0;
    rec[3 * blockIdx.x + 2] = t1;
  }
}

}  // namespace

namespace bil_internal {

int check_targets_host(const int64_t* targets, int64_t n, int64_t ignore_index, int64_t vocab,
                       cudaStream_t stream) {
  return ::check_targets_host(targets, n, ignore_index, vocab, stream);
}

int temperature_rcp(float temperature, float* rcp) { return ::temperature_rcp(temperature, rcp); }

int elem_bytes(int dtype) { return ::elem_bytes(dtype); }

bool extent_ok(int64_t rows, int64_t pitch, int64_t eb) { return ::extent_ok(rows, pitch, eb); }

int check_tile(int dtype, int64_t vocab, int32_t tile_v, int64_t* num_tiles) {
  return ::check_tile(dtype, vocab, tile_v, num_tiles);
}

int device_limits(int* sms, int* max_smem_optin) {
  DeviceInfo dev;
  if (int st = device_info(&dev)) return st;
  *sms = dev.sms;
  *max_smem_optin = dev.max_smem_optin;
  return BIL_OK;
}

}  // namespace bil_internal

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------

extern "C" {

const char* bil_contract_id(void) {
  return "bil.v4"
         ";tile=fixed tile_v columns, valid columns < vocab"
         ";rcp=float32(1/temperature) (rcp=1: no multiply)"
         ";lanes=32x8: lane l takes 8-element groups l, l+32, ... in order"
         ";max=exact, on x: m_x; m_t=m_x*rn rcp"
         ";tile_term=e=ex2.approx.ftz.f32(t), t=(x-rn m_x)*rn c, c=rcp*rn log2e"
         ";exp(a)=ex2.approx.ftz.f32(a*rn log2e) (merge, backward)"
         ";lane_sum=8 slot accumulators, ((a0+a1)+(a2+a3))+((a4+a5)+(a6+a7))"
         ";warp_sum=butterfly xor 16,8,4,2,1"
         ";entropy_sum=u_j=fma(e,max(t,-FLT_MAX),u_j), same trees; u_t=sum*rn ln2"
         ";merge=M=max m_t; w_t=exp(m_t-M); S=fma(s_t,w_t,S) t=0..T-1; LSE=M+rn logf(S)"
         ";merge_entropy=U=fma(fma(max(m_t-M,-FLT_MAX),s_t,u_t),w_t,U); H=logf(S)-rn(U/rn S)"
         ";logp=z_t-rn LSE, z_t=x_t*rn rcp"
         ";bwd=a=fma(x,rcp,-lse) (rcp=1: x-rn lse); p=exp(a); d=g*(onehot-p), with entropy"
         " d=fma(g,onehot-p,-(gh*(p*(max(a,-FLT_MAX)+H)))); [*rcp]; store rn"
         ";linear=z=fp32 tcgen05 sum over K blocks of 64 in order; tile 256, one thread per row,"
         " 8 slots over columns 8g+j, g in order, ((a0+a1)+(a2+a3))+((a4+a5)+(a6+a7))";
}

const char* bil_status_string(int status) {
  switch (status) {
    case BIL_OK: return "ok";
    case BIL_E_INVALID_ARG: return "invalid argument";
    case BIL_E_DTYPE: return "unsupported element type";
    case BIL_E_ALIGN: return "pointer not aligned to its element size";
    case BIL_E_TARGET_RANGE: return "active target outside [0, vocab)";
    case BIL_E_CUDA: return "CUDA runtime error";
    case BIL_E_UNSUPPORTED: return "beyond the library's limits";
    default: return "unknown status";
  }
}

int bil_logp_fwd(const void* logits, int dtype, int64_t n_rows, int64_t vocab, int64_t ld,
                 const int64_t* target_ids, int64_t ignore_index, int32_t tile_v, float temperature, float* logp,
                 float* lse, float* entropy, int validate, bil_stream_t stream) {
  bil_internal::NvtxRange nvtx_range("bil_logp_fwd");
  if (n_rows < 0 || vocab < 1 || ld < vocab) return BIL_E_INVALID_ARG;
  int64_t num_tiles = 0;
  if (int st = check_tile(dtype, vocab, tile_v, &num_tiles)) return st;
  if (!extent_ok(n_rows, ld, elem_bytes(dtype))) return BIL_E_UNSUPPORTED;
  float rcp = 1.0f;
  if (int st = temperature_rcp(temperature, &rcp)) return st;
  if (n_rows == 0) return BIL_OK;
  if (logits == nullptr || target_ids == nullptr || logp == nullptr) return BIL_E_INVALID_ARG;
  const int eb = elem_bytes(dtype);
  if (!aligned(logits, eb) || !aligned(target_ids, 8) || !aligned(logp, 4) || (lse && !aligned(lse, 4)) ||
      (entropy && !aligned(entropy, 4)))
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
  p.rcp = rcp;
  p.logp = logp;
  p.lse = lse;
  p.entropy = entropy;
  if (use_split(dtype, p)) return launch_split(dtype, entropy != nullptr, p, s);
  return launch_stream<true>(dtype, entropy != nullptr, p, s);
}

int bil_logp_tile_partials(const void* logits, int dtype, int64_t n_rows, int64_t vocab, int64_t ld,
                           int32_t tile_v, int32_t tile_begin, int32_t tile_end, float temperature,
                           const int64_t* target_ids, int64_t ignore_index, float* part_max, float* part_sum,
                           float* part_ent, int64_t ld_part, float* target_logit, bil_stream_t stream) {
  bil_internal::NvtxRange nvtx_range("bil_logp_tile_partials");
  if (n_rows < 0 || vocab < 1) return BIL_E_INVALID_ARG;
  int64_t num_tiles = 0;
  if (int st = check_tile(dtype, vocab, tile_v, &num_tiles)) return st;
  float rcp = 1.0f;
  if (int st = temperature_rcp(temperature, &rcp)) return st;
  if (tile_begin < 0 || tile_end <= tile_begin || tile_end > num_tiles) return BIL_E_INVALID_ARG;
  if (ld_part < num_tiles) return BIL_E_INVALID_ARG;
  // The shard holds global columns [tile_begin*tile_v, min(tile_end*tile_v, vocab)).
  const int64_t shard_cols = std::min<int64_t>(static_cast<int64_t>(tile_end) * tile_v, vocab) -
                             static_cast<int64_t>(tile_begin) * tile_v;
  if (ld < shard_cols) return BIL_E_INVALID_ARG;
  if (!extent_ok(n_rows, ld, elem_bytes(dtype)) || !extent_ok(n_rows, ld_part, 4)) return BIL_E_UNSUPPORTED;
  if (n_rows == 0) return BIL_OK;
  if (logits == nullptr || target_ids == nullptr || part_max == nullptr || part_sum == nullptr ||
      target_logit == nullptr)
    return BIL_E_INVALID_ARG;
  const int eb = elem_bytes(dtype);
  if (!aligned(logits, eb) || !aligned(target_ids, 8) || !aligned(part_max, 4) || !aligned(part_sum, 4) ||
      !aligned(target_logit, 4) || (part_ent && !aligned(part_ent, 4)))
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
  p.rcp = rcp;
  p.part_max = part_max;
  p.part_sum = part_sum;
  p.part_ent = part_ent;
  p.ld_part = ld_part;
  p.target_logit = target_logit;
  return launch_stream<false>(dtype, part_ent != nullptr, p, reinterpret_cast<cudaStream_t>(stream));
}

int bil_logp_merge(const float* part_max, const float* part_sum, const float* part_ent, int64_t n_rows,
                   int32_t num_tiles, int64_t ld_part, const float* target_logit, const int64_t* target_ids,
                   int64_t ignore_index, int64_t vocab, float* logp, float* lse, float* entropy, int validate,
                   bil_stream_t stream) {
  bil_internal::NvtxRange nvtx_range("bil_logp_merge");
  if (n_rows < 0 || num_tiles < 1 || ld_part < num_tiles || vocab < 1) return BIL_E_INVALID_ARG;
  if ((entropy != nullptr) != (part_ent != nullptr)) return BIL_E_INVALID_ARG;
  if (!extent_ok(n_rows, ld_part, 4)) return BIL_E_UNSUPPORTED;
  if (n_rows == 0) return BIL_OK;
  if (part_max == nullptr || part_sum == nullptr || target_logit == nullptr || target_ids == nullptr ||
      logp == nullptr)
    return BIL_E_INVALID_ARG;
  if (!aligned(part_max, 4) || !aligned(part_sum, 4) || !aligned(target_logit, 4) || !aligned(target_ids, 8) ||
      !aligned(logp, 4) || (lse && !aligned(lse, 4)) || (part_ent && !aligned(part_ent, 4)) ||
      (entropy && !aligned(entropy, 4)))
    return BIL_E_ALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (validate) {
    if (int st = check_targets_host(target_ids, n_rows, ignore_index, vocab, s)) return st;
  }
  DeviceInfo dev;
  if (int st = device_info(&dev)) return st;
  const int threads = 256;  // merge_kernel's shared scratch has one slot per warp of 256 threads
  // A few rows of many tiles: a block per row (the same bits, the partials' loads in one round).
  const size_t block_smem = static_cast<size_t>(num_tiles) * (entropy != nullptr ? 4 : 2) * sizeof(float);
  if (n_rows <= static_cast<int64_t>(dev.sms) && num_tiles >= kMergeBlockMinTiles && block_smem <= 48 * 1024) {
    const cudaError_t e =
        entropy != nullptr
            ? launch_pdl(merge_block_kernel<true>, n_rows, threads, block_smem, s, 1, part_max, part_sum, part_ent,
                         n_rows, num_tiles, ld_part, target_logit, target_ids, ignore_index, vocab, logp, lse, entropy)
            : launch_pdl(merge_block_kernel<false>, n_rows, threads, block_smem, s, 1, part_max, part_sum,
                         static_cast<const float*>(nullptr), n_rows, num_tiles, ld_part, target_logit, target_ids,
                         ignore_index, vocab, logp, lse, static_cast<float*>(nullptr));
    if (e != cudaSuccess) return BIL_E_CUDA;
    return cudaGetLastError() == cudaSuccess ? BIL_OK : BIL_E_CUDA;
  }
  const int64_t rows_per_block = threads / kLanes;
  const int64_t grid = std::max<int64_t>(
      1, std::min<int64_t>((n_rows + rows_per_block - 1) / rows_per_block, static_cast<int64_t>(dev.sms) * 8));
  const cudaError_t e =
      entropy != nullptr
          ? launch_pdl(merge_kernel<true>, grid, threads, 0, s, 1, part_max, part_sum, part_ent, n_rows, num_tiles,
                       ld_part, target_logit, target_ids, ignore_index, vocab, logp, lse, entropy)
          : launch_pdl(merge_kernel<false>, grid, threads, 0, s, 1, part_max, part_sum, static_cast<const float*>(nullptr),
                       n_rows, num_tiles, ld_part, target_logit, target_ids, ignore_index, vocab, logp, lse,
                       static_cast<float*>(nullptr));
  if (e != cudaSuccess) return BIL_E_CUDA;
  return cudaGetLastError() == cudaSuccess ? BIL_OK : BIL_E_CUDA;
}

int bil_logp_bwd(const void* logits, int dtype, int64_t n_rows, int64_t vocab, int64_t ld,
                 const int64_t* target_ids, int64_t ignore_index, float temperature, const float* lse,
                 const float* grad_logp, const float* entropy, const float* grad_entropy, void* dlogits,
                 int dlogits_dtype, int64_t ld_out, int64_t out_cols, bil_stream_t stream) {
  bil_internal::NvtxRange nvtx_range("bil_logp_bwd");
  const int eb = elem_bytes(dtype);
  const int ob = elem_bytes(dlogits_dtype);
  if (eb == 0 || ob == 0) return BIL_E_DTYPE;
  if (n_rows < 0 || vocab < 1 || ld < vocab || out_cols < vocab || ld_out < out_cols) return BIL_E_INVALID_ARG;
  if (!extent_ok(n_rows, ld, eb) || !extent_ok(n_rows, ld_out, ob)) return BIL_E_UNSUPPORTED;
  float rcp = 1.0f;
  if (int st = temperature_rcp(temperature, &rcp)) return st;
  if ((entropy != nullptr) != (grad_entropy != nullptr)) return BIL_E_INVALID_ARG;
  if (n_rows == 0) return BIL_OK;
  if (logits == nullptr || target_ids == nullptr || lse == nullptr || grad_logp == nullptr || dlogits == nullptr)
    return BIL_E_INVALID_ARG;
  if (!aligned(logits, eb) || !aligned(target_ids, 8) || !aligned(lse, 4) || !aligned(grad_logp, 4) ||
      !aligned(dlogits, ob) || (entropy && !aligned(entropy, 4)) || (grad_entropy && !aligned(grad_entropy, 4)))
    return BIL_E_ALIGN;
  const bool vec = rows_aligned16(logits, n_rows, ld, eb) && rows_aligned16(dlogits, n_rows, ld_out, ob);
  // input and output rows at the same offset from a 16-byte boundary, row after row
  const bool shared_offsets =
      eb == ob && (reinterpret_cast<uintptr_t>(logits) - reinterpret_cast<uintptr_t>(dlogits)) % 16 == 0 &&
      (n_rows <= 1 || ((ld - ld_out) * eb) % 16 == 0);
  const int rows = vec ? kBwdAligned : shared_offsets ? kBwdSharedOffsets : kBwdScalar;
  BwdParams bp{};
  bp.logits = static_cast<const unsigned char*>(logits);
  bp.n_rows = n_rows;
  bp.vocab = vocab;
  bp.ld = ld;
  bp.targets = target_ids;
  bp.ignore_index = ignore_index;
  bp.lse = lse;
  bp.grad = grad_logp;
  bp.entropy = entropy;
  bp.grad_entropy = grad_entropy;
  bp.rcp = rcp;
  bp.dlogits = static_cast<unsigned char*>(dlogits);
  bp.ld_out = ld_out;
  bp.out_cols = out_cols;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (dtype) {
    case BIL_BF16: return launch_bwd_dt<BIL_BF16>(dlogits_dtype, rows, bp, s);
    case BIL_F16: return launch_bwd_dt<BIL_F16>(dlogits_dtype, rows, bp, s);
    case BIL_F32: return launch_bwd_dt<BIL_F32>(dlogits_dtype, rows, bp, s);
    default: return BIL_E_DTYPE;
  }
}

int bil_stream_shape(int dtype, int32_t tile_v, int64_t num_tiles, int fused, int entropy, int* stages,
                     int* consumers, int64_t* smem_bytes) {
  const int eb = elem_bytes(dtype);
  if (eb == 0) return BIL_E_DTYPE;
  if (tile_v <= 0 || tile_v % kGroup != 0 || num_tiles < 1 || stages == nullptr || consumers == nullptr ||
      smem_bytes == nullptr)
    return BIL_E_INVALID_ARG;
  if (static_cast<int64_t>(tile_v) * eb > BIL_MAX_TILE_BYTES) return BIL_E_UNSUPPORTED;
  const StreamShape shape =
      stream_shape(static_cast<unsigned>(tile_v * eb), static_cast<int>(num_tiles), fused != 0, entropy != 0);
  *stages = shape.stages;
  *consumers = shape.consumers;
  *smem_bytes = static_cast<int64_t>(shape.smem);
  return BIL_OK;
}

int bil_watchdog_selftest(bil_stream_t stream) {
  bil_internal::NvtxRange nvtx_range("bil_watchdog_selftest");
  watchdog_selftest_kernel<<<1, kLanes, 0, reinterpret_cast<cudaStream_t>(stream)>>>();
  return cudaGetLastError() == cudaSuccess ? BIL_OK : BIL_E_CUDA;
}

int bil_probe_exp_rate(int32_t blocks, int32_t iters, float* sink, int64_t* records, bil_stream_t stream) {
  bil_internal::NvtxRange nvtx_range("bil_probe_exp_rate");
  if (blocks < 1 || iters < 1 || sink == nullptr || records == nullptr) return BIL_E_INVALID_ARG;
  if (!aligned(sink, 4) || !aligned(records, 8)) return BIL_E_ALIGN;
  exp_rate_kernel<<<static_cast<unsigned>(blocks), kExpRateThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      iters, sink, reinterpret_cast<long long*>(records));
  return cudaGetLastError() == cudaSuccess ? BIL_OK : BIL_E_CUDA;
}

int bil_watchdog_status(unsigned int* flags, int clear) {
  bil_internal::NvtxRange nvtx_range("bil_watchdog_status");
  if (flags == nullptr) return BIL_E_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return BIL_E_CUDA;
  if (cudaMemcpyFromSymbol(flags, g_watchdog, sizeof(unsigned int)) != cudaSuccess) return BIL_E_CUDA;
  if (clear) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_watchdog, &zero, sizeof(unsigned int)) != cudaSuccess) return BIL_E_CUDA;
  }
  unsigned int linear = 0;
  if (int st = bil_internal::linear_watchdog(&linear, clear)) return st;
  *flags |= linear;
  return BIL_OK;
}

}  // extern "C"
