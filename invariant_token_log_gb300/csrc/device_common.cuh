// Device helpers shared by the library's kernels: the contract's exponential,
// mbarrier operations and bounded waits.  Everything here is inline and in an
// anonymous namespace, so each translation unit gets its own copy (the
// library is built without relocatable device code).
#pragma once

#include <stdint.h>

namespace {

constexpr int kLanes = 32;

// log2(e) rounded to float32: exp(a) is evaluated as 2^(a * log2(e)).
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.693147180559945309f;  // ln 2 rounded to float32: the tile entropy sum's unit
// The most negative finite float32.
constexpr float kNegMax = -3.40282346638528859811704183484516925e38f;

__device__ __forceinline__ float ex2_approx(float a) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
  return r;
}

// Packed float32 pairs (sm_100 family): each half is an independent IEEE
// round-to-nearest operation, bit for bit what __fadd_rn / __fsub_rn /
// __fmul_rn give.  A pair is held as a 64-bit word, first element low.
__device__ __forceinline__ uint64_t pk(float lo, float hi) {
  return static_cast<uint64_t>(__float_as_uint(lo)) | (static_cast<uint64_t>(__float_as_uint(hi)) << 32);
}
__device__ __forceinline__ float lo_of(uint64_t a) { return __uint_as_float(static_cast<uint32_t>(a)); }
__device__ __forceinline__ float hi_of(uint64_t a) { return __uint_as_float(static_cast<uint32_t>(a >> 32)); }
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may be scheduled while the kernel before it in the stream is
// still finishing.  griddep_wait() returns once that kernel has completed and
// its memory operations are visible, so every thread calls it before its
// first access to global memory; griddep_launch_dependents() lets the next
// kernel in the stream be scheduled early in turn.  Without the launch
// attribute both return at once.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// exp(a) of the contract: one rounded multiply, then the hardware base-2
// exponential (flushes results below 2^-126 to zero).
__device__ __forceinline__ float contract_exp(float a) { return ex2_approx(__fmul_rn(a, kLog2e)); }

// What one row of the backward needs: its target, saved LSE, the upstream
// gradients of logp (g) and of the entropy (gh, with the row's entropy H),
// and the temperature's reciprocal.
struct RowMeta {
  int64_t target;
  float lse, g, H, gh;
};

// One element of the gradient:
//   a = x * rcp - lse (one fused multiply-add; rcp = 1: x - lse);  p = exp(a)
//   d = g * (onehot - p)
//   with entropy:  d = g * (onehot - p) - gh * (p * (a + H)), the product with
//                  g and the subtraction fused (d H / d z = -p (log p + H))
//   with a temperature:  d = d * rcp                (d z / d x = rcp)
// Every multiply whose result meets an add is an explicit fused multiply-add,
// in this scalar form and in the packed pairs of the vectorised kernels, so
// both produce the same bits whatever the code generator contracts.
__device__ __forceinline__ float grad_elem(float x, const RowMeta& m, bool is_target, float rcp, bool ent) {
  const bool scaled = rcp != 1.0f;
  const float a = scaled ? __fmaf_rn(x, rcp, -m.lse) : __fsub_rn(x, m.lse);
  const float p = contract_exp(a);
  const float om = __fsub_rn(is_target ? 1.0f : 0.0f, p);
  float d;
  if (ent) {
    // p (log p + H) -> 0 as p -> 0: a clamped to the largest finite magnitude
    // makes the term of an -inf logit 0 instead of 0 * inf
    const float t3 = __fmul_rn(m.gh, __fmul_rn(p, __fadd_rn(fmaxf(a, kNegMax), m.H)));
    d = __fmaf_rn(m.g, om, -t3);
  } else {
    d = __fmul_rn(m.g, om);
  }
  return scaled ? __fmul_rn(d, rcp) : d;
}

// ---------------------------------------------------------------------------
// mbarriers and bounded waits.  Every wait polls with a time limit; one that
// runs out records a bit in the caller's watchdog word and reports failure,
// so that the kernel can stop instead of hanging.
// ---------------------------------------------------------------------------

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

// As mbar_try_wait, but a thread whose phase has not completed sleeps until it
// completes or `hint_ns` pass, instead of returning at once: a waiting warp
// then takes no issue slots from the warps doing the arithmetic.
constexpr unsigned kSuspendHintNs = 200000;

__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Warp-wide wait until the phase with parity `parity` has completed.  Every
// lane polls (so every lane gets the barrier's acquire ordering) and the warp
// leaves together.  Returns false if the wait ran out (then `code` is set in
// *watch and *abort is raised), or if another warp of the block gave up
// (*abort set); the caller then stops.
__device__ __forceinline__ bool warp_wait_watch(uint64_t* bar, unsigned parity, volatile int* abort,
                                                unsigned code, unsigned int* watch) {
  long long start = 0;
  for (unsigned spin = 0;; ++spin) {
    const bool done = mbar_try_wait_sleep(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    if ((spin & 15u) == 15u) {
      int stop = 0;
      if ((threadIdx.x % kLanes) == 0) {
        const long long now = global_ns();
        if (start == 0) {
          start = now;
        } else if (*abort) {
          stop = 1;
        } else if (now - start > kWaitLimitNs) {
          atomicOr(watch, code);
          *abort = 1;
          stop = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
  }
}

// The same wait for one thread.  With check_abort false the wait ignores
// *abort (a thread waiting for its own asynchronous operations to finish
// before the block exits) but is still bounded.
__device__ __forceinline__ bool thread_wait_watch(uint64_t* bar, unsigned parity, volatile int* abort,
                                                  unsigned code, unsigned int* watch, bool check_abort) {
  long long start = 0;
  for (unsigned spin = 0;; ++spin) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if ((spin & 15u) == 15u) {
      const long long now = global_ns();
      if (start == 0) {
        start = now;
      } else if (check_abort && *abort) {
        return false;
      } else if (now - start > kWaitLimitNs) {
        atomicOr(watch, code);
        *abort = 1;
        return false;
      }
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

}  // namespace
