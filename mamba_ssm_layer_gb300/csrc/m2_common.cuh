// m2_common.cuh -- device helpers shared by the library's kernels: bf16 and
// E4M3 conversions, mbarrier / bulk-copy PTX wrappers with bounded waits,
// warp reductions, and the device status word.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "m2_kernels.h"

namespace m2 {

// ------------------------------------------------------------------ status

// Default limit of a bounded wait, in SM clock cycles (about 2 s): a correct
// pipeline completes its waits in microseconds.
constexpr long long kWaitCycles = 4000000000LL;

// First in-kernel failure (M2_ERR_TIMEOUT) recorded on this device, and the
// limit of the pipeline waits (m2_set_wait_limit).  Each translation unit has
// its own copies (no relocatable device code is needed); each defines host
// accessors (status_<unit>, wait_limit_<unit>) built on tu_status and
// tu_set_wait_limit below.
namespace {
__device__ int g_status = 0;
__device__ long long g_wait_limit = kWaitCycles;
}

__device__ __forceinline__ void record_timeout() { atomicCAS(&g_status, 0, -8); }

// Host side: this unit's status word (clear != 0 resets it) and wait limit.
static inline int tu_status(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return -4;
  if (clear) {
    const int z = 0;
    cudaMemcpyToSymbol(g_status, &z, sizeof(int));
  }
  return v;
}
static inline cudaError_t tu_set_wait_limit(long long cycles) {
  return cudaMemcpyToSymbol(g_wait_limit, &cycles, sizeof(cycles));
}

// ------------------------------------------------------------------ bf16

__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Round to nearest even (NaN stays NaN) via the hardware conversion.
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Error-free accumulation in two fp32 words (Knuth's two-sum): hi + lo holds
// the running sum to ~2^-48 relative, independent of the summation order to
// that accuracy.  Used for the RMSNorm sums of squares (x^2 of a bf16 x is
// exact in fp32), so that r = 1/sqrt(mean + eps) matches a double evaluation.
__device__ __forceinline__ void two_sum_acc(float& hi, float& lo, float p) {
  const float s = hi + p;
  const float z = s - hi;
  lo += (hi - (s - z)) + (p - z);
  hi = s;
}
__device__ __forceinline__ void two_sum_warp(float& hi, float& lo) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ohi = __shfl_xor_sync(0xffffffffu, hi, o);
    const float olo = __shfl_xor_sync(0xffffffffu, lo, o);
    two_sum_acc(hi, lo, ohi);
    lo += olo;
  }
}

// r = 1/sqrt(S/K + eps) of an RMSNorm row as an unevaluated pair hi + lo
// (relative error about 2^-43), from its sum of squares S = h + l, in fp32
// arithmetic only: 1/K and S/K carry their (fma-computed) errors, and one Newton
// step with an fma-exact residual refines rsqrtf.  Every thread of a row
// computes the same pair.
struct NormR {
  float hi, lo;
};
__device__ __forceinline__ NormR norm_r(float h, float l, int K, float eps) {
  const float kf = (float)K;
  const float ik = __frcp_rn(kf);
  const float ik_lo = fmaf(-ik, kf, 1.0f) * ik;  // 1/K - ik, to ~2^-24 of itself
  const float m = h * ik;                                   // S/K = m + me
  const float me = fmaf(h, ik_lo, fmaf(l, ik, fmaf(h, ik, -m)));
  const float v = m + eps;                                  // S/K + eps = v + ve
  const float z = v - m;
  const float ve = ((m - (v - z)) + (eps - z)) + me;
  const float r0 = rsqrtf(v);
  const float q = r0 * r0;                                  // r0^2 = q + qe
  const float qe = fmaf(r0, r0, -q);
  float d = fmaf(-v, q, 1.0f);                              // 1 - (v + ve) * r0^2
  d = fmaf(-v, qe, d);
  d = fmaf(-ve, q, d);
  NormR r;
  r.hi = r0;
  r.lo = 0.5f * r0 * d;
  return r;
}
// bf16(x * w * r), correctly rounded: x * w is exact in fp32 (both are bf16
// values), its product with the pair r is carried as s + t, and t decides the
// rounding where s lies exactly halfway between two bf16 values.  The result
// equals the rounding of the exact product unless that lies within about
// 2^-43 (relative) of a rounding boundary, and it does not depend on the
// order in which the sum of squares was accumulated.
__device__ __forceinline__ uint16_t norm_round_bf16(float x, float w, const NormR& r) {
  const float xw = x * w;
  const float p = xw * r.hi;
  const float e = fmaf(xw, r.lo, fmaf(xw, r.hi, -p));
  const float s = p + e;  // |e| << |p|: s + t = p + e exactly
  const float t = e - (s - p);
  const uint32_t b = __float_as_uint(s);
  const uint16_t rn = f32_to_bf16(s);
  const uint16_t dir = (uint16_t)((b >> 16) + ((t > 0.0f) == (s > 0.0f) ? 1u : 0u));  // away from zero iff |s + t| > |s|
  return ((b & 0xFFFFu) == 0x8000u && t != 0.0f) ? dir : rn;
}

// ------------------------------------------------------------------ E4M3

// Two E4M3 bytes -> two fp32, exactly: the hardware E4M3 -> f16 conversion is
// exact (every E4M3 value is an f16 normal), and f16 -> f32 is exact.
__device__ __forceinline__ void e4m3x2_to_f32(uint16_t v, float& lo, float& hi) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h2));
}

// ------------------------------------------------------------------ math

__device__ __forceinline__ float silu_f(float v) { return v / (1.0f + expf(-v)); }
__device__ __forceinline__ float softplus_f(float v) { return v > 20.0f ? v : log1pf(expf(v)); }

// Per-head scalars of the SSM step from the raw dt projection output:
// dt = clamp(softplus(dt_raw + dt_bias), 1e-9, 1e9), dA = exp(dt * A), A = -exp(A_log).
__device__ __forceinline__ void ssm_dt_dA(float dt_raw, float dt_bias, float A_log, float& dt, float& dA) {
  float d = softplus_f(dt_raw + dt_bias);
  d = fminf(fmaxf(d, 1e-9f), 1e9f);
  dt = d;
  dA = expf(d * -expf(A_log));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Potentially blocking test: the thread may be suspended until the phase
// completes, for at most about `hint_ns` nanoseconds.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
// Polls until the phase with the given parity completes or `limit` SM clocks
// pass; on a timeout records M2_ERR_TIMEOUT and returns false.  Polls suspend
// the thread (try_wait, at most about 1 us each; the hardware may hold it
// longer while the phase is pending), except under a limit below 1e6 clocks,
// where they only test, so that the clock is read often enough to end the wait
// in time.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, long long limit) {
  const long long t0 = clock64();
  const bool suspend = limit >= 1000000;
  for (;;) {
    if (suspend ? mbar_try_wait(bar, parity, 1000u) : mbar_test_wait(bar, parity)) return true;
    if (clock64() - t0 > limit) break;
  }
  record_timeout();
  return false;
}
// Bounded wait of the pipeline (a stage filled, a slot freed, a k block
// done): gives up after this device's wait limit (default kWaitCycles).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_test_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, *reinterpret_cast<volatile long long*>(&g_wait_limit));
}
// Wait for this thread's own asynchronous work (copies or MMAs it issued)
// before the CTA exits or frees what that work writes.  Such work always
// completes, so the limit is the fixed default, never the (possibly lowered)
// pipeline limit: a CTA that gave up on its pipeline still leaves nothing in
// flight behind it.
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity) {
  if (mbar_test_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, kWaitCycles);
}

// ------------------------------------------------------------------ bulk copy

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes).
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Programmatic dependent launch: wait until the previous grid in the stream
// has completed and its writes are visible / let the next grid start early.
// Both are no-ops for a kernel launched without the PDL attribute.  A kernel
// launched this way may already run while its predecessor writes, so data the
// predecessor produces must be read with ordinary (coherent) loads after
// pdl_wait(), never through the non-coherent read-only path (__ldg /
// ld.global.nc), which requires the data to stay unchanged for the whole
// lifetime of the reading kernel.  Every kernel here triggers its successor
// only after its own wait has returned, so at most two consecutive kernels of
// a chain run at once and a kernel's pre-wait reads can only race with its
// immediate predecessor.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Named barrier among `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace m2
