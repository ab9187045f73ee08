// k_mixer.cu -- the non-GEMM steps of the Mamba-2 mixer: conv1d update
// (decode and prefill), the SSM decode step, the sequential prefill scan, and
// the gated RMSNorm.  All are memory- or latency-bound elementwise/reduction
// kernels; the layouts keep every global access coalesced.
//
// Formulas (source listing "spark_model/layers/nemotron_mamba2.rs", module
// header steps 3-6, and its `conv1d_update_biased` / `ssm_decode` launchers):
//   conv:  u = silu(b + sum_j w[j] * window[j]), window = the d_conv-1
//          previous xBC tokens (oldest first) then the current one
//   SSM:   dt = clamp(softplus(dt_raw + dt_bias), 1e-9, 1e9), dA = exp(-dt*exp(A_log))
//          h = dA*h + dt*x*B;  y = C.h + D*x           (head h uses group h/(H/G))
//   gate:  g = rms_norm(y) * w * silu(z)
#include <cuda_runtime.h>
#include <stdint.h>

#include "m2_common.cuh"
#include "m2_kernels.h"

namespace m2 {

// ------------------------------------------------------------------ conv

__global__ void __launch_bounds__(256) conv_update_kernel(uint16_t* __restrict__ ring,
                                                          const int32_t* __restrict__ pos,
                                                          const uint16_t* __restrict__ x, int ldx,
                                                          const uint16_t* __restrict__ w,
                                                          const uint16_t* __restrict__ bias,
                                                          uint16_t* __restrict__ out, int ldo, int C, int dconv,
                                                          int silu) {
  const int c = blockIdx.x * 256 + threadIdx.x;
  const int b = blockIdx.y;
  if (c >= C) return;
  const int L = dconv - 1;
  const int p = pos[b];
  uint16_t* rg = ring + (size_t)b * L * C;
  const uint16_t xv = x[(size_t)b * ldx + c];
  float s = bias ? bf16_to_f32(bias[c]) : 0.0f;
  for (int j = 0; j < L; ++j) s += bf16_to_f32(w[(size_t)c * dconv + j]) * bf16_to_f32(rg[(size_t)((p + j) % L) * C + c]);
  s += bf16_to_f32(w[(size_t)c * dconv + L]) * bf16_to_f32(xv);
  out[(size_t)b * ldo + c] = f32_to_bf16(silu ? silu_f(s) : s);
  rg[(size_t)(p % L) * C + c] = xv;
}

__global__ void conv_pos_kernel(int32_t* pos, int B, int add) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) pos[b] += add;
}

cudaError_t launch_conv_update(uint16_t* ring, const int32_t* pos, const uint16_t* x, int32_t ldx,
                               const uint16_t* w, const uint16_t* b, uint16_t* out, int32_t ldo, int32_t B,
                               int32_t C, int32_t dconv, int32_t silu, cudaStream_t s) {
  trace_pre(K_CONV_UPDATE, s);
  conv_update_kernel<<<dim3((C + 255) / 256, B), 256, 0, s>>>(ring, pos, x, ldx, w, b, out, ldo, C, dconv, silu);
  trace_post(K_CONV_UPDATE, s);
  return cudaGetLastError();
}

cudaError_t launch_conv_pos(int32_t* pos, int32_t B, int32_t add, cudaStream_t s) {
  trace_pre(K_CONV_POS, s);
  conv_pos_kernel<<<(B + 127) / 128, 128, 0, s>>>(pos, B, add);
  trace_post(K_CONV_POS, s);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ staging copy

// Stream-ordered copy by a kernel (device memory and/or pinned host memory
// reached through its unified address).  Launched as a programmatic dependent:
// it waits for the previous kernel (which may still read dst or write src)
// before touching either, and lets the next kernel start its own prologue.
__global__ void __launch_bounds__(256) copy16_kernel(const uint4* src, uint4* dst, size_t n16) {
  pdl_wait();
  pdl_trigger();
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

cudaError_t launch_copy16(const void* src, void* dst, size_t n16, cudaStream_t s) {
  size_t blocks = (n16 + 255) / 256;
  if (blocks > (size_t)num_sms()) blocks = (size_t)num_sms();
  if (blocks < 1) blocks = 1;
  trace_pre(K_COPY, s);
  const cudaError_t e = launch_k(copy16_kernel, dim3((unsigned)blocks), dim3(256), 0, s, true,
                                 static_cast<const uint4*>(src), static_cast<uint4*>(dst), n16);
  trace_post(K_COPY, s);
  return e;
}

// Sequence of token row t in a varlen batch: the i with cu[i] <= t < cu[i+1]
// (sequences of length 0 are skipped by taking the last such i).
__device__ __forceinline__ int seq_of(const int32_t* cu, int n, int t) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Prefill conv over a varlen batch of sequences (token rows cu[i] .. cu[i+1]-1
// belong to sequence i, whose ring and position are ring[i], pos[i]).  A thread
// owns two adjacent channels and 8 consecutive token rows; the taps before a
// sequence's first token come from its ring.  The ring is not written here
// (other CTAs may still read it): conv_ring_store runs afterwards.
__global__ void __launch_bounds__(256) conv_prefill_kernel(const uint16_t* __restrict__ ring,
                                                           const int32_t* __restrict__ pos,
                                                           const uint16_t* __restrict__ xbc, int ldx,
                                                           const uint16_t* __restrict__ w,
                                                           const uint16_t* __restrict__ bias,
                                                           uint16_t* __restrict__ u, int ldu, int T, int C,
                                                           int dconv, const int32_t* __restrict__ cu, int nseq) {
  const int c = (blockIdx.x * 32 + (threadIdx.x & 31)) * 2;
  const int tb = (blockIdx.y * 8 + (threadIdx.x >> 5)) * 8;
  const int L = dconv - 1;
  if (c >= C || tb >= T) return;
  float w0[8], w1[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    w0[j] = j < dconv ? bf16_to_f32(w[(size_t)c * dconv + j]) : 0.0f;
    w1[j] = j < dconv ? bf16_to_f32(w[(size_t)(c + 1) * dconv + j]) : 0.0f;
  }
  const float b0 = bias ? bf16_to_f32(bias[c]) : 0.0f, b1 = bias ? bf16_to_f32(bias[c + 1]) : 0.0f;
  if (tb + 7 < T && dconv == 4) {
    const int i = seq_of(cu, nseq, tb);
    if (cu[i] <= tb - 3 && tb + 7 < cu[i + 1]) {
      // common case: the 8 tokens and their 3 predecessors are rows of one
      // sequence: the 11-row window is loaded once
      uint32_t win[11];
#pragma unroll
      for (int r = 0; r < 11; ++r) win[r] = *reinterpret_cast<const uint32_t*>(xbc + (size_t)(tb - 3 + r) * ldx + c);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float s0 = b0, s1 = b1;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          s0 = fmaf(w0[j], bf16lo(win[k + j]), s0);
          s1 = fmaf(w1[j], bf16hi(win[k + j]), s1);
        }
        *reinterpret_cast<uint32_t*>(u + (size_t)(tb + k) * ldu + c) = pack_bf16x2(silu_f(s0), silu_f(s1));
      }
      return;
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int t = tb + k;
    if (t < T) {
      const int i = seq_of(cu, nseq, t);
      const int start = cu[i];
      float s0 = b0, s1 = b1;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j <= L) {
          const int src = t - L + j;  // j == L: the current token
          uint32_t v;
          if (src >= start) {
            v = *reinterpret_cast<const uint32_t*>(xbc + (size_t)src * ldx + c);
          } else {  // history: the (start - src)-th token before the block, from the ring
            const int slot = (((pos[i] + (src - start)) % L) + L) % L;
            v = *reinterpret_cast<const uint32_t*>(ring + ((size_t)i * L + slot) * C + c);
          }
          s0 = fmaf(w0[j], bf16lo(v), s0);
          s1 = fmaf(w1[j], bf16hi(v), s1);
        }
      }
      *reinterpret_cast<uint32_t*>(u + (size_t)t * ldu + c) = pack_bf16x2(silu_f(s0), silu_f(s1));
    }
  }
}

// After the conv: each sequence's ring takes its last min(L, T_i) tokens, token
// k of the block (0-based) into slot (pos[i] + k) mod L.  pos is not advanced.
__global__ void __launch_bounds__(256) conv_ring_store_kernel(uint16_t* __restrict__ ring,
                                                              const int32_t* __restrict__ pos,
                                                              const uint16_t* __restrict__ xbc, int ldx, int C,
                                                              int dconv, const int32_t* __restrict__ cu) {
  const int i = blockIdx.y;
  const int L = dconv - 1;
  const int start = cu[i], len = cu[i + 1] - cu[i];
  const int first = len > L ? len - L : 0;
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < (len - first) * C; idx += gridDim.x * blockDim.x) {
    const int k = first + idx / C, c = idx % C;
    ring[((size_t)i * L + (pos[i] + k) % L) * C + c] = xbc[(size_t)(start + k) * ldx + c];
  }
}

cudaError_t launch_conv_prefill(uint16_t* ring, const int32_t* pos, const uint16_t* xbc, int32_t ldx,
                                const uint16_t* w, const uint16_t* b, uint16_t* u, int32_t ldu, int32_t T,
                                int32_t C, int32_t dconv, const int32_t* cu, int32_t nseq, cudaStream_t s) {
  trace_pre(K_CONV_PREFILL, s);
  const dim3 grid((C / 2 + 31) / 32, (T + 63) / 64);
  conv_prefill_kernel<<<grid, 256, 0, s>>>(ring, pos, xbc, ldx, w, b, u, ldu, T, C, dconv, cu, nseq);
  trace_post(K_CONV_PREFILL, s);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) {
    trace_pre(K_CONV_RING, s);
    conv_ring_store_kernel<<<dim3((C * (dconv - 1) + 255) / 256, nseq), 256, 0, s>>>(ring, pos, xbc, ldx, C, dconv,
                                                                                  cu);
    trace_post(K_CONV_RING, s);
    e = cudaGetLastError();
  }
  return e;
}

// ------------------------------------------------------------------ SSM step

// Thread layout shared by the SSM kernels: a row p of the state (N fp32) is
// covered by LPR = N/4 lanes holding 4 consecutive n each (one float4), so a
// warp covers 32/LPR rows and the 8 warps 8*32/LPR rows per pass.
__device__ __forceinline__ float4 ld4bf(const uint16_t* p) {
  const uint2 v = *reinterpret_cast<const uint2*>(p);
  return make_float4(bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y));
}

__device__ __forceinline__ void head_scalars(const uint16_t* dt_row, const float* dt_bias, const float* A_log, int h,
                                             float& dt, float& dA) {
  ssm_dt_dA(bf16_to_f32(dt_row[h]), dt_bias[h], A_log[h], dt, dA);
}

template <int LPR, int ROWS>
__global__ void __launch_bounds__(256) ssm_step_kernel(const SsmArgs a, int psplit) {
  // A CTA covers 8 * RPW * ROWS consecutive rows p of one head; each thread
  // ROWS rows, whose state loads are all issued before any is used.
  constexpr int RPW = 32 / LPR;
  constexpr int CTA_ROWS = 8 * RPW * ROWS;
  const int b = blockIdx.y;
  const int h = blockIdx.x / psplit;
  const int pc = blockIdx.x % psplit;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n4 = (lane % LPR) * 4;
  const int g = h / (a.H / a.G);
  float* hb = a.h + ((size_t)b * a.H + h) * a.P * a.N;
  const int p0 = pc * CTA_ROWS + warp * RPW + lane / LPR;
  if (a.l2_prefetch_bytes && threadIdx.x == 0) {
    // this CTA's share of the L2 prefetch range, in 16-byte units
    const size_t units = a.l2_prefetch_bytes / 16, nct = (size_t)gridDim.x * gridDim.y;
    const size_t cta = (size_t)blockIdx.y * gridDim.x + blockIdx.x;
    const size_t u0 = units * cta / nct, u1 = units * (cta + 1) / nct;
    const char* base = static_cast<const char*>(a.l2_prefetch);
    for (size_t u = u0; u < u1; u += 4096) {  // at most 64 KB per request
      const size_t n = (u1 - u < 4096 ? u1 - u : 4096) * 16;
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base + u * 16), "r"((uint32_t)n) : "memory");
    }
  }
  float4 hv[ROWS];
  // The state is written only by the SSM kernels of earlier steps, which have
  // completed by now (every kernel of the chain lets its successor launch only
  // after its own wait), so it can be fetched before waiting on the in_proj.
#pragma unroll
  for (int i = 0; i < ROWS; ++i) {
    const int p = p0 + i * 8 * RPW;
    if (p < a.P) hv[i] = *reinterpret_cast<const float4*>(hb + (size_t)p * a.N + n4);
  }
  pdl_wait();  // x, B, C, dt come from the previous kernel
  pdl_trigger();
  const uint16_t* xr = a.x + (size_t)b * a.ld_in;
  float dt, dA;
  head_scalars(a.dt + (size_t)b * a.ld_in, a.dt_bias, a.A_log, h, dt, dA);
  const float Dh = a.D[h];
  const float4 Bv = ld4bf(a.Bm + (size_t)b * a.ld_in + (size_t)g * a.N + n4);
  const float4 Cv = ld4bf(a.Cm + (size_t)b * a.ld_in + (size_t)g * a.N + n4);
  float xv[ROWS];
#pragma unroll
  for (int i = 0; i < ROWS; ++i) {
    const int p = p0 + i * 8 * RPW;
    xv[i] = p < a.P ? bf16_to_f32(xr[(size_t)h * a.P + p]) : 0.0f;
  }
#pragma unroll
  for (int i = 0; i < ROWS; ++i) {
    const int p = p0 + i * 8 * RPW;
    const bool live = p < a.P;  // uniform across the lanes of one row
    if (live) {
      const float dtx = dt * xv[i];
      hv[i].x = fmaf(dA, hv[i].x, dtx * Bv.x);
      hv[i].y = fmaf(dA, hv[i].y, dtx * Bv.y);
      hv[i].z = fmaf(dA, hv[i].z, dtx * Bv.z);
      hv[i].w = fmaf(dA, hv[i].w, dtx * Bv.w);
      *reinterpret_cast<float4*>(hb + (size_t)p * a.N + n4) = hv[i];
    }
    float yp = live ? Cv.x * hv[i].x + Cv.y * hv[i].y + Cv.z * hv[i].z + Cv.w * hv[i].w : 0.0f;
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) yp += __shfl_xor_sync(0xffffffffu, yp, o);
    if (live && (lane % LPR) == 0) a.y[(size_t)b * a.ldy + (size_t)h * a.P + p] = yp + Dh * xv[i];
  }
  if (a.pos_inc && blockIdx.x == 0 && threadIdx.x == 0) a.pos_inc[b] += 1;
}

template <int LPR>
static cudaError_t launch_ssm_lpr(const SsmArgs& a, cudaStream_t s, bool pdl) {
  // rows per thread: doubled from 1 (up to 8, or one CTA per head) while the
  // grid has more CTAs than the GPU has SMs
  constexpr int RPW = 32 / LPR;
  const long long heads = (long long)a.B * a.H;
  const int max_rows = (a.P + 8 * RPW - 1) / (8 * RPW);  // rows per thread with one CTA per head
  // A batch-1 step then leaves each SM room for the next kernel's CTA, which
  // launches early (programmatic dependent launch) and starts streaming its
  // weights while this one runs.
  int rows = 1;
  while (rows < 8 && rows < max_rows && heads * ((a.P + 8 * RPW * rows - 1) / (8 * RPW * rows)) > num_sms()) rows *= 2;
  const int cta_rows = 8 * RPW * rows;
  const int psplit = (a.P + cta_rows - 1) / cta_rows;
  dim3 grid(a.H * psplit, a.B);
  switch (rows) {
    case 1: return launch_k(ssm_step_kernel<LPR, 1>, grid, dim3(256), 0, s, pdl, a, psplit);
    case 2: return launch_k(ssm_step_kernel<LPR, 2>, grid, dim3(256), 0, s, pdl, a, psplit);
    case 4: return launch_k(ssm_step_kernel<LPR, 4>, grid, dim3(256), 0, s, pdl, a, psplit);
    default: return launch_k(ssm_step_kernel<LPR, 8>, grid, dim3(256), 0, s, pdl, a, psplit);
  }
}

cudaError_t launch_ssm_step(const SsmArgs& a, cudaStream_t s) {
  const bool pdl = a.pdl != 0;
  cudaError_t e;
  trace_pre(K_SSM_STEP, s);
  switch (a.N / 4) {
    case 4: e = launch_ssm_lpr<4>(a, s, pdl); break;
    case 8: e = launch_ssm_lpr<8>(a, s, pdl); break;
    case 16: e = launch_ssm_lpr<16>(a, s, pdl); break;
    default: e = launch_ssm_lpr<32>(a, s, pdl); break;
  }
  trace_post(K_SSM_STEP, s);
  return e;
}

// ------------------------------------------------------------------ sequential scan

// T steps of the recurrence for one sequence; the CTA's slice of the state
// (one row per thread group) lives in registers for the whole block of tokens.
// Inputs of step t+1 are fetched while step t is computed.
template <int LPR>
__global__ void __launch_bounds__(256) ssm_scan_seq_kernel(const ScanArgs a, int psplit) {
  constexpr int RPW = 32 / LPR;
  constexpr int ROWS = 8 * RPW;  // rows per CTA
  const int h = blockIdx.x / psplit;
  const int pc = blockIdx.x % psplit;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n4 = (lane % LPR) * 4;
  const int g = h / (a.H / a.G);
  const int p = pc * ROWS + warp * RPW + lane / LPR;
  const bool active = p < a.P;
  const int pp = active ? p : 0;
  const float Dh = a.D[h];
  const float Ah = -expf(a.A_log[h]);
  const float dtb = a.dt_bias[h];
  float4* hp = reinterpret_cast<float4*>(a.h + ((size_t)h * a.P + pp) * a.N + n4);
  float4 hv = active ? *hp : make_float4(0.f, 0.f, 0.f, 0.f);

  const size_t xoff = (size_t)h * a.P + pp;
  const size_t boff = (size_t)g * a.N + n4;
  // prefetch step 0
  float x_n = bf16_to_f32(a.x[xoff]);
  float dr_n = bf16_to_f32(a.dt[h]);
  float4 B_n = ld4bf(a.Bm + boff), C_n = ld4bf(a.Cm + boff);
  for (int t = 0; t < a.T; ++t) {
    const float xv = x_n, dr = dr_n;
    const float4 Bv = B_n, Cv = C_n;
    if (t + 1 < a.T) {
      x_n = bf16_to_f32(a.x[(size_t)(t + 1) * a.ld_in + xoff]);
      dr_n = bf16_to_f32(a.dt[(size_t)(t + 1) * a.ld_dt + h]);
      B_n = ld4bf(a.Bm + (size_t)(t + 1) * a.ld_in + boff);
      C_n = ld4bf(a.Cm + (size_t)(t + 1) * a.ld_in + boff);
    }
    float dt = softplus_f(dr + dtb);
    dt = fminf(fmaxf(dt, 1e-9f), 1e9f);
    const float dA = expf(dt * Ah);
    const float dtx = dt * xv;
    hv.x = fmaf(dA, hv.x, dtx * Bv.x);
    hv.y = fmaf(dA, hv.y, dtx * Bv.y);
    hv.z = fmaf(dA, hv.z, dtx * Bv.z);
    hv.w = fmaf(dA, hv.w, dtx * Bv.w);
    float yp = Cv.x * hv.x + Cv.y * hv.y + Cv.z * hv.z + Cv.w * hv.w;
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) yp += __shfl_xor_sync(0xffffffffu, yp, o);
    if (active && (lane % LPR) == 0) a.y[(size_t)t * a.ldy + xoff] = yp + Dh * xv;
  }
  if (active) *hp = hv;
  if (a.pos_inc && blockIdx.x == 0 && threadIdx.x == 0) a.pos_inc[0] += a.T;
}

cudaError_t launch_ssm_scan_seq(const ScanArgs& a, cudaStream_t s) {
  const int lpr = a.N / 4;
  const int rows = 8 * (32 / lpr);
  const int psplit = (a.P + rows - 1) / rows;
  trace_pre(K_SSM_SCAN_SEQ, s);
  switch (lpr) {
    case 4: ssm_scan_seq_kernel<4><<<a.H * psplit, 256, 0, s>>>(a, psplit); break;
    case 8: ssm_scan_seq_kernel<8><<<a.H * psplit, 256, 0, s>>>(a, psplit); break;
    case 16: ssm_scan_seq_kernel<16><<<a.H * psplit, 256, 0, s>>>(a, psplit); break;
    default: ssm_scan_seq_kernel<32><<<a.H * psplit, 256, 0, s>>>(a, psplit); break;
  }
  trace_post(K_SSM_SCAN_SEQ, s);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ activation prep

// The norm that produces a GEMV's or GEMM's activation rows:
//   PREP_RMSNORM  x * r * w,            r = 1/sqrt(mean(x^2) + eps)   (source
//                 listing "nemotron_mamba2.rs", module header step 1: weight*x)
//   PREP_GATED    y * r * w * silu(z),  r over groups of `group`      (step 6:
//                 rms_norm(y, ssm_norm) * silu(z))
// rounded to bf16 (the layer's rounding point), then stored as bf16 or, for an
// E4M3-weight GEMV, as f16 after the exact row prescale 2^j (max |v| * 2^j in
// [2^14, 2^15); unscale = 2^-j).  The RMSNorm sum of squares is an error-free
// fp32 pair and r an fp32 pair, so its outputs are the correct roundings of
// the exact products whatever the summation order (norm_round_bf16).
constexpr int kPrepMaxPer = 32;  // elements per thread: K <= 32 * threads

// Bytes of one row's staged inputs: per chunk of 8 elements and thread, the
// fp32 y (32 B) and bf16 z (16 B) of the gated norm, or the bf16 x (16 B).
__host__ __device__ constexpr int prep_stage_bytes(int threads, bool gated) {
  return threads * (kPrepMaxPer / 8) * (gated ? 48 : 16);
}

// silu of the gated norm.  Its bf16 output is a rounding point whose
// decisions are held to 2^-12 of the exact value, so the hardware exp2 and
// divide approximations (relative errors of a few 2^-23) serve; for z below
// about -87 the gate is 0 (the exact value is below 1e-36).
__device__ __forceinline__ float silu_gate(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Persistent CTAs of kPrepThreads threads (128 for K <= 4096, 256 for K <=
// 8192, 512 above, and 512 whenever the rows are no more than the SMs) walk
// rows m = blockIdx.x, + gridDim.x, ...  While a row is
// computed, the next row's inputs are copied into the other of two shared
// stages (cp.async); each thread copies exactly the 16-byte pieces it later
// reads, so the hand-over needs no barrier.  The norm weight is read once per
// CTA.
template <int kPrepThreads>
__device__ __forceinline__ void prep_fetch_row(const PrepArgs& a, int m, uint8_t* st, int tid) {
  const bool gated = a.mode == PREP_GATED;
#pragma unroll
  for (int c = 0; c < kPrepMaxPer / 8; ++c) {
    const int k0 = (tid + kPrepThreads * c) * 8;
    const int u = c * kPrepThreads + tid;  // this thread's piece of chunk c
    if (k0 < a.K) {
      if (gated) {
        cp_async16(st + u * 32, a.y + (size_t)m * a.ldy + k0);
        cp_async16(st + u * 32 + 16, a.y + (size_t)m * a.ldy + k0 + 4);
        cp_async16(st + kPrepThreads * (kPrepMaxPer / 8) * 32 + u * 16, a.z + (size_t)m * a.ldz + k0);
      } else {
        cp_async16(st + u * 16, a.x + (size_t)m * a.ldx + k0);
      }
    }
  }
}

template <int kPrepThreads>
__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const PrepArgs a) {
  constexpr int kW = kPrepThreads / 32;  // warps
  extern __shared__ __align__(16) uint8_t prep_stage[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ float s_hi[kW], s_lo[kW], s_max[kW];
  __shared__ float part[kPrepThreads * kPrepMaxPer / 8];  // gated mode: per-run sums of squares
  const int K = a.K;
  const bool gated = a.mode == PREP_GATED;
  const int sbytes = prep_stage_bytes(kPrepThreads, gated);
  uint4 wv[kPrepMaxPer / 8];  // the norm weight: not an output of the previous kernel
#pragma unroll
  for (int c = 0; c < kPrepMaxPer / 8; ++c) {
    const int k0 = (tid + kPrepThreads * c) * 8;
    wv[c] = (k0 < K && a.mode != PREP_QUANT) ? *reinterpret_cast<const uint4*>(a.w + k0) : make_uint4(0u, 0u, 0u, 0u);
  }
  pdl_wait();
  pdl_trigger();
  if ((int)blockIdx.x < a.M) prep_fetch_row<kPrepThreads>(a, blockIdx.x, prep_stage, tid);
  cp_async_commit();
  int it = 0;
  for (int m = blockIdx.x; m < a.M; m += gridDim.x, ++it) {
    uint8_t* cur = prep_stage + (it & 1) * sbytes;
    if (m + (int)gridDim.x < a.M) prep_fetch_row<kPrepThreads>(a, m + gridDim.x, prep_stage + ((it + 1) & 1) * sbytes, tid);
    cp_async_commit();
    cp_async_wait1();  // this thread's pieces of row m have landed
    float v[kPrepMaxPer];
    uint4 zv[kPrepMaxPer / 8];
    // element e of this thread: k = (tid + kPrepThreads * (e / 8)) * 8 + e % 8
#pragma unroll
    for (int c = 0; c < kPrepMaxPer / 8; ++c) {
      const int k0 = (tid + kPrepThreads * c) * 8;
      const int u = c * kPrepThreads + tid;
      zv[c] = make_uint4(0u, 0u, 0u, 0u);
      if (k0 < K) {
        if (!gated) {
          const uint4 x4 = *reinterpret_cast<const uint4*>(cur + u * 16);
          const uint32_t w4[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            v[c * 8 + 2 * e] = bf16lo(w4[e]);
            v[c * 8 + 2 * e + 1] = bf16hi(w4[e]);
          }
        } else {
          const float4 f0 = *reinterpret_cast<const float4*>(cur + u * 32);
          const float4 f1 = *reinterpret_cast<const float4*>(cur + u * 32 + 16);
          zv[c] = *reinterpret_cast<const uint4*>(cur + kPrepThreads * (kPrepMaxPer / 8) * 32 + u * 16);
          v[c * 8 + 0] = f0.x; v[c * 8 + 1] = f0.y; v[c * 8 + 2] = f0.z; v[c * 8 + 3] = f0.w;
          v[c * 8 + 4] = f1.x; v[c * 8 + 5] = f1.y; v[c * 8 + 6] = f1.z; v[c * 8 + 7] = f1.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[c * 8 + e] = 0.0f;
      }
    }
    if (a.mode == PREP_QUANT) {
      // rows as they are
    } else if (a.mode == PREP_RMSNORM) {
      // one error-free pair per 8-element chunk (independent chains), then
      // the chunks' pairs in order: the pair holds the sum to about 2^-48
      // whatever the order
      float hs[kPrepMaxPer / 8], ls[kPrepMaxPer / 8];
#pragma unroll
      for (int c = 0; c < kPrepMaxPer / 8; ++c) {
        hs[c] = ls[c] = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) two_sum_acc(hs[c], ls[c], v[c * 8 + e] * v[c * 8 + e]);
      }
      float hi = hs[0], lo = ls[0];
#pragma unroll
      for (int c = 1; c < kPrepMaxPer / 8; ++c) {
        two_sum_acc(hi, lo, hs[c]);
        lo += ls[c];
      }
      two_sum_warp(hi, lo);
      if (lane == 0) {
        s_hi[warp] = hi;
        s_lo[warp] = lo;
      }
      __syncthreads();
      if (tid == 0) {
        // combine the warps' pairs in a fixed order
        float h = 0.0f, l = 0.0f;
        for (int w = 0; w < kW; ++w) {
          two_sum_acc(h, l, s_hi[w]);
          l += s_lo[w];
        }
        s_hi[0] = h;
        s_lo[0] = l;
      }
      __syncthreads();
      const NormR nr = norm_r(s_hi[0], s_lo[0], K, a.eps);
#pragma unroll
      for (int c = 0; c < kPrepMaxPer / 8; ++c) {
        const int k0 = (tid + kPrepThreads * c) * 8;
        if (k0 < K) {
          const uint4 u = wv[c];
          const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            v[c * 8 + 2 * e] = bf16_to_f32(norm_round_bf16(v[c * 8 + 2 * e], bf16lo(w4[e]), nr));
            v[c * 8 + 2 * e + 1] = bf16_to_f32(norm_round_bf16(v[c * 8 + 2 * e + 1], bf16hi(w4[e]), nr));
          }
        }
      }
    } else {
      // sum of squares per group in a fixed order (results do not depend on
      // scheduling, so equal rows give equal outputs): each run of 8 elements
      // in sequence, then either warp butterflies and the warps' chunks of 256
      // in index order (group % 256 == 0), or a pairwise tree over the runs of
      // each group
      const int nrun = K / 8;  // runs of 8 in the row; a run never straddles a group (group % 16 == 0)
      float ssr[kPrepMaxPer / 8];
#pragma unroll
      for (int c = 0; c < kPrepMaxPer / 8; ++c) {
        float ss = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(v[c * 8 + e], v[c * 8 + e], ss);
        ssr[c] = ss;  // zero past K
      }
      int gstride;  // part[] index of group j's sum = j * gstride
      if (a.group % 256 == 0) {
#pragma unroll
        for (int c = 0; c < kPrepMaxPer / 8; ++c) {
          const float ws = warp_sum(ssr[c]);
          if (lane == 0) part[c * kW + warp] = ws;  // chunk of 256 elements starting at (warp + kW c) * 256
        }
        __syncthreads();
        const int cpg = a.group / 256, ngroups = K / a.group;
        float gs = 0.0f;
        if (tid < ngroups)
          for (int j = 0; j < cpg; ++j) gs += part[tid * cpg + j];
        __syncthreads();
        if (tid < ngroups) part[tid] = gs;
        gstride = 1;
      } else {
        const int R = a.group / 8;
#pragma unroll
        for (int c = 0; c < kPrepMaxPer / 8; ++c) {
          const int run = tid + kPrepThreads * c;
          if (run < nrun) part[run] = ssr[c];
        }
        __syncthreads();
        for (int st = 1; st < R; st <<= 1) {
          for (int run = tid; run < nrun; run += kPrepThreads) {
            const int li = run % R;
            if ((li & (2 * st - 1)) == 0 && li + st < R) part[run] += part[run + st];
          }
          __syncthreads();
        }
        gstride = R;
      }
      __syncthreads();
#pragma unroll
      for (int c = 0; c < kPrepMaxPer / 8; ++c) {
        const int k0 = (tid + kPrepThreads * c) * 8;
        if (k0 < K) {
          const float r = rsqrtf(part[(k0 / a.group) * gstride] / (float)a.group + a.eps);
          const uint4 u = wv[c];
          const uint4 zz = zv[c];
          const uint32_t w4[4] = {u.x, u.y, u.z, u.w}, z4[4] = {zz.x, zz.y, zz.z, zz.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float g0 = v[c * 8 + 2 * e] * r * bf16lo(w4[e]) * silu_gate(bf16lo(z4[e]));
            const float g1 = v[c * 8 + 2 * e + 1] * r * bf16hi(w4[e]) * silu_gate(bf16hi(z4[e]));
            v[c * 8 + 2 * e] = bf16_to_f32(f32_to_bf16(g0));
            v[c * 8 + 2 * e + 1] = bf16_to_f32(f32_to_bf16(g1));
          }
        }
      }
    }
    if (a.q8) {
      // W8A8 activations: a 128-element block is the 8-element runs of 16
      // consecutive threads (one half-warp)
#pragma unroll
      for (int c = 0; c < kPrepMaxPer / 8; ++c) {
        const int k0 = (tid + kPrepThreads * c) * 8;
        float bm = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) bm = fmaxf(bm, fabsf(v[c * 8 + e]));  // v = 0 past K
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
        if (k0 < K) {
          const float inv = bm > 0.0f ? 448.0f / bm : 0.0f;
          uint32_t q[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint16_t h;
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
                : "=h"(h)
                : "f"(v[c * 8 + 2 * e + 1] * inv), "f"(v[c * 8 + 2 * e] * inv));
            q[e] = h;
          }
          *reinterpret_cast<uint2*>(a.q8 + (size_t)m * a.ldq + k0) = make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
          if ((tid & 15) == 0) a.sq[(size_t)(k0 >> 7) * a.ldsq + m] = bm / 448.0f;
        }
      }
    }
    if (a.out) {
    float up = 1.0f;
    if (a.f16) {
      float mx = 0.0f;
#pragma unroll
      for (int e = 0; e < kPrepMaxPer; ++e) mx = fmaxf(mx, fabsf(v[e]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if (lane == 0) s_max[warp] = mx;
      __syncthreads();
      mx = 0.0f;
#pragma unroll
      for (int w = 0; w < kW; ++w) mx = fmaxf(mx, s_max[w]);
      const unsigned bits = __float_as_uint(mx);
      const int ex = bits ? (int)((bits >> 23) & 0xFF) - 127 : 14;
      const int jx = max(-120, min(120, 14 - ex));
      up = ldexpf(1.0f, jx);
      if (tid == 0) a.unscale[m] = ldexpf(1.0f, -jx);
    } else if (a.unscale && tid == 0) {
      a.unscale[m] = 1.0f;
    }
#pragma unroll
    for (int c = 0; c < kPrepMaxPer / 8; ++c) {
      const int k0 = (tid + kPrepThreads * c) * 8;
      if (k0 < K) {
        uint32_t o4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (a.f16) {
            uint32_t h;
            asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(v[c * 8 + 2 * e + 1] * up), "f"(v[c * 8 + 2 * e] * up));
            o4[e] = h;
          } else {
            o4[e] = pack_bf16x2(v[c * 8 + 2 * e], v[c * 8 + 2 * e + 1]);
          }
        }
        *reinterpret_cast<uint4*>(a.out + (size_t)m * a.ldo + k0) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
    }
    }
    __syncthreads();  // the shared reduction scratch is reused by the next row
  }
}

// Grid of the persistent prep kernel: as many CTAs as fit on the SMs (from the
// occupancy query, cached per variant and stage size), at most one per row.
template <int T>
static cudaError_t launch_prep_t(const PrepArgs& a, cudaStream_t s) {
  static int done_mask[64] = {0};
  static int cached_smem[2] = {-1, -1}, cached_nb[2] = {0, 0};
  const bool gated = a.mode == PREP_GATED;
  const int smem = 2 * prep_stage_bytes(T, gated);
  cudaError_t e = set_smem_once((const void*)prep_kernel<T>, smem, done_mask);
  if (e != cudaSuccess) return e;
  int& nb = cached_nb[gated ? 1 : 0];
  if (cached_smem[gated ? 1 : 0] != smem) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, prep_kernel<T>, T, smem);
    if (e != cudaSuccess) return e;
    if (nb < 1) nb = 1;
    cached_smem[gated ? 1 : 0] = smem;
  }
  int grid = nb * num_sms();
  if (grid > a.M) grid = a.M;
  return launch_k(prep_kernel<T>, dim3(grid), dim3(T), smem, s, a.pdl != 0, a);
}

cudaError_t launch_prep(const PrepArgs& a0, cudaStream_t s) {
  const PrepArgs& a = a0;
  if (a.M <= 0) return cudaSuccess;
  trace_pre(K_PREP, s);
  cudaError_t e;
  // rows no more than the SMs (batched decode): one 512-thread CTA per row,
  // each thread with a short share of the row (the results do not depend on
  // the thread count); else the smallest CTA that covers K, several rows per SM
  if (a.M <= num_sms() || a.K > 256 * kPrepMaxPer) e = launch_prep_t<512>(a, s);
  else if (a.K <= 128 * kPrepMaxPer) e = launch_prep_t<128>(a, s);
  else e = launch_prep_t<256>(a, s);
  trace_post(K_PREP, s);
  return e;
}

int status_mixer(int clear) { return tu_status(clear); }

cudaError_t wait_limit_mixer(long long cycles) { return tu_set_wait_limit(cycles); }

}  // namespace m2
