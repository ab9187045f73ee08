// k_gemv_mma.cu -- decode GEMV (batch <= 8) on warp-level MMA, weights
// streamed from HBM into shared memory by bulk copies.
//
// Same contract as the CUDA-core GEMV in k_gemv.cu (GemvArgs: w8a16 E4M3
// block-scaled or bf16 weights, plain or prepared activations, store /
// residual / conv-update epilogue), for K % 64 == 0, K <= 8192 and up to 8
// batch rows.  The GEMV is HBM-bound.  Register-destination loads keep too few
// bytes in flight per SM to reach the HBM rate, so one producer warp streams
// the weights with 1-D bulk copies (async proxy, mbarrier completion) through
// a ring of shared-memory stages, each 16 rows x KC bytes: one copy of the 16
// whole rows when a row is at most 4 KB, else one copy per row with rows
// padded by 64 bytes (conflict-free fragment loads); the producer starts
// before the dependency wait, since weights are never the previous kernel's
// output.
//
// 16 consumer warps split each stage's 64-element groups.  Lane (g, t) =
// (lane/4, lane%4) reads, per group, the 16 weight bytes [16t, 16t+16) (E4M3;
// 32 bytes for bf16) of rows g and g+8, converts E4M3 exactly to f16 and
// issues 4 m16n8k16 MMAs against the activations (up to 8 batch rows in the
// 8 MMA columns); the k order inside a group is permuted identically for both
// operands, which a dot product allows.  One m16n8k16 consumes 256 weights,
// so a weight costs a fraction of an instruction.  Activations (f16 with the
// exact per-row prescale for E4M3, or bf16) sit in shared memory; E4M3
// partials are scaled per 128-element block; each warp leaves its 16 x MB tile
// per row group in shared memory, and at the end all threads add the 16
// warps' tiles in a fixed order (deterministic) and run the epilogue.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "m2_common.cuh"
#include "m2_kernels.h"
#include "m2_tc.cuh"

namespace m2 {

constexpr int kMmaWarps = 16;                // consumer warps
constexpr int kMmaThreads = (kMmaWarps + 1) * 32;  // + one producer warp
constexpr int kMmaRows = 16;                 // rows per group (MMA M)
constexpr int kRowPad = 64;                  // bytes of padding per staged row
constexpr int kMaxStages = 8;

struct MmaTail {
  unsigned amax[8];
  float unscale[8];
  int32_t pos[8];
  float red[48];  // the norm's cross-warp partials
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t epi_bar;   // epilogue inputs staged by bulk copies
  uint64_t epi_bar2;  // fused decode step: the residual rows of the out_proj epilogue
};

// Shared-memory layout.  kc: bytes of a row per stage (a multiple of 64
// elements); stages: ring depth.
struct MmaLayout {
  int act_ld, tail, act, tot, epi, stage, stage_bytes, kc, pitch, stages, total;
  bool whole;  // a stage is one contiguous block of 16 whole rows (one copy, no row padding)
  bool tma;    // a stage of row pieces arrives as one 3-D tensor copy, rows unpadded
};
// tma: stages of row pieces (rows longer than 4 KB) come as one 3-D tensor
// copy into unpadded rows; kc, and with it which k each warp sums, is the
// same either way.
__host__ __device__ inline MmaLayout mma_layout(int K, int es, int rows_max, int mb, int epi, int dconv,
                                                bool tma = false) {
  MmaLayout L;
  L.act_ld = K + 8;  // elements per activation row (the pad spreads rows over banks)
  L.tail = 0;
  L.act = (int)((sizeof(MmaTail) + 127) / 128 * 128);
  L.tot = L.act + (mb * L.act_ld * 2 + 127) / 128 * 128;  // activation rows (lanes past the batch read row 0)
  L.epi = L.tot + (rows_max * kMmaWarps * mb * 4 + 127) / 128 * 128;  // per-warp partials
  int epi_bytes = 0;
  // conv: taps [rows_max][dconv], bias [rows_max], ring slots [mb][dconv-1][rows_max] (storage order)
  if (epi == EPI_INPROJ_CONV) epi_bytes = rows_max * dconv * 2 + rows_max * 2 + mb * rows_max * (dconv - 1) * 2;
  if (epi == EPI_RESID) epi_bytes = mb * rows_max * 2;
  L.stage = L.epi + (epi_bytes + 127) / 128 * 128;
  const int budget = 227 * 1024 - L.stage;
  const int row_bytes = K * es;
  // Rows of at most 4 KB whose 16-row groups fit 3 stages travel as one copy
  // per row group (fewer, larger copies stream faster; the unpadded rows cost
  // a 2-way bank conflict in the fragment loads).  Otherwise: the largest chunk
  // (<= 4 KB of a row, rows padded) that leaves at least 3 stages.
  L.whole = row_bytes <= 4096 && budget / (kMmaRows * row_bytes) >= 3;
  int kc = row_bytes < 4096 ? row_bytes : 4096;
  if (!L.whole)
    while (kc > 64 * es && budget / (kMmaRows * (kc + kRowPad)) < 3) kc = (kc / 2 + 64 * es - 1) / (64 * es) * (64 * es);
  L.kc = kc;
  L.tma = tma && !L.whole;
  L.pitch = L.whole ? row_bytes : (L.tma ? kc : kc + kRowPad);
  L.stage_bytes = kMmaRows * L.pitch;
  L.stages = budget / L.stage_bytes;
  if (L.stages > kMaxStages) L.stages = kMaxStages;
  L.total = L.stage + L.stages * L.stage_bytes;
  return L;
}

__device__ __forceinline__ uint32_t cvt_e4m3x2(uint32_t two_bytes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)two_bytes));
  return h2;
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

template <bool FP8>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  if constexpr (FP8) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// Fused activation norm for the decode GEMV (consumer threads only, nC of
// them; `red` is 64 floats of shared scratch).  Row m of the activation is
// computed into act (bf16, or f16 after the exact power-of-two prescale for
// E4M3 weights, unscale[m] = 2^-j).  Same arithmetic as the separate norm
// kernel (k_mixer.cu): the RMSNorm sum of squares as error-free fp32 pairs
// and near-tie decisions in double, so its rounding decisions do not depend on
// the order; the gated sum in a fixed order (every CTA computes the same row
// identically).  One exchange through shared memory: each warp leaves its
// partial sums and the largest |product| it will scale; every thread then
// combines the warps' values in the same fixed order itself (no second round
// and no single-thread combine).  The f16 prescale comes from that largest
// product times the norm factor, enlarged by 2^-20 so that it never falls
// below the largest rounded output: the rows' maximum lands in [2^13, 2^15)
// and every bf16 value within 2^30 of it stays exact in f16.
// The norm's inputs that never come from the immediately preceding kernel:
// the weight, and (gated norm) z, which the in_proj two launches back wrote.
// Loaded before the dependency wait, so that their latency -- long while the
// weight stream fills the memory system -- overlaps the wait.
constexpr int kNormPer = 2;  // 16-byte chunks of 8 elements per thread (K <= 8192 with 512 threads)
struct NormPre {
  uint4 wv[kNormPer];
  float sz[kNormPer * 8];  // gated: silu(z)
  bool w, z;               // which of them are loaded
};
__device__ __forceinline__ void norm_preload(const GemvArgs& a, int m, int tid, int nC, bool z, NormPre& pre) {
  pre.z = z && a.norm == NORM_GATED;
  uint4 zv[kNormPer];
#pragma unroll
  for (int c = 0; c < kNormPer; ++c) {
    const int k0 = (tid + nC * c) * 8;
    pre.wv[c] = zv[c] = make_uint4(0u, 0u, 0u, 0u);
    if (k0 < a.K) {
      pre.wv[c] = __ldg(reinterpret_cast<const uint4*>(a.norm_w + k0));
      if (pre.z) zv[c] = __ldcg(reinterpret_cast<const uint4*>(a.gz + (size_t)m * a.ldgz + k0));
    }
  }
  if (pre.z) {
#pragma unroll
    for (int c = 0; c < kNormPer; ++c) {
      const uint32_t z4[4] = {zv[c].x, zv[c].y, zv[c].z, zv[c].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        pre.sz[c * 8 + 2 * e] = silu_f(bf16lo(z4[e]));
        pre.sz[c * 8 + 2 * e + 1] = silu_f(bf16hi(z4[e]));
      }
    }
  }
  pre.w = true;
}

// 2^j for |j| <= 126, exactly
__device__ __forceinline__ float exp2i(int j) { return __uint_as_float((uint32_t)(127 + j) << 23); }

// One activation row's norm into shared memory.  red: 48 floats of scratch
// (not aliasing act or zero); zero[0, nzero): a region this call clears while
// the row's loads are in flight (the caller's accumulators).
template <bool F16>
__device__ void fused_norm_row(const GemvArgs& a, int m, uint16_t* act, float* red, float* unscale, int tid,
                               int nC, const NormPre* pre = nullptr, float* zero = nullptr, int nzero = 0) {
  const int K = a.K, warp = tid >> 5, lane = tid & 31;
  const int nw = nC / 32;
  constexpr int kPer = kNormPer;
  float v[kPer * 8];
  uint4 wv[kPer], zv[kPer];
  // chunk c of this thread holds elements k0 = (tid + nC * c) * 8 ..; chunks
  // past K (uniform across a warp when K is a multiple of 256) are skipped
  auto live = [&](int c) { return (tid + nC * c) * 8 < K; };
  const bool zpre = pre && pre->z && m == 0;
#pragma unroll
  for (int c = 0; c < kPer; ++c) {
    const int k0 = (tid + nC * c) * 8;
    wv[c] = zv[c] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[c * 8 + e] = 0.0f;
    if (k0 < K) {
      wv[c] = (pre && pre->w) ? pre->wv[c] : __ldg(reinterpret_cast<const uint4*>(a.norm_w + k0));
      if (a.norm == NORM_RMS) {
        const uint4 u = *reinterpret_cast<const uint4*>(a.A + (size_t)m * a.lda + k0);  // coherent: previous kernel
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[c * 8 + 2 * e] = bf16lo(w4[e]);
          v[c * 8 + 2 * e + 1] = bf16hi(w4[e]);
        }
      } else {
        if (!zpre) zv[c] = __ldcg(reinterpret_cast<const uint4*>(a.gz + (size_t)m * a.ldgz + k0));
        // L2 loads: y may come from other CTAs of the same launch (fused step)
        const float4 f0 = __ldcg(reinterpret_cast<const float4*>(a.gy + (size_t)m * a.ldgy + k0));
        const float4 f1 = __ldcg(reinterpret_cast<const float4*>(a.gy + (size_t)m * a.ldgy + k0 + 4));
        v[c * 8 + 0] = f0.x; v[c * 8 + 1] = f0.y; v[c * 8 + 2] = f0.z; v[c * 8 + 3] = f0.w;
        v[c * 8 + 4] = f1.x; v[c * 8 + 5] = f1.y; v[c * 8 + 6] = f1.z; v[c * 8 + 7] = f1.w;
      }
    }
  }
  for (int i = tid; i < nzero; i += nC) zero[i] = 0.0f;
  // silu(z) (gated), and the largest |v * w (* silu(z))|
  float sz[kPer * 8];
  float pm = 0.0f;
#pragma unroll
  for (int c = 0; c < kPer; ++c) {
    const uint32_t w4[4] = {wv[c].x, wv[c].y, wv[c].z, wv[c].w}, z4[4] = {zv[c].x, zv[c].y, zv[c].z, zv[c].w};
#pragma unroll
    for (int e = 0; e < 8; ++e) sz[c * 8 + e] = 1.0f;
    if (!live(c)) continue;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (a.norm != NORM_RMS) {
        sz[c * 8 + 2 * e] = zpre ? pre->sz[c * 8 + 2 * e] : silu_f(bf16lo(z4[e]));
        sz[c * 8 + 2 * e + 1] = zpre ? pre->sz[c * 8 + 2 * e + 1] : silu_f(bf16hi(z4[e]));
      }
      if (F16) {
        pm = fmaxf(pm, fabsf(v[c * 8 + 2 * e] * bf16lo(w4[e]) * sz[c * 8 + 2 * e]));
        pm = fmaxf(pm, fabsf(v[c * 8 + 2 * e + 1] * bf16hi(w4[e]) * sz[c * 8 + 2 * e + 1]));
      }
    }
  }
  if (F16) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, o));
  }
  uint16_t o[kPer * 8];
  float r;  // the norm factor as the rounding uses it
  if (a.norm == NORM_RMS) {
    float hi = 0.0f, lo = 0.0f;
#pragma unroll
    for (int c = 0; c < kPer; ++c) {
      if (!live(c)) continue;
#pragma unroll
      for (int e = 0; e < 8; ++e) two_sum_acc(hi, lo, v[c * 8 + e] * v[c * 8 + e]);
    }
    two_sum_warp(hi, lo);
    if (lane == 0) {
      red[warp] = hi;
      red[16 + warp] = lo;
      red[32 + warp] = pm;
    }
    named_bar(1, nC);
    // the warps' partials combined by a fixed butterfly (lanes 16..31 mirror
    // 0..15); every thread then takes lane 0's result
    const int src = lane & 15;
    float h = src < nw ? red[src] : 0.0f, l = src < nw ? red[16 + src] : 0.0f;
    pm = src < nw ? red[32 + src] : 0.0f;
#pragma unroll
    for (int sh = 8; sh > 0; sh >>= 1) {
      const float oh = __shfl_xor_sync(0xffffffffu, h, sh), ol = __shfl_xor_sync(0xffffffffu, l, sh);
      two_sum_acc(h, l, oh);
      l += ol;
      pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, sh));
    }
    h = __shfl_sync(0xffffffffu, h, 0);
    l = __shfl_sync(0xffffffffu, l, 0);
    pm = __shfl_sync(0xffffffffu, pm, 0);
    const NormR nr = norm_r(h, l, K, a.norm_eps);
    r = nr.hi;
#pragma unroll
    for (int c = 0; c < kPer; ++c) {
      if (!live(c)) continue;
      const uint32_t w4[4] = {wv[c].x, wv[c].y, wv[c].z, wv[c].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        o[c * 8 + 2 * e] = norm_round_bf16(v[c * 8 + 2 * e], bf16lo(w4[e]), nr);
        o[c * 8 + 2 * e + 1] = norm_round_bf16(v[c * 8 + 2 * e + 1], bf16hi(w4[e]), nr);
      }
    }
  } else {
    // sum of squares in the order of the separate gated-norm kernel: runs of 8
    // in sequence, warp butterflies, then the 256-element chunks in index order
#pragma unroll
    for (int c = 0; c < kPer; ++c) {
      float ss = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(v[c * 8 + e], v[c * 8 + e], ss);
      ss = warp_sum(ss);
      if (lane == 0) red[c * nw + warp] = ss;  // chunk (warp + 16c) of 256 elements
    }
    if (lane == 0) red[kPer * nw + warp] = pm;
    named_bar(1, nC);
    // the 256-element chunks' sums and the warps' maxima, combined by fixed
    // butterflies; every thread then takes lane 0's result
    float gs = lane < kPer * nw ? red[lane] : 0.0f;
    pm = lane < nw ? red[kPer * nw + lane] : 0.0f;
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) {
      gs += __shfl_xor_sync(0xffffffffu, gs, sh);
      pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, sh));
    }
    gs = __shfl_sync(0xffffffffu, gs, 0);
    pm = __shfl_sync(0xffffffffu, pm, 0);
    r = 1.0f / sqrtf(gs / (float)K + a.norm_eps);
#pragma unroll
    for (int c = 0; c < kPer; ++c) {
      if (!live(c)) continue;
      const uint32_t w4[4] = {wv[c].x, wv[c].y, wv[c].z, wv[c].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        o[c * 8 + 2 * e] = f32_to_bf16(v[c * 8 + 2 * e] * r * bf16lo(w4[e]) * sz[c * 8 + 2 * e]);
        o[c * 8 + 2 * e + 1] = f32_to_bf16(v[c * 8 + 2 * e + 1] * r * bf16hi(w4[e]) * sz[c * 8 + 2 * e + 1]);
      }
    }
  }
  float up = 1.0f;
  if (F16) {
    // exponent of an upper bound of the largest rounded output
    const float mx = pm * r * (1.0f + 0x1p-20f);
    const unsigned bits = __float_as_uint(mx);
    const int ex = bits ? (int)((bits >> 23) & 0xFF) - 127 : 14;
    const int jx = max(-120, min(120, 14 - ex));
    up = exp2i(jx);
    if (tid == 0) unscale[m] = exp2i(-jx);
  } else if (tid == 0) {
    unscale[m] = 1.0f;
  }
#pragma unroll
  for (int c = 0; c < kPer; ++c) {
    const int k0 = (tid + nC * c) * 8;
    if (k0 < K) {
      uint32_t o4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (F16) {
          o4[e] = pack_h2(bf16_to_f32(o[c * 8 + 2 * e]) * up, bf16_to_f32(o[c * 8 + 2 * e + 1]) * up);
        } else {
          o4[e] = (uint32_t)o[c * 8 + 2 * e] | ((uint32_t)o[c * 8 + 2 * e + 1] << 16);
        }
      }
      *reinterpret_cast<uint4*>(act + k0) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
    }
  }
  named_bar(1, nC);  // act is complete, and red[] may be reused by the next row
}

template <bool FP8, int MB>
__global__ void __launch_bounds__(kMmaThreads, 1)
    gemv_mma_kernel(const GemvArgs a, int rows_max, const __grid_constant__ CUtensorMap tmW, int tma) {
  constexpr int ES = FP8 ? 1 : 2;  // bytes per weight
  extern __shared__ __align__(128) uint8_t smem[];
  const int kb = (a.K + 127) / 128;
  const MmaLayout lay = mma_layout(a.K, ES, rows_max, MB, a.epi, a.dconv, tma != 0);
  MmaTail* tail = reinterpret_cast<MmaTail*>(smem + lay.tail);
  uint16_t* act_s = reinterpret_cast<uint16_t*>(smem + lay.act);  // [MB][act_ld]
  float* tot = reinterpret_cast<float*>(smem + lay.tot);
  uint8_t* epi_s = smem + lay.epi;
  uint8_t* stg = smem + lay.stage;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = gridDim.x;
  const int nrg_all = (a.N + kMmaRows - 1) / kMmaRows;
  const int rg_begin = (int)(((long long)nrg_all * blockIdx.x) / G);
  const int rg_end = (int)(((long long)nrg_all * (blockIdx.x + 1)) / G);
  const int row_begin = rg_begin * kMmaRows;
  const int row_end = min(a.N, rg_end * kMmaRows);
  const int nrows = row_end - row_begin;
  const int nrg = rg_end - rg_begin;
  const int mvalid = min(MB, a.M);
  const int L = a.dconv - 1;
  const int row_bytes = a.K * ES;
  const int nch = (row_bytes + lay.kc - 1) / lay.kc;  // chunks (stages) per row group
  const int nst = nrg * nch;                          // stages this CTA streams
  const int pitch = lay.pitch;
  const int S = lay.stages;
  // epilogue input regions of shared memory
  uint16_t* cwS = reinterpret_cast<uint16_t*>(epi_s);  // conv taps [rows_max][dconv]
  uint16_t* bS = cwS + (size_t)rows_max * a.dconv;      // conv bias [rows_max]
  uint16_t* rgS = bS + rows_max;                         // ring slots [MB][L][rows_max], storage order
  uint16_t* rsS = reinterpret_cast<uint16_t*>(epi_s);  // residual rows [MB][rows_max]
  // this CTA's conv rows: local rows [rx0, rx0 + nx) = channels [cx0, cx0 + nx)
  const int xa = max(row_begin, a.xbc0), xb = min(row_end, a.xbc0 + a.d_xbc);
  const int nx = (a.epi == EPI_INPROJ_CONV && xb > xa) ? xb - xa : 0;
  const int rx0 = nx ? xa - row_begin : 0, cx0 = nx ? xa - a.xbc0 : 0;
  auto al16p = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  bool epi_bulk;
  if (a.epi == EPI_INPROJ_CONV)
    epi_bulk = nx > 0 && nx % 8 == 0 && cx0 % 8 == 0 && rx0 % 8 == 0 && a.d_xbc % 8 == 0 && a.conv_b &&
               al16p(a.conv_w) && al16p(a.conv_b) && al16p(a.ring);
  else if (a.epi == EPI_RESID)
    epi_bulk = nrows % 8 == 0 && row_begin % 8 == 0 && a.ldr % 8 == 0 && al16p(a.resid);
  else
    epi_bulk = false;

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&tail->full[i], 1);
      mbar_init(&tail->empty[i], kMmaWarps);
    }
    mbar_init(&tail->epi_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();

  bool dead = false;
  if (warp == kMmaWarps) {
    // ------------------------------------------------ producer warp
    // Weights are never written by the previous kernel: stream without waiting.
    const uint64_t pol = a.evict_first ? policy_evict_first() : policy_evict_normal();
    const uint8_t* W = static_cast<const uint8_t*>(a.W);
    if (epi_bulk && lane == 0) {
      // epilogue inputs of this CTA's rows, a few contiguous ranges (weights,
      // or state written by launches before the immediately preceding kernel)
      const uint64_t pn = policy_evict_normal();
      uint32_t bytes = 0;
      if (a.epi == EPI_INPROJ_CONV) bytes = (uint32_t)(nx * (a.dconv + 1) * 2 + mvalid * L * nx * 2);
      else bytes = (uint32_t)(mvalid * nrows * 2);
      mbar_arrive_expect_tx(&tail->epi_bar, bytes);
      if (a.epi == EPI_INPROJ_CONV) {
        bulk_g2s(cwS + (size_t)rx0 * a.dconv, a.conv_w + (size_t)cx0 * a.dconv, (uint32_t)(nx * a.dconv * 2),
                 &tail->epi_bar, pn);
        bulk_g2s(bS + rx0, a.conv_b + cx0, (uint32_t)(nx * 2), &tail->epi_bar, pn);
        for (int m = 0; m < mvalid; ++m)
          for (int jj = 0; jj < L; ++jj)
            bulk_g2s(rgS + ((size_t)m * L + jj) * rows_max + rx0, a.ring + ((size_t)m * L + jj) * a.d_xbc + cx0,
                     (uint32_t)(nx * 2), &tail->epi_bar, pn);
      } else {
        for (int m = 0; m < mvalid; ++m)
          bulk_g2s(rsS + (size_t)m * rows_max, a.resid + (size_t)m * a.ldr + row_begin, (uint32_t)(nrows * 2),
                   &tail->epi_bar, pn);
      }
    }
    // a later launch's bytes (a hint): this CTA's share is pulled toward L2
    // once its own ring is issued
    auto pull_ahead = [&]() {
      if (lane != 0 || !a.l2_ahead_bytes) return;
      const size_t units = a.l2_ahead_bytes / 16;
      const size_t u0 = units * blockIdx.x / G, u1 = units * (blockIdx.x + 1) / G;
      for (size_t u = u0; u < u1; u += 4096) {  // at most 64 KB per request
        const uint32_t n = (uint32_t)((u1 - u < 4096 ? u1 - u : 4096) * 16);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.l2_ahead + u * 16), "r"(n) : "memory");
      }
    };
    int j = 0;
    bool waited = false;
    // a tensor copy needs a 128-byte aligned destination (the layout keeps
    // every stage at a multiple of 128 from the base): if the base is not,
    // stop here -- the consumers' waits then time out and report it
    if (lay.tma && (smem_addr(stg) & 127u)) {
      if (lane == 0) record_timeout();
      dead = true;
    }
    for (; j < nst && !dead; ++j) {
      const int s = j % S;
      if (j == S) {
        // the ring is full: now take part in the dependency protocol
        pull_ahead();
        pdl_wait();
        pdl_trigger();
        waited = true;
      }
      // every lane waits; the warp goes on only if all saw the slot freed
      if (j >= S && !__all_sync(0xffffffffu, mbar_wait(&tail->empty[s], ((j / S) - 1) & 1))) dead = true;
      if (dead) break;
      const int rg = rg_begin + j / nch, ch = j % nch;
      const int cb = min(lay.kc, row_bytes - ch * lay.kc);  // bytes of each row in this chunk
      if (lay.whole) {
        // rows rg*16 .. min(N, rg*16+16) are contiguous: one copy (rows past N stay stale, results unused)
        if (lane == 0) {
          const int nr = min(kMmaRows, a.N - rg * kMmaRows);
          mbar_arrive_expect_tx(&tail->full[s], (uint32_t)(nr * row_bytes));
          bulk_g2s(stg + (size_t)s * lay.stage_bytes, W + (size_t)rg * kMmaRows * row_bytes, (uint32_t)(nr * row_bytes),
                   &tail->full[s], pol);
        }
      } else if (lay.tma) {
        // 16 rows x kc bytes in one copy (pieces past a row's end and rows past
        // N arrive as zeros; the whole box counts)
        if (lane == 0) {
          mbar_arrive_expect_tx(&tail->full[s], (uint32_t)(kMmaRows * lay.kc));
          tma_load_3d(stg + (size_t)s * lay.stage_bytes, &tmW, 0, ch * (lay.kc / 256), rg * kMmaRows, &tail->full[s],
                      pol);
        }
      } else {
        if (lane == 0) mbar_arrive_expect_tx(&tail->full[s], (uint32_t)(kMmaRows * cb));
        __syncwarp();
        if (lane < kMmaRows) {
          const int r = min(rg * kMmaRows + lane, a.N - 1);  // rows past N repeat row N-1 (results unused)
          bulk_g2s(stg + (size_t)s * lay.stage_bytes + (size_t)lane * pitch,
                   W + (size_t)r * row_bytes + (size_t)ch * lay.kc, (uint32_t)cb, &tail->full[s], pol);
        }
      }
    }
    if (!waited) {
      if (!dead) pull_ahead();
      pdl_wait();
      pdl_trigger();
    }
    // drain: every copy this warp issued has landed before the CTA may exit
    // (also after a timeout, when the consumers may have stopped reading)
    for (int k = max(0, j - S); k < j; ++k)
      if (!mbar_drain(&tail->full[k % S], (k / S) & 1)) break;
    if (epi_bulk && lane == 0) mbar_drain(&tail->epi_bar, 0);
    __syncthreads();  // pairs with the consumers' barrier before the epilogue
    return;
  }

  // ------------------------------------------------ consumers: prologue
  // Epilogue inputs of this CTA's rows.  Under programmatic dependent launch
  // they come from launches before the immediately preceding kernel, which have
  // completed by now, so they are staged before the wait (L2 loads: not L1).
  constexpr int kC = kMmaWarps * 32;  // consumer threads
  // Epilogue inputs of this CTA's rows.  Under programmatic dependent launch
  // they come from launches before the immediately preceding kernel, which have
  // completed by now, so they may be read before the wait: by the producer's
  // bulk copies when aligned (waited for only before the epilogue), else here
  // (L2 loads: not L1).  The positions stay in registers until the epilogue.
  const int pos_r = (a.epi == EPI_INPROJ_CONV && tid < mvalid) ? __ldcg(a.pos + tid) : 0;
  if (!epi_bulk && a.epi == EPI_INPROJ_CONV) {
    for (int r = rx0 + tid; r < rx0 + nx; r += kC) {
      const int c = cx0 + (r - rx0);
      for (int jj = 0; jj < a.dconv; ++jj) cwS[r * a.dconv + jj] = __ldg(a.conv_w + (size_t)c * a.dconv + jj);
      bS[r] = a.conv_b ? __ldg(a.conv_b + c) : (uint16_t)0;
      for (int m = 0; m < mvalid; ++m)
        for (int jj = 0; jj < L; ++jj)
          rgS[((size_t)m * L + jj) * rows_max + r] = __ldcg(a.ring + ((size_t)m * L + jj) * a.d_xbc + c);
    }
  } else if (!epi_bulk && a.epi == EPI_RESID) {
    for (int i = tid; i < nrows * mvalid; i += kC) {
      const int m = i / nrows, r = i % nrows;
      rsS[m * rows_max + r] = __ldcg(a.resid + (size_t)m * a.ldr + row_begin + r);
    }
  }
  NormPre pre;
  // before the wait; silu(z) only for a single row (registers)
  if (a.norm != NORM_NONE) norm_preload(a, 0, tid, kC, MB == 1 && mvalid == 1, pre);
  pdl_wait();
  pdl_trigger();
  const int ntot = rows_max * kMmaWarps * MB;
  if (a.norm != NORM_NONE) {
    // the activation rows are this kernel's own norm of its inputs; the
    // accumulators are cleared while the first row's loads are in flight
    // (the norm's barriers order that before the main loop)
    for (int m = 0; m < mvalid; ++m)
      fused_norm_row<FP8>(a, m, act_s + (size_t)m * lay.act_ld, tail->red, tail->unscale, tid, kC, &pre,
                          m == 0 ? tot : nullptr, m == 0 ? ntot : 0);
  } else {
    for (int i = tid; i < ntot; i += kC) tot[i] = 0.0f;
    if (tid < 8) tail->amax[tid] = 0u;
    named_bar(1, kC);
    // activations -> shared memory (coherent loads: written by the previous kernel)
    const int kv = a.K / 8;  // 16-byte vectors per row
    for (int i = tid; i < mvalid * kv; i += kC) {
      const int m = i / kv, k8 = (i % kv) * 8;
      uint4 v = *reinterpret_cast<const uint4*>(a.A + (size_t)m * a.lda + k8);
      if (FP8 && a.act == ACT_PLAIN) {
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
        float mx = 0.0f;
#pragma unroll
        for (int e = 0; e < 4; ++e) mx = fmaxf(mx, fmaxf(fabsf(bf16lo(w4[e])), fabsf(bf16hi(w4[e]))));
        atomicMax(&tail->amax[m], __float_as_uint(mx));
      }
      *reinterpret_cast<uint4*>(act_s + (size_t)m * lay.act_ld + k8) = v;
    }
    named_bar(1, kC);
    if (FP8 && a.act == ACT_PLAIN) {
      // plain bf16 rows: per-row prescale into the f16 range, converted in place
      for (int i = tid; i < mvalid * kv; i += kC) {
        const int m = i / kv, k8 = (i % kv) * 8;
        const unsigned bits = tail->amax[m];
        const int ex = bits ? (int)((bits >> 23) & 0xFF) - 127 : 14;
        const float up = ldexpf(1.0f, max(-120, min(120, 14 - ex)));
        uint4* p = reinterpret_cast<uint4*>(act_s + (size_t)m * lay.act_ld + k8);
        uint4 v = *p;
        v.x = pack_h2(bf16lo(v.x) * up, bf16hi(v.x) * up);
        v.y = pack_h2(bf16lo(v.y) * up, bf16hi(v.y) * up);
        v.z = pack_h2(bf16lo(v.z) * up, bf16hi(v.z) * up);
        v.w = pack_h2(bf16lo(v.w) * up, bf16hi(v.w) * up);
        *p = v;
      }
      if (tid < 8) {
        const unsigned bits = tail->amax[tid];
        const int ex = bits ? (int)((bits >> 23) & 0xFF) - 127 : 14;
        tail->unscale[tid] = ldexpf(1.0f, -max(-120, min(120, 14 - ex)));
      }
    } else if (tid < 8) {
      tail->unscale[tid] = (a.act == ACT_PREPARED && tid < mvalid) ? a.unscale[tid] : 1.0f;
    }
    named_bar(1, kC);
  }

  // ------------------------------------------------ consumers: main loop
  // MMA column g is batch row g; lanes past the batch read row 0 into columns
  // that are never stored
  const uint16_t* act_g = act_s + (size_t)(g < mvalid ? g : 0) * lay.act_ld;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < nst && !dead; ++j) {
    const int s = j % S;
    const int rg = rg_begin + j / nch, ch = j % nch;
    const int cb = min(lay.kc, row_bytes - ch * lay.kc);
    const int ng = cb / (64 * ES);                      // 64-element groups in this chunk
    const int q0 = (ng * warp) / kMmaWarps, q1 = (ng * (warp + 1)) / kMmaWarps;
    const int kel0 = ch * (lay.kc / ES);                // first k of the chunk
    // the MMAs below are warp-collective: the warp decides together
    if (!__all_sync(0xffffffffu, mbar_wait(&tail->full[s], (j / S) & 1))) {
      dead = true;
      break;
    }
    const uint8_t* st0 = stg + (size_t)s * lay.stage_bytes + (size_t)g * pitch;
    const uint8_t* st8 = st0 + (size_t)8 * pitch;
    const int r0 = min(rg * kMmaRows + g, row_end - 1), r8 = min(rg * kMmaRows + g + 8, row_end - 1);
    for (int q = q0; q < q1; ++q) {
      const int k0 = kel0 + q * 64;  // first k of the group
      const uint4 bl = *reinterpret_cast<const uint4*>(act_g + k0 + 16 * t);
      const uint4 bh = *reinterpret_cast<const uint4*>(act_g + k0 + 16 * t + 8);
      const uint32_t bw[8] = {bl.x, bl.y, bl.z, bl.w, bh.x, bh.y, bh.z, bh.w};
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (FP8) {
        const uint4 v0 = *reinterpret_cast<const uint4*>(st0 + q * 64 + 16 * t);
        const uint4 v8 = *reinterpret_cast<const uint4*>(st8 + q * 64 + 16 * t);
        const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w};
        const uint32_t w8[4] = {v8.x, v8.y, v8.z, v8.w};
#pragma unroll
        for (int sp = 0; sp < 4; ++sp)
          mma16816<FP8>(d, cvt_e4m3x2(w0[sp]), cvt_e4m3x2(w8[sp]), cvt_e4m3x2(w0[sp] >> 16),
                        cvt_e4m3x2(w8[sp] >> 16), bw[2 * sp], bw[2 * sp + 1]);
        // one 128-element scale block per group; rows g and g+8 may sit in different n-blocks
        const int kbk = k0 >> 7;
        const float s0 = bf16_to_f32(__ldg(a.S + (size_t)(r0 >> 7) * kb + kbk));  // read-only: L1 hits
        const float s8 = bf16_to_f32(__ldg(a.S + (size_t)(r8 >> 7) * kb + kbk));
        acc[0] = fmaf(d[0], s0, acc[0]);
        acc[1] = fmaf(d[1], s0, acc[1]);
        acc[2] = fmaf(d[2], s8, acc[2]);
        acc[3] = fmaf(d[3], s8, acc[3]);
      } else {
        const uint4 v0a = *reinterpret_cast<const uint4*>(st0 + q * 128 + 32 * t);
        const uint4 v0b = *reinterpret_cast<const uint4*>(st0 + q * 128 + 32 * t + 16);
        const uint4 v8a = *reinterpret_cast<const uint4*>(st8 + q * 128 + 32 * t);
        const uint4 v8b = *reinterpret_cast<const uint4*>(st8 + q * 128 + 32 * t + 16);
        const uint32_t w0[8] = {v0a.x, v0a.y, v0a.z, v0a.w, v0b.x, v0b.y, v0b.z, v0b.w};
        const uint32_t w8[8] = {v8a.x, v8a.y, v8a.z, v8a.w, v8b.x, v8b.y, v8b.z, v8b.w};
#pragma unroll
        for (int sp = 0; sp < 4; ++sp)
          mma16816<FP8>(d, w0[2 * sp], w8[2 * sp], w0[2 * sp + 1], w8[2 * sp + 1], bw[2 * sp], bw[2 * sp + 1]);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] += d[i];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&tail->empty[s]);
    if (ch == nch - 1) {
      // row group done: this warp's 16 x MB tile goes to its own slots; the
      // epilogue adds the 16 warps in a fixed order (deterministic results)
      const int lr = (rg - rg_begin) * kMmaRows;
      const int c0 = 2 * t, c1 = 2 * t + 1;
      // tot [warp][rows_max][MB]: the epilogue's threads (consecutive rows) read
      // consecutive words
      float* t0 = tot + ((size_t)warp * rows_max + lr + g) * MB;
      float* t8 = tot + ((size_t)warp * rows_max + lr + g + 8) * MB;
      if (c0 < MB) {
        t0[c0] = acc[0];
        t8[c0] = acc[2];
      }
      if (c1 < MB) {
        t0[c1] = acc[1];
        t8[c1] = acc[3];
      }
      acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
    }
  }
  if (tid < 8) tail->pos[tid] = pos_r;
  if (epi_bulk && !mbar_wait(&tail->epi_bar, 0)) dead = true;
  __syncthreads();  // all consumers and the producer (after its drain)

  // ------------------------------------------------ epilogue (consumer threads)
  for (int i = tid; i < nrows * mvalid; i += kC) {
    const int r = i / mvalid, m = i % mvalid;
    const int n = row_begin + r;
    float sum = 0.0f;
#pragma unroll
    for (int w = 0; w < kMmaWarps; ++w) sum += tot[((size_t)w * rows_max + r) * MB + m];
    const float accv = sum * tail->unscale[m];
    uint16_t* o = a.out + (size_t)m * a.ldo + n;
    if (a.epi == EPI_RESID) {
      const float res = bf16_to_f32(rsS[m * rows_max + r]);
      *o = f32_to_bf16(res + accv);
    } else if (a.epi == EPI_INPROJ_CONV && n >= a.xbc0 && n < a.xbc0 + a.d_xbc) {
      // conv1d update with bias + SiLU; this thread alone owns (sequence m,
      // channel c) in this call, and the ring taps were staged before any write
      const uint16_t vb = f32_to_bf16(accv);  // rounding point of the in_proj output
      const int c = n - a.xbc0;
      const uint16_t* w = cwS + r * a.dconv;
      const int p = tail->pos[m];
      float s = bf16_to_f32(bS[r]);
      for (int j = 0; j < L; ++j) s += bf16_to_f32(w[j]) * bf16_to_f32(rgS[((size_t)m * L + (p + j) % L) * rows_max + r]);
      s += bf16_to_f32(w[L]) * bf16_to_f32(vb);
      *o = f32_to_bf16(silu_f(s));
      a.ring[(size_t)m * L * a.d_xbc + (size_t)(tail->pos[m] % L) * a.d_xbc + c] = vb;
    } else {
      *o = f32_to_bf16(accv);
    }
  }
}

template <bool FP8, int MB>
static cudaError_t launch_mma_one(const GemvArgs& a, cudaStream_t s) {
  static int done_mask[64] = {0};
  const int nrg = (a.N + kMmaRows - 1) / kMmaRows;
  // the fewest CTAs whose largest share of row groups is that of one CTA per
  // SM: the step takes as long, every CTA finishes at about the same time,
  // and the SMs left over take the next kernel's CTAs early
  const int per = (nrg + num_sms() - 1) / num_sms();
  const int grid = (nrg + per - 1) / per;
  const int rows_max = per * kMmaRows;
  // rows longer than 4 KB: each stage (16 row pieces) as one 3-D tensor copy
  // instead of 16 row copies, when the rows split into 256-byte pieces
  CUtensorMap tmW;
  memset(&tmW, 0, sizeof(tmW));
  const int row_bytes = a.K * (FP8 ? 1 : 2);
  const MmaLayout plain = mma_layout(a.K, FP8 ? 1 : 2, rows_max, MB, a.epi, a.dconv);
  const int tma = (!plain.whole && row_bytes % 256 == 0 && plain.kc % 256 == 0 &&
                   encode_rows_3d(&tmW, a.W, (uint64_t)row_bytes, (uint64_t)a.N, 256, plain.kc / 256, kMmaRows))
                      ? 1
                      : 0;
  const MmaLayout lay = mma_layout(a.K, FP8 ? 1 : 2, rows_max, MB, a.epi, a.dconv, tma != 0);
  if (lay.stages < 2 || lay.total > 227 * 1024) return cudaErrorInvalidConfiguration;
  auto kern = gemv_mma_kernel<FP8, MB>;
  cudaError_t e = set_smem_once((const void*)kern, lay.total, done_mask);
  if (e != cudaSuccess) return e;
  const int id = (FP8 ? K_GEMV_FP8 : K_GEMV_BF16) + (a.epi == EPI_INPROJ_CONV ? 1 : (a.epi == EPI_RESID ? 2 : 0));
  trace_pre(id, s);
  e = launch_k(kern, dim3(grid), dim3(kMmaThreads), lay.total, s, a.pdl != 0, a, rows_max, tmW, tma);
  trace_post(id, s);
  return e;
}

bool gemv_mma_supported(int M, int K) { return M >= 1 && M <= 8 && K % 64 == 0 && K <= 8192; }

cudaError_t launch_gemv_mma(const GemvArgs& a, bool fp8, cudaStream_t s) {
  if (!gemv_mma_supported(a.M, a.K)) return cudaErrorInvalidValue;
  const int mb = a.M <= 1 ? 1 : (a.M <= 2 ? 2 : (a.M <= 4 ? 4 : 8));
  if (fp8) {
    switch (mb) {
      case 1: return launch_mma_one<true, 1>(a, s);
      case 2: return launch_mma_one<true, 2>(a, s);
      case 4: return launch_mma_one<true, 4>(a, s);
      default: return launch_mma_one<true, 8>(a, s);
    }
  }
  switch (mb) {
    case 1: return launch_mma_one<false, 1>(a, s);
    case 2: return launch_mma_one<false, 2>(a, s);
    case 4: return launch_mma_one<false, 4>(a, s);
    default: return launch_mma_one<false, 8>(a, s);
  }
}

// ------------------------------------------------------------------ fused decode step, batch 1
//
// The whole layer step of one sequence in one cooperative launch, one CTA per
// SM, all CTAs resident:
//   phase 1  in_proj GEMV, input RMSNorm in the prologue, conv1d update with
//            bias and SiLU in the epilogue (this CTA's row groups)
//   grid barrier
//   phase 2  SSM step of this CTA's share of the H*P state rows
//   grid barrier
//   phase 3  out_proj GEMV, gated RMSNorm in the prologue, residual add in the
//            epilogue (in place on the hidden row)
// The producer warp streams both projections' weight rows through one ring
// without a break, so the out_proj rows land in shared memory while the SSM
// phase and the barriers run; the three-kernel chain pays a launch ramp and a
// drain per kernel instead.  Row groups, the per-group MMA work and the
// fixed-order reductions are those of gemv_mma_kernel, so the outputs are
// bit-identical to the three-kernel chain.

// One GEMV's share of this CTA: row groups [rg_begin, rg_end), streamed in
// nst stages of kc bytes per row (whole 16-row groups when a row is <= 4 KB).
struct MmaPlan {
  int rg_begin, rg_end, row_begin, row_end, nrows, nrg, nch, nst, row_bytes, kc, pitch;
  bool whole;
};

// kc / whole: the chunking the stand-alone GEMV launch would choose for this
// projection (it decides which k each warp sums, hence the rounding).
__device__ __forceinline__ MmaPlan mma_plan(const GemvArgs& a, int es, int kc, bool whole) {
  MmaPlan p;
  const int G = gridDim.x;
  const int nrg_all = (a.N + kMmaRows - 1) / kMmaRows;
  p.rg_begin = (int)(((long long)nrg_all * blockIdx.x) / G);
  p.rg_end = (int)(((long long)nrg_all * (blockIdx.x + 1)) / G);
  p.row_begin = p.rg_begin * kMmaRows;
  p.row_end = min(a.N, p.rg_end * kMmaRows);
  p.nrows = max(0, p.row_end - p.row_begin);
  p.nrg = p.rg_end - p.rg_begin;
  p.row_bytes = a.K * es;
  p.whole = whole;
  p.kc = kc;
  p.pitch = p.whole ? p.row_bytes : p.kc + kRowPad;
  p.nch = (p.row_bytes + p.kc - 1) / p.kc;
  p.nst = p.nrg * p.nch;
  return p;
}

constexpr int kFusedStride = kMmaRows * (4096 + kRowPad);  // bytes per ring stage

struct FusedLayout {
  int act, tot, epc, epr, stage, stages, total;
};
// k_in / k_out: the projections' K; rows_in / rows_out: row capacity per CTA.
__host__ __device__ inline FusedLayout fused_layout(int k_in, int k_out, int rows_in, int rows_out, int dconv) {
  FusedLayout L;
  const int kmax = k_in > k_out ? k_in : k_out;
  const int rmax = rows_in > rows_out ? rows_in : rows_out;
  L.act = (int)((sizeof(MmaTail) + 127) / 128 * 128);
  L.tot = L.act + ((kmax + 8) * 2 + 127) / 128 * 128;               // one activation row
  L.epc = L.tot + (rmax * kMmaWarps * 4 + 127) / 128 * 128;          // per-warp row totals
  L.epr = L.epc + (rows_in * (2 * dconv + 1) * 2 + 127) / 128 * 128;  // conv taps, bias, ring slots
  L.stage = L.epr + (rows_out * 2 + 127) / 128 * 128;                // residual rows
  L.stages = (227 * 1024 - L.stage) / kFusedStride;
  if (L.stages > kMaxStages) L.stages = kMaxStages;
  L.total = L.stage + L.stages * kFusedStride;
  return L;
}

// Issue the bulk copies of stage jl of plan p (whole warp; lane 0 arms the barrier).
__device__ __forceinline__ void mma_produce(const GemvArgs& a, const MmaPlan& p, int jl, uint8_t* dst, uint64_t* full,
                                            uint64_t pol, int lane) {
  const uint8_t* W = static_cast<const uint8_t*>(a.W);
  const int rg = p.rg_begin + jl / p.nch, ch = jl % p.nch;
  const int cb = min(p.kc, p.row_bytes - ch * p.kc);
  if (p.whole) {
    if (lane == 0) {
      const int nr = min(kMmaRows, a.N - rg * kMmaRows);
      mbar_arrive_expect_tx(full, (uint32_t)(nr * p.row_bytes));
      bulk_g2s(dst, W + (size_t)rg * kMmaRows * p.row_bytes, (uint32_t)(nr * p.row_bytes), full, pol);
    }
  } else {
    if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)(kMmaRows * cb));
    __syncwarp();
    if (lane < kMmaRows) {
      const int r = min(rg * kMmaRows + lane, a.N - 1);
      bulk_g2s(dst + (size_t)lane * p.pitch, W + (size_t)r * p.row_bytes + (size_t)ch * p.kc, (uint32_t)cb, full, pol);
    }
  }
}

// Consume this CTA's stages of plan p (ring slots j0 + jl); one batch row
// (act), totals per warp into tot [warp][rows_max].  False on a timeout.
template <bool FP8>
__device__ __forceinline__ bool mma_consume(const GemvArgs& a, const MmaPlan& p, int j0, int S, uint8_t* stg,
                                            MmaTail* tail, const uint16_t* act, float* tot, int rows_max, int warp,
                                            int lane) {
  constexpr int ES = FP8 ? 1 : 2;
  const int g = lane >> 2, t = lane & 3;
  const int kb = (a.K + 127) / 128;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int jl = 0; jl < p.nst; ++jl) {
    const int j = j0 + jl, s = j % S;
    const int rg = p.rg_begin + jl / p.nch, ch = jl % p.nch;
    const int cb = min(p.kc, p.row_bytes - ch * p.kc);
    const int ng = cb / (64 * ES);
    const int q0 = (ng * warp) / kMmaWarps, q1 = (ng * (warp + 1)) / kMmaWarps;
    const int kel0 = ch * (p.kc / ES);
    if (!__all_sync(0xffffffffu, mbar_wait(&tail->full[s], (j / S) & 1))) return false;  // warp-collective MMAs follow
    const uint8_t* st0 = stg + (size_t)s * kFusedStride + (size_t)g * p.pitch;
    const uint8_t* st8 = st0 + (size_t)8 * p.pitch;
    const int r0 = min(rg * kMmaRows + g, p.row_end - 1), r8 = min(rg * kMmaRows + g + 8, p.row_end - 1);
    for (int q = q0; q < q1; ++q) {
      const int k0 = kel0 + q * 64;
      // every MMA column reads the one batch row; only column 0 is stored
      const uint4 bl = *reinterpret_cast<const uint4*>(act + k0 + 16 * t);
      const uint4 bh = *reinterpret_cast<const uint4*>(act + k0 + 16 * t + 8);
      const uint32_t bw[8] = {bl.x, bl.y, bl.z, bl.w, bh.x, bh.y, bh.z, bh.w};
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (FP8) {
        const uint4 v0 = *reinterpret_cast<const uint4*>(st0 + q * 64 + 16 * t);
        const uint4 v8 = *reinterpret_cast<const uint4*>(st8 + q * 64 + 16 * t);
        const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w};
        const uint32_t w8[4] = {v8.x, v8.y, v8.z, v8.w};
#pragma unroll
        for (int sp = 0; sp < 4; ++sp)
          mma16816<FP8>(d, cvt_e4m3x2(w0[sp]), cvt_e4m3x2(w8[sp]), cvt_e4m3x2(w0[sp] >> 16),
                        cvt_e4m3x2(w8[sp] >> 16), bw[2 * sp], bw[2 * sp + 1]);
        const int kbk = k0 >> 7;
        const float s0 = bf16_to_f32(__ldg(a.S + (size_t)(r0 >> 7) * kb + kbk));
        const float s8 = bf16_to_f32(__ldg(a.S + (size_t)(r8 >> 7) * kb + kbk));
        acc[0] = fmaf(d[0], s0, acc[0]);
        acc[2] = fmaf(d[2], s8, acc[2]);
      } else {
        const uint4 v0a = *reinterpret_cast<const uint4*>(st0 + q * 128 + 32 * t);
        const uint4 v0b = *reinterpret_cast<const uint4*>(st0 + q * 128 + 32 * t + 16);
        const uint4 v8a = *reinterpret_cast<const uint4*>(st8 + q * 128 + 32 * t);
        const uint4 v8b = *reinterpret_cast<const uint4*>(st8 + q * 128 + 32 * t + 16);
        const uint32_t w0[8] = {v0a.x, v0a.y, v0a.z, v0a.w, v0b.x, v0b.y, v0b.z, v0b.w};
        const uint32_t w8[8] = {v8a.x, v8a.y, v8a.z, v8a.w, v8b.x, v8b.y, v8b.z, v8b.w};
#pragma unroll
        for (int sp = 0; sp < 4; ++sp)
          mma16816<FP8>(d, w0[2 * sp], w8[2 * sp], w0[2 * sp + 1], w8[2 * sp + 1], bw[2 * sp], bw[2 * sp + 1]);
        acc[0] += d[0];
        acc[2] += d[2];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&tail->empty[s]);
    if (ch == p.nch - 1) {
      const int lr = (rg - p.rg_begin) * kMmaRows;
      if (t == 0) {  // column 0: the batch row
        tot[(size_t)warp * rows_max + lr + g] = acc[0];
        tot[(size_t)warp * rows_max + lr + g + 8] = acc[2];
      }
      acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
    }
  }
  return true;
}

// Grid-wide barrier of the fused step (all CTAs resident: cooperative launch).
// One 64-bit arrival counter that only grows: an arrival that finds the count
// at c waits until it reaches the next multiple of the grid size above c.
// Every CTA arrives exactly once at each barrier, timed out or not (a timeout
// only ends the wait: the status word is set and the CTA goes on), so the
// count is a multiple of the grid size again when a launch ends, and the next
// launch's barriers line up however the previous one ended; nothing has to be
// reset between launches.
__device__ unsigned long long g_fused_arrivals;

__device__ __forceinline__ unsigned long long ld_acquire_gpu_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __noinline__ void fused_grid_barrier(int tid, int nthreads) {
  named_bar(1, nthreads);
  if (tid == 0) {
    const unsigned long long G = gridDim.x;
    __threadfence();  // this CTA's writes before its arrival
    const unsigned long long c = atomicAdd(&g_fused_arrivals, 1ull);
    const unsigned long long target = (c / G + 1) * G;
    const long long limit = *reinterpret_cast<volatile long long*>(&g_wait_limit);
    const long long t0 = clock64();
    while (ld_acquire_gpu_u64(&g_fused_arrivals) < target) {
      if (clock64() - t0 > limit) {
        record_timeout();
        break;
      }
    }
    __threadfence();
  }
  named_bar(1, nthreads);
}

// Chunking of the two projections (as the stand-alone GEMV launches choose it).
struct FusedChunks {
  int kc_in, whole_in, kc_out, whole_out;
};

template <bool FP8>
__global__ void __launch_bounds__(kMmaThreads, 1)
    decode_step_fused_kernel(const FusedStepArgs fa, int rows_in, int rows_out, const FusedChunks ck) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int ES = FP8 ? 1 : 2;
  constexpr int kC = kMmaWarps * 32;  // consumer threads
  const GemvArgs& a1 = fa.in;
  const GemvArgs& a3 = fa.out;
  const SsmArgs& sa = fa.ssm;
  const FusedLayout lay = fused_layout(a1.K, a3.K, rows_in, rows_out, a1.dconv);
  MmaTail* tail = reinterpret_cast<MmaTail*>(smem);
  uint16_t* act_s = reinterpret_cast<uint16_t*>(smem + lay.act);
  float* tot = reinterpret_cast<float*>(smem + lay.tot);
  uint16_t* cwS = reinterpret_cast<uint16_t*>(smem + lay.epc);  // conv taps [rows_in][dconv]
  uint16_t* bS = cwS + (size_t)rows_in * a1.dconv;                // conv bias [rows_in]
  uint16_t* rgS = bS + rows_in;                                   // ring slots [L][rows_in], storage order
  uint16_t* rsS = reinterpret_cast<uint16_t*>(smem + lay.epr);  // residual row [rows_out]
  uint8_t* stg = smem + lay.stage;
  const int S = lay.stages;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const MmaPlan p1 = mma_plan(a1, ES, ck.kc_in, ck.whole_in != 0), p3 = mma_plan(a3, ES, ck.kc_out, ck.whole_out != 0);
  const int L = a1.dconv - 1;
  // this CTA's conv rows in phase 1: local rows [rx0, rx0 + nx) = channels [cx0, cx0 + nx)
  const int xa = max(p1.row_begin, a1.xbc0), xb = min(p1.row_end, a1.xbc0 + a1.d_xbc);
  const int nx = xb > xa ? xb - xa : 0;
  const int rx0 = nx ? xa - p1.row_begin : 0, cx0 = nx ? xa - a1.xbc0 : 0;
  auto al16p = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  const bool bulk1 = nx > 0 && nx % 8 == 0 && cx0 % 8 == 0 && rx0 % 8 == 0 && a1.d_xbc % 8 == 0 && a1.conv_b &&
                     al16p(a1.conv_w) && al16p(a1.conv_b) && al16p(a1.ring);
  const bool bulk3 = p3.nrows > 0 && p3.nrows % 8 == 0 && p3.row_begin % 8 == 0 && al16p(a3.resid);
  // phase-2 rows of this CTA: [sr0, sr1) of the H*P state rows
  const int nsr = sa.H * sa.P;
  const int sr0 = (int)(((long long)nsr * blockIdx.x) / gridDim.x);
  const int sr1 = (int)(((long long)nsr * (blockIdx.x + 1)) / gridDim.x);

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&tail->full[i], 1);
      mbar_init(&tail->empty[i], kMmaWarps);
    }
    mbar_init(&tail->epi_bar, 1);
    mbar_init(&tail->epi_bar2, 1);
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kMmaWarps) {
    // ------------------------------------------------ producer warp
    // Weights are never written by a kernel: the ring fills before the
    // dependency wait.  Everything else (ring, residual) after it.
    const uint64_t pol1 = a1.evict_first ? policy_evict_first() : policy_evict_normal();
    const uint64_t pol3 = a3.evict_first ? policy_evict_first() : policy_evict_normal();
    if (lane == 0 && sr1 > sr0) {
      // this CTA's phase-2 state rows into L2 (one contiguous range)
      const char* base = reinterpret_cast<const char*>(sa.h + (size_t)sr0 * sa.N);
      const size_t bytes = (size_t)(sr1 - sr0) * sa.N * 4;
      for (size_t o = 0; o < bytes; o += 65536) {
        const uint32_t n = (uint32_t)(bytes - o < 65536 ? bytes - o : 65536);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base + o), "r"(n) : "memory");
      }
    }
    auto epi_copies = [&]() {
      if (lane != 0) return;
      const uint64_t pn = policy_evict_normal();
      if (bulk1) {
        mbar_arrive_expect_tx(&tail->epi_bar, (uint32_t)(nx * (a1.dconv + 1) * 2 + L * nx * 2));
        bulk_g2s(cwS + (size_t)rx0 * a1.dconv, a1.conv_w + (size_t)cx0 * a1.dconv, (uint32_t)(nx * a1.dconv * 2),
                 &tail->epi_bar, pn);
        bulk_g2s(bS + rx0, a1.conv_b + cx0, (uint32_t)(nx * 2), &tail->epi_bar, pn);
        for (int jj = 0; jj < L; ++jj)
          bulk_g2s(rgS + (size_t)jj * rows_in + rx0, a1.ring + (size_t)jj * a1.d_xbc + cx0, (uint32_t)(nx * 2),
                   &tail->epi_bar, pn);
      }
      if (bulk3) {
        mbar_arrive_expect_tx(&tail->epi_bar2, (uint32_t)(p3.nrows * 2));
        bulk_g2s(rsS, a3.resid + p3.row_begin, (uint32_t)(p3.nrows * 2), &tail->epi_bar2, pn);
      }
    };
    bool dead = false, waited = false;
    const int nst = p1.nst + p3.nst;
    int j = 0;
    for (; j < nst && !dead; ++j) {
      const int s = j % S;
      if (j == S) {
        pdl_wait();
        pdl_trigger();
        waited = true;
        epi_copies();
      }
      if (j >= S && !__all_sync(0xffffffffu, mbar_wait(&tail->empty[s], ((j / S) - 1) & 1))) dead = true;
      if (dead) break;
      uint8_t* dst = stg + (size_t)s * kFusedStride;
      if (j < p1.nst) mma_produce(a1, p1, j, dst, &tail->full[s], pol1, lane);
      else mma_produce(a3, p3, j - p1.nst, dst, &tail->full[s], pol3, lane);
    }
    if (!waited) {
      pdl_wait();
      pdl_trigger();
      epi_copies();
    }
    // drain: the weight stages and epilogue copies this warp issued have
    // landed before the CTA may exit (also after a timeout)
    for (int k = max(0, j - S); k < j; ++k)
      if (!mbar_drain(&tail->full[k % S], (k / S) & 1)) break;
    if (lane == 0 && bulk1) mbar_drain(&tail->epi_bar, 0);
    if (lane == 0 && bulk3) mbar_drain(&tail->epi_bar2, 0);
    __syncthreads();
    return;
  }

  // ------------------------------------------------ consumers
  pdl_wait();  // hidden, conv ring and position, SSM state: the previous launch's
  pdl_trigger();
  const int pos_r = __ldcg(a1.pos);
  if (!bulk1) {
    for (int r = rx0 + tid; r < rx0 + nx; r += kC) {
      const int c = cx0 + (r - rx0);
      for (int jj = 0; jj < a1.dconv; ++jj) cwS[r * a1.dconv + jj] = __ldg(a1.conv_w + (size_t)c * a1.dconv + jj);
      bS[r] = a1.conv_b ? __ldg(a1.conv_b + c) : (uint16_t)0;
      for (int jj = 0; jj < L; ++jj) rgS[(size_t)jj * rows_in + r] = __ldcg(a1.ring + (size_t)jj * a1.d_xbc + c);
    }
  }
  if (!bulk3)
    for (int r = tid; r < p3.nrows; r += kC) rsS[r] = __ldcg(a3.resid + p3.row_begin + r);
  bool dead = false;

  // ---- phase 1: in_proj
  fused_norm_row<FP8>(a1, 0, act_s, tot, tail->unscale, tid, kC);
  for (int i = tid; i < rows_in * kMmaWarps; i += kC) tot[i] = 0.0f;
  named_bar(1, kC);
  if (!mma_consume<FP8>(a1, p1, 0, S, stg, tail, act_s, tot, rows_in, warp, lane)) dead = true;
  if (bulk1 && !dead && !mbar_wait(&tail->epi_bar, 0)) dead = true;
  named_bar(1, kC);
  {
    const float us = tail->unscale[0];
    for (int r = tid; r < p1.nrows; r += kC) {
      const int n = p1.row_begin + r;
      float sum = 0.0f;
#pragma unroll
      for (int w = 0; w < kMmaWarps; ++w) sum += tot[(size_t)w * rows_in + r];
      const float accv = sum * us;
      uint16_t* o = a1.out + n;
      if (n >= a1.xbc0 && n < a1.xbc0 + a1.d_xbc) {
        const uint16_t vb = f32_to_bf16(accv);  // rounding point of the in_proj output
        const int c = n - a1.xbc0;
        const uint16_t* w = cwS + r * a1.dconv;
        float sc = bf16_to_f32(bS[r]);
        for (int jj = 0; jj < L; ++jj) sc += bf16_to_f32(w[jj]) * bf16_to_f32(rgS[(size_t)((pos_r + jj) % L) * rows_in + r]);
        sc += bf16_to_f32(w[L]) * bf16_to_f32(vb);
        *o = f32_to_bf16(silu_f(sc));
        a1.ring[(size_t)(pos_r % L) * a1.d_xbc + c] = vb;
      } else {
        *o = f32_to_bf16(accv);
      }
    }
  }
  fused_grid_barrier(tid, kC);

  // ---- phase 2: SSM step, rows [sr0, sr1); a row is N/4 lanes x 4 states
  {
    const int lpr = sa.N / 4, rpw = 32 / lpr;
    const int n4 = (lane % lpr) * 4;
    const int hpg = sa.H / sa.G;
    for (int rb = sr0 + warp * rpw; rb < sr1; rb += kMmaWarps * rpw) {
      const int r = rb + lane / lpr;
      const bool live = r < sr1;  // uniform across the lanes of one row
      const int rr = live ? r : sr1 - 1;
      const int h = rr / sa.P, p = rr % sa.P, gi = h / hpg;
      float* hp = sa.h + (size_t)rr * sa.N + n4;
      float4 hv = __ldcg(reinterpret_cast<const float4*>(hp));
      float dt, dA;
      ssm_dt_dA(bf16_to_f32(__ldcg(sa.dt + h)), __ldg(sa.dt_bias + h), __ldg(sa.A_log + h), dt, dA);
      const float xv = bf16_to_f32(__ldcg(sa.x + (size_t)h * sa.P + p));
      const uint2 bu = __ldcg(reinterpret_cast<const uint2*>(sa.Bm + (size_t)gi * sa.N + n4));
      const uint2 cu = __ldcg(reinterpret_cast<const uint2*>(sa.Cm + (size_t)gi * sa.N + n4));
      const float4 Bv = make_float4(bf16lo(bu.x), bf16hi(bu.x), bf16lo(bu.y), bf16hi(bu.y));
      const float4 Cv = make_float4(bf16lo(cu.x), bf16hi(cu.x), bf16lo(cu.y), bf16hi(cu.y));
      const float dtx = dt * xv;
      hv.x = fmaf(dA, hv.x, dtx * Bv.x);
      hv.y = fmaf(dA, hv.y, dtx * Bv.y);
      hv.z = fmaf(dA, hv.z, dtx * Bv.z);
      hv.w = fmaf(dA, hv.w, dtx * Bv.w);
      if (live) *reinterpret_cast<float4*>(hp) = hv;
      float yp = Cv.x * hv.x + Cv.y * hv.y + Cv.z * hv.z + Cv.w * hv.w;
      for (int o = lpr / 2; o > 0; o >>= 1) yp += __shfl_xor_sync(0xffffffffu, yp, o);
      if (live && (lane % lpr) == 0) sa.y[(size_t)h * sa.P + p] = yp + __ldg(sa.D + h) * xv;
    }
    if (blockIdx.x == 0 && tid == 0 && sa.pos_inc) sa.pos_inc[0] += 1;  // every CTA has read it
  }
  fused_grid_barrier(tid, kC);

  // ---- phase 3: out_proj
  fused_norm_row<FP8>(a3, 0, act_s, tot, tail->unscale, tid, kC);
  for (int i = tid; i < rows_out * kMmaWarps; i += kC) tot[i] = 0.0f;
  named_bar(1, kC);
  if (!dead && !mma_consume<FP8>(a3, p3, p1.nst, S, stg, tail, act_s, tot, rows_out, warp, lane)) dead = true;
  if (bulk3 && !dead && !mbar_wait(&tail->epi_bar2, 0)) dead = true;
  __syncthreads();  // all consumers and the producer (after its drain)
  {
    const float us = tail->unscale[0];
    for (int r = tid; r < p3.nrows; r += kC) {
      float sum = 0.0f;
#pragma unroll
      for (int w = 0; w < kMmaWarps; ++w) sum += tot[(size_t)w * rows_out + r];
      a3.out[p3.row_begin + r] = f32_to_bf16(bf16_to_f32(rsS[r]) + sum * us);
    }
  }
}

// The chunking gemv_mma_kernel's launch picks for projection a at batch 1.
static void chain_chunking(const GemvArgs& a, int es, int& kc, int& whole) {
  const int nrg = (a.N + kMmaRows - 1) / kMmaRows;
  int grid = num_sms();
  if (grid > nrg) grid = nrg;
  const int rows_max = ((nrg + grid - 1) / grid) * kMmaRows;
  const MmaLayout lay = mma_layout(a.K, es, rows_max, 1, a.epi, a.dconv);
  kc = lay.kc;
  whole = lay.whole ? 1 : 0;
}

bool decode_fused_supported(const FusedStepArgs& fa, bool fp8) {
  const GemvArgs& a1 = fa.in;
  const GemvArgs& a3 = fa.out;
  const SsmArgs& s = fa.ssm;
  if (a1.M != 1 || a3.M != 1 || !gemv_mma_supported(1, a1.K) || !gemv_mma_supported(1, a3.K)) return false;
  if (a1.epi != EPI_INPROJ_CONV || a3.epi != EPI_RESID || a1.norm != NORM_RMS || a3.norm != NORM_GATED) return false;
  if (a1.dconv < 2 || s.B != 1 || s.N % 4 != 0 || s.N < 4 || s.N > 128 || ((s.N / 4) & (s.N / 4 - 1)) != 0) return false;
  if (s.G < 1 || s.H % s.G != 0) return false;
  int coop = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess)
    return false;
  if (!coop) return false;
  const int G = num_sms();
  const int rin = (((a1.N + kMmaRows - 1) / kMmaRows + G - 1) / G) * kMmaRows;
  const int rout = (((a3.N + kMmaRows - 1) / kMmaRows + G - 1) / G) * kMmaRows;
  const FusedLayout lay = fused_layout(a1.K, a3.K, rin, rout, a1.dconv);
  int kc, whole;
  for (const GemvArgs* g : {&a1, &a3}) {  // a stage of the stand-alone chunking fits the ring stride
    chain_chunking(*g, fp8 ? 1 : 2, kc, whole);
    const int sb = whole ? kMmaRows * g->K * (fp8 ? 1 : 2) : kMmaRows * (kc + kRowPad);
    if (sb > kFusedStride) return false;
  }
  return lay.stages >= 2 && lay.total <= 227 * 1024;
}

// Per device: whether the cooperative launch accepts the PDL attribute (-1
// untried, 1 yes, 0 cooperative alone) and the occupancy probed for a layout.
struct FusedLaunchInfo {
  int pdl_mode = -1;
  int occ_smem = -1;
  int occ_blocks = 0;
};
static std::mutex g_fused_mu;

template <bool FP8>
static cudaError_t launch_fused_one(const FusedStepArgs& fa, cudaStream_t st) {
  static int done_mask[64] = {0};
  static FusedLaunchInfo info[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_fused_mu);
  FusedLaunchInfo& fi = info[dev];
  const int G = num_sms();
  const int rin = (((fa.in.N + kMmaRows - 1) / kMmaRows + G - 1) / G) * kMmaRows;
  const int rout = (((fa.out.N + kMmaRows - 1) / kMmaRows + G - 1) / G) * kMmaRows;
  const FusedLayout lay = fused_layout(fa.in.K, fa.out.K, rin, rout, fa.in.dconv);
  if (lay.stages < 2 || lay.total > 227 * 1024) return cudaErrorInvalidConfiguration;
  auto kern = decode_step_fused_kernel<FP8>;
  cudaError_t e = set_smem_once((const void*)kern, lay.total, done_mask);
  if (e != cudaSuccess) return e;
  if (fi.occ_smem != lay.total) {  // all CTAs must be resident at once
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fi.occ_blocks, kern, kMmaThreads, lay.total)) !=
        cudaSuccess)
      return e;
    fi.occ_smem = lay.total;
  }
  if (fi.occ_blocks < 1) return cudaErrorCooperativeLaunchTooLarge;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(kMmaThreads);
  cfg.dynamicSmemBytes = lay.total;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  trace_pre(K_DECODE_FUSED, st);
  cfg.numAttrs = fi.pdl_mode == 0 ? 1 : 2;
  FusedChunks ck;
  chain_chunking(fa.in, FP8 ? 1 : 2, ck.kc_in, ck.whole_in);
  chain_chunking(fa.out, FP8 ? 1 : 2, ck.kc_out, ck.whole_out);
  e = cudaLaunchKernelEx(&cfg, kern, fa, rin, rout, ck);
  if (e != cudaSuccess && fi.pdl_mode == -1) {
    cudaGetLastError();  // the attribute pair was refused: cooperative alone from now on
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, fa, rin, rout, ck);
    if (e == cudaSuccess) fi.pdl_mode = 0;
  } else if (e == cudaSuccess && fi.pdl_mode == -1) {
    fi.pdl_mode = 1;
  }
  trace_post(K_DECODE_FUSED, st);
  return e;
}

cudaError_t launch_decode_fused(const FusedStepArgs& fa, bool fp8, cudaStream_t s) {
  return fp8 ? launch_fused_one<true>(fa, s) : launch_fused_one<false>(fa, s);
}

int status_gemv_mma(int clear) { return tu_status(clear); }

cudaError_t wait_limit_gemv_mma(long long cycles) { return tu_set_wait_limit(cycles); }

}  // namespace m2
