// k_gemv_mma.cu -- decode GEMV (batch <= 8) on warp-level MMA, weights
// streamed straight from HBM into registers.
//
// Same contract as the CUDA-core GEMV in k_gemv.cu (GemvArgs: w8a16 E4M3
// block-scaled or bf16 weights, plain or prepared activations, store /
// residual / conv-update epilogue), for K % 64 == 0, K <= 8192 and up to 8
// batch rows.  The GEMV is HBM-bound; the MMA only replaces the per-weight
// multiply-adds: one m16n8k16 instruction consumes 256 weights (16 rows x 16
// k), so a weight costs well under one instruction (its half of an exact
// E4M3->f16x2 conversion plus a share of the load and the MMA) instead of ~4
// on the FMA pipes, and the 8 MMA columns carry up to 8 batch rows for free.
//
// One CTA (16 warps) per SM over a contiguous range of 16-row groups.  Warp w
// owns a k-slice of every row (a run of 64-element groups).  Lane (g, t) =
// (lane/4, lane%4) loads, per group, the 16 weight bytes [16t, 16t+16) of rows
// g and g+8 with one 128-bit load each (4 lanes cover a row's 64 contiguous
// bytes), converts them to the A fragments and issues 4 MMAs; the k order
// inside a group is permuted identically for A and B, which a dot product
// allows.  Loads for the next unit of work are issued before the current one
// is computed (two register buffers), so each warp keeps 8 x 16 B per lane in
// flight, and L2 prefetches run four units further ahead.  Activations (f16
// with the exact per-row prescale for E4M3, or bf16) sit in shared memory;
// E4M3 partials are scaled per 128-element block; each warp leaves its 16 x MB
// tile per row group in shared memory, and at the end all threads add the 16
// warps' tiles in a fixed order (deterministic) and run the epilogue.
#include <cuda_runtime.h>
#include <stdint.h>

#include "m2_common.cuh"
#include "m2_kernels.h"

namespace m2 {

constexpr int kMmaWarps = 16;
constexpr int kMmaThreads = kMmaWarps * 32;  // 512
constexpr int kMmaRows = 16;                 // rows per group (MMA M)
// Weight matrices up to this size are prefetched into L2 whole at launch.
constexpr size_t kSlabPrefetchMax = 96ull << 20;

struct MmaTail {
  unsigned amax[8];
  float unscale[8];
  int32_t pos[8];
};

struct MmaLayout {
  int act_ld, tail, act, tot, epi, total;
};
// act_ld: elements per activation row in shared memory (K + 8 pads the rows
// onto different banks).
__host__ __device__ inline MmaLayout mma_layout(int K, int rows_max, int mb, int kb, int epi, int dconv) {
  MmaLayout L;
  L.act_ld = K + 8;
  L.tail = 0;
  L.act = (int)((sizeof(MmaTail) + 127) / 128 * 128);
  L.tot = L.act + ((mb + 1) * L.act_ld * 2 + 15) / 16 * 16;  // + one zero row for lanes past the batch
  (void)kb;
  L.epi = L.tot + (rows_max * kMmaWarps * mb * 4 + 15) / 16 * 16;  // per-warp partials
  int epi_bytes = 0;
  if (epi == EPI_INPROJ_CONV) epi_bytes = rows_max * (dconv + 1) * 2 + mb * rows_max * (dconv - 1) * 2;
  if (epi == EPI_RESID) epi_bytes = mb * rows_max * 2;
  L.total = L.epi + (epi_bytes + 15) / 16 * 16;
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

// 64-element groups per unit of work: 4 for E4M3 (16 bytes per lane per row
// and group), 2 for bf16 (32 bytes), so that a unit's weights take 32
// registers per lane in both cases.
template <bool FP8>
struct Unit {
  static constexpr int kGroups = FP8 ? 4 : 2;
};
// Weight registers of one unit: kGroups groups x rows {g, g+8}.
template <bool FP8>
struct WBuf {
  uint4 r0[4];
  uint4 r8[4];
};

template <bool FP8, int MB>
__global__ void __launch_bounds__(kMmaThreads, 1)
    gemv_mma_kernel(const GemvArgs a, int rows_max) {
  constexpr int ES = FP8 ? 1 : 2;  // bytes per weight
  constexpr int kMmaUnit = Unit<FP8>::kGroups;
  extern __shared__ __align__(128) uint8_t smem[];
  const int kb = (a.K + 127) / 128;
  const MmaLayout lay = mma_layout(a.K, rows_max, MB, kb, a.epi, a.dconv);
  MmaTail* tail = reinterpret_cast<MmaTail*>(smem + lay.tail);
  uint16_t* act_s = reinterpret_cast<uint16_t*>(smem + lay.act);  // [MB + 1][act_ld]
  float* tot = reinterpret_cast<float*>(smem + lay.tot);
  uint8_t* epi_s = smem + lay.epi;

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
  // this warp's 64-element groups [q0, q1) of every row, processed in units
  const int ngrp = a.K / 64;
  const int q0 = (ngrp * warp) / kMmaWarps, q1 = (ngrp * (warp + 1)) / kMmaWarps;
  const int nunit_rg = (q1 - q0 + kMmaUnit - 1) / kMmaUnit;  // units per row group
  const int nunit = nunit_rg * nrg;

  const uint8_t* W = static_cast<const uint8_t*>(a.W);
  // loads of unit u into buffer b (rows past N load row N-1; groups past q1 load nothing)
  auto load_unit = [&](int u, WBuf<FP8>& b) {
    const int rg = rg_begin + u / nunit_rg;
    const int qb = q0 + (u % nunit_rg) * kMmaUnit;
    const int r0 = min(rg * kMmaRows + g, a.N - 1), r8 = min(rg * kMmaRows + g + 8, a.N - 1);
    const uint8_t* p0 = W + ((size_t)r0 * a.K + (size_t)qb * 64 + 16 * t) * ES;
    const uint8_t* p8 = W + ((size_t)r8 * a.K + (size_t)qb * 64 + 16 * t) * ES;
#pragma unroll
    for (int i = 0; i < kMmaUnit; ++i) {
      if (qb + i < q1) {
#pragma unroll
        for (int h = 0; h < ES; ++h) {
          b.r0[i * ES + h] = __ldcs(reinterpret_cast<const uint4*>(p0 + (size_t)i * 64 * ES) + h);
          b.r8[i * ES + h] = __ldcs(reinterpret_cast<const uint4*>(p8 + (size_t)i * 64 * ES) + h);
        }
      }
    }
  };
  // L2 prefetch of a whole unit (16 rows x the unit's k-range), one bulk
  // prefetch per row from lanes 0..15: keeps HBM busy beyond the two register
  // buffers, including while the prologue below waits and stages.
  auto prefetch_unit = [&](int u) {
    if (u >= nunit || lane >= kMmaRows) return;
    const int rg = rg_begin + u / nunit_rg;
    const int qb = q0 + (u % nunit_rg) * kMmaUnit;
    const int ng = min(kMmaUnit, q1 - qb);
    const int r = min(rg * kMmaRows + lane, a.N - 1);
    const uint8_t* p = W + ((size_t)r * a.K + (size_t)qb * 64) * ES;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"((uint32_t)(ng * 64 * ES)) : "memory");
  };
  constexpr int kPrefetchUnits = 4;
  WBuf<FP8> buf0, buf1;  // two named buffers: register arrays must be indexed statically
  if (nunit > 0) load_unit(0, buf0);  // weights never depend on the previous kernel
  // L2 prefetch: a weight matrix that fits comfortably in L2 is requested
  // whole at launch (this CTA's contiguous rows, 32 KB per request), so HBM
  // streams at full rate while this kernel waits for its activations and the
  // register loads then hit L2; larger matrices are prefetched a few units
  // ahead of each warp instead.
  const bool whole = (size_t)a.N * a.K * ES <= kSlabPrefetchMax;
  if (whole) {
    const size_t slab0 = (size_t)row_begin * a.K * ES, slab = (size_t)nrows * a.K * ES;
    for (size_t off = (size_t)tid * 32768; off < slab; off += (size_t)kMmaThreads * 32768) {
      const uint32_t n = (uint32_t)(slab - off < 32768 ? slab - off : 32768);
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(W + slab0 + off), "r"(n) : "memory");
    }
  } else {
    for (int u = 1; u <= kPrefetchUnits; ++u) prefetch_unit(u);
  }

  // ------------------------------------------------ prologue
  // Epilogue inputs of this CTA's rows.  Under programmatic dependent launch
  // they come from launches before the immediately preceding kernel, which have
  // completed by now, so they are staged before the wait (L2 loads: not L1).
  if (tid < 8) tail->pos[tid] = (a.epi == EPI_INPROJ_CONV && tid < mvalid) ? __ldcg(a.pos + tid) : 0;
  if (a.epi == EPI_INPROJ_CONV) {
    uint16_t* cw = reinterpret_cast<uint16_t*>(epi_s);  // [rows_max][dconv+1]
    uint16_t* rgs = cw + (size_t)rows_max * (a.dconv + 1);  // [MB][L][rows_max]
    for (int r = tid; r < nrows; r += kMmaThreads) {
      const int n = row_begin + r;
      if (n < a.xbc0 || n >= a.xbc0 + a.d_xbc) continue;
      const int c = n - a.xbc0;
      uint16_t wv[9];
#pragma unroll
      for (int j = 0; j < 8; ++j) wv[j] = j < a.dconv ? __ldg(a.conv_w + (size_t)c * a.dconv + j) : (uint16_t)0;
      wv[8] = a.conv_b ? __ldg(a.conv_b + c) : (uint16_t)0;
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        if (m < mvalid) {
          const int p = __ldcg(a.pos + m);
          const uint16_t* ring = a.ring + (size_t)m * L * a.d_xbc;
          uint16_t rv[7];
#pragma unroll
          for (int j = 0; j < 7; ++j) rv[j] = j < L ? __ldcg(ring + (size_t)((p + j) % L) * a.d_xbc + c) : (uint16_t)0;
#pragma unroll
          for (int j = 0; j < 7; ++j)
            if (j < L) rgs[((size_t)m * L + j) * rows_max + r] = rv[j];
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < a.dconv) cw[r * (a.dconv + 1) + j] = wv[j];
      cw[r * (a.dconv + 1) + a.dconv] = wv[8];
    }
  } else if (a.epi == EPI_RESID) {
    uint16_t* rs = reinterpret_cast<uint16_t*>(epi_s);  // [MB][rows_max]
    for (int i = tid; i < nrows * mvalid; i += kMmaThreads) {
      const int m = i / nrows, r = i % nrows;
      rs[m * rows_max + r] = __ldcg(a.resid + (size_t)m * a.ldr + row_begin + r);
    }
  }
  pdl_wait();
  pdl_trigger();
  for (int i = tid; i < rows_max * kMmaWarps * MB; i += kMmaThreads) tot[i] = 0.0f;
  if (tid < 8) tail->amax[tid] = 0u;
  __syncthreads();
  // activations -> shared memory (coherent loads: written by the previous kernel)
  const int kv = a.K / 8;  // 16-byte vectors per row
  for (int i = tid; i < (MB + 1) * kv; i += kMmaThreads) {
    const int m = i / kv, k8 = (i % kv) * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (m < mvalid) v = *reinterpret_cast<const uint4*>(a.A + (size_t)m * a.lda + k8);
    if (FP8 && a.act == ACT_PLAIN && m < mvalid) {
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
      float mx = 0.0f;
#pragma unroll
      for (int e = 0; e < 4; ++e) mx = fmaxf(mx, fmaxf(fabsf(bf16lo(w4[e])), fabsf(bf16hi(w4[e]))));
      atomicMax(&tail->amax[m], __float_as_uint(mx));
    }
    *reinterpret_cast<uint4*>(act_s + (size_t)m * lay.act_ld + k8) = v;
  }
  __syncthreads();
  if (FP8 && a.act == ACT_PLAIN) {
    // plain bf16 rows: per-row prescale into the f16 range, converted in place
    for (int i = tid; i < mvalid * kv; i += kMmaThreads) {
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
  __syncthreads();

  // ------------------------------------------------ main loop
  const uint16_t* act_g = act_s + (size_t)(g < mvalid ? g : MB) * lay.act_ld;  // zero row past the batch
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  auto process = [&](int u, const WBuf<FP8>& cur) {
    const int rg = rg_begin + u / nunit_rg;
    const int qb = q0 + (u % nunit_rg) * kMmaUnit;
#pragma unroll
    for (int i = 0; i < kMmaUnit; ++i) {
      const int q = qb + i;
      if (q < q1) {
        const uint4 bl = *reinterpret_cast<const uint4*>(act_g + q * 64 + 16 * t);
        const uint4 bh = *reinterpret_cast<const uint4*>(act_g + q * 64 + 16 * t + 8);
        const uint32_t bw[8] = {bl.x, bl.y, bl.z, bl.w, bh.x, bh.y, bh.z, bh.w};
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (FP8) {
          const uint32_t w0[4] = {cur.r0[i].x, cur.r0[i].y, cur.r0[i].z, cur.r0[i].w};
          const uint32_t w8[4] = {cur.r8[i].x, cur.r8[i].y, cur.r8[i].z, cur.r8[i].w};
#pragma unroll
          for (int sp = 0; sp < 4; ++sp)
            mma16816<FP8>(d, cvt_e4m3x2(w0[sp]), cvt_e4m3x2(w8[sp]), cvt_e4m3x2(w0[sp] >> 16),
                          cvt_e4m3x2(w8[sp] >> 16), bw[2 * sp], bw[2 * sp + 1]);
          // one 128-element scale block per group; rows g and g+8 may sit in different n-blocks
          const int kbk = q >> 1;
          const int r0 = min(rg * kMmaRows + g, row_end - 1), r8 = min(rg * kMmaRows + g + 8, row_end - 1);
          const float s0 = bf16_to_f32(__ldg(a.S + (size_t)(r0 >> 7) * kb + kbk));  // read-only: L1 hits
          const float s8 = bf16_to_f32(__ldg(a.S + (size_t)(r8 >> 7) * kb + kbk));
          acc[0] = fmaf(d[0], s0, acc[0]);
          acc[1] = fmaf(d[1], s0, acc[1]);
          acc[2] = fmaf(d[2], s8, acc[2]);
          acc[3] = fmaf(d[3], s8, acc[3]);
        } else {
          const uint32_t w0[8] = {cur.r0[2 * i].x, cur.r0[2 * i].y, cur.r0[2 * i].z, cur.r0[2 * i].w,
                                  cur.r0[2 * i + 1].x, cur.r0[2 * i + 1].y, cur.r0[2 * i + 1].z, cur.r0[2 * i + 1].w};
          const uint32_t w8[8] = {cur.r8[2 * i].x, cur.r8[2 * i].y, cur.r8[2 * i].z, cur.r8[2 * i].w,
                                  cur.r8[2 * i + 1].x, cur.r8[2 * i + 1].y, cur.r8[2 * i + 1].z, cur.r8[2 * i + 1].w};
#pragma unroll
          for (int sp = 0; sp < 4; ++sp)
            mma16816<FP8>(d, w0[2 * sp], w8[2 * sp], w0[2 * sp + 1], w8[2 * sp + 1], bw[2 * sp], bw[2 * sp + 1]);
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[j] += d[j];
        }
      }
    }
    if ((u % nunit_rg) == nunit_rg - 1) {
      // row group done: this warp's 16 x MB tile goes to its own slots; the
      // epilogue adds the 16 warps in a fixed order (deterministic results)
      const int lr = (rg - rg_begin) * kMmaRows;
      const int c0 = 2 * t, c1 = 2 * t + 1;
      float* t0 = tot + ((size_t)(lr + g) * kMmaWarps + warp) * MB;
      float* t8 = tot + ((size_t)(lr + g + 8) * kMmaWarps + warp) * MB;
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
  };
  // loads of the next unit are in flight while the current one is computed
  for (int u = 0; u < nunit; u += 2) {
    if (u + 1 < nunit) load_unit(u + 1, buf1);
    if (!whole) prefetch_unit(u + 1 + kPrefetchUnits);
    process(u, buf0);
    if (u + 1 < nunit) {
      if (u + 2 < nunit) load_unit(u + 2, buf0);
      if (!whole) prefetch_unit(u + 2 + kPrefetchUnits);
      process(u + 1, buf1);
    }
  }
  __syncthreads();

  // ------------------------------------------------ epilogue (all threads)
  const uint16_t* cw = reinterpret_cast<const uint16_t*>(epi_s);
  const uint16_t* rgp = cw + (size_t)rows_max * (a.dconv + 1);
  for (int i = tid; i < nrows * mvalid; i += kMmaThreads) {
    const int r = i / mvalid, m = i % mvalid;
    const int n = row_begin + r;
    float sum = 0.0f;
#pragma unroll
    for (int w = 0; w < kMmaWarps; ++w) sum += tot[((size_t)r * kMmaWarps + w) * MB + m];
    const float accv = sum * tail->unscale[m];
    uint16_t* o = a.out + (size_t)m * a.ldo + n;
    if (a.epi == EPI_RESID) {
      const float res = bf16_to_f32(reinterpret_cast<const uint16_t*>(epi_s)[m * rows_max + r]);
      *o = f32_to_bf16(res + accv);
    } else if (a.epi == EPI_INPROJ_CONV && n >= a.xbc0 && n < a.xbc0 + a.d_xbc) {
      // conv1d update with bias + SiLU; this thread alone owns (sequence m,
      // channel c) in this call, and the ring taps were staged before any write
      const uint16_t vb = f32_to_bf16(accv);  // rounding point of the in_proj output
      const int c = n - a.xbc0;
      const uint16_t* w = cw + r * (a.dconv + 1);
      float s = bf16_to_f32(w[a.dconv]);
      for (int j = 0; j < L; ++j) s += bf16_to_f32(w[j]) * bf16_to_f32(rgp[((size_t)m * L + j) * rows_max + r]);
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
  int grid = num_sms();
  if (grid > nrg) grid = nrg;
  const int rows_max = ((nrg + grid - 1) / grid) * kMmaRows;
  const int kb = (a.K + 127) / 128;
  const MmaLayout lay = mma_layout(a.K, rows_max, MB, kb, a.epi, a.dconv);
  if (lay.total > 227 * 1024) return cudaErrorInvalidConfiguration;
  auto kern = gemv_mma_kernel<FP8, MB>;
  cudaError_t e = set_smem_once((const void*)kern, lay.total, done_mask);
  if (e != cudaSuccess) return e;
  const int id = (FP8 ? K_GEMV_FP8 : K_GEMV_BF16) + (a.epi == EPI_INPROJ_CONV ? 1 : (a.epi == EPI_RESID ? 2 : 0));
  trace_pre(id, s);
  e = launch_k(kern, dim3(grid), dim3(kMmaThreads), lay.total, s, a.pdl != 0, a, rows_max);
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

int status_gemv_mma(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return -4;
  if (clear) {
    const int z = 0;
    cudaMemcpyToSymbol(g_status, &z, sizeof(int));
  }
  return v;
}

}  // namespace m2
