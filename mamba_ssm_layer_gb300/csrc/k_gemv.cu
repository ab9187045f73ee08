// k_gemv.cu -- CUDA-core w8a16 / bf16 GEMV for small batches (decode).
//
// Computes out[m][n] = sum_k A[m][k] * W~[n][k] with W~ = E4M3(W)*S[n/128][k/128]
// (page "Struct Qwen3SsmLayer", `set_fp8_decode_weights`; scale index of
// "Struct NemotronMamba2Layer", `set_fp8_weights`) or W~ = bf16 W (native BF16
// projections).  The decode GEMV is HBM-bound: every weight byte is read once
// per call, so the design keeps ~180 KB of weight reads in flight per SM and
// keeps every latency (activation prologue, reductions, epilogue inputs) off
// the streaming loop.
//
// One CTA per SM, persistent over a contiguous range of rows:
//   warp 16     producer: one lane streams R whole weight rows per stage
//               (R*K contiguous bytes) into a shared-memory ring with 1-D bulk
//               copies (cp.async.bulk, mbarrier completion, L2 evict-first);
//   warps 0..15 consumers, two groups of 8 warps that take alternate stages
//               (two warps per scheduler per group hide the load/convert/FMA
//               latencies): thread t of a group owns the 16-byte chunks t,
//               t+256, ... of every row, so its activations stay in registers
//               for the whole call.  Per row a thread
//               forms 16-element partial dot products, multiplies each by the
//               chunk's block scale and accumulates; per stage the R*MB sums
//               are reduced with a transposing warp butterfly and handed to
//               the helper through a shared-memory slot;
//   warp 17     helper: stages the block scales and the epilogue inputs (conv
//               taps and ring, residual) into shared memory, then adds the 8
//               warps' partials of every stage into the row totals.
// After the loop all threads run the epilogue (store / residual add / the
// conv1d update with bias and SiLU) from shared memory.
// E4M3 is decoded in registers with the exact hardware E4M3->f16 conversion
// and multiplied by f16 activations with fp32 accumulation (fma.rn.f32.f16).
#include <cuda_runtime.h>
#include <stdint.h>

#include "m2_common.cuh"
#include "m2_kernels.h"

namespace m2 {

constexpr int kGemvConsumerWarps = 8;                    // warps per consumer group
constexpr int kGemvGroups = 2;                           // groups take alternate stages
constexpr int kGemvConsumers = kGemvConsumerWarps * 32;  // 256 threads per group
constexpr int kGemvAllConsumers = kGemvGroups * kGemvConsumers;
constexpr int kGemvProducerWarp = kGemvGroups * kGemvConsumerWarps;  // warp 16
constexpr int kGemvHelperWarp = kGemvProducerWarp + 1;               // warp 17
constexpr int kGemvThreads = kGemvAllConsumers + 64;                 // 576
constexpr int kGemvStageBudget = 184320;                 // bytes of weight ring
constexpr int kGemvMaxStages = 8;
constexpr int kGemvSlots = 4;                            // reduction slots

struct GemvSmemTail {
  uint64_t full[kGemvMaxStages];
  uint64_t empty[kGemvMaxStages];
  uint64_t red_full[kGemvSlots];
  uint64_t red_empty[kGemvSlots];
  float red[kGemvSlots][kGemvConsumerWarps][32];
  unsigned amax[4];           // max |activation| per batch row (float bits)
  float unscale[4];           // 2^-j undoing the f16 prescale of row m
};

// Mixed-precision multiply-add with fp32 accumulation (a*b+c, one rounding):
// two f16 (or bf16) pairs against two fp32 chains.
__device__ __forceinline__ void fma2_f16(uint32_t w2, uint32_t a2, float& c0, float& c1) {
  asm("{\n\t.reg .f16 wl, wh, al, ah;\n\tmov.b32 {wl, wh}, %2;\n\tmov.b32 {al, ah}, %3;\n\t"
      "fma.rn.f32.f16 %0, wl, al, %0;\n\tfma.rn.f32.f16 %1, wh, ah, %1;\n\t}"
      : "+f"(c0), "+f"(c1)
      : "r"(w2), "r"(a2));
}
__device__ __forceinline__ void fma2_bf16(uint32_t w2, uint32_t a2, float& c0, float& c1) {
  asm("{\n\t.reg .b16 wl, wh, al, ah;\n\tmov.b32 {wl, wh}, %2;\n\tmov.b32 {al, ah}, %3;\n\t"
      "fma.rn.f32.bf16 %0, wl, al, %0;\n\tfma.rn.f32.bf16 %1, wh, ah, %1;\n\t}"
      : "+f"(c0), "+f"(c1)
      : "r"(w2), "r"(a2));
}
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  return h2;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

template <bool FP8>
struct WTraits;
template <>
struct WTraits<true> {
  static constexpr int kEpc = 16;  // elements per 16-byte chunk
  static constexpr int kEsize = 1;
};
template <>
struct WTraits<false> {
  static constexpr int kEpc = 8;
  static constexpr int kEsize = 2;
};

template <int V>
struct Log2 {
  static constexpr int value = 1 + Log2<V / 2>::value;
};
template <>
struct Log2<1> {
  static constexpr int value = 0;
};

// One level of the transposing warp reduction: lanes with bit `O` set keep the
// upper half of the CNT live values, the others the lower half, each adding
// the partner lane's copy of the half it keeps.  Once one value is left the
// remaining levels are plain xor-reductions.  Afterwards lane l holds the warp
// total of value index l >> (5 - log2(CNT)).
template <int CNT, int O>
struct Butterfly {
  static __device__ __forceinline__ void run(float* v, int lane) {
    if constexpr (CNT > 1) {
      const bool upper = (lane & O) != 0;
#pragma unroll
      for (int i = 0; i < CNT / 2; ++i) {
        const float send = upper ? v[i] : v[i + CNT / 2];
        const float keep = upper ? v[i + CNT / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
      }
      if constexpr (O > 1) Butterfly<CNT / 2, O / 2>::run(v, lane);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
      if constexpr (O > 1) Butterfly<1, O / 2>::run(v, lane);
    }
  }
};

// Shared-memory layout beyond the weight ring (offsets in bytes, host and
// device agree through this function).
struct GemvLayout {
  int tail, sc, tot, epi, total;
};
__host__ __device__ inline GemvLayout gemv_layout(int stages, int stage_bytes, int rows_max, int mb, int kb,
                                                  int epi, int dconv) {
  GemvLayout L;
  L.tail = stages * stage_bytes;
  L.sc = L.tail + (int)((sizeof(GemvSmemTail) + 15) / 16 * 16);
  const int nbs = rows_max / 128 + 2;  // n-blocks a row range can touch
  L.tot = L.sc + (nbs * kb * 4 + 15) / 16 * 16;
  L.epi = L.tot + (rows_max * mb * 4 + 15) / 16 * 16;
  int epi_bytes = 0;
  if (epi == EPI_INPROJ_CONV) epi_bytes = rows_max * (dconv + 1) * 2 + mb * rows_max * (dconv - 1) * 2 + 16 * 4;
  if (epi == EPI_RESID) epi_bytes = mb * rows_max * 2;
  L.total = L.epi + (epi_bytes + 15) / 16 * 16;
  return L;
}

template <bool FP8, int MB, int CPT, int R>
__global__ void __launch_bounds__(kGemvThreads, 1)
    gemv_kernel(const GemvArgs a, int m0, int stages, int rows_max) {
  using T = WTraits<FP8>;
  constexpr int V = R * MB;
  constexpr int LOGV = Log2<V>::value;
  static_assert((1 << LOGV) == V && V <= 32, "R*MB must be a power of two <= 32");

  extern __shared__ __align__(128) uint8_t smem[];
  const int rowbytes = a.K * T::kEsize;
  const int stage_bytes = R * rowbytes;
  const int kb = (a.K + 127) / 128;
  const GemvLayout lay = gemv_layout(stages, stage_bytes, rows_max, MB, kb, a.epi, a.dconv);
  GemvSmemTail* tail = reinterpret_cast<GemvSmemTail*>(smem + lay.tail);
  float* sc = reinterpret_cast<float*>(smem + lay.sc);
  float* tot = reinterpret_cast<float*>(smem + lay.tot);
  uint8_t* epi_s = smem + lay.epi;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  const int row_begin = (int)(((long long)a.N * blockIdx.x) / G);
  const int row_end = (int)(((long long)a.N * (blockIdx.x + 1)) / G);
  const int nrows = row_end - row_begin;
  const int niter = (nrows + R - 1) / R;
  const int nchunks = rowbytes / 16;
  const int mvalid = min(MB, a.M - m0);
  const int nb0 = row_begin >> 7;
  const int L = a.dconv - 1;

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&tail->full[s], 1);
      mbar_init(&tail->empty[s], kGemvConsumerWarps);
    }
    for (int s = 0; s < kGemvSlots; ++s) {
      mbar_init(&tail->red_full[s], kGemvConsumerWarps);
      mbar_init(&tail->red_empty[s], 1);
    }
    for (int m = 0; m < 4; ++m) tail->amax[m] = 0u;
    fence_mbar_init();
  }
  __syncthreads();

  const uint64_t pol = a.evict_first ? policy_evict_first() : policy_evict_normal();
  const uint8_t* wbase = static_cast<const uint8_t*>(a.W) + (size_t)row_begin * rowbytes;
  // the producer puts the first stages in flight before anything else: weights
  // do not depend on the previous kernel
  if (warp == kGemvProducerWarp && lane == 0) {
    for (int it = 0; it < niter && it < stages; ++it) {
      const int rows = min(R, nrows - it * R);
      const uint32_t bytes = (uint32_t)(rows * rowbytes);
      mbar_arrive_expect_tx(&tail->full[it], bytes);
      bulk_g2s(smem + (size_t)it * stage_bytes, wbase + (size_t)it * R * rowbytes, bytes, &tail->full[it], pol);
    }
  }
  if (warp == kGemvHelperWarp && FP8) {
    // block scales of the n-blocks this row range touches, as fp32
    const int nbs = ((row_end - 1) >> 7) - nb0 + 1;
    for (int i = lane; i < nbs * kb; i += 32)
      sc[i] = bf16_to_f32(__ldg(a.S + (size_t)(nb0 + i / kb) * kb + (i % kb)));
  }

  // ------------------------------------------------ activation prologue
  // Activations are cached in registers as packed pairs: f16 for E4M3
  // weights (E4M3 -> f16 is exact, and the products then run as
  // fma.rn.f32.f16 at full FFMA rate), bf16 for bf16 weights.  f16 rows carry
  // an exact power-of-two prescale 2^j that puts the row maximum in
  // [2^14, 2^15): every bf16 value within 2^31 of the row maximum is then
  // exactly representable; 2^-j is applied to the row totals.  Prepared
  // activations (ACT_PREPARED) arrive in that form; plain bf16 rows are
  // converted here.
  uint32_t acth[MB][CPT][T::kEpc / 2];
  const int grp = warp / kGemvConsumerWarps;  // consumer group (consumers only)
  const int gtid = tid % kGemvConsumers;      // thread index within the group
  const int gwarp = warp % kGemvConsumerWarps;
  if (warp < kGemvGroups * kGemvConsumerWarps) {
    pdl_wait();  // A comes from the previous kernel
#pragma unroll
    for (int m = 0; m < MB; ++m)
#pragma unroll
      for (int j = 0; j < CPT; ++j) {
        const int c = gtid + j * kGemvConsumers;
        if (m < mvalid && c < nchunks) {
          const uint4* src = reinterpret_cast<const uint4*>(a.A + (size_t)(m0 + m) * a.lda + (size_t)c * T::kEpc);
#pragma unroll
          for (int q = 0; q < T::kEpc / 8; ++q) {
            const uint4 v = src[q];  // coherent load: written by the PDL predecessor
            acth[m][j][4 * q] = v.x;
            acth[m][j][4 * q + 1] = v.y;
            acth[m][j][4 * q + 2] = v.z;
            acth[m][j][4 * q + 3] = v.w;
          }
        } else {
#pragma unroll
          for (int e = 0; e < T::kEpc / 2; ++e) acth[m][j][e] = 0u;
        }
      }
    if (a.act == ACT_PREPARED) {
      if (tid < 4) tail->unscale[tid] = tid < mvalid ? a.unscale[m0 + tid] : 1.0f;
    } else if constexpr (FP8) {
      // plain bf16 rows: find each row's prescale, convert to f16
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        float mx = 0.0f;
#pragma unroll
        for (int j = 0; j < CPT; ++j)
#pragma unroll
          for (int e = 0; e < T::kEpc / 2; ++e)
            mx = fmaxf(mx, fmaxf(fabsf(bf16lo(acth[m][j][e])), fabsf(bf16hi(acth[m][j][e]))));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0 && grp == 0) atomicMax(&tail->amax[m], __float_as_uint(mx));
      }
      named_bar(1, kGemvAllConsumers);
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        const unsigned bits = tail->amax[m];
        // amax in [2^e, 2^(e+1)) -> j = 14 - e; zero rows keep j = 0
        const int e = bits ? (int)((bits >> 23) & 0xFF) - 127 : 14;
        const int jx = max(-120, min(120, 14 - e));
        const float up = ldexpf(1.0f, jx);
        if (tid == 0) tail->unscale[m] = ldexpf(1.0f, -jx);
#pragma unroll
        for (int j = 0; j < CPT; ++j)
#pragma unroll
          for (int e2 = 0; e2 < T::kEpc / 2; ++e2)
            acth[m][j][e2] = pack_f16x2(bf16lo(acth[m][j][e2]) * up, bf16hi(acth[m][j][e2]) * up);
      }
    } else {
      if (tid < 4) tail->unscale[tid] = 1.0f;  // bf16 weights use the bf16 rows as they are
    }
  }
  if (warp == kGemvHelperWarp) {
    pdl_wait();  // ring / pos / residual may be written by the previous kernel
    // epilogue inputs of this CTA's rows
    if (a.epi == EPI_INPROJ_CONV) {
      uint16_t* cw = reinterpret_cast<uint16_t*>(epi_s);              // [rows_max][dconv+1]
      uint16_t* rg = cw + (size_t)rows_max * (a.dconv + 1);            // [MB][L][rows_max]
      int32_t* ps = reinterpret_cast<int32_t*>(
          (reinterpret_cast<uintptr_t>(rg + (size_t)MB * L * rows_max) + 3) & ~uintptr_t(3));
      if (lane < MB) ps[lane] = lane < mvalid ? a.pos[m0 + lane] : 0;
      __syncwarp();
      for (int r = lane; r < nrows; r += 32) {
        const int n = row_begin + r;
        if (n < a.xbc0 || n >= a.xbc0 + a.d_xbc) continue;
        const int c = n - a.xbc0;
        for (int j = 0; j < a.dconv; ++j) cw[r * (a.dconv + 1) + j] = a.conv_w[(size_t)c * a.dconv + j];
        cw[r * (a.dconv + 1) + a.dconv] = a.conv_b ? a.conv_b[c] : (uint16_t)0;
        for (int m = 0; m < mvalid; ++m) {
          const int p = ps[m];
          const uint16_t* ring = a.ring + (size_t)(m0 + m) * L * a.d_xbc;
          for (int j = 0; j < L; ++j) rg[((size_t)m * L + j) * rows_max + r] = ring[(size_t)((p + j) % L) * a.d_xbc + c];
        }
      }
    } else if (a.epi == EPI_RESID) {
      uint16_t* rs = reinterpret_cast<uint16_t*>(epi_s);  // [MB][rows_max]
      for (int i = lane; i < nrows * mvalid; i += 32) {
        const int m = i / nrows, r = i % nrows;
        rs[m * rows_max + r] = a.resid[(size_t)(m0 + m) * a.ldr + row_begin + r];
      }
    }
  }
  __syncthreads();  // scales staged; epilogue inputs staged
  pdl_trigger();    // every consumer has passed its wait

  bool dead = false;
  if (warp == kGemvProducerWarp) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      int it = stages;
      for (; it < niter; ++it) {
        const int s = it % stages;
        if (!mbar_wait(&tail->empty[s], ((it / stages) - 1) & 1)) break;  // status recorded
        const int rows = min(R, nrows - it * R);
        const uint32_t bytes = (uint32_t)(rows * rowbytes);
        mbar_arrive_expect_tx(&tail->full[s], bytes);
        bulk_g2s(smem + (size_t)s * stage_bytes, wbase + (size_t)it * R * rowbytes, bytes, &tail->full[s], pol);
      }
      // drain: the copies issued (stages [0, it)) have landed before the CTA
      // may exit, also when the consumers stopped after a timeout
      const int issued = min(it, niter);
      for (int k = max(0, issued - stages); k < issued; ++k)
        if (!mbar_drain(&tail->full[k % stages], (k / stages) & 1)) break;
    }
  } else if (warp == kGemvHelperWarp) {
    // ---------------------------------------------------------- helper
    for (int it = 0; it < niter; ++it) {
      const int slot = it % kGemvSlots;
      // the lanes meet at __syncwarp below: the warp decides together
      if (!dead && !__all_sync(0xffffffffu, mbar_wait(&tail->red_full[slot], (it / kGemvSlots) & 1))) dead = true;
      if (!dead && lane < V) {
        float t = 0.0f;
#pragma unroll
        for (int w = 0; w < kGemvConsumerWarps; ++w) t += tail->red[slot][w][lane];
        tot[(it * R + lane / MB) * MB + (lane % MB)] = t;  // rows beyond nrows land in the padding
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->red_empty[slot]);
    }
  } else {
    // ---------------------------------------------------------- consumers
    for (int it = grp; it < niter; it += kGemvGroups) {
      const int s = it % stages;
      const int row0 = row_begin + it * R;
      const int rows = min(R, nrows - it * R);
      // shuffles and __syncwarp follow: the warp decides together
      if (!dead && !__all_sync(0xffffffffu, mbar_wait(&tail->full[s], (it / stages) & 1))) dead = true;
      const uint8_t* st = smem + (size_t)s * stage_bytes;

      float v[V];
#pragma unroll
      for (int i = 0; i < V; ++i) v[i] = 0.0f;
      if (!dead) {
        // rows past `rows` in a partial last stage compute on stale shared
        // memory; their sums are discarded (the butterfly keeps rows apart)
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int n = min(row0 + r, row_end - 1);
#pragma unroll
          for (int j = 0; j < CPT; ++j) {
            const int c = gtid + j * kGemvConsumers;
            if (c < nchunks) {
              const uint4 wv = *reinterpret_cast<const uint4*>(st + (size_t)r * rowbytes + (size_t)c * 16);
              const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
              float p0[MB], p1[MB];
#pragma unroll
              for (int m = 0; m < MB; ++m) p0[m] = p1[m] = 0.0f;
              if constexpr (FP8) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const uint32_t h2 = e4m3x2_to_f16x2((uint16_t)(w4[e >> 1] >> ((e & 1) * 16)));
#pragma unroll
                  for (int m = 0; m < MB; ++m) fma2_f16(h2, acth[m][j][e], p0[m], p1[m]);
                }
                const float scv = sc[((n >> 7) - nb0) * kb + ((c * 16) >> 7)];
#pragma unroll
                for (int m = 0; m < MB; ++m) v[r * MB + m] = fmaf(p0[m] + p1[m], scv, v[r * MB + m]);
              } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
#pragma unroll
                  for (int m = 0; m < MB; ++m) fma2_bf16(w4[e], acth[m][j][e], p0[m], p1[m]);
#pragma unroll
                for (int m = 0; m < MB; ++m) v[r * MB + m] += p0[m] + p1[m];
              }
            }
          }
        }
      }
      // stage consumed: hand it back to the producer before reducing
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->empty[s]);
      Butterfly<V, 16>::run(v, lane);
      const int slot = it % kGemvSlots;
      if (it >= kGemvSlots && !dead &&
          !__all_sync(0xffffffffu, mbar_wait(&tail->red_empty[slot], ((it / kGemvSlots) - 1) & 1)))
        dead = true;
      if ((lane & ((1 << (5 - LOGV)) - 1)) == 0) tail->red[slot][gwarp][lane >> (5 - LOGV)] = v[0];
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->red_full[slot]);
    }
  }
  __syncthreads();  // all row totals are in shared memory
  if (dead) return;

  // ------------------------------------------------ epilogue (all threads)
  const uint16_t* cw = reinterpret_cast<const uint16_t*>(epi_s);
  const uint16_t* rg = cw + (size_t)rows_max * (a.dconv + 1);
  const int32_t* ps = reinterpret_cast<const int32_t*>(
      (reinterpret_cast<uintptr_t>(rg + (size_t)MB * L * rows_max) + 3) & ~uintptr_t(3));
  for (int i = tid; i < nrows * mvalid; i += kGemvThreads) {
    const int r = i / mvalid, m = i % mvalid;
    const int n = row_begin + r;
    const float acc = tot[r * MB + m] * tail->unscale[m];
    uint16_t* o = a.out + (size_t)(m0 + m) * a.ldo + n;
    if (a.epi == EPI_RESID) {
      const float res = bf16_to_f32(reinterpret_cast<const uint16_t*>(epi_s)[m * rows_max + r]);
      *o = f32_to_bf16(res + acc);
    } else if (a.epi == EPI_INPROJ_CONV && n >= a.xbc0 && n < a.xbc0 + a.d_xbc) {
      // conv1d update with bias + SiLU; this thread alone owns (sequence m,
      // channel c) in this call, and the ring taps were staged before any write
      const uint16_t vb = f32_to_bf16(acc);  // rounding point of the in_proj output
      const int c = n - a.xbc0;
      const uint16_t* w = cw + r * (a.dconv + 1);
      float s = bf16_to_f32(w[a.dconv]);
      for (int j = 0; j < L; ++j) s += bf16_to_f32(w[j]) * bf16_to_f32(rg[((size_t)m * L + j) * rows_max + r]);
      s += bf16_to_f32(w[L]) * bf16_to_f32(vb);
      *o = f32_to_bf16(silu_f(s));
      a.ring[(size_t)(m0 + m) * L * a.d_xbc + (size_t)(ps[m] % L) * a.d_xbc + c] = vb;
    } else {
      *o = f32_to_bf16(acc);
    }
  }
}

template <bool FP8, int MB, int CPT, int R>
static cudaError_t launch_one(const GemvArgs& a, int m0, cudaStream_t s) {
  static int done_mask[64] = {0};
  using T = WTraits<FP8>;
  const int rowbytes = a.K * T::kEsize;
  const int stage_bytes = R * rowbytes;
  int grid = num_sms();
  const int maxg = (a.N + R - 1) / R;
  if (grid > maxg) grid = maxg;
  const int rows_max = (a.N + grid - 1) / grid + R;  // stage padding of the last range
  const int kb = (a.K + 127) / 128;
  int stages = kGemvStageBudget / stage_bytes;
  if (stages > kGemvMaxStages) stages = kGemvMaxStages;
  if (stages < 1) stages = 1;
  GemvLayout lay = gemv_layout(stages, stage_bytes, rows_max, MB, kb, a.epi, a.dconv);
  while (lay.total > 227 * 1024 && stages > 1) lay = gemv_layout(--stages, stage_bytes, rows_max, MB, kb, a.epi, a.dconv);
  if (lay.total > 227 * 1024) return cudaErrorInvalidConfiguration;
  auto kern = gemv_kernel<FP8, MB, CPT, R>;
  cudaError_t e = set_smem_once((const void*)kern, lay.total, done_mask);
  if (e != cudaSuccess) return e;
  // EPI_STORE / EPI_RESID / EPI_INPROJ_CONV -> trace ids store / resid / conv
  const int id = (FP8 ? K_GEMV_FP8 : K_GEMV_BF16) + (a.epi == EPI_INPROJ_CONV ? 1 : (a.epi == EPI_RESID ? 2 : 0));
  trace_pre(id, s);
  e = launch_k(kern, dim3(grid), dim3(kGemvThreads), lay.total, s, a.pdl != 0, a, m0, stages, rows_max);
  trace_post(id, s);
  return e;
}

// Launches one pass over the weights for batch rows [m0, m0 + rows) and
// returns the number of rows it covered.  Register budget of the activation
// cache: MB * CPT <= 4 (CPT = 16-byte chunks per consumer thread per row).
template <bool FP8>
static int launch_group(const GemvArgs& a, int m0, cudaStream_t s, cudaError_t* err) {
  // stages of ~32 KB: R = 32 KB / row bytes rows per stage
  const int rowbytes = a.K * WTraits<FP8>::kEsize;
  const int cpt = (rowbytes + 4095) / 4096;
  const int rem = a.M - m0;
  if (cpt == 1) {
    if (rem >= 3) { *err = launch_one<FP8, 4, 1, 8>(a, m0, s); return 4; }
    if (rem == 2) { *err = launch_one<FP8, 2, 1, 8>(a, m0, s); return 2; }
    *err = launch_one<FP8, 1, 1, 8>(a, m0, s);
    return 1;
  }
  if (cpt == 2) {
    if (rem >= 2) { *err = launch_one<FP8, 2, 2, 4>(a, m0, s); return 2; }
    *err = launch_one<FP8, 1, 2, 4>(a, m0, s);
    return 1;
  }
  if (cpt <= 4) { *err = launch_one<FP8, 1, 4, 2>(a, m0, s); return 1; }
  if constexpr (!FP8) { *err = launch_one<FP8, 1, 8, 1>(a, m0, s); return 1; }
  *err = cudaErrorInvalidValue;
  return 1;
}

cudaError_t launch_gemv(const GemvArgs& a, bool fp8, cudaStream_t s) {
  // more than 8 rows: the tcgen05 tensor-core GEMM (k_gemm_tc.cu)
  if (gemm_tc_supported(a.M, a.N, a.K, fp8)) return launch_gemm_tc(a, fp8, s);
  // batches of up to 8 rows with K % 64 == 0, K <= 8192: one weight pass on
  // the warp-MMA GEMV (k_gemv_mma.cu)
  if (gemv_mma_supported(a.M, a.K)) return launch_gemv_mma(a, fp8, s);
  for (int m0 = 0; m0 < a.M;) {
    cudaError_t e = cudaSuccess;
    GemvArgs b = a;
    if (m0 > 0) b.pdl = 0;  // later passes follow a GEMV of this call
    m0 += fp8 ? launch_group<true>(b, m0, s, &e) : launch_group<false>(b, m0, s, &e);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Largest batch row count one GEMV pass covers for a K-wide row (the fused
// norm prologue needs the whole batch in one pass).
int gemv_rows_per_pass(int K, bool fp8) {
  if (gemv_mma_supported(8, K)) return 8;
  const int cpt = (K * (fp8 ? 1 : 2) + 4095) / 4096;
  return cpt == 1 ? 4 : (cpt == 2 ? 2 : 1);
}

int status_gemv(int clear) { return tu_status(clear); }

cudaError_t wait_limit_gemv(long long cycles) { return tu_set_wait_limit(cycles); }

}  // namespace m2
