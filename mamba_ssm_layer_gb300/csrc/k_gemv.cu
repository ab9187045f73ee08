// k_gemv.cu -- CUDA-core w8a16 / bf16 GEMV for small batches (decode).
//
// Computes out[m][n] = sum_k A[m][k] * W~[n][k] with W~ = E4M3(W)*S[n/128][k/128]
// (page "Struct Qwen3SsmLayer", `set_fp8_decode_weights`; scale index of
// "Struct NemotronMamba2Layer", `set_fp8_weights`) or W~ = bf16 W (native BF16
// projections).  The decode GEMV is HBM-bound: every weight byte is read once
// per call, so the design goal is to keep ~200 KB of weight reads in flight per
// SM and to spend few instructions per byte.
//
// Layout of one CTA (one per SM, persistent over a contiguous row range):
//   warp 8      producer: one lane streams R whole weight rows per stage
//               (R*K contiguous bytes) into a shared-memory ring with 1-D bulk
//               copies (cp.async.bulk, mbarrier completion, L2 evict-first);
//   warps 0..7  consumers: thread t owns the 16-byte chunks t, t+256, ... of
//               every row, so its activations (<= 64 fp32) stay in registers
//               for the whole call; per row it forms 16-element partial dot
//               products, multiplies each by the chunk's block scale and
//               accumulates.  Per stage the R*MB partial sums are reduced
//               with a transposing warp butterfly and one shared-memory pass.
// E4M3 is decoded in registers with the exact hardware E4M3->f16 conversion.
#include <cuda_runtime.h>
#include <stdint.h>

#include "m2_common.cuh"
#include "m2_kernels.h"

namespace m2 {

constexpr int kGemvConsumerWarps = 8;
constexpr int kGemvConsumers = kGemvConsumerWarps * 32;  // 256
constexpr int kGemvThreads = kGemvConsumers + 32;        // + producer warp
constexpr int kGemvStageBudget = 196608;                 // bytes of weight ring
constexpr int kGemvMaxStages = 8;

struct GemvSmemTail {
  uint64_t full[kGemvMaxStages];
  uint64_t empty[kGemvMaxStages];
  float red[2][kGemvConsumerWarps][32];
};

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
// remaining levels are plain xor-reductions.
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
template <int V, int O>
__device__ __forceinline__ void butterfly(float* v, int lane) {
  Butterfly<V, O>::run(v, lane);
}

// Epilogue for one output element (row n, batch row m).
__device__ __forceinline__ void gemv_epilogue(const GemvArgs& a, int n, int m, float acc) {
  if (a.epi == EPI_RESID) {
    float r = bf16_to_f32(a.resid[(size_t)m * a.ldr + n]);
    a.out[(size_t)m * a.ldo + n] = f32_to_bf16(r + acc);
    return;
  }
  uint16_t vb = f32_to_bf16(acc);  // rounding point of the in_proj output
  if (a.epi == EPI_INPROJ_CONV && n >= a.xbc0 && n < a.xbc0 + a.d_xbc) {
    // conv1d update with bias + SiLU for channel c; this thread owns channel c
    // of sequence m for the whole call, so reading the ring and then writing
    // its oldest slot is race-free.
    const int c = n - a.xbc0;
    const int L = a.dconv - 1;
    const int p = a.pos[m];
    uint16_t* rg = a.ring + (size_t)m * L * a.d_xbc;
    const uint16_t* wc = a.conv_w + (size_t)c * a.dconv;
    float s = a.conv_b ? bf16_to_f32(a.conv_b[c]) : 0.0f;
    for (int j = 0; j < L; ++j) s += bf16_to_f32(wc[j]) * bf16_to_f32(rg[(size_t)((p + j) % L) * a.d_xbc + c]);
    s += bf16_to_f32(wc[L]) * bf16_to_f32(vb);
    a.out[(size_t)m * a.ldo + n] = f32_to_bf16(silu_f(s));
    rg[(size_t)(p % L) * a.d_xbc + c] = vb;
    return;
  }
  a.out[(size_t)m * a.ldo + n] = vb;
}

template <bool FP8, int MB, int CPT, int R>
__global__ void __launch_bounds__(kGemvThreads, 1) gemv_kernel(const GemvArgs a, int m0, int stages) {
  using T = WTraits<FP8>;
  constexpr int V = R * MB;
  constexpr int LOGV = Log2<V>::value;
  static_assert((1 << LOGV) == V && V <= 32, "R*MB must be a power of two <= 32");

  extern __shared__ __align__(128) uint8_t smem[];
  const int rowbytes = a.K * T::kEsize;
  const int stage_bytes = R * rowbytes;
  GemvSmemTail* tail = reinterpret_cast<GemvSmemTail*>(smem + (size_t)stages * stage_bytes);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  const int row_begin = (int)(((long long)a.N * blockIdx.x) / G);
  const int row_end = (int)(((long long)a.N * (blockIdx.x + 1)) / G);
  const int nrows = row_end - row_begin;
  const int niter = (nrows + R - 1) / R;
  const int nchunks = rowbytes / 16;
  const int kb = (a.K + 127) / 128;
  const int mvalid = min(MB, a.M - m0);

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&tail->full[s], 1);
      mbar_init(&tail->empty[s], kGemvConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kGemvConsumerWarps) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = a.evict_first ? policy_evict_first() : policy_evict_normal();
      const uint8_t* wbase = static_cast<const uint8_t*>(a.W) + (size_t)row_begin * rowbytes;
      for (int it = 0; it < niter; ++it) {
        const int s = it % stages;
        if (it >= stages && !mbar_wait(&tail->empty[s], ((it / stages) - 1) & 1)) return;  // status recorded
        const int rows = min(R, nrows - it * R);
        const uint32_t bytes = (uint32_t)(rows * rowbytes);
        mbar_arrive_expect_tx(&tail->full[s], bytes);
        bulk_g2s(smem + (size_t)s * stage_bytes, wbase + (size_t)it * R * rowbytes, bytes, &tail->full[s], pol);
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  // activations of my chunks, fp32 in registers
  float act[MB][CPT][T::kEpc];
#pragma unroll
  for (int m = 0; m < MB; ++m)
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
      const int c = tid + j * kGemvConsumers;
      if (m < mvalid && c < nchunks) {
        const uint4* src = reinterpret_cast<const uint4*>(a.A + (size_t)(m0 + m) * a.lda + (size_t)c * T::kEpc);
#pragma unroll
        for (int q = 0; q < T::kEpc / 8; ++q) {
          const uint4 v = __ldg(src + q);
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            act[m][j][q * 8 + 2 * e] = bf16lo(w4[e]);
            act[m][j][q * 8 + 2 * e + 1] = bf16hi(w4[e]);
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < T::kEpc; ++e) act[m][j][e] = 0.0f;
      }
    }

  // After a timed-out wait a warp stops touching memory but keeps taking part
  // in the named barrier, so that no other warp waits on it forever.
  bool dead = false;
  for (int it = 0; it < niter; ++it) {
    const int s = it % stages;
    const int row0 = row_begin + it * R;
    const int rows = dead ? 0 : min(R, nrows - it * R);
    if (!dead && !mbar_wait(&tail->full[s], (it / stages) & 1)) dead = true;
    const uint8_t* st = smem + (size_t)s * stage_bytes;

    float v[V];
#pragma unroll
    for (int i = 0; i < V; ++i) v[i] = 0.0f;

#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (r < rows && !dead) {
        const int n = row0 + r;
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
          const int c = tid + j * kGemvConsumers;
          if (c < nchunks) {
            const uint4 wv = *reinterpret_cast<const uint4*>(st + (size_t)r * rowbytes + (size_t)c * 16);
            const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
            float p[MB];
#pragma unroll
            for (int m = 0; m < MB; ++m) p[m] = 0.0f;
            if constexpr (FP8) {
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                float w0, w1;
                e4m3x2_to_f32((uint16_t)(w4[e >> 1] >> ((e & 1) * 16)), w0, w1);
#pragma unroll
                for (int m = 0; m < MB; ++m) {
                  p[m] = fmaf(w0, act[m][j][2 * e], p[m]);
                  p[m] = fmaf(w1, act[m][j][2 * e + 1], p[m]);
                }
              }
              const float sc = bf16_to_f32(__ldg(a.S + (size_t)(n >> 7) * kb + ((c * 16) >> 7)));
#pragma unroll
              for (int m = 0; m < MB; ++m) v[r * MB + m] = fmaf(p[m], sc, v[r * MB + m]);
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float w0 = bf16lo(w4[e]), w1 = bf16hi(w4[e]);
#pragma unroll
                for (int m = 0; m < MB; ++m) {
                  p[m] = fmaf(w0, act[m][j][2 * e], p[m]);
                  p[m] = fmaf(w1, act[m][j][2 * e + 1], p[m]);
                }
              }
#pragma unroll
              for (int m = 0; m < MB; ++m) v[r * MB + m] += p[m];
            }
          }
        }
      }
    }
    // stage consumed: hand it back to the producer before reducing
    __syncwarp();
    if (lane == 0) mbar_arrive(&tail->empty[s]);

    // transposing butterfly: after it, lane l holds the warp total of value
    // index l >> (5 - LOGV)
    butterfly<V, 16>(v, lane);
    const int buf = it & 1;
    if ((lane & ((1 << (5 - LOGV)) - 1)) == 0) tail->red[buf][warp][lane >> (5 - LOGV)] = v[0];
    named_bar(1, kGemvConsumers);
    if (tid < V) {
      float tot = 0.0f;
#pragma unroll
      for (int w = 0; w < kGemvConsumerWarps; ++w) tot += tail->red[buf][w][tid];
      const int r = tid / MB, m = tid % MB;
      if (!dead && r < rows && m < mvalid) gemv_epilogue(a, row0 + r, m0 + m, tot);
    }
  }
}

template <bool FP8, int MB, int CPT, int R>
static cudaError_t launch_one(const GemvArgs& a, int m0, cudaStream_t s) {
  static int done_mask[64] = {0};
  using T = WTraits<FP8>;
  const int rowbytes = a.K * T::kEsize;
  const int stage_bytes = R * rowbytes;
  int stages = kGemvStageBudget / stage_bytes;
  if (stages > kGemvMaxStages) stages = kGemvMaxStages;
  if (stages < 1) stages = 1;
  const int smem = stages * stage_bytes + (int)sizeof(GemvSmemTail);
  auto kern = gemv_kernel<FP8, MB, CPT, R>;
  cudaError_t e = set_smem_once((const void*)kern, smem, done_mask);
  if (e != cudaSuccess) return e;
  int grid = num_sms();
  const int maxg = (a.N + R - 1) / R;
  if (grid > maxg) grid = maxg;
  // EPI_STORE / EPI_RESID / EPI_INPROJ_CONV -> trace ids store / resid / conv
  const int id = (FP8 ? K_GEMV_FP8 : K_GEMV_BF16) + (a.epi == EPI_INPROJ_CONV ? 1 : (a.epi == EPI_RESID ? 2 : 0));
  trace_pre(id, s);
  kern<<<grid, kGemvThreads, smem, s>>>(a, m0, stages);
  trace_post(id, s);
  return cudaGetLastError();
}

// Launches one pass over the weights for batch rows [m0, m0 + rows) and
// returns the number of rows it covered.  Register budget of the activation
// cache: MB * CPT <= 4 (CPT = 16-byte chunks per consumer thread per row).
template <bool FP8>
static int launch_group(const GemvArgs& a, int m0, cudaStream_t s, cudaError_t* err) {
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
    if (rem >= 2) { *err = launch_one<FP8, 2, 2, 8>(a, m0, s); return 2; }
    *err = launch_one<FP8, 1, 2, 8>(a, m0, s);
    return 1;
  }
  if (cpt <= 4) { *err = launch_one<FP8, 1, 4, 4>(a, m0, s); return 1; }
  if constexpr (!FP8) { *err = launch_one<FP8, 1, 8, 2>(a, m0, s); return 1; }
  *err = cudaErrorInvalidValue;
  return 1;
}

cudaError_t launch_gemv(const GemvArgs& a, bool fp8, cudaStream_t s) {
  for (int m0 = 0; m0 < a.M;) {
    cudaError_t e = cudaSuccess;
    m0 += fp8 ? launch_group<true>(a, m0, s, &e) : launch_group<false>(a, m0, s, &e);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// ------------------------------------------------------------------ RMSNorm

// Input RMSNorm, weight * x scaling (source listing "nemotron_mamba2.rs",
// module header step 1): out = bf16( x / sqrt(mean(x^2) + eps) * w ).
__global__ void __launch_bounds__(256) rmsnorm_kernel(const uint16_t* __restrict__ x, int ldx,
                                                      const uint16_t* __restrict__ w, uint16_t* __restrict__ out,
                                                      int ldo, int K, float eps) {
  const uint16_t* xr = x + (size_t)blockIdx.x * ldx;
  __shared__ float red[8];
  float ss = 0.0f;
  for (int k = threadIdx.x * 8; k < K; k += 256 * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + k);
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a0 = bf16lo(w4[e]), a1 = bf16hi(w4[e]);
      ss = fmaf(a0, a0, ss);
      ss = fmaf(a1, a1, ss);
    }
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) tot += red[i];
  const float r = 1.0f / sqrtf(tot / (float)K + eps);
  uint16_t* o = out + (size_t)blockIdx.x * ldo;
  for (int k = threadIdx.x * 8; k < K; k += 256 * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + k);
    const uint4 g = *reinterpret_cast<const uint4*>(w + k);
    const uint32_t x4[4] = {v.x, v.y, v.z, v.w}, g4[4] = {g.x, g.y, g.z, g.w};
    uint32_t o4[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      o4[e] = pack_bf16x2(bf16lo(x4[e]) * r * bf16lo(g4[e]), bf16hi(x4[e]) * r * bf16hi(g4[e]));
    *reinterpret_cast<uint4*>(o + k) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
  }
}

cudaError_t launch_rmsnorm(const uint16_t* x, int32_t ldx, const uint16_t* w, uint16_t* out, int32_t ldo,
                           int32_t M, int32_t K, float eps, cudaStream_t s) {
  trace_pre(K_RMSNORM, s);
  rmsnorm_kernel<<<M, 256, 0, s>>>(x, ldx, w, out, ldo, K, eps);
  trace_post(K_RMSNORM, s);
  return cudaGetLastError();
}

int status_gemv(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return -4;
  if (clear) {
    const int z = 0;
    cudaMemcpyToSymbol(g_status, &z, sizeof(int));
  }
  return v;
}

}  // namespace m2
