// k_ssd.cu -- chunked SSD prefill scan (state-space dual form) for one
// sequence of T tokens.
//
// The recurrence of the SSM decode step (source listing
// "spark_model/layers/nemotron_mamba2.rs", `ssm_decode`; "SSD chunked prefill
// scan ... ceil(T/64) serial links instead of T" in its kernel table)
//   h_t = exp(dt_t A) h_{t-1} + dt_t x_t B_t^T,   y_t = h_t C_t + D x_t
// unrolls, inside a chunk of Q tokens starting at c0 with state h_in, into
//   a_t = dt_t A,  s_t = sum_{r=c0..t} a_r                  (inclusive cumsum)
//   y_t = sum_{s=c0..t} (C_t . B_s) exp(s_t - s_s) dt_s x_s + exp(s_t) h_in C_t + D x_t
//   h_out = exp(s_last) h_in + sum_s exp(s_last - s_s) dt_s x_s B_s^T
// so only the chunk states are sequential.  Three kernels:
//   ssd_chunk_state  per (head, chunk): dH_c = sum_s w_s x_s B_s^T, w_s = exp(s_last - s_s) dt_s,
//                    and the chunk decay exp(s_last)
//   ssd_state_pass   per state element: h_in(c) for every chunk (sequential over
//                    chunks, parallel over H*P*N), final state, conv position
//   ssd_chunk_out    per (head, chunk): G = C B^T (masked, decay-weighted) times
//                    X, plus exp(s_t) C h_in(c)^T, plus D x
// fp32 arithmetic throughout (bf16 inputs are exact in fp32); the chunk length
// is 128 (the layer's prefill chunk).
#include <cuda_runtime.h>
#include <stdint.h>

#include "m2_common.cuh"
#include "m2_kernels.h"

namespace m2 {

constexpr int kQ = 128;  // chunk length
constexpr int kSsdThreads = 256;

// dt, inclusive cumulative log-decay and the last value for one chunk of one
// head, into shared memory (Qc <= 128 valid tokens; the rest are zero).
__device__ __forceinline__ void chunk_decay(const SsdArgs& a, int h, int t0, int qc, float* dt_s, float* cs_s) {
  const int tid = threadIdx.x;
  const float A = -expf(a.A_log[h]);
  const float bias = a.dt_bias[h];
  if (tid < kQ) {
    float dt = 0.0f;
    if (tid < qc) {
      dt = softplus_f(bf16_to_f32(a.dt[(size_t)(t0 + tid) * a.ld_dt + h]) + bias);
      dt = fminf(fmaxf(dt, 1e-9f), 1e9f);
    }
    dt_s[tid] = dt;
    cs_s[tid] = dt * A;
  }
  __syncthreads();
  // inclusive prefix sum over 128 values (Hillis-Steele, fp32)
  for (int o = 1; o < kQ; o <<= 1) {
    float v = 0.0f;
    if (tid < kQ && tid >= o) v = cs_s[tid - o];
    __syncthreads();
    if (tid < kQ) cs_s[tid] += v;
    __syncthreads();
  }
}

// ------------------------------------------------------------------ chunk states

// dH[h][c][p][n] = sum_s exp(s_last - s_s) dt_s x_s[p] B_s[n]; decay[h][c] = exp(s_last).
// Thread tile: 8 p x 4 n (P = 64, N = 128 -> 256 threads; other shapes loop).
__global__ void __launch_bounds__(kSsdThreads) ssd_chunk_state_kernel(const SsdArgs a) {
  const int h = blockIdx.x, c = blockIdx.y;
  const int t0 = c * kQ, qc = min(kQ, a.T - t0);
  const int g = h / (a.H / a.G);
  __shared__ float dt_s[kQ], cs_s[kQ], w_s[kQ];
  extern __shared__ float dyn[];
  float* xs = dyn;                  // [Q][P]
  float* bs = dyn + kQ * a.P;       // [Q][N]
  chunk_decay(a, h, t0, qc, dt_s, cs_s);
  const float last = cs_s[max(qc - 1, 0)];
  for (int i = threadIdx.x; i < kQ; i += blockDim.x) w_s[i] = i < qc ? expf(last - cs_s[i]) * dt_s[i] : 0.0f;
  for (int i = threadIdx.x; i < kQ * a.P; i += blockDim.x) {
    const int s = i / a.P, p = i % a.P;
    xs[i] = s < qc ? bf16_to_f32(a.x[(size_t)(t0 + s) * a.ld_in + (size_t)h * a.P + p]) : 0.0f;
  }
  for (int i = threadIdx.x; i < kQ * a.N; i += blockDim.x) {
    const int s = i / a.N, n = i % a.N;
    bs[i] = s < qc ? bf16_to_f32(a.Bm[(size_t)(t0 + s) * a.ld_in + (size_t)g * a.N + n]) : 0.0f;
  }
  __syncthreads();
  float* out = a.dH + (((size_t)h * a.nchunks + c) * a.P) * a.N;
  for (int tile = threadIdx.x; tile < (a.P / 8) * (a.N / 4); tile += blockDim.x) {
    const int p0 = (tile / (a.N / 4)) * 8, n0 = (tile % (a.N / 4)) * 4;
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
    for (int s = 0; s < qc; ++s) {
      const float w = w_s[s];
      const float4 b = *reinterpret_cast<const float4*>(bs + s * a.N + n0);
      float xv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) xv[i] = xs[s * a.P + p0 + i] * w;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        acc[i][0] = fmaf(xv[i], b.x, acc[i][0]);
        acc[i][1] = fmaf(xv[i], b.y, acc[i][1]);
        acc[i][2] = fmaf(xv[i], b.z, acc[i][2]);
        acc[i][3] = fmaf(xv[i], b.w, acc[i][3]);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
      *reinterpret_cast<float4*>(out + (size_t)(p0 + i) * a.N + n0) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  }
  if (threadIdx.x == 0) a.decay[(size_t)h * a.nchunks + c] = expf(last);
}

// ------------------------------------------------------------------ state pass

// Sequential over chunks for each state element (float4 of n): replaces dH[c]
// with the state entering chunk c, and writes the final state into h.
__global__ void __launch_bounds__(256) ssd_state_pass_kernel(const SsdArgs a) {
  const size_t per_head = (size_t)a.P * a.N / 4;
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < (size_t)a.H * per_head) {
    const int h = (int)(i / per_head);
    const size_t e = i % per_head;
    float4* st = reinterpret_cast<float4*>(a.h) + i;
    float4 cur = *st;
    for (int c = 0; c < a.nchunks; ++c) {
      float4* d = reinterpret_cast<float4*>(a.dH + ((size_t)h * a.nchunks + c) * a.P * a.N) + e;
      const float4 dh = *d;
      const float dec = a.decay[(size_t)h * a.nchunks + c];
      *d = cur;  // state entering chunk c
      cur.x = fmaf(dec, cur.x, dh.x);
      cur.y = fmaf(dec, cur.y, dh.y);
      cur.z = fmaf(dec, cur.z, dh.z);
      cur.w = fmaf(dec, cur.w, dh.w);
    }
    *st = cur;
  }
  if (a.pos_inc && blockIdx.x == 0 && threadIdx.x == 0) a.pos_inc[0] += a.T;
}

// ------------------------------------------------------------------ chunk outputs

// y[t][h*P+p] for the chunk.  L[s][t] = (C_t . B_s) exp(s_t - s_s) dt_s for
// s <= t (kept transposed, s-major, for contiguous reads) is formed in one 8x8
// tile per thread (16 x 16 tiles of the 128 x 128 chunk), then
// y = L^T X + exp(s_t) C h_in^T + D x in 4 t x 8 p tiles.
__global__ void __launch_bounds__(kSsdThreads) ssd_chunk_out_kernel(const SsdArgs a) {
  static_assert(kSsdThreads == (kQ / 8) * (kQ / 8), "one L tile per thread");
  const int h = blockIdx.x, c = blockIdx.y;
  const int t0 = c * kQ, qc = min(kQ, a.T - t0);
  const int g = h / (a.H / a.G);
  const int tid = threadIdx.x;
  __shared__ float dt_s[kQ], cs_s[kQ];
  extern __shared__ float dyn[];
  float* ct = dyn;                   // C^T [N][Q]
  float* bt = ct + a.N * kQ;         // B^T [N][Q], then L^T [Q (s)][Q (t)]
  float* xs = bt + max(a.N, kQ) * kQ;  // X [Q][P]
  float* Ht = xs + kQ * a.P;         // h_in^T [N][P]
  float* Lt = bt;                    // reuses B^T once C B^T is in registers
  chunk_decay(a, h, t0, qc, dt_s, cs_s);
  for (int i = tid; i < kQ * a.N; i += blockDim.x) {
    const int t = i / a.N, n = i % a.N;
    const size_t row = (size_t)(t0 + t) * a.ld_in + (size_t)g * a.N + n;
    ct[n * kQ + t] = t < qc ? bf16_to_f32(a.Cm[row]) : 0.0f;
    bt[n * kQ + t] = t < qc ? bf16_to_f32(a.Bm[row]) : 0.0f;
  }
  for (int i = tid; i < kQ * a.P; i += blockDim.x) {
    const int s = i / a.P, p = i % a.P;
    xs[i] = s < qc ? bf16_to_f32(a.x[(size_t)(t0 + s) * a.ld_in + (size_t)h * a.P + p]) : 0.0f;
  }
  const float* hin = a.dH + (((size_t)h * a.nchunks + c) * a.P) * a.N;
  for (int i = tid; i < a.P * a.N; i += blockDim.x) {
    const int p = i / a.N, n = i % a.N;
    Ht[n * a.P + p] = hin[i];
  }
  __syncthreads();
  {
    const int s0 = (tid / (kQ / 8)) * 8, tt0 = (tid % (kQ / 8)) * 8;
    float gacc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) gacc[i][j] = 0.0f;
    if (s0 <= tt0) {
      for (int n = 0; n < a.N; ++n) {
        const float4 b0 = *reinterpret_cast<const float4*>(bt + n * kQ + s0);
        const float4 b1 = *reinterpret_cast<const float4*>(bt + n * kQ + s0 + 4);
        const float4 c0 = *reinterpret_cast<const float4*>(ct + n * kQ + tt0);
        const float4 c1 = *reinterpret_cast<const float4*>(ct + n * kQ + tt0 + 4);
        const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        const float cv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) gacc[i][j] = fmaf(bv[i], cv[j], gacc[i][j]);
      }
    }
    __syncthreads();  // every read of B^T is done before L^T overwrites it
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int s = s0 + i;
      float r[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int t = tt0 + j;
        // masked before exp: for s > t the exponent is positive
        r[j] = (s <= t) ? gacc[i][j] * expf(cs_s[t] - cs_s[s]) * dt_s[s] : 0.0f;
      }
      *reinterpret_cast<float4*>(Lt + s * kQ + tt0) = make_float4(r[0], r[1], r[2], r[3]);
      *reinterpret_cast<float4*>(Lt + s * kQ + tt0 + 4) = make_float4(r[4], r[5], r[6], r[7]);
    }
  }
  __syncthreads();
  const float Dh = a.D[h];
  for (int tile = tid; tile < (kQ / 4) * (a.P / 8); tile += blockDim.x) {
    const int tq = (tile / (a.P / 8)) * 4, p0 = (tile % (a.P / 8)) * 8;
    float acc[4][8], inter[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = inter[i][j] = 0.0f;
    const int smax = min(tq + 3, qc - 1);
    for (int s = 0; s <= smax; ++s) {
      const float4 l = *reinterpret_cast<const float4*>(Lt + s * kQ + tq);
      const float lv[4] = {l.x, l.y, l.z, l.w};
      const float4 x0 = *reinterpret_cast<const float4*>(xs + s * a.P + p0);
      const float4 x1 = *reinterpret_cast<const float4*>(xs + s * a.P + p0 + 4);
      const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(lv[i], xv[j], acc[i][j]);
    }
    for (int n = 0; n < a.N; ++n) {
      const float4 cc = *reinterpret_cast<const float4*>(ct + n * kQ + tq);
      const float cv[4] = {cc.x, cc.y, cc.z, cc.w};
      const float4 h0 = *reinterpret_cast<const float4*>(Ht + n * a.P + p0);
      const float4 h1 = *reinterpret_cast<const float4*>(Ht + n * a.P + p0 + 4);
      const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) inter[i][j] = fmaf(cv[i], hv[j], inter[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = tq + i;
      if (t < qc) {
        const float e = expf(cs_s[t]);
        float* yo = a.y + (size_t)(t0 + t) * a.ldy + (size_t)h * a.P + p0;
        float r[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) r[j] = acc[i][j] + e * inter[i][j] + Dh * xs[t * a.P + p0 + j];
        *reinterpret_cast<float4*>(yo) = make_float4(r[0], r[1], r[2], r[3]);
        *reinterpret_cast<float4*>(yo + 4) = make_float4(r[4], r[5], r[6], r[7]);
      }
    }
  }
}

static int smem_state_bytes(int P, int N) { return (kQ * P + kQ * N) * 4; }
static int smem_out_bytes(int P, int N) { return (N * kQ + (N > kQ ? N : kQ) * kQ + kQ * P + N * P) * 4; }

bool ssd_supported(int H, int P, int N, int G) {
  if (G <= 0 || H % G || P % 8 || N % 4) return false;
  return smem_out_bytes(P, N) <= 227 * 1024 && smem_state_bytes(P, N) <= 227 * 1024;
}

size_t ssd_workspace_bytes(int T, int H, int P, int N) {
  const size_t nc = (size_t)(T + kQ - 1) / kQ;
  return ((nc * H * P * N * 4 + 255) / 256) * 256 + ((nc * H * 4 + 255) / 256) * 256;
}

static int done_state[64], done_out[64];

cudaError_t launch_ssd(const SsdArgs& a0, cudaStream_t s) {
  SsdArgs a = a0;
  a.nchunks = (a.T + kQ - 1) / kQ;
  const int smem_state = smem_state_bytes(a.P, a.N);
  const int smem_out = smem_out_bytes(a.P, a.N);
  cudaError_t e = set_smem_once((const void*)ssd_chunk_state_kernel, smem_state, done_state);
  if (e != cudaSuccess) return e;
  e = set_smem_once((const void*)ssd_chunk_out_kernel, smem_out, done_out);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.H, a.nchunks);
  trace_pre(K_SSD_CHUNK_STATE, s);
  ssd_chunk_state_kernel<<<grid, kSsdThreads, smem_state, s>>>(a);
  trace_post(K_SSD_CHUNK_STATE, s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const size_t n4 = (size_t)a.H * a.P * a.N / 4;
  trace_pre(K_SSD_STATE_PASS, s);
  ssd_state_pass_kernel<<<(unsigned)((n4 + 255) / 256), 256, 0, s>>>(a);
  trace_post(K_SSD_STATE_PASS, s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  trace_pre(K_SSD_CHUNK_OUT, s);
  ssd_chunk_out_kernel<<<grid, kSsdThreads, smem_out, s>>>(a);
  trace_post(K_SSD_CHUNK_OUT, s);
  return cudaGetLastError();
}

}  // namespace m2
