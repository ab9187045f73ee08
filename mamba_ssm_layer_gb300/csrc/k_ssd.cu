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
#include "m2_tc.cuh"

namespace m2 {

constexpr int kQ = 128;  // chunk length
constexpr int kSsdThreads = 256;

// Global chunk id -> sequence, first token row, valid tokens (<= 128), and the
// sequence's token offset.
__device__ __forceinline__ void chunk_info(const SsdArgs& a, int cid, int& seq, int& t0, int& qc) {
  int lo = 0, hi = a.nseq - 1;
  while (lo < hi) {  // last i with cprefix[i] <= cid
    const int mid = (lo + hi + 1) >> 1;
    if (a.cprefix[mid] <= cid) lo = mid;
    else hi = mid - 1;
  }
  seq = lo;
  t0 = a.cu[lo] + (cid - a.cprefix[lo]) * kQ;
  qc = min(kQ, a.cu[lo + 1] - t0);
}

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
  int seq, t0, qc;
  chunk_info(a, c, seq, t0, qc);
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

// Sequential over each sequence's chunks for each state element (float4 of n):
// replaces dH[c] with the state entering chunk c and writes the final state
// back.  Grid: (elements, sequences).
__global__ void __launch_bounds__(256) ssd_state_pass_kernel(const SsdArgs a) {
  const int seq = blockIdx.y;
  const size_t per_head = (size_t)a.P * a.N / 4;
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int c0 = a.cprefix[seq], c1 = a.cprefix[seq + 1];
  if (i < (size_t)a.H * per_head) {
    const int h = (int)(i / per_head);
    const size_t e = i % per_head;
    float4* st = reinterpret_cast<float4*>(a.h + (size_t)seq * a.H * a.P * a.N) + i;
    float4 cur = *st;
    // the chunk states of up to 8 chunks are loaded together (independent of
    // the carried state), then folded in order
    for (int cb = c0; cb < c1; cb += 8) {
      float4 dh[8];
      float dec[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (cb + k < c1) {
          dh[k] = *(reinterpret_cast<const float4*>(a.dH + ((size_t)h * a.nchunks + cb + k) * a.P * a.N) + e);
          dec[k] = a.decay[(size_t)h * a.nchunks + cb + k];
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (cb + k < c1) {
          *(reinterpret_cast<float4*>(a.dH + ((size_t)h * a.nchunks + cb + k) * a.P * a.N) + e) = cur;  // state entering the chunk
          cur.x = fmaf(dec[k], cur.x, dh[k].x);
          cur.y = fmaf(dec[k], cur.y, dh[k].y);
          cur.z = fmaf(dec[k], cur.z, dh[k].z);
          cur.w = fmaf(dec[k], cur.w, dh[k].w);
        }
      }
    }
    *st = cur;
  }
  if (a.pos_inc && blockIdx.x == 0 && threadIdx.x == 0) a.pos_inc[seq] += a.cu[seq + 1] - a.cu[seq];
}

// ------------------------------------------------------------------ chunk outputs

// y[t][h*P+p] for the chunk.  L[s][t] = (C_t . B_s) exp(s_t - s_s) dt_s for
// s <= t (kept transposed, s-major, for contiguous reads) is formed in one 8x8
// tile per thread (16 x 16 tiles of the 128 x 128 chunk), then
// y = L^T X + exp(s_t) C h_in^T + D x in 4 t x 8 p tiles.
__global__ void __launch_bounds__(kSsdThreads) ssd_chunk_out_kernel(const SsdArgs a) {
  static_assert(kSsdThreads == (kQ / 8) * (kQ / 8), "one L tile per thread");
  const int h = blockIdx.x, c = blockIdx.y;
  int seq, t0, qc;
  chunk_info(a, c, seq, t0, qc);
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

// ------------------------------------------------------------------ tensor-core chunk kernels
//
// The same three products on warp MMA (m16n8k16, bf16 operands, fp32
// accumulation).  x, B and C are bf16 values (the conv output's rounding
// point), so C B^T, C h^T and x-side operands enter the MMA exactly.  The fp32
// operands (the decay-weighted L, the carried state h_in and w_s x_s) are split
// into two bf16 parts, v = hi + lo with hi = bf16(v), lo = bf16(v - hi), so each
// product keeps about 16 significant bits and the sums stay fp32.  Shared
// arrays are row-major with rows padded by 16 bytes (conflict-free ldmatrix).

__device__ __forceinline__ void ldsm_x4(const void* p, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"((uint32_t)__cvta_generic_to_shared(p)));
}
__device__ __forceinline__ void ldsm_x4_t(const void* p, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"((uint32_t)__cvta_generic_to_shared(p)));
}
__device__ __forceinline__ void ldsm_x2_t(const void* p, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"((uint32_t)__cvta_generic_to_shared(p)));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// v = hi + lo, both bf16 (packed pairs)
__device__ __forceinline__ void split2(float v0, float v1, uint32_t& hi, uint32_t& lo) {
  const uint16_t h0 = f32_to_bf16(v0), h1 = f32_to_bf16(v1);
  hi = (uint32_t)h0 | ((uint32_t)h1 << 16);
  lo = (uint32_t)f32_to_bf16(v0 - bf16_to_f32(h0)) | ((uint32_t)f32_to_bf16(v1 - bf16_to_f32(h1)) << 16);
}

// Row-major bf16 tile [rows][cols] from global rows (ld elements apart) into
// shared memory with pitch cols + 8; rows >= valid are zero.
template <int COLS>
__device__ __forceinline__ void stage_rows(uint16_t* dst, const uint16_t* src, size_t ld, int rows, int valid) {
  constexpr int V = COLS / 8;  // 16-byte vectors per row
  for (int i = threadIdx.x; i < rows * V; i += blockDim.x) {
    const int r = i / V, v = i % V;
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (r < valid) x = *reinterpret_cast<const uint4*>(src + (size_t)r * ld + v * 8);
    *reinterpret_cast<uint4*>(dst + r * (COLS + 8) + v * 8) = x;
  }
}

// dH[h][c] = sum_s w_s x_s B_s^T (P x N), w_s = exp(s_last - s_s) dt_s; decay = exp(s_last).
template <int P, int N>
__global__ void __launch_bounds__(kSsdThreads) ssd_state_mma_kernel(const SsdArgs a) {
  constexpr int BP = N + 8, XP = P + 8;
  const int h = blockIdx.x, c = blockIdx.y;
  int seq, t0, qc;
  chunk_info(a, c, seq, t0, qc);
  const int g = h / (a.H / a.G);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ float dt_s[kQ], cs_s[kQ];
  extern __shared__ __align__(16) uint16_t sm16[];
  uint16_t* Bs = sm16;                 // [Q][BP]
  uint16_t* Wh = Bs + kQ * BP;         // [Q][XP]  hi part of w_s x_s
  uint16_t* Wl = Wh + kQ * XP;         // [Q][XP]  lo part
  chunk_decay(a, h, t0, qc, dt_s, cs_s);
  stage_rows<N>(Bs, a.Bm + (size_t)t0 * a.ld_in + (size_t)g * N, a.ld_in, kQ, qc);
  const float last = cs_s[max(qc - 1, 0)];
  for (int i = threadIdx.x; i < kQ * (P / 2); i += blockDim.x) {
    const int s_ = i / (P / 2), p2 = (i % (P / 2)) * 2;
    float v0 = 0.0f, v1 = 0.0f;
    if (s_ < qc) {
      const uint32_t xx = *reinterpret_cast<const uint32_t*>(a.x + (size_t)(t0 + s_) * a.ld_in + (size_t)h * P + p2);
      const float w = expf(last - cs_s[s_]) * dt_s[s_];
      v0 = w * bf16lo(xx);
      v1 = w * bf16hi(xx);
    }
    uint32_t hi, lo;
    split2(v0, v1, hi, lo);
    *reinterpret_cast<uint32_t*>(Wh + s_ * XP + p2) = hi;
    *reinterpret_cast<uint32_t*>(Wl + s_ * XP + p2) = lo;
  }
  __syncthreads();
  float* out = a.dH + ((size_t)h * a.nchunks + c) * P * N;
  const int gq = lane >> 2, tq = lane & 3;
  constexpr int units = (P / 16) * (N / 8);
  for (int u = warp; u < units; u += kSsdThreads / 32) {
    const int mp = u / (N / 8), j = u % (N / 8);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < kQ / 16; ++kk) {
      uint32_t ah[4], al[4], b0, b1;
      const int ar = 16 * kk + (lane & 7) + ((lane >> 4) & 1) * 8, ac = 16 * mp + ((lane >> 3) & 1) * 8;
      ldsm_x4_t(Wh + ar * XP + ac, ah);
      ldsm_x4_t(Wl + ar * XP + ac, al);
      ldsm_x2_t(Bs + (16 * kk + (lane & 7) + ((lane >> 3) & 1) * 8) * BP + 8 * j, b0, b1);
      mma_bf16(acc, ah, b0, b1);
      mma_bf16(acc, al, b0, b1);
    }
    const int p0 = 16 * mp + gq, n0 = 8 * j + 2 * tq;
    *reinterpret_cast<float2*>(out + (size_t)p0 * N + n0) = make_float2(acc[0], acc[1]);
    *reinterpret_cast<float2*>(out + (size_t)(p0 + 8) * N + n0) = make_float2(acc[2], acc[3]);
  }
  if (threadIdx.x == 0) a.decay[(size_t)h * a.nchunks + c] = expf(last);
}

// y for the chunk: warp w owns the 16 tokens [16w, 16w+16).
//   G = C B^T (only s <= t), L = G * exp(s_t - s_s) * dt_s (mask s <= t),
//   y = L x + exp(s_t) * (C h_in^T) + D x.
template <int P, int N>
__global__ void __launch_bounds__(kSsdThreads) ssd_out_mma_kernel(const SsdArgs a) {
  constexpr int CP = N + 8, XP = P + 8;
  static_assert(kSsdThreads / 32 * 16 == kQ, "one 16-token strip per warp");
  const int h = blockIdx.x, c = blockIdx.y;
  int seq, t0, qc;
  chunk_info(a, c, seq, t0, qc);
  const int g = h / (a.H / a.G);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  __shared__ float dt_s[kQ], cs_s[kQ];
  extern __shared__ __align__(16) uint16_t sm16[];
  uint16_t* Cs = sm16;             // [Q][CP]
  uint16_t* Bs = Cs + kQ * CP;     // [Q][CP]
  uint16_t* Xs = Bs + kQ * CP;     // [Q][XP]
  uint16_t* Hh = Xs + kQ * XP;     // [P][CP]  hi part of h_in
  uint16_t* Hl = Hh + P * CP;      // [P][CP]  lo part
  chunk_decay(a, h, t0, qc, dt_s, cs_s);
  stage_rows<N>(Cs, a.Cm + (size_t)t0 * a.ld_in + (size_t)g * N, a.ld_in, kQ, qc);
  stage_rows<N>(Bs, a.Bm + (size_t)t0 * a.ld_in + (size_t)g * N, a.ld_in, kQ, qc);
  stage_rows<P>(Xs, a.x + (size_t)t0 * a.ld_in + (size_t)h * P, a.ld_in, kQ, qc);
  const float* hin = a.dH + ((size_t)h * a.nchunks + c) * P * N;
  for (int i = threadIdx.x; i < P * N / 2; i += blockDim.x) {
    const int pp = i / (N / 2), n2 = (i % (N / 2)) * 2;
    const float2 v = *reinterpret_cast<const float2*>(hin + (size_t)pp * N + n2);
    uint32_t hi, lo;
    split2(v.x, v.y, hi, lo);
    *reinterpret_cast<uint32_t*>(Hh + pp * CP + n2) = hi;
    *reinterpret_cast<uint32_t*>(Hl + pp * CP + n2) = lo;
  }
  __syncthreads();
  const int w = warp;
  const int tr0 = 16 * w + gq, tr1 = tr0 + 8;  // this thread's two token rows
  // ---- G = C B^T for s tiles 0 .. 2w+1
  float G[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) G[j][0] = G[j][1] = G[j][2] = G[j][3] = 0.0f;
#pragma unroll
  for (int kk = 0; kk < N / 16; ++kk) {
    uint32_t af[4];
    ldsm_x4(Cs + (16 * w + (lane & 15)) * CP + 16 * kk + (lane >> 4) * 8, af);
#pragma unroll
    for (int jp = 0; jp < 8; ++jp) {
      if (jp <= w) {
        uint32_t bf[4];
        ldsm_x4(Bs + (16 * jp + (lane & 7) + ((lane >> 4) << 3)) * CP + 16 * kk + ((lane >> 3) & 1) * 8, bf);
        mma_bf16(G[2 * jp], af, bf[0], bf[1]);
        mma_bf16(G[2 * jp + 1], af, bf[2], bf[3]);
      }
    }
  }
  // ---- L (in place)
  const float cs0 = cs_s[tr0], cs1 = cs_s[tr1];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (j <= 2 * w + 1) {
      const int s0 = 8 * j + 2 * tq, s1 = s0 + 1;
      const float e00 = expf(fminf(cs0 - cs_s[s0], 0.0f)) * dt_s[s0], e01 = expf(fminf(cs0 - cs_s[s1], 0.0f)) * dt_s[s1];
      const float e10 = expf(fminf(cs1 - cs_s[s0], 0.0f)) * dt_s[s0], e11 = expf(fminf(cs1 - cs_s[s1], 0.0f)) * dt_s[s1];
      G[j][0] = s0 <= tr0 ? G[j][0] * e00 : 0.0f;
      G[j][1] = s1 <= tr0 ? G[j][1] * e01 : 0.0f;
      G[j][2] = s0 <= tr1 ? G[j][2] * e10 : 0.0f;
      G[j][3] = s1 <= tr1 ? G[j][3] * e11 : 0.0f;
    }
  }
  // ---- y_intra = L x
  float Y[P / 8][4];
#pragma unroll
  for (int q = 0; q < P / 8; ++q) Y[q][0] = Y[q][1] = Y[q][2] = Y[q][3] = 0.0f;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    if (kk <= w) {
      uint32_t ah[4], al[4];
      split2(G[2 * kk][0], G[2 * kk][1], ah[0], al[0]);
      split2(G[2 * kk][2], G[2 * kk][3], ah[1], al[1]);
      split2(G[2 * kk + 1][0], G[2 * kk + 1][1], ah[2], al[2]);
      split2(G[2 * kk + 1][2], G[2 * kk + 1][3], ah[3], al[3]);
#pragma unroll
      for (int qp = 0; qp < P / 16; ++qp) {
        uint32_t bf[4];
        ldsm_x4_t(Xs + (16 * kk + (lane & 7) + ((lane >> 3) & 1) * 8) * XP + 16 * qp + (lane >> 4) * 8, bf);
        mma_bf16(Y[2 * qp], ah, bf[0], bf[1]);
        mma_bf16(Y[2 * qp], al, bf[0], bf[1]);
        mma_bf16(Y[2 * qp + 1], ah, bf[2], bf[3]);
        mma_bf16(Y[2 * qp + 1], al, bf[2], bf[3]);
      }
    }
  }
  // ---- y_inter = C h_in^T
  float Yi[P / 8][4];
#pragma unroll
  for (int q = 0; q < P / 8; ++q) Yi[q][0] = Yi[q][1] = Yi[q][2] = Yi[q][3] = 0.0f;
#pragma unroll
  for (int kk = 0; kk < N / 16; ++kk) {
    uint32_t af[4];
    ldsm_x4(Cs + (16 * w + (lane & 15)) * CP + 16 * kk + (lane >> 4) * 8, af);
#pragma unroll
    for (int qp = 0; qp < P / 16; ++qp) {
      uint32_t bh[4], bl[4];
      const int hr = 16 * qp + (lane & 7) + ((lane >> 4) << 3), hc = 16 * kk + ((lane >> 3) & 1) * 8;
      ldsm_x4(Hh + hr * CP + hc, bh);
      ldsm_x4(Hl + hr * CP + hc, bl);
      mma_bf16(Yi[2 * qp], af, bh[0], bh[1]);
      mma_bf16(Yi[2 * qp], af, bl[0], bl[1]);
      mma_bf16(Yi[2 * qp + 1], af, bh[2], bh[3]);
      mma_bf16(Yi[2 * qp + 1], af, bl[2], bl[3]);
    }
  }
  // ---- y = y_intra + exp(s_t) y_inter + D x
  const float Dh = a.D[h];
  const float ex0 = expf(cs0), ex1 = expf(cs1);
#pragma unroll
  for (int q = 0; q < P / 8; ++q) {
    const int p0 = 8 * q + 2 * tq;
    if (tr0 < qc) {
      const uint32_t xx = *reinterpret_cast<const uint32_t*>(Xs + tr0 * XP + p0);
      float* yo = a.y + (size_t)(t0 + tr0) * a.ldy + (size_t)h * P + p0;
      *reinterpret_cast<float2*>(yo) =
          make_float2(Y[q][0] + ex0 * Yi[q][0] + Dh * bf16lo(xx), Y[q][1] + ex0 * Yi[q][1] + Dh * bf16hi(xx));
    }
    if (tr1 < qc) {
      const uint32_t xx = *reinterpret_cast<const uint32_t*>(Xs + tr1 * XP + p0);
      float* yo = a.y + (size_t)(t0 + tr1) * a.ldy + (size_t)h * P + p0;
      *reinterpret_cast<float2*>(yo) =
          make_float2(Y[q][2] + ex1 * Yi[q][2] + Dh * bf16lo(xx), Y[q][3] + ex1 * Yi[q][3] + Dh * bf16hi(xx));
    }
  }
}

// ------------------------------------------------------------------ tcgen05 chunk kernels
//
// The chunk products of the 128-state shape on the 5th-generation tensor
// cores: operands in shared memory in the K-major, 128-byte-swizzled layout
// (sw128_desc), one thread issuing tcgen05.mma (kind::f16, bf16 operands,
// fp32 accumulation in tensor memory), four warps draining tensor memory
// (warp w reads lanes 32w..32w+31).  Operand rounding as in the warp-MMA
// kernels: x, B, C enter exactly; the fp32 operands (the decay-weighted L,
// w_s x_s, h_in) as hi + lo bf16 pairs, two MMAs each.
//   state: dH^T [n][p] = B^T [n][s] (w x)^T [p][s]^T   (M = 128 n, N = P, K = 128 s)
//   out:   S = C [t][n] B [s][n]^T                      (M = 128 t, N = 128 s, K = 128 n)
//          Yi = C [t][n] h_in [p][n]^T                  (N = P, K = 128 n)
//          Y  = L [t][s] x^T [p][s]^T                   (N = P, K = 128 s), L = mask(S) * exp(s_t - s_s) * dt_s
// Every wait is bounded; the issuing thread drains its MMAs before tensor
// memory is freed.
constexpr int kSsdTcThreads = 128;     // state kernel: 4 warps, one per TMEM lane quarter
constexpr int kSsdTcOutThreads = 256;  // output kernel: 8 warps, two per lane quarter (column halves)

// Stores the 8 bf16 values v[0..7] of K positions k0..k0+7 of row r of a
// K-major swizzled tile of R rows (k0 % 8 == 0).
__device__ __forceinline__ void sw_store8(uint8_t* tile, int R, int r, int k0, const uint4& v) {
  *reinterpret_cast<uint4*>(tile + sw128_chunk(R, r, k0 >> 3)) = v;
}
// 8 x 8 block of 16-bit values: in[r] holds row r (8 values, packed in
// pairs), out[c] receives column c (the 8 rows' values).
__device__ __forceinline__ void transpose8x8(const uint4 (&in)[8], uint4 (&out)[8]) {
  uint32_t w[8][4];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    w[r][0] = in[r].x;
    w[r][1] = in[r].y;
    w[r][2] = in[r].z;
    w[r][3] = in[r].w;
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // rows 2j and 2j+1 of column c: low or high half of word c/2
      const uint32_t sel = (c & 1) ? 0x7632u : 0x5410u;
      o[j] = __byte_perm(w[2 * j][c >> 1], w[2 * j + 1][c >> 1], sel);
    }
    out[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// 8 fp32 values -> hi and lo bf16 parts, v = hi + lo (packed in pairs).
__device__ __forceinline__ void split8(const float (&v)[8], uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) split2(v[2 * i], v[2 * i + 1], h[i], l[i]);
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// MMAs of an M = 128 tile: K = 128 (8 steps of 16) from K-major swizzled A
// (128 rows) and B (NB rows) into tensor memory at d; accumulate onto d when
// acc0 (else the first step overwrites).
__device__ __forceinline__ void tc_mma_k128(uint32_t d, const uint8_t* A, const uint8_t* B, int NB, uint32_t idesc,
                                            int acc0) {
  const uint32_t a0 = smem_addr(A), b0 = smem_addr(B);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const int atom = kk >> 2, within = (kk & 3) * 32;
    tc_mma(d, sw128_desc(a0 + atom * 128 * 128 + within), sw128_desc(b0 + atom * NB * 128 + within), idesc,
           (acc0 || kk > 0) ? 1 : 0);
  }
}

template <int P>
__global__ void __launch_bounds__(kSsdTcThreads, 1) ssd_state_tc_kernel(const SsdArgs a) {
  constexpr int N = 128;
  const int h = blockIdx.x, c = blockIdx.y;
  int seq, t0, qc;
  chunk_info(a, c, seq, t0, qc);
  const int g = h / (a.H / a.G);
  const int tid = threadIdx.x, warp = tid >> 5;
  __shared__ float dt_s[kQ], cs_s[kQ];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_slot;
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Bt = sm;                   // B^T [128 n][128 s]
  uint8_t* Wh = Bt + N * kQ * 2;      // (w x)^T hi [P][128 s]
  uint8_t* Wl = Wh + P * kQ * 2;      // lo
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_slot, P < 32 ? 32 : P);
  chunk_decay(a, h, t0, qc, dt_s, cs_s);  // ends with __syncthreads
  const float last = cs_s[max(qc - 1, 0)];
  // B^T and (w x)^T, zero past the chunk's tokens, in 8 x 8 blocks (16-byte
  // loads, a register transpose, 16-byte stores; block (sb, nb) of a thread:
  // the eight lanes of a store phase hold eight different sb, so their
  // swizzled chunks differ)
  for (int i = tid; i < (kQ / 8) * (N / 8); i += kSsdTcThreads) {
    const int s0 = (i % (kQ / 8)) * 8, n0 = (i / (kQ / 8)) * 8;
    uint4 rows[8], cols[8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
      rows[r] = s0 + r < qc ? *reinterpret_cast<const uint4*>(a.Bm + (size_t)(t0 + s0 + r) * a.ld_in + (size_t)g * N + n0)
                            : make_uint4(0u, 0u, 0u, 0u);
    transpose8x8(rows, cols);
#pragma unroll
    for (int c = 0; c < 8; ++c) sw_store8(Bt, N, n0 + c, s0, cols[c]);
  }
  for (int i = tid; i < (kQ / 8) * (P / 8); i += kSsdTcThreads) {
    const int s0 = (i % (kQ / 8)) * 8, p0 = (i / (kQ / 8)) * 8;
    uint4 rh[8], rl[8], ch[8], cl[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int s_ = s0 + r;
      float v[8];
      if (s_ < qc) {
        const uint4 xv = *reinterpret_cast<const uint4*>(a.x + (size_t)(t0 + s_) * a.ld_in + (size_t)h * P + p0);
        const float w = expf(last - cs_s[s_]) * dt_s[s_];
        const uint32_t x4[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[2 * e] = w * bf16lo(x4[e]);
          v[2 * e + 1] = w * bf16hi(x4[e]);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = 0.0f;
      }
      split8(v, rh[r], rl[r]);
    }
    transpose8x8(rh, ch);
    transpose8x8(rl, cl);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      sw_store8(Wh, P, p0 + c, s0, ch[c]);
      sw_store8(Wl, P, p0 + c, s0, cl[c]);
    }
  }
  fence_proxy_async();  // generic-proxy stores -> visible to the tensor cores
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (tid == 0) {
    constexpr uint32_t idesc = tc_idesc(128, P);
    tc_mma_k128(tmem, Bt, Wh, P, idesc, 0);
    tc_mma_k128(tmem, Bt, Wl, P, idesc, 1);
    tc_commit(&bar);
  }
  // tcgen05.ld is warp-collective (.sync.aligned): every lane of a warp takes
  // the same branch around it
  const bool ok = __all_sync(0xffffffffu, mbar_wait(&bar, 0));
  tc_fence_after();
  if (ok) {
    // thread (warp w, lane l) holds row n = 32 w + l: P columns
    const int n = tid;
    float* out = a.dH + ((size_t)h * a.nchunks + c) * P * N;
#pragma unroll
    for (int c0 = 0; c0 < P; c0 += 16) {
      float v[16];
      tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + c0, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) out[(size_t)(c0 + j) * N + n] = v[j];
    }
  }
  if (tid == 0) {
    a.decay[(size_t)h * a.nchunks + c] = expf(last);
    mbar_drain(&bar, 0);  // no MMA still writes tensor memory when it is freed
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_free(tmem, P < 32 ? 32 : P);
  }
}

template <int P>
// two CTAs per SM: 97 KB of shared memory and 256 TMEM columns each
__global__ void __launch_bounds__(kSsdTcOutThreads, 2) ssd_out_tc_kernel(const SsdArgs a) {
  constexpr int N = 128;
  constexpr uint32_t kCols = 256;  // S: 128, Yi: P, Y: P
  const int h = blockIdx.x, c = blockIdx.y;
  int seq, t0, qc;
  chunk_info(a, c, seq, t0, qc);
  const int g = h / (a.H / a.G);
  const int tid = threadIdx.x, warp = tid >> 5;
  __shared__ float dt_s[kQ], cs_s[kQ];
  __shared__ __align__(8) uint64_t bar[2];
  __shared__ uint32_t tmem_slot;
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
  // 96 KB at P = 64 (two CTAs per SM): the space of C and B takes L once S
  // and Yi are done, that of h_in takes x^T
  uint8_t* Cs = sm;                   // C [128 t][128 n], then L hi [128 t][128 s]
  uint8_t* Bs = Cs + kQ * N * 2;      // B [128 s][128 n], then L lo
  uint8_t* Hh = Bs + kQ * N * 2;      // h_in hi [P][128 n], then x^T [P][128 s]
  uint8_t* Hl = Hh + P * N * 2;       // h_in lo
  uint8_t* Xt = Hh;
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_slot, kCols);
  // C, B rows (zero past the chunk), x^T, h_in split.  Each thread issues a
  // batch of its loads before any of the stores that use them (the stores go
  // through generic pointers, so the compiler keeps a later iteration's loads
  // behind an earlier iteration's stores: one L2 round trip per iteration),
  // and the first batch before the chunk's decays, whose dt loads and prefix
  // sum then overlap it.
  constexpr int kCb = kQ * (N / 8) / kSsdTcOutThreads;  // 8 row pieces of C and of B per thread
  constexpr int kHp = P * (N / 8) / kSsdTcOutThreads;   // row pieces of h_in per thread
  static_assert(kQ * (N / 8) % kSsdTcOutThreads == 0 && kCb % 2 == 0, "C/B pieces per thread");
  static_assert(P * (N / 8) % kSsdTcOutThreads == 0, "h_in pieces per thread");
  const float* hin = a.dH + ((size_t)h * a.nchunks + c) * P * N;
  uint4 cv[kCb / 2], bv[kCb / 2];
  float4 f[2 * kHp];
  auto load_cb = [&](int bt) {
#pragma unroll
    for (int j = 0; j < kCb / 2; ++j) {
      const int i = tid + kSsdTcOutThreads * (bt * (kCb / 2) + j);
      const int r = i / (N / 8), n0 = (i % (N / 8)) * 8;
      cv[j] = bv[j] = make_uint4(0u, 0u, 0u, 0u);
      if (r < qc) {
        const size_t row = (size_t)(t0 + r) * a.ld_in + (size_t)g * N + n0;
        cv[j] = *reinterpret_cast<const uint4*>(a.Cm + row);
        bv[j] = *reinterpret_cast<const uint4*>(a.Bm + row);
      }
    }
  };
  auto store_cb = [&](int bt) {
#pragma unroll
    for (int j = 0; j < kCb / 2; ++j) {
      const int i = tid + kSsdTcOutThreads * (bt * (kCb / 2) + j);
      const int r = i / (N / 8), n0 = (i % (N / 8)) * 8;
      sw_store8(Cs, kQ, r, n0, cv[j]);
      sw_store8(Bs, kQ, r, n0, bv[j]);
    }
  };
  load_cb(0);
#pragma unroll
  for (int j = 0; j < kHp; ++j) {
    const int i = tid + kSsdTcOutThreads * j;
    const int pp = i / (N / 8), n0 = (i % (N / 8)) * 8;
    f[2 * j] = *reinterpret_cast<const float4*>(hin + (size_t)pp * N + n0);
    f[2 * j + 1] = *reinterpret_cast<const float4*>(hin + (size_t)pp * N + n0 + 4);
  }
  chunk_decay(a, h, t0, qc, dt_s, cs_s);
  store_cb(0);
  load_cb(1);
  store_cb(1);
#pragma unroll
  for (int j = 0; j < kHp; ++j) {
    const int i = tid + kSsdTcOutThreads * j;
    const int pp = i / (N / 8), n0 = (i % (N / 8)) * 8;
    const float v[8] = {f[2 * j].x, f[2 * j].y, f[2 * j].z, f[2 * j].w,
                        f[2 * j + 1].x, f[2 * j + 1].y, f[2 * j + 1].z, f[2 * j + 1].w};
    uint4 hi, lo;
    split8(v, hi, lo);
    sw_store8(Hh, P, pp, n0, hi);
    sw_store8(Hl, P, pp, n0, lo);
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t tS = tmem, tYi = tmem + 128, tY = tmem + 128 + P;
  if (tid == 0) {
    tc_mma_k128(tS, Cs, Bs, kQ, tc_idesc(128, 128), 0);  // S = C B^T
    tc_mma_k128(tYi, Cs, Hh, P, tc_idesc(128, P), 0);    // Yi = C h_in^T
    tc_mma_k128(tYi, Cs, Hl, P, tc_idesc(128, P), 1);
    tc_commit(&bar[0]);
  }
  // x^T goes into the space of h_in once the MMAs above have read it, in
  // 8 x 8 blocks (one per thread at most); its rows are loaded while they run
  static_assert((kQ / 8) * (P / 8) <= kSsdTcOutThreads, "one x^T block per thread");
  const bool xb = tid < (kQ / 8) * (P / 8);
  const int xs0 = (tid % (kQ / 8)) * 8, xp0 = (tid / (kQ / 8)) * 8;
  uint4 xrows[8];
#pragma unroll
  for (int r = 0; r < 8; ++r)
    xrows[r] = (xb && xs0 + r < qc)
                   ? *reinterpret_cast<const uint4*>(a.x + (size_t)(t0 + xs0 + r) * a.ld_in + (size_t)h * P + xp0)
                   : make_uint4(0u, 0u, 0u, 0u);
  // tcgen05.ld is warp-collective (.sync.aligned): every lane of a warp loads,
  // whatever its own row; only stores depend on the row
  bool ok = __all_sync(0xffffffffu, mbar_wait(&bar[0], 0));
  tc_fence_after();
  if (xb) {
    uint4 cols[8];
    transpose8x8(xrows, cols);
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) sw_store8(Xt, P, xp0 + c8, xs0, cols[c8]);
  }
  // L row t = 32 (w mod 4) + l, columns [64 (w / 4), +64) (C and B are no
  // longer read: their space takes L)
  const int q = warp & 3, half = warp >> 2;
  const int t = 32 * q + (tid & 31);
  const uint32_t lane_base = (uint32_t)(32 * q) << 16;
  {
    const float cst = cs_s[t];
#pragma unroll 1
    for (int s0 = 64 * half; s0 < 64 * half + 64; s0 += 16) {
      // columns s0 .. s0 + 15 lie above the diagonal for all of this warp's
      // rows t < 32 (q + 1) when s0 >= 32 (q + 1): zeros, nothing to compute
      if (s0 >= 32 * (q + 1)) {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        sw_store8(Cs, kQ, t, s0, z);
        sw_store8(Bs, kQ, t, s0, z);
        sw_store8(Cs, kQ, t, s0 + 8, z);
        sw_store8(Bs, kQ, t, s0 + 8, z);
        continue;
      }
      float v[16];
      if (ok) {
        tmem_ld16(tS + lane_base + s0, v);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = 0.0f;
      }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float l8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int s_ = s0 + 8 * half + j;
          // the hardware exp2 approximation (relative error a few 2^-23): L
          // enters the MMA as a bf16 hi + lo pair, about 16 significant bits
          l8[j] = (s_ <= t) ? v[8 * half + j] * __expf(cst - cs_s[s_]) * dt_s[s_] : 0.0f;
        }
        uint4 hi, lo;
        split8(l8, hi, lo);
        sw_store8(Cs, kQ, t, s0 + 8 * half, hi);
        sw_store8(Bs, kQ, t, s0 + 8 * half, lo);
      }
    }
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    tc_mma_k128(tY, Cs, Xt, P, tc_idesc(128, P), 0);  // Y = L x
    tc_mma_k128(tY, Bs, Xt, P, tc_idesc(128, P), 1);
    tc_commit(&bar[1]);
  }
  ok = __all_sync(0xffffffffu, mbar_wait(&bar[1], 0)) && ok;
  tc_fence_after();
  // y = Y + exp(s_t) Yi + D x through shared memory (the space of L, whose
  // MMAs are done; x from the x^T tile): each thread its row's half, then
  // each warp stores whole rows
  constexpr int kYp = P + 1;  // row pitch in floats: a warp's 32 rows fall in 32 banks
  float* Ys = reinterpret_cast<float*>(Cs);
  static_assert(kQ * (P + 1) * 4 <= 2 * kQ * N * 2, "y tile in the space of L");
  if (ok) {
    const float Dh = a.D[h];
    const float ex = expf(cs_s[t]);
#pragma unroll
    for (int c0 = half * (P / 2); c0 < (half + 1) * (P / 2); c0 += 16) {
      float y1[16], yi[16];
      tmem_ld16(tY + lane_base + c0, y1);
      tmem_ld16(tYi + lane_base + c0, yi);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int pp = c0 + j;
        const uint16_t xv = *reinterpret_cast<const uint16_t*>(Xt + sw128_chunk(P, pp, t >> 3) + (t & 7) * 2);
        Ys[t * kYp + pp] = y1[j] + ex * yi[j] + Dh * bf16_to_f32(xv);
      }
    }
  }
  __syncthreads();
  if (ok) {
    for (int r = warp; r < qc; r += kSsdTcOutThreads / 32) {
      float* yo = a.y + (size_t)(t0 + r) * a.ldy + (size_t)h * P;
#pragma unroll
      for (int pp = (tid & 31); pp < P; pp += 32) yo[pp] = Ys[r * kYp + pp];
    }
  }
  if (tid == 0) mbar_drain(&bar[1], 0);  // no MMA still writes tensor memory when it is freed
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_free(tmem, kCols);
  }
}

template <int P>
constexpr int ssd_state_tc_smem() { return (128 * kQ + 2 * P * kQ) * 2 + 1024; }
template <int P>
constexpr int ssd_out_tc_smem() { return (2 * kQ * 128 + 2 * P * 128) * 2 + 1024; }

template <int P>
static cudaError_t launch_ssd_tc_t(const SsdArgs& a, const dim3& grid, int which, cudaStream_t s) {
  static int done_s[64], done_o[64];
  if (which == 0) {
    constexpr int smem = ssd_state_tc_smem<P>();
    cudaError_t e = set_smem_once((const void*)ssd_state_tc_kernel<P>, smem, done_s);
    if (e != cudaSuccess) return e;
    ssd_state_tc_kernel<P><<<grid, kSsdTcThreads, smem, s>>>(a);
  } else {
    constexpr int smem = ssd_out_tc_smem<P>();
    cudaError_t e = set_smem_once((const void*)ssd_out_tc_kernel<P>, smem, done_o);
    if (e != cudaSuccess) return e;
    ssd_out_tc_kernel<P><<<grid, kSsdTcOutThreads, smem, s>>>(a);
  }
  return cudaGetLastError();
}

// Shapes on the tcgen05 chunk kernels: 128 states (M = 128 for the state
// product), head dims 32 and 64.
static bool ssd_tc_shape(int P, int N) { return N == 128 && (P == 64 || P == 32); }

template <int P, int N>
constexpr int ssd_state_mma_smem() { return (kQ * (N + 8) + 2 * kQ * (P + 8)) * 2; }
template <int P, int N>
constexpr int ssd_out_mma_smem() { return (2 * kQ * (N + 8) + kQ * (P + 8) + 2 * P * (N + 8)) * 2; }

// Shapes with tensor-core chunk kernels.
static bool ssd_mma_shape(int P, int N) {
  return (P == 64 && N == 128) || (P == 32 && N == 16) || (P == 64 && N == 64) || (P == 32 && N == 128);
}

template <int P, int N>
static cudaError_t launch_ssd_mma_t(const SsdArgs& a, const dim3& grid, int which, cudaStream_t s) {
  static int done_s[64], done_o[64];
  if (which == 0) {
    constexpr int smem = ssd_state_mma_smem<P, N>();
    cudaError_t e = set_smem_once((const void*)ssd_state_mma_kernel<P, N>, smem, done_s);
    if (e != cudaSuccess) return e;
    ssd_state_mma_kernel<P, N><<<grid, kSsdThreads, smem, s>>>(a);
  } else {
    constexpr int smem = ssd_out_mma_smem<P, N>();
    cudaError_t e = set_smem_once((const void*)ssd_out_mma_kernel<P, N>, smem, done_o);
    if (e != cudaSuccess) return e;
    ssd_out_mma_kernel<P, N><<<grid, kSsdThreads, smem, s>>>(a);
  }
  return cudaGetLastError();
}

static cudaError_t launch_ssd_mma(const SsdArgs& a, const dim3& grid, int which, cudaStream_t s) {
  if (a.P == 64 && a.N == 128) return launch_ssd_mma_t<64, 128>(a, grid, which, s);
  if (a.P == 32 && a.N == 16) return launch_ssd_mma_t<32, 16>(a, grid, which, s);
  if (a.P == 64 && a.N == 64) return launch_ssd_mma_t<64, 64>(a, grid, which, s);
  return launch_ssd_mma_t<32, 128>(a, grid, which, s);
}

bool ssd_supported(int H, int P, int N, int G) {
  if (G <= 0 || H % G || P % 8 || N % 4) return false;
  return smem_out_bytes(P, N) <= 227 * 1024 && smem_state_bytes(P, N) <= 227 * 1024;
}

int32_t ssd_chunk_table(const int32_t* cu, int32_t nseq, int32_t* tab) {
  int32_t nc = 0;
  for (int i = 0; i <= nseq; ++i) tab[i] = cu[i];
  for (int i = 0; i < nseq; ++i) {
    tab[nseq + 1 + i] = nc;
    nc += (cu[i + 1] - cu[i] + kQ - 1) / kQ;
  }
  tab[2 * nseq + 1] = nc;
  return nc;
}

size_t ssd_workspace_bytes(int nchunks, int H, int P, int N) {
  const size_t nc = (size_t)nchunks;
  return ((nc * H * P * N * 4 + 255) / 256) * 256 + ((nc * H * 4 + 255) / 256) * 256;
}

static int done_state[64], done_out[64];

cudaError_t launch_ssd(const SsdArgs& a0, cudaStream_t s) {
  SsdArgs a = a0;
  const int smem_state = smem_state_bytes(a.P, a.N);
  const int smem_out = smem_out_bytes(a.P, a.N);
  cudaError_t e = set_smem_once((const void*)ssd_chunk_state_kernel, smem_state, done_state);
  if (e != cudaSuccess) return e;
  e = set_smem_once((const void*)ssd_chunk_out_kernel, smem_out, done_out);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.H, a.nchunks);
  const bool tc = ssd_tc_shape(a.P, a.N);
  const bool mma = ssd_mma_shape(a.P, a.N);
  trace_pre(K_SSD_CHUNK_STATE, s);
  if (tc) {
    e = a.P == 64 ? launch_ssd_tc_t<64>(a, grid, 0, s) : launch_ssd_tc_t<32>(a, grid, 0, s);
  } else if (mma) {
    e = launch_ssd_mma(a, grid, 0, s);
  } else {
    ssd_chunk_state_kernel<<<grid, kSsdThreads, smem_state, s>>>(a);
    e = cudaGetLastError();
  }
  trace_post(K_SSD_CHUNK_STATE, s);
  if (e != cudaSuccess) return e;
  const size_t n4 = (size_t)a.H * a.P * a.N / 4;
  trace_pre(K_SSD_STATE_PASS, s);
  ssd_state_pass_kernel<<<dim3((unsigned)((n4 + 255) / 256), a.nseq), 256, 0, s>>>(a);
  trace_post(K_SSD_STATE_PASS, s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  trace_pre(K_SSD_CHUNK_OUT, s);
  if (tc) {
    e = a.P == 64 ? launch_ssd_tc_t<64>(a, grid, 1, s) : launch_ssd_tc_t<32>(a, grid, 1, s);
  } else if (mma) {
    e = launch_ssd_mma(a, grid, 1, s);
  } else {
    ssd_chunk_out_kernel<<<grid, kSsdThreads, smem_out, s>>>(a);
    e = cudaGetLastError();
  }
  trace_post(K_SSD_CHUNK_OUT, s);
  return e;
}

}  // namespace m2
