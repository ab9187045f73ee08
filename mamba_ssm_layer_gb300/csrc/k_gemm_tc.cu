// k_gemm_tc.cu -- tensor-core (tcgen05) w8a16 / bf16 GEMM for prefill and
// batched decode: out[m][n] = sum_k A[m][k] * W~[n][k] for M > 8 token rows.
//
// W~ = E4M3(W) * S[n/128][k/128] (page "Struct Qwen3SsmLayer",
// `set_fp8_decode_weights`; scale index of "Struct NemotronMamba2Layer",
// `set_fp8_weights`), or bf16 W.  tcgen05 has no 16-bit x E4M3 MMA and E4M3
// activations would change the numbers, so each E4M3 weight tile is converted
// exactly (every E4M3 value is an f16 and a bf16 value) and multiplied by the
// 16-bit activations with kind::f16 (fp32 accumulation in TMEM).  The
// converted tile goes to tensor memory, the MMA's A operand there: the
// converters read 16 KB of shared memory per k block and the MMA reads only
// the activation tile from shared memory.  The 128x128 block scale is not a
// power of two and varies with the k block, so it cannot ride on the MMA:
// each 128-wide k block is accumulated alone into a TMEM buffer and the
// epilogue promotes it, acc += s * partial.
//
// The MMA computes D^T: UMMA M = 128 weight rows (one scale row block), UMMA N
// = NT token rows, so one tile is [128 weight rows] x [NT tokens]; NT is 16,
// 32, 64 or 128, the narrowest that holds the rows (the activation tile is
// copied and multiplied whole).
// Persistent CTAs walk work items (a tile, or a k range of a tile when the
// tiles alone would leave most SMs idle) weight-tile major, so the token tiles
// of one weight tile are adjacent and its bytes are re-read from L2.  Roles
// (each ring has its own fill and free barriers; the MMA issuer frees the
// slots it read with one commit each per k block):
//   warp 0      weight producer (lane 0): TMA of the E4M3 tile [128][128]
//               (128-byte swizzle) into a ring; bf16 weights go straight into a
//               ring of 128-byte-swizzled tiles, the MMA's A operand.  It does
//               not wait for the previous kernel: weights are never its output.
//   warp 22     activation producer (lane 0): after the dependency wait, one
//               3-D tensor copy per k block of the 16-bit activation tile
//               [NT][128] (two 64-wide halves, 128-byte swizzle = the UMMA
//               K-major canonical layout) into a ring;
//   warps 2-5   converters (E4M3 weights): one weight row per thread (its TMEM
//               lane), E4M3 -> f16 (prescaled f16 activations) or bf16, stored
//               with tcgen05.st into one of the A stages in TMEM;
//   warp 1      TMEM allocation; lane 0 issues 8 MMAs (K = 16 each) per k block
//               into one of the TMEM partial buffers, then commits per ring;
//   warps 6-21  epilogue, four warps per TMEM lane quarter (each a quarter of
//               the token columns): per k block, TMEM -> registers, acc += s * partial;
//               per item, the store / residual / conv-update epilogue, or fp32
//               partials that a second kernel sums in split order.
// Every wait is bounded (see mbar_wait); TMEM is freed on every exit path.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "m2_common.cuh"
#include "m2_kernels.h"
#include "m2_tc.cuh"

namespace m2 {

constexpr int kTcEpiWarps = 16;  // four per TMEM lane quarter, each a quarter of the token columns
constexpr int kTcAWarp = 6 + kTcEpiWarps;       // activation producer
constexpr int kTcThreads = (kTcAWarp + 1) * 32;  // 23 warps
constexpr int kTcBM = 128;       // weight rows per tile (UMMA M)
constexpr int kTcBK = 128;       // k per block (= scale block)

struct TcBars {
  static constexpr int kMaxRing = 8, kMaxTmem = 4;
  uint64_t w_full[kMaxRing], w_empty[kMaxRing];
  uint64_t a_full[kMaxRing], a_empty[kMaxRing];
  uint64_t ta_full[kMaxTmem], ta_empty[kMaxTmem];
  uint64_t mma_done[kMaxTmem], tmem_empty[kMaxTmem];
  uint32_t tmem_base;
};

// Shared memory (offsets from a 1024-byte aligned base) and tensor memory of
// one CTA.  E4M3 weights (FP8): raw 16 KB tiles in the weight ring, converted
// tiles in TMEM (64 columns each, after the partial buffers), so both rings
// fill shared memory.  bf16 weights: 32 KB swizzled tiles.
template <int NT, bool FP8>
struct TcLayout {
  static constexpr int kWStages = FP8 ? (NT <= 32 ? 8 : (NT <= 64 ? 6 : 4)) : 4;
  static constexpr int kWBytes = FP8 ? kTcBM * kTcBK : kTcBM * kTcBK * 2;
  static constexpr int kAStages = FP8 ? (NT <= 32 ? 8 : (NT <= 64 ? 6 : 5)) : (NT <= 64 ? 4 : 3);
  static constexpr int kABytes = NT * kTcBK * 2;  // one activation stage
  static constexpr int kTBufs = (FP8 && NT > 64) ? 3 : 4;  // k-block partials in TMEM
  static constexpr int kTAStages = FP8 ? (NT <= 64 ? 4 : 2) : 0;  // converted weight tiles in TMEM
  static constexpr int kTACol = kTBufs * NT;  // first column of the A stages
  static constexpr int kTmemCols = FP8 ? 512 : kTBufs * NT;
  static constexpr int kW = 0;
  static constexpr int kA = kWStages * kWBytes;
  static constexpr int kBars = kA + kAStages * kABytes;
  static_assert(kTACol + kTAStages * (kTcBK / 2) <= kTmemCols && kTmemCols <= 512, "TMEM budget");
  static_assert(kWStages <= TcBars::kMaxRing && kAStages <= TcBars::kMaxRing, "ring barriers");
  static_assert(kTAStages <= TcBars::kMaxTmem && kTBufs <= TcBars::kMaxTmem, "TMEM barriers");
  static_assert(kBars + (int)sizeof(TcBars) + 1024 <= 232448, "shared memory");
};


template <int NT, bool FP8>
constexpr int tc_smem_bytes() {
  return TcLayout<NT, FP8>::kBars + (int)sizeof(TcBars) + 1024;  // + alignment slack
}

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Two E4M3 -> two bf16, exactly (E4M3 -> f16 -> f32 -> bf16 are all exact).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two_bytes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)two_bytes));
  float lo, hi;
  asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h2));
  return pack_bf16x2(lo, hi);
}

// Two E4M3 -> two f16, exactly (every E4M3 value is an f16 normal).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)two_bytes));
  return h2;
}

// Conv taps of one channel: history taps 0..L-1 (oldest first) and the tap
// of the current token, in registers (indexed with compile-time indices only).
struct ConvTaps {
  float hist[7];
  float cur, bias;
};

__device__ __forceinline__ void load_taps(const GemvArgs& a, int c, int L, ConvTaps& t) {
#pragma unroll
  for (int j = 0; j < 7; ++j) t.hist[j] = j < L ? bf16_to_f32(a.conv_w[(size_t)c * a.dconv + j]) : 0.0f;
  t.cur = bf16_to_f32(a.conv_w[(size_t)c * a.dconv + L]);
  t.bias = a.conv_b ? bf16_to_f32(a.conv_b[c]) : 0.0f;
}

// The store / residual / conv-update epilogue of one output (token m, row n).
// Conv rows: this thread alone owns (sequence m, channel c), so the ring taps
// it reads are the previous tokens' and the slot it writes is its own.
__device__ __forceinline__ void tc_epi_elem(const GemvArgs& a, int m, int n, float acc, bool conv,
                                            const ConvTaps& t, int L) {
  uint16_t* o = a.out + (size_t)m * a.ldo + n;
  if (a.epi == EPI_RESID) {
    *o = f32_to_bf16(bf16_to_f32(a.resid[(size_t)m * a.ldr + n]) + acc);
  } else if (conv) {
    const uint16_t vb = f32_to_bf16(acc);  // rounding point of the in_proj output
    const int c = n - a.xbc0;
    uint16_t* rg = a.ring + (size_t)m * L * a.d_xbc;
    const int p = a.pos[m];
    float sv = t.bias;
#pragma unroll
    for (int j = 0; j < 7; ++j)
      if (j < L) sv += t.hist[j] * bf16_to_f32(rg[(size_t)((p + j) % L) * a.d_xbc + c]);
    sv += t.cur * bf16_to_f32(vb);
    *o = f32_to_bf16(silu_f(sv));
    rg[(size_t)(p % L) * a.d_xbc + c] = vb;
  } else {
    *o = f32_to_bf16(acc);
  }
}

// The end-of-item epilogue of one thread: weight row n, token columns m0 ..
// m0 + HC - 1 of acc.  The mode is decided once, outside the per-column loops,
// so that each unrolled loop stays a few hundred instructions (every epilogue
// warp runs it once per item; one loop holding all modes' code, 64 times over,
// ran from instruction-cache misses).  Loads come before the stores of the
// same columns: `out` may alias `resid` (and the conv ring is written here), so
// a load placed after a store could not be moved ahead of it, and each column
// would wait one memory round trip behind the previous column's store.  Each
// element is read and written by this thread alone, so reading all first is
// exact.
template <int HC>
__device__ __forceinline__ void tc_item_store(const GemvArgs& a, int ksplit, float* part, int ks, int n, int m0,
                                              const float (&acc)[HC], int L) {
  if (n >= a.N) return;
  const int mc = min(HC, a.M - m0);
  if (ksplit > 1) {
    float* pp = part + ((size_t)ks * a.M + m0) * a.N + n;
#pragma unroll
    for (int j = 0; j < HC; ++j)
      if (j < mc) pp[(size_t)j * a.N] = acc[j];
  } else if (a.epi == EPI_RESID) {
    uint16_t* o = a.out + (size_t)m0 * a.ldo + n;
    const uint16_t* r = a.resid + (size_t)m0 * a.ldr + n;
    constexpr int G = HC < 8 ? HC : (HC >= 64 ? 4 : 8);  // columns whose loads are in flight together
#pragma unroll
    for (int j0 = 0; j0 < HC; j0 += G) {
      uint16_t rv[G];
#pragma unroll
      for (int g = 0; g < G; ++g) rv[g] = j0 + g < mc ? r[(size_t)(j0 + g) * a.ldr] : (uint16_t)0;
#pragma unroll
      for (int g = 0; g < G; ++g)
        if (j0 + g < mc) o[(size_t)(j0 + g) * a.ldo] = f32_to_bf16(bf16_to_f32(rv[g]) + acc[j0 + g]);
    }
  } else if (a.epi == EPI_INPROJ_CONV && n >= a.xbc0 && n < a.xbc0 + a.d_xbc) {
    // conv update of channel c for each token column (a sequence in batched
    // decode), G columns at a time: their positions and ring taps are loaded,
    // then their outputs and new ring slots stored
    constexpr int G = 4;
    const int c = n - a.xbc0;
    ConvTaps t;
    load_taps(a, c, L, t);
    float v[HC];
#pragma unroll
    for (int j = 0; j < HC; ++j) v[j] = acc[j];
#pragma unroll 1
    for (int j0 = 0; j0 < mc; j0 += G) {
      int p[G];
      float hv[G][7];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        p[g] = j0 + g < mc ? a.pos[m0 + j0 + g] : 0;
        const uint16_t* rg = a.ring + (size_t)(m0 + j0 + g) * L * a.d_xbc + c;
#pragma unroll
        for (int i = 0; i < 7; ++i)
          hv[g][i] = (i < L && j0 + g < mc) ? bf16_to_f32(rg[(size_t)((p[g] + i) % L) * a.d_xbc]) : 0.0f;
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        if (j0 + g >= mc) break;
        const int m = m0 + j0 + g;
        const uint16_t vb = f32_to_bf16(v[j0 + g]);  // rounding point of the in_proj output
        float sv = t.bias;
#pragma unroll
        for (int i = 0; i < 7; ++i)
          if (i < L) sv += t.hist[i] * hv[g][i];
        sv += t.cur * bf16_to_f32(vb);
        a.out[(size_t)m * a.ldo + n] = f32_to_bf16(silu_f(sv));
        a.ring[(size_t)m * L * a.d_xbc + (size_t)(p[g] % L) * a.d_xbc + c] = vb;
      }
    }
  } else {
    uint16_t* o = a.out + (size_t)m0 * a.ldo + n;
#pragma unroll
    for (int j = 0; j < HC; ++j)
      if (j < mc) o[(size_t)j * a.ldo] = f32_to_bf16(acc[j]);
  }
}

// ------------------------------------------------------------------ kernel

struct TcArgs {
  GemvArgs g;      // operand pointers, sizes, epilogue
  int32_t m_tiles, n_tiles, kblocks;
  int32_t fp8;
  int32_t f16;     // fp8 weights with prescaled f16 activations: f16 x f16 MMAs, columns unscaled
  int32_t ksplit;  // > 1: k blocks split over work items, fp32 partials to `part`
  float* part;     // [ksplit][M][N]
};

// Work item i: weight tile, token tile and k range, weight-tile major so that
// the token tiles of one weight tile are adjacent and its bytes are re-read
// from L2.
__device__ __forceinline__ void tc_item(const TcArgs& ta, int item, int& nt, int& mt, int& kb0, int& kb1) {
  const int tile = item / ta.ksplit, ks = item % ta.ksplit;
  nt = tile / ta.m_tiles;
  mt = tile % ta.m_tiles;
  kb0 = (int)((long long)ta.kblocks * ks / ta.ksplit);
  kb1 = (int)((long long)ta.kblocks * (ks + 1) / ta.ksplit);
}

template <int NT, bool FP8>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA, const TcArgs ta) {
  using Lay = TcLayout<NT, FP8>;
  constexpr int SW = Lay::kWStages, SA = Lay::kAStages, TB = Lay::kTBufs, NA = Lay::kTAStages;
  const GemvArgs& a = ta.g;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  TcBars* bars = reinterpret_cast<TcBars*>(smem + Lay::kBars);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nitems = ta.m_tiles * ta.n_tiles * ta.ksplit;
  const int cid = blockIdx.x, ncl = gridDim.x;
  const int L = a.dconv - 1;

  if (tid == 0) {
    for (int s = 0; s < SW; ++s) {
      mbar_init(&bars->w_full[s], 1);
      mbar_init(&bars->w_empty[s], FP8 ? 4 : 1);  // the converter warps, or the MMA issuer's commit
    }
    for (int s = 0; s < SA; ++s) {
      mbar_init(&bars->a_full[s], 1);
      mbar_init(&bars->a_empty[s], 1);
    }
    for (int s = 0; s < NA; ++s) {
      mbar_init(&bars->ta_full[s], 4);
      mbar_init(&bars->ta_empty[s], 1);
    }
    for (int b = 0; b < TB; ++b) {
      mbar_init(&bars->mma_done[b], 1);
      mbar_init(&bars->tmem_empty[b], kTcEpiWarps);
    }
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&bars->tmem_base, Lay::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  bool dead = false;

  if (warp == 0) {
    // -------------------------------------------------------- weight producer
    // Weights never come from the previous kernel: no dependency wait, so the
    // first tiles stream in while that kernel finishes.
    if (lane == 0) {
      const uint64_t polw = policy_evict_normal();  // weight tiles are re-read by the token tiles
      int gk = 0;
      for (int item = cid; item < nitems && !dead; item += ncl) {
        int nt, mt, kb0, kb1;
        tc_item(ta, item, nt, mt, kb0, kb1);
        for (int kb = kb0; kb < kb1 && !dead; ++kb, ++gk) {
          const int s = gk % SW;
          if (gk >= SW && !mbar_wait(&bars->w_empty[s], ((gk / SW) - 1) & 1)) dead = true;
          if (dead) break;
          uint8_t* wbuf = smem + Lay::kW + s * Lay::kWBytes;
          mbar_arrive_expect_tx(&bars->w_full[s], Lay::kWBytes);
          if constexpr (FP8) {  // E4M3 tile, 128-byte swizzle, for the converters
            tma_load_2d(wbuf, &tmW, kb * kTcBK, nt * kTcBM, &bars->w_full[s], polw);
          } else {
            tma_load_2d(wbuf, &tmW, kb * kTcBK, nt * kTcBM, &bars->w_full[s], polw);
            tma_load_2d(wbuf + kTcBM * 128, &tmW, kb * kTcBK + 64, nt * kTcBM, &bars->w_full[s], polw);
          }
        }
      }
      // drain: the tiles issued (k blocks [0, gk)) have landed before the CTA
      // may exit, also after a timeout stopped their consumers
      for (int k = max(0, gk - SW); k < gk; ++k)
        if (!mbar_drain(&bars->w_full[k % SW], (k / SW) & 1)) break;
    }
  } else if (warp == kTcAWarp) {
    // -------------------------------------------------------- activation producer
    pdl_wait();  // A is written by the previous kernel
    if (lane == 0) {
      const uint64_t pola = policy_evict_last();  // activations are re-read by every weight tile
      int gk = 0;
      for (int item = cid; item < nitems && !dead; item += ncl) {
        int nt, mt, kb0, kb1;
        tc_item(ta, item, nt, mt, kb0, kb1);
        for (int kb = kb0; kb < kb1 && !dead; ++kb, ++gk) {
          const int s = gk % SA;
          if (gk >= SA && !mbar_wait(&bars->a_empty[s], ((gk / SA) - 1) & 1)) dead = true;
          if (dead) break;
          uint8_t* abuf = smem + Lay::kA + s * Lay::kABytes;
          mbar_arrive_expect_tx(&bars->a_full[s], Lay::kABytes);
          tma_load_3d(abuf, &tmA, 0, mt * NT, kb * 2, &bars->a_full[s], pola);  // both halves
        }
      }
      // drain: everything issued has landed before the CTA may exit
      for (int k = max(0, gk - SA); k < gk; ++k)
        if (!mbar_drain(&bars->a_full[k % SA], (k / SA) & 1)) break;
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = ta.f16 ? tc_idesc_f16(kTcBM, NT) : tc_idesc(kTcBM, NT);
      int gk = 0;
      for (int item = cid; item < nitems && !dead; item += ncl) {
        int nt, mt, kb0, kb1;
        tc_item(ta, item, nt, mt, kb0, kb1);
        for (int kb = kb0; kb < kb1 && !dead; ++kb, ++gk) {
          const int s = gk % SW, sa = gk % SA, tb = gk % TB;
          const int na = FP8 ? gk % NA : 0;
          if constexpr (FP8) {
            if (!mbar_wait(&bars->ta_full[na], (gk / NA) & 1)) dead = true;
          } else {
            if (!mbar_wait(&bars->w_full[s], (gk / SW) & 1)) dead = true;
          }
          if (!dead && !mbar_wait(&bars->a_full[sa], (gk / SA) & 1)) dead = true;
          if (!dead && gk >= TB && !mbar_wait(&bars->tmem_empty[tb], ((gk / TB) - 1) & 1)) dead = true;
          if (dead) break;
          tc_fence_after();
          const uint32_t ab = smem_addr(smem + Lay::kA + sa * Lay::kABytes);
#pragma unroll
          for (int kk = 0; kk < kTcBK / 16; ++kk) {
            const int atom = kk >> 2, within = (kk & 3) * 32;  // 64-k atoms of 128 bytes per row
            const uint64_t bd = sw128_desc(ab + atom * NT * 128 + within);
            if constexpr (FP8) {
              // converted tile: k = 16 kk .. 16 kk + 15 in columns 8 kk .. 8 kk + 7
              tc_mma_ts(tmem + tb * NT, tmem + Lay::kTACol + na * (kTcBK / 2) + kk * 8, bd, idesc, kk > 0 ? 1 : 0);
            } else {
              const uint32_t wb = smem_addr(smem + Lay::kW + s * Lay::kWBytes);
              tc_mma(tmem + tb * NT, sw128_desc(wb + atom * kTcBM * 128 + within), bd, idesc, kk > 0 ? 1 : 0);
            }
          }
          // commits: the partial is done (epilogue), and the operand slots this
          // k block read are free (their producers wait on them)
          tc_commit(&bars->mma_done[tb]);
          tc_commit(&bars->a_empty[sa]);
          tc_commit(FP8 ? &bars->ta_empty[na] : &bars->w_empty[s]);
        }
      }
      // drain: no MMA of this thread is still running when TMEM is freed
      // (the last commit tracks all earlier MMAs)
      if (gk > 0) mbar_drain(&bars->mma_done[(gk - 1) % TB], ((gk - 1) / TB) & 1);
    }
  } else if (warp < 6) {
    // -------------------------------------------------------- converters
    if constexpr (FP8) {
      // warp w reaches TMEM lanes 32 (w % 4) .. + 31: one weight row per thread
      const int q = warp & 3, row = 32 * q + lane, r8 = row & 7;
      const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16) + Lay::kTACol;
      int gk = 0;
      for (int item = cid; item < nitems && !dead; item += ncl) {
        int nt, mt, kb0, kb1;
        tc_item(ta, item, nt, mt, kb0, kb1);
        for (int kb = kb0; kb < kb1 && !dead; ++kb, ++gk) {
          const int s = gk % SW, na = gk % NA;
          // each warp decides together (the TMEM stores are warp-collective)
          if (!__all_sync(0xffffffffu, mbar_wait(&bars->w_full[s], (gk / SW) & 1))) dead = true;
          if (!dead && gk >= NA && !__all_sync(0xffffffffu, mbar_wait(&bars->ta_empty[na], ((gk / NA) - 1) & 1)))
            dead = true;  // k block gk - NA read this A stage
          if (dead) break;
          tc_fence_after();
          // row `row` of the raw tile: 16-byte chunk j (k = 16j .. 16j+15) at
          // chunk position j ^ (row mod 8) (128-byte swizzle; a warp's 32 rows
          // spread over all banks)
          const uint8_t* rr = smem + Lay::kW + s * Lay::kWBytes + row * kTcBK;
#pragma unroll
          for (int h = 0; h < 4; ++h) {  // 32 k -> 16 columns
            const uint4 v0 = *reinterpret_cast<const uint4*>(rr + (((2 * h) ^ r8) << 4));
            const uint4 v1 = *reinterpret_cast<const uint4*>(rr + (((2 * h + 1) ^ r8) << 4));
            const uint32_t w8[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            uint32_t o[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              if (ta.f16) {  // one exact conversion per pair
                o[2 * i] = e4m3x2_to_f16x2(w8[i]);
                o[2 * i + 1] = e4m3x2_to_f16x2(w8[i] >> 16);
              } else {
                o[2 * i] = e4m3x2_to_bf16x2(w8[i]);
                o[2 * i + 1] = e4m3x2_to_bf16x2(w8[i] >> 16);
              }
            }
            tmem_st16(trow + na * (kTcBK / 2) + 16 * h, o);
          }
          // the raw tile is in registers: its slot is free
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->w_empty[s]);
          // the A stage is written before the MMA issuer may read it
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->ta_full[na]);
        }
      }
    }
  } else {
    // -------------------------------------------------------- epilogue
    // warps 6..21: TMEM lane quarter warp % 4 (a warp reaches only its own
    // quarter), token columns [hf * HC, (hf + 1) * HC); each drains its part of
    // a k block's partial with one TMEM load and one wait
    constexpr int EPG = kTcEpiWarps / 4;  // warps per lane quarter
    constexpr int HC = NT / EPG;
    const int q = warp & 3;
    const int hf = (warp - 6) >> 2;
    const int row = 32 * q + lane;  // weight row within the tile
    pdl_wait();
    // Per item, lane l holds the weight-tile scales of k blocks kb0 + l and
    // kb0 + 32 + l, and the unscale of this warp's token column l; they are
    // loaded one item ahead, so that no load latency falls between items.
    struct ItemConsts {
      float s0, s1, u;
    };
    auto load_consts = [&](int item) {
      ItemConsts c{1.0f, 1.0f, 1.0f};
      if (item < nitems) {
        int nt, mt, kb0, kb1;
        tc_item(ta, item, nt, mt, kb0, kb1);
        if (FP8) {
          const uint16_t* srow = a.S + (size_t)nt * ta.kblocks;
          if (kb0 + lane < kb1) c.s0 = bf16_to_f32(__ldg(srow + kb0 + lane));
          if (kb0 + 32 + lane < kb1) c.s1 = bf16_to_f32(__ldg(srow + kb0 + 32 + lane));
        }
        const int mc0 = mt * NT + hf * HC;
        if (ta.f16 && lane < HC && mc0 + lane < a.M) c.u = __ldg(a.unscale + mc0 + lane);
      }
      return c;
    };
    ItemConsts cur = load_consts(cid);
    float acc[HC];
    int gk = 0;
    for (int item = cid; item < nitems && !dead; item += ncl) {
      int nt, mt, kb0, kb1;
      tc_item(ta, item, nt, mt, kb0, kb1);
      const int ks = item % ta.ksplit;
      const ItemConsts nxt = load_consts(item + ncl);
#pragma unroll
      for (int j = 0; j < HC; ++j) acc[j] = 0.0f;
      for (int kb = kb0; kb < kb1 && !dead; ++kb, ++gk) {
        const int tb = gk % TB;
        const int i = kb - kb0;
        float s = 1.0f;
        if (FP8)
          s = i < 64 ? __shfl_sync(0xffffffffu, i < 32 ? cur.s0 : cur.s1, i & 31)
                     : bf16_to_f32(__ldg(a.S + (size_t)nt * ta.kblocks + kb));
        // the TMEM loads below are warp-collective: the warp decides together.
        // The phase awaited cannot alias a later one: k block gk + TB needs the
        // TMEM buffer this warp frees below.
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->mma_done[tb], (gk / TB) & 1))) dead = true;
        if (dead) break;
        tc_fence_after();
        // at most 16 columns per TMEM load: two loads in flight before one
        // wait at HC = 32 would hold 32 more registers than the 80 a thread
        // has here
        const uint32_t ta_ = tmem + ((uint32_t)(32 * q) << 16) + tb * NT + hf * HC;
        constexpr int CH = HC < 16 ? HC : 16;
#pragma unroll
        for (int c0 = 0; c0 < HC; c0 += CH) {
          float v[CH];
          if constexpr (CH == 16) tmem_ld16(ta_ + c0, v);
          else if constexpr (CH == 8) tmem_ld8(ta_ + c0, v);
          else tmem_ld4(ta_ + c0, v);
#pragma unroll
          for (int i = 0; i < CH; ++i) acc[c0 + i] = fmaf(s, v[i], acc[c0 + i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->tmem_empty[tb]);
      }
      if (dead) break;
      const int m0 = mt * NT + hf * HC;
      if (ta.f16) {  // the activation rows' prescale 2^j, undone exactly
#pragma unroll
        for (int j = 0; j < HC; ++j) acc[j] *= __shfl_sync(0xffffffffu, cur.u, j);
      }
      cur = nxt;
      tc_item_store<HC>(a, ta.ksplit, ta.part, ks, nt * kTcBM + row, m0, acc, L);
    }
  }
  tc_fence_before();
  __syncthreads();
  pdl_trigger();
  if (warp == 1) {
    tc_fence_after();
    tmem_free(tmem, Lay::kTmemCols);
  }
}

// ------------------------------------------------------------------ W8A8 kernel
//
// E4M3 weights x E4M3 activation codes (kind::f8f6f4) in tiles of 128 weight
// rows x NT tokens (UMMA N = NT, up to 256), one k block per stage.  What
// bounds this product is the operands' path from L2 into the SM, so the tile
// is as wide as TMEM allows: at NT = 256 a k block moves 48 KB for 8.4 MFLOP
// (32 KB for 4.2 at NT = 128).  A bulk copy also costs the thread that issues
// it a fixed time, so each operand has its own issuing thread.  Roles:
//   warp 0, lane 0   weight tiles [128][128] (128-byte swizzle) into a ring of S stages
//   warp 0, lane 1   activation tiles [NT][128] (128-byte swizzle), same ring positions
//   warp 0, lane 2   the token scales of each k block (fp32 [NT]) into S slots
//   warp 1           TMEM; lane 0 issues 4 MMAs (K = 32) per k block into one of the
//                    partial buffers, then commits twice: the stage is free, the
//                    partial is done
//   warps 2-17       epilogue, four warps per TMEM lane quarter, NT/4 token columns
//                    each: per k block, c = s_w * s_a for its columns (into its own
//                    scratch, which frees the scale slot), then acc += c * partial,
//                    two columns per fma; per item, the store epilogue or split-k
//                    partials
// Every wait is bounded; every issuing thread waits for its own copies and
// MMAs before the CTA frees TMEM and exits.
constexpr int kW8Warps = 18;
constexpr int kW8Threads = kW8Warps * 32;
constexpr int kW8EpiWarp0 = 2;
constexpr int kW8EpiWarps = 16;
constexpr int kW8Ring = 196608;  // operand ring bytes

template <int NT>
struct W8Cfg {
  static constexpr int kWBytes = kTcBM * kTcBK;                  // 16 KB of E4M3 weights
  static constexpr int kABytes = NT * kTcBK;                     // NT x 128 E4M3 codes
  static constexpr int kStages = kW8Ring / (kWBytes + kABytes);  // 256: 4, 128: 6, 64: 8
  static constexpr int kBufs = NT >= 256 ? 2 : 4;                // TMEM partials of NT columns
  static constexpr int kTmemCols = NT >= 128 ? 512 : 256;
  static constexpr int kW = 0;
  static constexpr int kA = kW + kStages * kWBytes;
  static constexpr int kSc = kA + kStages * kABytes;             // [kStages][NT] fp32
  static constexpr int kC = kSc + kStages * NT * 4;              // [16 warps][NT / 4] fp32
  static constexpr int kBars = kC + kW8EpiWarps * (NT / 4) * 4;
};

struct W8Bars {
  static constexpr int kMaxRing = 8, kMaxTmem = 4;
  uint64_t w_full[kMaxRing], a_full[kMaxRing], stage_empty[kMaxRing];
  uint64_t sc_full[kMaxRing], sc_empty[kMaxRing];
  uint64_t mma_done[kMaxTmem], tmem_empty[kMaxTmem];
  uint32_t tmem_base;
};

template <int NT>
constexpr int w8_smem_bytes() {
  static_assert(W8Cfg<NT>::kStages <= W8Bars::kMaxRing && W8Cfg<NT>::kBufs <= W8Bars::kMaxTmem, "barriers");
  static_assert(W8Cfg<NT>::kBars + (int)sizeof(W8Bars) + 1024 <= 232448, "shared memory");
  return W8Cfg<NT>::kBars + (int)sizeof(W8Bars) + 1024;  // + alignment slack
}

template <int NT>
__global__ void __launch_bounds__(kW8Threads, 1)
    gemm_w8a8_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmS, const TcArgs ta) {
  using Cfg = W8Cfg<NT>;
  constexpr int S = Cfg::kStages, NB = Cfg::kBufs;
  static_assert(S <= 8 && NB <= 4, "barrier arrays");
  const GemvArgs& a = ta.g;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  W8Bars* bars = reinterpret_cast<W8Bars*>(smem + Cfg::kBars);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nitems = ta.m_tiles * ta.n_tiles * ta.ksplit;
  const int cid = blockIdx.x, ncl = gridDim.x;
  const int L = a.dconv - 1;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&bars->w_full[s], 1);
      mbar_init(&bars->a_full[s], 1);
      mbar_init(&bars->stage_empty[s], 1);
      mbar_init(&bars->sc_full[s], 1);
      mbar_init(&bars->sc_empty[s], kW8EpiWarps);
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(&bars->mma_done[b], 1);
      mbar_init(&bars->tmem_empty[b], kW8EpiWarps);
    }
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&bars->tmem_base, Cfg::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  bool dead = false;

  if (warp == 0 && lane < 3) {
    // -------------------------------------------------------- operand issuers
    // lane 0: weights (never the previous kernel's output: no dependency wait);
    // lanes 1, 2: activation codes and token scales (written by the previous kernel)
    if (lane > 0) pdl_wait();
    const uint64_t pol = lane == 0 ? policy_evict_normal() : policy_evict_last();
    uint64_t* full = lane == 0 ? bars->w_full : (lane == 1 ? bars->a_full : bars->sc_full);
    uint64_t* empty = lane == 2 ? bars->sc_empty : bars->stage_empty;
    const uint32_t bytes = lane == 0 ? Cfg::kWBytes : (lane == 1 ? Cfg::kABytes : NT * 4);
    int gk = 0;
    for (int item = cid; item < nitems && !dead; item += ncl) {
      int nt, mt, kb0, kb1;
      tc_item(ta, item, nt, mt, kb0, kb1);
      for (int kb = kb0; kb < kb1; ++kb, ++gk) {
        const int s = gk % S;
        if (gk >= S && !mbar_wait(&empty[s], ((gk / S) - 1) & 1)) {
          dead = true;
          break;
        }
        mbar_arrive_expect_tx(&full[s], bytes);
        if (lane == 0)
          tma_load_2d(smem + Cfg::kW + s * Cfg::kWBytes, &tmW, kb * kTcBK, nt * kTcBM, &full[s], pol);
        else if (lane == 1)
          tma_load_2d(smem + Cfg::kA + s * Cfg::kABytes, &tmA, kb * kTcBK, mt * NT, &full[s], pol);
        else
          tma_load_2d(smem + Cfg::kSc + s * NT * 4, &tmS, mt * NT, kb, &full[s], pol);
      }
    }
    // drain: every copy this thread issued has landed
    for (int k = max(0, gk - S); k < gk; ++k)
      if (!mbar_drain(&full[k % S], (k / S) & 1)) break;
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc8 = tc_idesc_f8(kTcBM, NT);
      int gk = 0;
      for (int item = cid; item < nitems && !dead; item += ncl) {
        int nt, mt, kb0, kb1;
        tc_item(ta, item, nt, mt, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb, ++gk) {
          const int s = gk % S, tb = gk % NB;
          if (!mbar_wait(&bars->w_full[s], (gk / S) & 1) || !mbar_wait(&bars->a_full[s], (gk / S) & 1) ||
              (gk >= NB && !mbar_wait(&bars->tmem_empty[tb], ((gk / NB) - 1) & 1))) {
            dead = true;
            break;
          }
          tc_fence_after();
          const uint32_t wb = smem_addr(smem + Cfg::kW + s * Cfg::kWBytes);
          const uint32_t ab = smem_addr(smem + Cfg::kA + s * Cfg::kABytes);
#pragma unroll
          for (int kk = 0; kk < kTcBK / 32; ++kk)
            tc_mma_f8(tmem + tb * NT, sw128_desc(wb + kk * 32), sw128_desc(ab + kk * 32), idesc8, kk > 0 ? 1 : 0);
          tc_commit(&bars->stage_empty[s]);  // the stage's tiles have been read
          tc_commit(&bars->mma_done[tb]);    // the partial is complete
        }
      }
      if (gk > 0) mbar_drain(&bars->mma_done[(gk - 1) % NB], ((gk - 1) / NB) & 1);
    }
  } else if (warp >= kW8EpiWarp0 && warp < kW8EpiWarp0 + kW8EpiWarps) {
    // -------------------------------------------------------- epilogue
    constexpr int HC = NT / 4;  // token columns of this warp
    const int q = warp & 3;     // TMEM lane quarter this warp may access
    const int hf = (warp - kW8EpiWarp0) >> 2;
    const int row = 32 * q + lane;
    pdl_wait();
    float acc[HC];
    float* cw = reinterpret_cast<float*>(smem + Cfg::kC) + (warp - kW8EpiWarp0) * HC;  // this warp's c
    const uint32_t cws = smem_addr(cw);
    int gk = 0;
    for (int item = cid; item < nitems && !dead; item += ncl) {
      int nt, mt, kb0, kb1;
      tc_item(ta, item, nt, mt, kb0, kb1);
      const int ks = item % ta.ksplit;
#pragma unroll
      for (int j = 0; j < HC; ++j) acc[j] = 0.0f;
      for (int kb = kb0; kb < kb1; ++kb, ++gk) {
        const int s = gk % S, tb = gk % NB;
        const float sw = bf16_to_f32(__ldg(a.S + (size_t)nt * ta.kblocks + kb));
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->sc_full[s], (gk / S) & 1))) {
          dead = true;
          break;
        }
        const float* sa = reinterpret_cast<const float*>(smem + Cfg::kSc + s * NT * 4) + hf * HC;
#pragma unroll
        for (int j = lane; j < HC; j += 32) cw[j] = sw * sa[j];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->sc_empty[s]);  // the slot is read
        // the TMEM loads below are warp-collective: the warp decides together
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->mma_done[tb], (gk / NB) & 1))) {
          dead = true;
          break;
        }
        tc_fence_after();
        const uint32_t tadr = tmem + ((uint32_t)(32 * q) << 16) + tb * NT + hf * HC;
        // 8 columns per TMEM load: the NT = 256 accumulators leave few registers
#pragma unroll
        for (int c0 = 0; c0 < HC; c0 += 8) {
          float v[8];
          tmem_ld8(tadr + c0, v);
#pragma unroll
          for (int i4 = 0; i4 < 2; ++i4) {
            const float4 c4 = lds_f4_ordered(cws + (c0 + 4 * i4) * 4);
            const int j = c0 + 4 * i4;
            const float2 a0 = ffma2(make_float2(c4.x, c4.y), make_float2(v[4 * i4], v[4 * i4 + 1]),
                                    make_float2(acc[j], acc[j + 1]));
            const float2 a1 = ffma2(make_float2(c4.z, c4.w), make_float2(v[4 * i4 + 2], v[4 * i4 + 3]),
                                    make_float2(acc[j + 2], acc[j + 3]));
            acc[j] = a0.x;
            acc[j + 1] = a0.y;
            acc[j + 2] = a1.x;
            acc[j + 3] = a1.y;
          }
        }
        tc_fence_before();
        __syncwarp();  // also: every lane has read cw before the next k block rewrites it
        if (lane == 0) mbar_arrive(&bars->tmem_empty[tb]);
      }
      if (dead) break;
      tc_item_store<HC>(a, ta.ksplit, ta.part, ks, nt * kTcBM + row, mt * NT + hf * HC, acc, L);
    }
  }
  tc_fence_before();
  __syncthreads();
  pdl_trigger();
  if (warp == 1) {
    tc_fence_after();
    tmem_free(tmem, Cfg::kTmemCols);
  }
}

// Split-k reduction: sums the k-split partials of each output in split order
// (deterministic) and runs the epilogue.  vec4: four adjacent outputs per
// thread (store and residual epilogues with 4-aligned rows), the splits'
// loads issued together.
__global__ void __launch_bounds__(256) gemm_tc_reduce_kernel(const GemvArgs a, const float* part, int ksplit,
                                                              int vec4) {
  pdl_wait();
  pdl_trigger();
  const int L = a.dconv - 1;
  if (vec4) {
    const int nq = a.N / 4;
    const size_t quads = (size_t)a.M * nq, sstride = (size_t)a.M * a.N;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < quads; i += (size_t)gridDim.x * blockDim.x) {
      const int m = (int)(i / nq), n = (int)(i % nq) * 4;
      uint2 r = make_uint2(0u, 0u);
      if (a.epi == EPI_RESID) r = *reinterpret_cast<const uint2*>(a.resid + (size_t)m * a.ldr + n);
      const float* pp = part + (size_t)m * a.N + n;
      float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 4
      for (int ks = 0; ks < ksplit; ++ks) {
        const float4 v = *reinterpret_cast<const float4*>(pp + ks * sstride);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      if (a.epi == EPI_RESID) {
        acc.x += bf16lo(r.x);
        acc.y += bf16hi(r.x);
        acc.z += bf16lo(r.y);
        acc.w += bf16hi(r.y);
      }
      *reinterpret_cast<uint2*>(a.out + (size_t)m * a.ldo + n) =
          make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
    }
    return;
  }
  const size_t total = (size_t)a.M * a.N;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int m = (int)(i / a.N), n = (int)(i % a.N);
    float acc = 0.0f;
    for (int ks = 0; ks < ksplit; ++ks) acc += part[((size_t)ks * a.M + m) * a.N + n];
    const bool conv = a.epi == EPI_INPROJ_CONV && n >= a.xbc0 && n < a.xbc0 + a.d_xbc;
    ConvTaps taps;
    if (conv) load_taps(a, n - a.xbc0, L, taps);
    tc_epi_elem(a, m, n, acc, conv, taps, L);
  }
}

// ------------------------------------------------------------------ host

// Whether the split-k reduction may take four adjacent outputs per thread.
static bool reduce_vec4(const GemvArgs& g) {
  if (g.epi == EPI_INPROJ_CONV || g.N % 4 || g.ldo % 4 || (reinterpret_cast<uintptr_t>(g.out) & 7)) return false;
  if (g.epi == EPI_RESID && (g.ldr % 4 || (reinterpret_cast<uintptr_t>(g.resid) & 7))) return false;
  return true;
}

bool gemm_tc_supported(int M, int N, int K, bool fp8) {
  (void)N;
  (void)fp8;
  return M > 8 && K % 16 == 0;
}

// Token tile: as narrow as the rows need (the activation tile is copied and
// multiplied whole), up to 128.
static int tc_nt(int M) { return M <= 16 ? 16 : (M <= 32 ? 32 : (M <= 64 ? 64 : 128)); }

// k split for grids that would leave most SMs idle (few weight tiles at small
// M): enough items to cover the SMs, at least 4 k blocks per item.
int gemm_tc_ksplit(int M, int N, int K) {
  const int nt = tc_nt(M);
  const int tiles = ((M + nt - 1) / nt) * ((N + kTcBM - 1) / kTcBM);
  const int kb = (K + kTcBK - 1) / kTcBK;
  int ks = num_sms() / tiles;
  if (ks > kb / 4) ks = kb / 4;
  return ks > 1 ? ks : 1;
}

size_t gemm_tc_partial_bytes(int M, int N, int K) {
  const int ks = gemm_tc_ksplit(M, N, K);
  return ks > 1 ? (size_t)ks * M * N * 4 : 0;
}

// Token tile of the W8A8 product: as wide as the token count needs, up to 256.
static int w8_nt(int M) { return M <= 64 ? 64 : (M <= 128 ? 128 : 256); }

// k split of the W8A8 product: as gemm_tc_ksplit, for its own tiles, and no
// more splits than `part_bytes` holds partials for.
static int w8_ksplit(int M, int N, int K, size_t part_bytes) {
  const int nt = w8_nt(M);
  const int tiles = ((M + nt - 1) / nt) * ((N + kTcBM - 1) / kTcBM);
  const int kb = (K + kTcBK - 1) / kTcBK;
  int ks = num_sms() / tiles;
  if (ks > kb / 4) ks = kb / 4;
  const size_t per = (size_t)M * N * 4;
  if (ks > 1 && (size_t)ks * per > part_bytes) ks = (int)(part_bytes / per);
  return ks > 1 ? ks : 1;
}

template <int NT>
static cudaError_t launch_w8a8(const GemvArgs& g, cudaStream_t s) {
  static int done_mask[64] = {0};
  CUtensorMap tmW, tmA, tmS;
  TcArgs ta;
  ta.g = g;
  ta.m_tiles = (g.M + NT - 1) / NT;
  ta.n_tiles = (g.N + kTcBM - 1) / kTcBM;
  ta.kblocks = (g.K + kTcBK - 1) / kTcBK;
  ta.fp8 = 1;
  ta.part = g.part;
  ta.ksplit = g.part ? w8_ksplit(g.M, g.N, g.K, g.part_bytes) : 1;
  if (!encode_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.W, g.K, g.N, (uint64_t)g.K, kTcBK, kTcBM,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.q8, g.K, g.M, (uint64_t)g.ldq, kTcBK, NT,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tmS, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, g.sq, (uint64_t)g.ldsq, (uint64_t)ta.kblocks,
                 (uint64_t)g.ldsq * 4, NT, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  const int smem = w8_smem_bytes<NT>();
  auto kern = gemm_w8a8_kernel<NT>;
  cudaError_t e = set_smem_once((const void*)kern, smem, done_mask);
  if (e != cudaSuccess) return e;
  const int nitems = ta.m_tiles * ta.n_tiles * ta.ksplit;
  int grid = num_sms();
  if (grid > nitems) grid = nitems;
  trace_pre(K_GEMM_TC, s);
  e = launch_k(kern, dim3(grid), dim3(kW8Threads), smem, s, g.pdl != 0, tmW, tmA, tmS, ta);
  trace_post(K_GEMM_TC, s);
  if (e != cudaSuccess || ta.ksplit == 1) return e;
  const size_t total = (size_t)g.M * g.N;
  int rgrid = (int)(((reduce_vec4(g) ? total / 4 : total) + 255) / 256);
  if (rgrid > 8 * num_sms()) rgrid = 8 * num_sms();
  trace_pre(K_GEMM_TC_REDUCE, s);
  e = launch_k(gemm_tc_reduce_kernel, dim3(rgrid), dim3(256), 0, s, g.pdl != 0, g, (const float*)ta.part,
               ta.ksplit, reduce_vec4(g) ? 1 : 0);
  trace_post(K_GEMM_TC_REDUCE, s);
  return e;
}

template <int NT, bool FP8>
static cudaError_t launch_tc(const GemvArgs& g, cudaStream_t s) {
  static int done_mask[64] = {0};
  constexpr bool fp8 = FP8;
  CUtensorMap tmW, tmA;
  if (fp8) {
    if (!encode_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.W, g.K, g.N, (uint64_t)g.K, kTcBK, kTcBM,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  } else {
    if (!encode_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.W, g.K, g.N, (uint64_t)g.K * 2, 64, kTcBM,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  TcArgs ta;
  ta.g = g;
  ta.m_tiles = (g.M + NT - 1) / NT;
  ta.n_tiles = (g.N + kTcBM - 1) / kTcBM;
  ta.kblocks = (g.K + kTcBK - 1) / kTcBK;
  ta.fp8 = fp8 ? 1 : 0;
  ta.f16 = (fp8 && g.act == ACT_PREPARED && g.unscale) ? 1 : 0;
  ta.ksplit = gemm_tc_ksplit(g.M, g.N, g.K);
  ta.part = g.part;
  if (ta.ksplit > 1 && (!g.part || g.part_bytes < gemm_tc_partial_bytes(g.M, g.N, g.K))) ta.ksplit = 1;
  {
    // bf16 activations as {64-element half of a k block, rows, halves}: one
    // copy of box {64, NT, 2} lands the two 128-byte-swizzled [NT][64] halves
    // of a k block back to back
    auto enc = tensor_map_encoder();
    const cuuint64_t dims[3] = {64, (cuuint64_t)g.M, (cuuint64_t)(g.K / 64)};
    const cuuint64_t strides[2] = {(cuuint64_t)g.lda * 2, 128};
    const cuuint32_t box[3] = {64, (cuuint32_t)NT, 2};
    const cuuint32_t es[3] = {1, 1, 1};
    if (!enc || g.K % 64 ||
        enc(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(g.A), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const int smem = tc_smem_bytes<NT, FP8>();
  auto kern = gemm_tc_kernel<NT, FP8>;
  cudaError_t e = set_smem_once((const void*)kern, smem, done_mask);
  if (e != cudaSuccess) return e;
  const int nitems = ta.m_tiles * ta.n_tiles * ta.ksplit;
  int grid = num_sms();
  if (grid > nitems) grid = nitems;
  trace_pre(K_GEMM_TC, s);
  e = launch_k(kern, dim3(grid), dim3(kTcThreads), smem, s, g.pdl != 0, tmW, tmA, ta);
  trace_post(K_GEMM_TC, s);
  if (e != cudaSuccess || ta.ksplit == 1) return e;
  const size_t total = (size_t)g.M * g.N;
  int rgrid = (int)(((reduce_vec4(g) ? total / 4 : total) + 255) / 256);
  if (rgrid > 8 * num_sms()) rgrid = 8 * num_sms();
  trace_pre(K_GEMM_TC_REDUCE, s);
  e = launch_k(gemm_tc_reduce_kernel, dim3(rgrid), dim3(256), 0, s, g.pdl != 0, g, (const float*)ta.part,
               ta.ksplit, reduce_vec4(g) ? 1 : 0);
  trace_post(K_GEMM_TC_REDUCE, s);
  return e;
}

// ------------------------------------------------------------------ wait-path check
//
// One CTA that holds tensor memory and has a bulk copy in flight waits, with
// the pipeline limit, on a barrier that nothing signals.  It must give up
// (M2_ERR_TIMEOUT in the status word), wait for its copy with the drain limit,
// pass the copied bytes to `out`, free its tensor memory and return.
__global__ void __launch_bounds__(128, 1) wait_check_kernel(const uint4* probe, uint4* out) {
  __shared__ __align__(128) uint4 buf;
  __shared__ __align__(8) uint64_t bar_copy, bar_never;
  __shared__ uint32_t tmem_base;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bar_copy, 1);
    mbar_init(&bar_never, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_base)),
                 "r"(32));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0 && lane == 0) {
    mbar_arrive_expect_tx(&bar_copy, 16);
    bulk_g2s(&buf, probe, 16, &bar_copy, policy_evict_normal());
    if (!mbar_wait(&bar_never, 0)) {  // nothing arrives: this times out
      if (mbar_drain(&bar_copy, 0)) *out = buf;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(32));
  }
}

cudaError_t launch_wait_check(const void* probe, void* out, cudaStream_t s) {
  trace_pre(K_WAIT_CHECK, s);
  const cudaError_t e = launch_k(wait_check_kernel, dim3(1), dim3(128), 0, s, false,
                                 static_cast<const uint4*>(probe), static_cast<uint4*>(out));
  trace_post(K_WAIT_CHECK, s);
  return e;
}

cudaError_t launch_gemm_tc(const GemvArgs& g, bool fp8, cudaStream_t s) {
  if (g.q8) {  // W8A8: E4M3 activation codes with per-(token, k block) scales
    if (!fp8 || g.K % 128 || g.ldq % 16 || g.ldsq % 128) return cudaErrorInvalidValue;
    const int nt = w8_nt(g.M);
    if (nt == 64) return launch_w8a8<64>(g, s);
    if (nt == 128) return launch_w8a8<128>(g, s);
    return launch_w8a8<256>(g, s);
  }
  switch (tc_nt(g.M)) {
    case 16: return fp8 ? launch_tc<16, true>(g, s) : launch_tc<16, false>(g, s);
    case 32: return fp8 ? launch_tc<32, true>(g, s) : launch_tc<32, false>(g, s);
    case 64: return fp8 ? launch_tc<64, true>(g, s) : launch_tc<64, false>(g, s);
    default: return fp8 ? launch_tc<128, true>(g, s) : launch_tc<128, false>(g, s);
  }
}

int status_gemm_tc(int clear) { return tu_status(clear); }

cudaError_t wait_limit_gemm_tc(long long cycles) { return tu_set_wait_limit(cycles); }

}  // namespace m2
