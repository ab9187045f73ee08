// m2_abi.cu -- the exported C ABI (include/mamba2.h): host-side validation,
// workspace carving, the launch sequence of the decode and prefill paths,
// launch counting, per-kernel event tracing and the device status word.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/mamba2.h"
#include "m2_kernels.h"

namespace m2 {

// ------------------------------------------------------------------ device info

static int g_sms[64];

int num_sms() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (g_sms[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
    g_sms[dev] = v;
  }
  return g_sms[dev];
}

cudaError_t set_smem_once(const void* func, int bytes, int* done_mask) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && done_mask[dev] >= bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done_mask[dev] = bytes;
  return e;
}

// ------------------------------------------------------------------ tracing

static std::atomic<int64_t> g_launches{0};
static std::mutex g_trace_mu;
struct TraceSlot {
  cudaEvent_t a, b;
  int32_t id;
};
static std::vector<TraceSlot> g_trace;
static int32_t g_trace_used = 0;
static bool g_trace_on = false;

void trace_pre(int32_t id, cudaStream_t s) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (!g_trace_on) return;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (g_trace_used < (int32_t)g_trace.size()) {
    g_trace[g_trace_used].id = id;
    cudaEventRecord(g_trace[g_trace_used].a, s);
  }
}

void trace_post(int32_t id, cudaStream_t s) {
  (void)id;
  if (!g_trace_on) return;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (g_trace_used < (int32_t)g_trace.size()) {
    cudaEventRecord(g_trace[g_trace_used].b, s);
    ++g_trace_used;
  }
}

static const char* kNames[K_COUNT] = {
    "norm_prep",     "gemv_fp8",        "gemv_fp8_inproj_conv", "gemv_fp8_outproj_resid",
    "gemv_bf16",     "gemv_bf16_inproj_conv", "gemv_bf16_outproj_resid", "conv_update",
    "conv_pos",      "ssm_step",        "conv_prefill",    "ssm_scan_seq",
    "gemm_tc",       "ssd_chunk_state", "ssd_state_pass",  "ssd_chunk_out",   "gemm_tc_reduce",
    "conv_ring_store", "decode_step_fused", "copy", "wait_check"};

// ------------------------------------------------------------------ helpers

static inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static inline bool al8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }
static inline size_t rup(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Derived {
  int d_inner, d_xbc, n_in, ldz;
};

static Derived derive(const m2_dims& d) {
  Derived r;
  r.d_inner = d.nheads * d.head_dim;
  r.d_xbc = r.d_inner + 2 * d.n_groups * d.d_state;
  r.n_in = r.d_inner + r.d_xbc + d.nheads;
  r.ldz = (int)rup((size_t)r.n_in, 8);
  return r;
}

static int check_dims(const m2_dims* d) {
  if (!d) return M2_ERR_ARG;
  if (d->hidden <= 0 || d->nheads <= 0 || d->head_dim <= 0 || d->d_state <= 0 || d->n_groups <= 0 || d->d_conv <= 0)
    return M2_ERR_ARG;
  if (d->nheads % d->n_groups) return M2_ERR_ARG;
  if (!(d->eps_in >= 0.0f) || !(d->eps_gated >= 0.0f)) return M2_ERR_ARG;
  const int d_inner = d->nheads * d->head_dim;
  if (d->hidden % 16 || d->hidden > 16384 || d_inner % 16 || d_inner > 16384) return M2_ERR_UNSUPPORTED;
  if (!(d->d_state == 16 || d->d_state == 32 || d->d_state == 64 || d->d_state == 128)) return M2_ERR_UNSUPPORTED;
  if (d->head_dim > 256 || d->d_conv < 2 || d->d_conv > 8) return M2_ERR_UNSUPPORTED;
  if (d->gnorm_group <= 0 || d_inner % d->gnorm_group || d->gnorm_group % 16) return M2_ERR_UNSUPPORTED;
  return M2_OK;
}

static int check_weight(const m2_weight& w, int n, int k) {
  if (!w.w) return M2_ERR_ARG;
  if (w.n != n || w.k != k) return M2_ERR_ARG;
  if (!al16(w.w)) return M2_ERR_ALIGN;
  if (w.fmt == M2_W_FP8_BLOCK128) {
    if (!w.scale) return M2_ERR_FORMAT;
    if (k % 16 || k > 16384) return M2_ERR_UNSUPPORTED;
  } else if (w.fmt == M2_W_BF16) {
    if (w.scale) return M2_ERR_FORMAT;
    if (k % 8 || k > 16384) return M2_ERR_UNSUPPORTED;
  } else {
    return M2_ERR_FORMAT;
  }
  return M2_OK;
}

// Workspace layouts (each region 256-byte aligned).
//   decode:  act_in [B][hidden] (2 B), zxu [B][ldz] bf16 (z | conv output u | dt),
//            y [B][d_inner] fp32, act_out [B][d_inner] (2 B), unscale [2][B] fp32
//   prefill: act_in [T][hidden], zx [T][ldz] (raw in_proj output), u [T][d_xbc],
//            y [T][d_inner] fp32, act_out [T][d_inner], unscale [2][T] fp32
// Scratch for the k-split partials of the tensor-core projections over M rows.
static size_t proj_part_bytes(const m2_dims& d, int M) {
  if (M <= 0 || !gemm_tc_supported(M, 0, 16, true)) return 0;
  const Derived r = derive(d);
  const size_t a = gemm_tc_partial_bytes(M, r.n_in, d.hidden), b = gemm_tc_partial_bytes(M, d.hidden, r.d_inner);
  return rup(a > b ? a : b, 256);
}

// Byte offsets of the decode workspace regions for B rows (each 256-aligned):
// xn [B][hidden] (2 B), zxu [B][ldz] bf16 (z | conv output u | dt), y
// [B][d_inner] fp32, g [B][d_inner] (2 B), unscale [2][B] fp32, then the
// optional k-split partials of the tensor-core projections at `end`.
struct DecodeMap {
  size_t xn, zxu, y, g, unscale, end;
};
static DecodeMap decode_map(const m2_dims& d, int B) {
  const Derived r = derive(d);
  DecodeMap m;
  m.xn = 0;
  m.zxu = rup(m.xn + (size_t)B * d.hidden * 2, 256);
  m.y = rup(m.zxu + (size_t)B * r.ldz * 2, 256);
  m.g = rup(m.y + (size_t)B * r.d_inner * 4, 256);
  m.unscale = rup(m.g + (size_t)B * r.d_inner * 2, 256);
  m.end = rup(m.unscale + (size_t)2 * B * 4, 256);
  return m;
}

// Decode workspace without (min) and with the tensor-core k-split partials;
// a workspace between the two runs the projections without the split.
static size_t decode_ws_min(const m2_dims& d, int B) { return decode_map(d, B).end; }
static size_t decode_ws(const m2_dims& d, int B) { return decode_ws_min(d, B) + proj_part_bytes(d, B); }

// Prefill workspace for T token rows in nseq sequences with nchunks SSD chunks
// in total (ceil(T_i / 128) summed; at most T / 128 + nseq).
// W8A8 activation codes and block scales (the larger of the two projections' inputs).
static size_t q8_ldq(const m2_dims& d) {
  const Derived r = derive(d);
  return rup((size_t)(d.hidden > r.d_inner ? d.hidden : r.d_inner), 16);
}
static size_t q8_bytes(const m2_dims& d, int T) {
  return rup((size_t)T * q8_ldq(d), 256) + rup(q8_ldq(d) / 128 * rup((size_t)T, 128) * 4, 256);
}

// Byte offsets of the prefill workspace regions for T token rows in nseq
// sequences with nchunks SSD chunks (each region 256-aligned): xn [T][hidden],
// zx [T][ldz] (raw in_proj output), u [T][d_xbc] (conv output), y [T][d_inner]
// fp32, g [T][d_inner], unscale [2][T] fp32, the sequence tables (token and
// chunk offsets), the SSD chunk states and decays, the tensor-core k-split
// partials, and (W8A8 arm) the E4M3 codes [T][ldq] and scales [K/128][rup(T, 128)].
struct PrefillMap {
  size_t xn, zx, u, y, g, unscale, tab, ssd, part, q8, sq, end, end_w8a8;
};
static PrefillMap prefill_map(const m2_dims& d, int T, int nseq, int nchunks) {
  const Derived r = derive(d);
  PrefillMap m;
  m.xn = 0;
  m.zx = rup(m.xn + (size_t)T * d.hidden * 2, 256);
  m.u = rup(m.zx + (size_t)T * r.ldz * 2, 256);
  m.y = rup(m.u + (size_t)T * r.d_xbc * 2, 256);
  m.g = rup(m.y + (size_t)T * r.d_inner * 4, 256);
  m.unscale = rup(m.g + (size_t)T * r.d_inner * 2, 256);
  m.tab = rup(m.unscale + (size_t)2 * T * 4, 256);
  m.ssd = rup(m.tab + (size_t)2 * (nseq + 1) * 4, 256);
  m.part = m.ssd;
  if (ssd_supported(d.nheads, d.head_dim, d.d_state, d.n_groups))
    m.part += ssd_workspace_bytes(nchunks, d.nheads, d.head_dim, d.d_state);  // chunk states + decays
  m.end = m.part + proj_part_bytes(d, T);
  m.q8 = rup(m.end, 256);
  m.sq = m.q8 + rup((size_t)T * q8_ldq(d), 256);
  m.end_w8a8 = m.q8 + q8_bytes(d, T);
  return m;
}

static size_t prefill_ws(const m2_dims& d, int T, int nseq, int nchunks, bool w8a8 = true) {
  const PrefillMap m = prefill_map(d, T, nseq, nchunks);
  return w8a8 ? m.end_w8a8 : m.end;
}
static size_t prefill_ws_bound(const m2_dims& d, int T, int nseq, bool w8a8 = true) {
  return prefill_ws(d, T, nseq, (T + 127) / 128 + nseq, w8a8);
}

// Whether a projection consumes f16 activation rows, each prescaled by an
// exact power of two (E4M3 weights: their f16 conversion is one instruction a
// pair, in the GEMV and in the tensor-core GEMM's f16 x f16 MMAs), or bf16 rows
// (bf16 weights: both MMA operands must have one type).
static bool proj_f16(const m2_weight& w, int M) {
  (void)M;
  return w.fmt == M2_W_FP8_BLOCK128;
}

static GemvArgs proj_args(const m2_weight& w, const uint16_t* A, int lda, int M, uint16_t* out, int ldo,
                          GemvEpi epi, const uint16_t* resid, int ldr, GemvArgs* extra = nullptr,
                          const float* unscale = nullptr, int pdl = 0, float* part = nullptr,
                          size_t part_bytes = 0) {
  GemvArgs a;
  memset(&a, 0, sizeof(a));
  if (extra) a = *extra;
  a.A = A;
  a.lda = lda;
  a.W = w.w;
  a.S = w.scale;
  a.M = M;
  a.N = w.n;
  a.K = w.k;
  a.out = out;
  a.ldo = ldo;
  a.epi = epi;
  a.resid = resid;
  a.ldr = ldr;
  // prepared f16 rows carry a prescale; prepared bf16 rows are plain bf16
  a.act = (unscale && proj_f16(w, M)) ? ACT_PREPARED : ACT_PLAIN;
  a.unscale = unscale;
  a.pdl = pdl;
  a.part = part;
  a.part_bytes = part_bytes;
  const int rowbytes = w.k * (w.fmt == M2_W_FP8_BLOCK128 ? 1 : 2);
  const int grp = rowbytes <= 4096 ? 4 : (rowbytes <= 8192 ? 2 : 1);
  a.evict_first = M <= grp ? 1 : 0;
  return a;
}

static cudaError_t proj(const m2_weight& w, const uint16_t* A, int lda, int M, uint16_t* out, int ldo,
                        GemvEpi epi, const uint16_t* resid, int ldr, cudaStream_t s, GemvArgs* extra = nullptr,
                        const float* unscale = nullptr, int pdl = 0, float* part = nullptr,
                        size_t part_bytes = 0) {
  const GemvArgs a = proj_args(w, A, lda, M, out, ldo, epi, resid, ldr, extra, unscale, pdl, part, part_bytes);
  return launch_gemv(a, w.fmt == M2_W_FP8_BLOCK128, s);
}

// Batch-1 decode as one cooperative launch (m2_set_fused_decode).  Off by
// default: measured on the 8B-like layer it takes 43 us per step against 32 us
// for the PDL-chained kernels, whose SSM and out_proj work hides under the
// neighbouring kernels while the single launch runs its phases back to back.
static int g_fused_decode = 0;

static int launch_status(cudaError_t e) {
  if (e != cudaSuccess) {
    cudaGetLastError();
    return M2_ERR_LAUNCH;
  }
  return M2_OK;
}

}  // namespace m2

using namespace m2;

extern "C" {

const char* m2_strerror(int status) {
  switch (status) {
    case M2_OK: return "ok";
    case M2_ERR_ARG: return "invalid argument (null pointer or bad size)";
    case M2_ERR_FORMAT: return "weight format tag or scale grid inconsistent";
    case M2_ERR_WORKSPACE: return "workspace missing or too small";
    case M2_ERR_LAUNCH: return "CUDA launch failed";
    case M2_ERR_UNSUPPORTED: return "shape outside the supported range";
    case M2_ERR_ALIGN: return "pointer not 16-byte aligned";
    case M2_ERR_DEVICE: return "no usable CUDA device";
    case M2_ERR_TIMEOUT: return "a bounded in-kernel wait timed out";
    case M2_ERR_SCRATCH: return "decode workspace larger than the built-in scratch of mamba2_layer_decode_noalloc";
    default: return "unknown status";
  }
}

int m2_validate(const m2_dims* dims, const m2_layer* L) {
  int st = check_dims(dims);
  if (st) return st;
  if (!L) return M2_ERR_ARG;
  const Derived r = derive(*dims);
  if (!L->norm_w || !L->conv_w || !L->A_log || !L->D || !L->dt_bias || !L->gnorm_w) return M2_ERR_ARG;
  if (!al16(L->norm_w) || !al16(L->gnorm_w)) return M2_ERR_ALIGN;
  if ((st = check_weight(L->in_proj, r.n_in, dims->hidden))) return st;
  if ((st = check_weight(L->out_proj, dims->hidden, r.d_inner))) return st;
  return M2_OK;
}

size_t m2_workspace_bytes(const m2_dims* dims, int32_t max_batch, int32_t max_tokens) {
  if (check_dims(dims) || max_batch < 0 || max_tokens < 0) return 0;
  const size_t a = max_batch > 0 ? decode_ws(*dims, max_batch) : 0;
  const size_t b = max_tokens > 0 ? prefill_ws_bound(*dims, max_tokens, 1, false) : 0;
  return a > b ? a : b;
}

static int decode_impl(const m2_dims* dims, const m2_layer* L, uint16_t* hidden, int32_t B, float* ssm_state,
                       uint16_t* conv_state, int32_t* conv_pos, void* ws, size_t ws_bytes, const char* ahead,
                       size_t ahead_bytes, cudaStream_t stream) {
  int st = m2_validate(dims, L);
  if (st) return st;
  if (B <= 0 || !hidden || !ssm_state || !conv_state || !conv_pos) return M2_ERR_ARG;
  if (!al16(hidden) || !al16(ssm_state) || !al8(conv_state)) return M2_ERR_ALIGN;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < decode_ws_min(*dims, B)) return M2_ERR_WORKSPACE;
  const m2_dims& d = *dims;
  const Derived r = derive(d);
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  const DecodeMap wm = decode_map(d, B);
  uint16_t* xn = reinterpret_cast<uint16_t*>(w8 + wm.xn);
  uint16_t* zxu = reinterpret_cast<uint16_t*>(w8 + wm.zxu);
  float* y = reinterpret_cast<float*>(w8 + wm.y);
  uint16_t* g = reinterpret_cast<uint16_t*>(w8 + wm.g);
  float* us_in = reinterpret_cast<float*>(w8 + wm.unscale);
  float* us_out = us_in + B;
  float* part = reinterpret_cast<float*>(w8 + wm.end);
  const size_t part_bytes = ws_bytes >= decode_ws(d, B) ? proj_part_bytes(d, B) : 0;  // 0: no k split

  cudaError_t e;
  // Each kernel is launched as a programmatic dependent of the previous one,
  // so that a GEMV streams its weights while its predecessor drains.  With the
  // decode GEMV (B <= 8) the two norms run inside the GEMVs' prologues: three
  // kernels per step (at B = 1 optionally one cooperative kernel for the whole
  // step).
  // Otherwise (tensor-core projections) a norm kernel precedes each
  // projection: five.
  const bool fuse = !gemm_tc_supported(B, r.n_in, d.hidden, true) && gemv_mma_supported(B, d.hidden) &&
                    gemv_mma_supported(B, r.d_inner) && d.gnorm_group == r.d_inner;
  // 1. input RMSNorm -> GEMV activation
  PrepArgs pa;
  memset(&pa, 0, sizeof(pa));
  if (!fuse) {
    pa.mode = PREP_RMSNORM;
    pa.x = hidden;
    pa.ldx = d.hidden;
    pa.w = L->norm_w;
    pa.eps = d.eps_in;
    pa.M = B;
    pa.K = d.hidden;
    pa.out = xn;
    pa.ldo = d.hidden;
    pa.f16 = proj_f16(L->in_proj, B) ? 1 : 0;
    pa.unscale = us_in;
    pa.pdl = 1;
    if ((e = launch_prep(pa, stream))) return launch_status(e);
  }
  // 2+3. in_proj, conv1d update (bias, SiLU) in its epilogue
  FusedStepArgs fa;
  memset(&fa, 0, sizeof(fa));
  GemvArgs ex;
  memset(&ex, 0, sizeof(ex));
  ex.ring = conv_state;
  ex.pos = conv_pos;
  ex.conv_w = L->conv_w;
  ex.conv_b = L->conv_b;
  ex.xbc0 = r.d_inner;
  ex.d_xbc = r.d_xbc;
  ex.dconv = d.d_conv;
  if (fuse) {
    ex.norm = NORM_RMS;
    ex.norm_w = L->norm_w;
    ex.norm_eps = d.eps_in;
  }
  fa.in = proj_args(L->in_proj, fuse ? hidden : xn, d.hidden, B, zxu, r.ldz, EPI_INPROJ_CONV, nullptr, 0, &ex,
                    fuse ? nullptr : us_in, 1, part, part_bytes);
  // 4+5. split and SSM step (advances conv_pos)
  SsmArgs sa;
  memset(&sa, 0, sizeof(sa));
  sa.h = ssm_state;
  sa.x = zxu + r.d_inner;
  sa.Bm = zxu + 2 * r.d_inner;
  sa.Cm = zxu + 2 * r.d_inner + d.n_groups * d.d_state;
  sa.dt = zxu + r.d_inner + r.d_xbc;
  sa.ld_in = r.ldz;
  sa.A_log = L->A_log;
  sa.D = L->D;
  sa.dt_bias = L->dt_bias;
  sa.y = y;
  sa.ldy = r.d_inner;
  sa.B = B;
  sa.H = d.nheads;
  sa.P = d.head_dim;
  sa.N = d.d_state;
  sa.G = d.n_groups;
  sa.pos_inc = conv_pos;
  sa.pdl = 1;
  {
    // the SSM kernel starts while the in_proj drains and moves little data
    // itself: it pulls the first rows of the out_proj weights into L2 for the
    // GEMV two launches on.  Only the first kSsmPrefetch bytes: the out_proj's
    // CTAs launch during the SSM step and fill their own rings, and more
    // prefetch traffic delays the SSM's state reads.  Measured on the 8B-like
    // layer at batch 1 (with the 8 MB next-layer hint of the prefetching
    // decode): 10 MB 30.06 us per step, 4 MB 30.65, the whole 33.5 MB 30.5;
    // without the hint: 10 MB 30.26, none 31.18, all 31.44.
    constexpr size_t kSsmPrefetch = 10ull << 20;
    const m2_weight& wo = L->out_proj;
    const size_t wo_bytes = (size_t)wo.n * wo.k * (wo.fmt == M2_W_BF16 ? 2 : 1);
    sa.l2_prefetch = wo.w;
    sa.l2_prefetch_bytes = wo_bytes < kSsmPrefetch ? wo_bytes : kSsmPrefetch;
  }
  // 7+8. out_proj with the residual add in its epilogue (in place on hidden)
  GemvArgs eo;
  memset(&eo, 0, sizeof(eo));
  if (fuse) {
    eo.norm = NORM_GATED;
    eo.norm_w = L->gnorm_w;
    eo.norm_eps = d.eps_gated;
    eo.gy = y;
    eo.ldgy = r.d_inner;
    eo.gz = zxu;
    eo.ldgz = r.ldz;
  }
  eo.l2_ahead = ahead;
  eo.l2_ahead_bytes = ahead_bytes;
  fa.out = proj_args(L->out_proj, g, r.d_inner, B, hidden, d.hidden, EPI_RESID, hidden, d.hidden, &eo,
                     fuse ? nullptr : us_out, 1, part, part_bytes);
  fa.ssm = sa;
  const bool fp8 = L->in_proj.fmt == M2_W_FP8_BLOCK128;
  if (fuse && B == 1 && g_fused_decode && L->in_proj.fmt == L->out_proj.fmt) {
    // the whole step in one launch: SSM state and the out_proj weights are
    // handled inside (no L2 prefetch hand-off needed)
    fa.ssm.l2_prefetch = nullptr;
    fa.ssm.l2_prefetch_bytes = 0;
    if (decode_fused_supported(fa, fp8)) return launch_status(launch_decode_fused(fa, fp8, stream));
  }
  if ((e = launch_gemv(fa.in, fp8, stream))) return launch_status(e);
  if ((e = launch_ssm_step(sa, stream))) return launch_status(e);
  // 6. gated RMSNorm -> GEMV activation
  if (!fuse) {
    memset(&pa, 0, sizeof(pa));
    pa.mode = PREP_GATED;
    pa.y = y;
    pa.ldy = r.d_inner;
    pa.z = zxu;
    pa.ldz = r.ldz;
    pa.w = L->gnorm_w;
    pa.eps = d.eps_gated;
    pa.group = d.gnorm_group;
    pa.M = B;
    pa.K = r.d_inner;
    pa.out = g;
    pa.ldo = r.d_inner;
    pa.f16 = proj_f16(L->out_proj, B) ? 1 : 0;
    pa.unscale = us_out;
    pa.pdl = 1;
    if ((e = launch_prep(pa, stream))) return launch_status(e);
  }
  if ((e = launch_gemv(fa.out, L->out_proj.fmt == M2_W_FP8_BLOCK128, stream))) return launch_status(e);
  return M2_OK;
}

}  // extern "C"

namespace m2 {

// Prefill of a varlen batch (cu: host token offsets, nseq + 1 entries).
static int prefill_impl(const m2_dims* dims, const m2_layer* L, uint16_t* hidden, int32_t nseq, const int32_t* cu,
                        float* ssm_state, uint16_t* conv_state, int32_t* conv_pos, void* ws, size_t ws_bytes,
                        cudaStream_t stream, bool w8a8) {
  int st = m2_validate(dims, L);
  if (st) return st;
  if (nseq <= 0 || !cu || !hidden || !ssm_state || !conv_state || !conv_pos) return M2_ERR_ARG;
  if (cu[0] != 0) return M2_ERR_ARG;
  for (int i = 0; i < nseq; ++i)
    if (cu[i + 1] < cu[i]) return M2_ERR_ARG;
  const int T = cu[nseq];
  if (T <= 0) return M2_ERR_ARG;
  if (!al16(hidden) || !al16(ssm_state) || !al8(conv_state)) return M2_ERR_ALIGN;
  const m2_dims& d = *dims;
  std::vector<int32_t> tab(2 * (size_t)(nseq + 1));
  const int nchunks = ssd_chunk_table(cu, nseq, tab.data());
  if (w8a8 && T <= 8) return M2_ERR_UNSUPPORTED;  // the W8A8 arm runs on the tensor-core projections
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < prefill_ws(d, T, nseq, nchunks, w8a8))
    return M2_ERR_WORKSPACE;
  const Derived r = derive(d);
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  const PrefillMap wm = prefill_map(d, T, nseq, nchunks);
  uint16_t* xn = reinterpret_cast<uint16_t*>(w8 + wm.xn);
  uint16_t* zx = reinterpret_cast<uint16_t*>(w8 + wm.zx);
  uint16_t* u = reinterpret_cast<uint16_t*>(w8 + wm.u);
  float* y = reinterpret_cast<float*>(w8 + wm.y);
  uint16_t* g = reinterpret_cast<uint16_t*>(w8 + wm.g);
  float* us_in = reinterpret_cast<float*>(w8 + wm.unscale);
  float* us_out = us_in + T;
  int32_t* dtab = reinterpret_cast<int32_t*>(w8 + wm.tab);  // cu, then chunk offsets
  const bool ssd = ssd_supported(d.nheads, d.head_dim, d.d_state, d.n_groups);
  float* ssd_dh = reinterpret_cast<float*>(w8 + wm.ssd);
  float* ssd_decay =
      reinterpret_cast<float*>(w8 + rup(wm.ssd + (size_t)nchunks * d.nheads * d.head_dim * d.d_state * 4, 256));
  float* part = reinterpret_cast<float*>(w8 + wm.part);
  const size_t part_bytes = proj_part_bytes(d, T);
  // W8A8: E4M3 codes [T][ldq] of the projection inputs, scales [K/128][rup(T, 128)]
  uint8_t* q8 = w8 + wm.q8;
  const int ldq = (int)q8_ldq(d);
  float* sq = reinterpret_cast<float*>(w8 + wm.sq);
  const int ldsq = (int)rup((size_t)T, 128);
  const bool q_in = w8a8 && L->in_proj.fmt == M2_W_FP8_BLOCK128;
  const bool q_out = w8a8 && L->out_proj.fmt == M2_W_FP8_BLOCK128;

  cudaError_t e;
  // the sequence tables, stream-ordered before the kernels that read them
  // (pageable source: the call returns once the bytes are staged)
  if ((e = cudaMemcpyAsync(dtab, tab.data(), tab.size() * 4, cudaMemcpyHostToDevice, stream)))
    return launch_status(e);
  PrepArgs pa;
  memset(&pa, 0, sizeof(pa));
  pa.mode = PREP_RMSNORM;
  pa.x = hidden;
  pa.ldx = d.hidden;
  pa.w = L->norm_w;
  pa.eps = d.eps_in;
  pa.M = T;
  pa.K = d.hidden;
  pa.out = xn;
  pa.ldo = d.hidden;
  pa.f16 = proj_f16(L->in_proj, T) ? 1 : 0;
  pa.unscale = us_in;
  if (q_in) {
    pa.out = nullptr;
    pa.q8 = q8;
    pa.ldq = ldq;
    pa.sq = sq;
    pa.ldsq = ldsq;
  }
  if ((e = launch_prep(pa, stream))) return launch_status(e);
  GemvArgs qa;
  memset(&qa, 0, sizeof(qa));
  if (q_in) {
    qa.q8 = q8;
    qa.ldq = ldq;
    qa.sq = sq;
    qa.ldsq = ldsq;
  }
  if ((e = proj(L->in_proj, xn, d.hidden, T, zx, r.ldz, EPI_STORE, nullptr, 0, stream, &qa, us_in, 0, part,
                part_bytes)))
    return launch_status(e);
  if ((e = launch_conv_prefill(conv_state, conv_pos, zx + r.d_inner, r.ldz, L->conv_w, L->conv_b, u, r.d_xbc, T,
                               r.d_xbc, d.d_conv, dtab, nseq, stream)))
    return launch_status(e);
  if (ssd) {
    SsdArgs sa;
    memset(&sa, 0, sizeof(sa));
    sa.h = ssm_state;
    sa.x = u;
    sa.Bm = u + r.d_inner;
    sa.Cm = u + r.d_inner + d.n_groups * d.d_state;
    sa.dt = zx + r.d_inner + r.d_xbc;
    sa.ld_in = r.d_xbc;
    sa.ld_dt = r.ldz;
    sa.A_log = L->A_log;
    sa.D = L->D;
    sa.dt_bias = L->dt_bias;
    sa.y = y;
    sa.ldy = r.d_inner;
    sa.T = T;
    sa.H = d.nheads;
    sa.P = d.head_dim;
    sa.N = d.d_state;
    sa.G = d.n_groups;
    sa.pos_inc = conv_pos;
    sa.dH = ssd_dh;
    sa.decay = ssd_decay;
    sa.nchunks = nchunks;
    sa.nseq = nseq;
    sa.cu = dtab;
    sa.cprefix = dtab + nseq + 1;
    if ((e = launch_ssd(sa, stream))) return launch_status(e);
  } else {
    // shapes without the chunked scan: the sequential scan, one sequence at a time
    const size_t hstride = (size_t)d.nheads * d.head_dim * d.d_state;
    for (int i = 0; i < nseq; ++i) {
      const int Ti = cu[i + 1] - cu[i];
      if (Ti == 0) continue;
      ScanArgs sa;
      memset(&sa, 0, sizeof(sa));
      sa.h = ssm_state + (size_t)i * hstride;
      sa.x = u + (size_t)cu[i] * r.d_xbc;
      sa.Bm = sa.x + r.d_inner;
      sa.Cm = sa.x + r.d_inner + d.n_groups * d.d_state;
      sa.dt = zx + (size_t)cu[i] * r.ldz + r.d_inner + r.d_xbc;
      sa.ld_in = r.d_xbc;
      sa.ld_dt = r.ldz;
      sa.A_log = L->A_log;
      sa.D = L->D;
      sa.dt_bias = L->dt_bias;
      sa.y = y + (size_t)cu[i] * r.d_inner;
      sa.ldy = r.d_inner;
      sa.T = Ti;
      sa.H = d.nheads;
      sa.P = d.head_dim;
      sa.N = d.d_state;
      sa.G = d.n_groups;
      sa.pos_inc = conv_pos + i;
      if ((e = launch_ssm_scan_seq(sa, stream))) return launch_status(e);
    }
  }
  memset(&pa, 0, sizeof(pa));
  pa.mode = PREP_GATED;
  pa.y = y;
  pa.ldy = r.d_inner;
  pa.z = zx;
  pa.ldz = r.ldz;
  pa.w = L->gnorm_w;
  pa.eps = d.eps_gated;
  pa.group = d.gnorm_group;
  pa.M = T;
  pa.K = r.d_inner;
  pa.out = g;
  pa.ldo = r.d_inner;
  pa.f16 = proj_f16(L->out_proj, T) ? 1 : 0;
  pa.unscale = us_out;
  if (q_out) {
    pa.out = nullptr;
    pa.q8 = q8;
    pa.ldq = ldq;
    pa.sq = sq;
    pa.ldsq = ldsq;
  }
  if ((e = launch_prep(pa, stream))) return launch_status(e);
  memset(&qa, 0, sizeof(qa));
  if (q_out) {
    qa.q8 = q8;
    qa.ldq = ldq;
    qa.sq = sq;
    qa.ldsq = ldsq;
  }
  if ((e = proj(L->out_proj, g, r.d_inner, T, hidden, d.hidden, EPI_RESID, hidden, d.hidden, stream, &qa, us_out,
                0, part, part_bytes)))
    return launch_status(e);
  return M2_OK;
}

}  // namespace m2

extern "C" {

int mamba2_layer_prefill(const m2_dims* dims, const m2_layer* L, uint16_t* hidden, int32_t T, float* ssm_state,
                         uint16_t* conv_state, int32_t* conv_pos, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (T <= 0) return M2_ERR_ARG;
  const int32_t cu[2] = {0, T};
  return prefill_impl(dims, L, hidden, 1, cu, ssm_state, conv_state, conv_pos, ws, ws_bytes, stream, false);
}

int mamba2_layer_prefill_varlen(const m2_dims* dims, const m2_layer* L, uint16_t* hidden, int32_t nseq,
                                const int32_t* cu_seqlens, float* ssm_state, uint16_t* conv_state, int32_t* conv_pos,
                                void* ws, size_t ws_bytes, cudaStream_t stream) {
  return prefill_impl(dims, L, hidden, nseq, cu_seqlens, ssm_state, conv_state, conv_pos, ws, ws_bytes, stream,
                      false);
}

int mamba2_layer_prefill_varlen_w8a8(const m2_dims* dims, const m2_layer* L, uint16_t* hidden, int32_t nseq,
                                     const int32_t* cu_seqlens, float* ssm_state, uint16_t* conv_state,
                                     int32_t* conv_pos, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return prefill_impl(dims, L, hidden, nseq, cu_seqlens, ssm_state, conv_state, conv_pos, ws, ws_bytes, stream,
                      true);
}

size_t m2_workspace_bytes_varlen(const m2_dims* dims, int32_t max_seqs, int32_t max_total_tokens) {
  if (check_dims(dims) || max_seqs <= 0 || max_total_tokens < 0) return 0;
  return prefill_ws_bound(*dims, max_total_tokens, max_seqs);
}

int w8a16_gemv(const uint16_t* A, const uint8_t* W, const uint16_t* S, uint16_t* out, int32_t M, int32_t N,
               int32_t K, cudaStream_t stream) {
  if (!A || !W || !S || !out || M <= 0 || N <= 0 || K <= 0) return M2_ERR_ARG;
  if (K % 16 || K > 16384) return M2_ERR_UNSUPPORTED;
  if (!al16(A) || !al16(W)) return M2_ERR_ALIGN;
  m2_weight w;
  w.w = W;
  w.scale = S;
  w.n = N;
  w.k = K;
  w.fmt = M2_W_FP8_BLOCK128;
  return launch_status(proj(w, A, K, M, out, N, EPI_STORE, nullptr, 0, stream));
}

size_t m2_w8a8_workspace_bytes(int32_t M, int32_t K) {
  if (M <= 0 || K <= 0) return 0;
  const size_t ldq = rup((size_t)K, 16);
  return rup((size_t)M * ldq, 256) + rup((size_t)(K + 127) / 128 * rup((size_t)M, 128) * 4, 256);
}

int w8a8_gemm(const uint16_t* A, const uint8_t* W, const uint16_t* S, uint16_t* out, int32_t M, int32_t N, int32_t K,
              void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!A || !W || !S || !out || M <= 0 || N <= 0 || K <= 0) return M2_ERR_ARG;
  if (K % 128 || K > 16384 || M <= 8) return M2_ERR_UNSUPPORTED;
  if (!al16(A) || !al16(W)) return M2_ERR_ALIGN;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < m2_w8a8_workspace_bytes(M, K))
    return M2_ERR_WORKSPACE;
  uint8_t* q8 = static_cast<uint8_t*>(ws);
  const int ldq = (int)rup((size_t)K, 16);
  float* sq = reinterpret_cast<float*>(q8 + rup((size_t)M * ldq, 256));
  const int ldsq = (int)rup((size_t)M, 128);
  PrepArgs pa;
  memset(&pa, 0, sizeof(pa));
  pa.mode = PREP_QUANT;
  pa.x = A;
  pa.ldx = K;
  pa.M = M;
  pa.K = K;
  pa.q8 = q8;
  pa.ldq = ldq;
  pa.sq = sq;
  pa.ldsq = ldsq;
  cudaError_t e = launch_prep(pa, stream);
  if (e) return launch_status(e);
  m2_weight w;
  w.w = W;
  w.scale = S;
  w.n = N;
  w.k = K;
  w.fmt = M2_W_FP8_BLOCK128;
  GemvArgs qa;
  memset(&qa, 0, sizeof(qa));
  qa.q8 = q8;
  qa.ldq = ldq;
  qa.sq = sq;
  qa.ldsq = ldsq;
  return launch_status(proj(w, A, K, M, out, N, EPI_STORE, nullptr, 0, stream, &qa));
}

// Device-accessible address of p: device memory as is; page-locked host memory
// through its unified address; nullptr for anything else (pageable host memory).
static const void* device_view(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return p;
  if (at.type == cudaMemoryTypeHost && at.devicePointer) {
    // the same offset into the page-locked allocation
    const char* hb = static_cast<const char*>(at.hostPointer);
    const char* db = static_cast<const char*>(at.devicePointer);
    return db + (static_cast<const char*>(p) - hb);
  }
  return nullptr;
}

// Whether [p, p + bytes) lies inside one allocation the driver knows: the
// allocation's address range when the driver reports it, else both ends must
// be device-accessible at the same offset of one mapping.
typedef CUresult (*PFN_pointer_get_attribute)(void*, CUpointer_attribute, CUdeviceptr);
static bool within_one_allocation(const void* p, size_t bytes) {
  static PFN_pointer_get_attribute fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_pointer_get_attribute>(f);
  });
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  if (bytes > UINTPTR_MAX - a) return false;
  if (fn) {
    CUdeviceptr base = 0;
    size_t size = 0;
    if (fn(&base, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, (CUdeviceptr)a) == CUDA_SUCCESS &&
        fn(&size, CU_POINTER_ATTRIBUTE_RANGE_SIZE, (CUdeviceptr)a) == CUDA_SUCCESS && size > 0)
      return a >= (uintptr_t)base && a - (uintptr_t)base <= size && bytes <= size - (a - (uintptr_t)base);
  }
  const char* first = static_cast<const char*>(device_view(p));
  const char* last = static_cast<const char*>(device_view(static_cast<const char*>(p) + bytes - 16));
  return first && last && last == first + (bytes - 16);
}

int m2_copy(void* dst, const void* src, size_t bytes, cudaStream_t stream) {
  if (!dst || !src) return M2_ERR_ARG;
  if (bytes == 0) return M2_OK;
  if (!al16(dst) || !al16(src) || bytes % 16) return M2_ERR_ALIGN;
  const void* s = device_view(src);
  void* d = const_cast<void*>(device_view(dst));
  if (!s || !d) return M2_ERR_ARG;
  if (!within_one_allocation(src, bytes) || !within_one_allocation(dst, bytes)) return M2_ERR_ARG;
  return launch_status(launch_copy16(s, d, bytes / 16, stream));
}

int conv1d_update(uint16_t* conv_state, int32_t* conv_pos, const uint16_t* x, int32_t ld_x, const uint16_t* w,
                  const uint16_t* bias, uint16_t* out, int32_t B, int32_t C, int32_t d_conv, int32_t silu,
                  cudaStream_t stream) {
  if (!conv_state || !conv_pos || !x || !w || !out || B <= 0 || C <= 0 || ld_x < C) return M2_ERR_ARG;
  if (d_conv < 2 || d_conv > 8) return M2_ERR_UNSUPPORTED;
  cudaError_t e = launch_conv_update(conv_state, conv_pos, x, ld_x, w, bias, out, C, B, C, d_conv, silu, stream);
  if (e) return launch_status(e);
  return launch_status(launch_conv_pos(conv_pos, B, 1, stream));
}

int mamba2_ssm_step(float* h, const uint16_t* x, const uint16_t* Bm, const uint16_t* Cm, const uint16_t* dt_raw,
                    int32_t ld_in, const float* A_log, const float* D, const float* dt_bias, float* y, int32_t B,
                    int32_t H, int32_t P, int32_t N, int32_t G, cudaStream_t stream) {
  if (!h || !x || !Bm || !Cm || !dt_raw || !A_log || !D || !dt_bias || !y) return M2_ERR_ARG;
  if (B <= 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G) return M2_ERR_ARG;
  if (!(N == 16 || N == 32 || N == 64 || N == 128) || P > 256) return M2_ERR_UNSUPPORTED;
  if (ld_in % 4 || ld_in < H * P) return M2_ERR_ARG;
  if (!al16(h) || !al8(Bm) || !al8(Cm)) return M2_ERR_ALIGN;
  SsmArgs sa;
  memset(&sa, 0, sizeof(sa));
  sa.h = h;
  sa.x = x;
  sa.Bm = Bm;
  sa.Cm = Cm;
  sa.dt = dt_raw;
  sa.ld_in = ld_in;
  sa.A_log = A_log;
  sa.D = D;
  sa.dt_bias = dt_bias;
  sa.y = y;
  sa.ldy = H * P;
  sa.B = B;
  sa.H = H;
  sa.P = P;
  sa.N = N;
  sa.G = G;
  sa.pos_inc = nullptr;
  return launch_status(launch_ssm_step(sa, stream));
}

int mamba2_layer_decode(const m2_dims* dims, const m2_layer* L, uint16_t* hidden, int32_t B, float* ssm_state,
                        uint16_t* conv_state, int32_t* conv_pos, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return decode_impl(dims, L, hidden, B, ssm_state, conv_state, conv_pos, ws, ws_bytes, nullptr, 0, stream);
}

int mamba2_layer_decode_prefetch(const m2_dims* dims, const m2_layer* L, uint16_t* hidden, int32_t B,
                                 float* ssm_state, uint16_t* conv_state, int32_t* conv_pos, void* ws,
                                 size_t ws_bytes, const void* prefetch, size_t prefetch_bytes, cudaStream_t stream) {
  size_t n = prefetch ? prefetch_bytes / 16 * 16 : 0;
  if (n) {
    if (!al16(prefetch)) return M2_ERR_ALIGN;
    if (n > (size_t)M2_PREFETCH_MAX_BYTES || !within_one_allocation(prefetch, n)) return M2_ERR_ARG;
  }
  return decode_impl(dims, L, hidden, B, ssm_state, conv_state, conv_pos, ws, ws_bytes,
                     static_cast<const char*>(prefetch), n, stream);
}

// Scratch of mamba2_layer_decode_noalloc: a fixed device array, so that
// callers who cannot allocate still get a workspace.  Host code must not use
// the symbol as an address; the device address is looked up once per device.
static __device__ __align__(256) uint8_t g_noalloc_scratch[M2_NOALLOC_SCRATCH_BYTES];
static void* g_noalloc_ptr[64];
static std::mutex g_noalloc_mu;

int mamba2_layer_decode_noalloc(const m2_dims* dims, const m2_layer* layer, uint16_t* hidden, int32_t B,
                                float* ssm_state, uint16_t* conv_state, int32_t* conv_pos, cudaStream_t stream) {
  int st = m2_validate(dims, layer);
  if (st) return st;
  if (B <= 0) return M2_ERR_ARG;
  const size_t need = decode_ws_min(*dims, B);
  if (need > (size_t)M2_NOALLOC_SCRATCH_BYTES) return M2_ERR_SCRATCH;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return M2_ERR_DEVICE;
  void* ptr;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
      // the current device is `dev`: this resolves the array's address there
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return M2_ERR_DEVICE;
      }
      g_noalloc_ptr[dev] = p;
    }
    ptr = g_noalloc_ptr[dev];
  }
  return mamba2_layer_decode(dims, layer, hidden, B, ssm_state, conv_state, conv_pos, ptr,
                             (size_t)M2_NOALLOC_SCRATCH_BYTES, stream);
}

int m2_device_status(int clear) {
  if (cudaDeviceSynchronize() != cudaSuccess) return M2_ERR_LAUNCH;
  const int parts[] = {status_gemv(clear), status_gemv_mma(clear), status_gemm_tc(clear), status_mixer(clear)};
  for (int v : parts)
    if (v != 0) return v;
  return M2_OK;
}

int m2_workspace_map(const m2_dims* dims, int32_t kind, int32_t n, const int32_t* cu_seqlens, size_t* offsets,
                     int32_t n_offsets) {
  if (check_dims(dims) || !offsets || n_offsets < M2_WS_COUNT || n <= 0) return M2_ERR_ARG;
  for (int i = 0; i < n_offsets; ++i) offsets[i] = SIZE_MAX;
  if (kind == M2_WS_KIND_DECODE) {
    const DecodeMap m = decode_map(*dims, n);
    offsets[M2_WS_XN] = m.xn;
    offsets[M2_WS_ZX] = m.zxu;
    offsets[M2_WS_Y] = m.y;
    offsets[M2_WS_G] = m.g;
    offsets[M2_WS_UNSCALE] = m.unscale;
    return M2_OK;
  }
  if (kind != M2_WS_KIND_PREFILL && kind != M2_WS_KIND_PREFILL_W8A8) return M2_ERR_ARG;
  if (!cu_seqlens || cu_seqlens[0] != 0) return M2_ERR_ARG;
  for (int i = 0; i < n; ++i)
    if (cu_seqlens[i + 1] < cu_seqlens[i]) return M2_ERR_ARG;
  const int T = cu_seqlens[n];
  if (T <= 0) return M2_ERR_ARG;
  std::vector<int32_t> tab(2 * (size_t)(n + 1));
  const int nchunks = ssd_chunk_table(cu_seqlens, n, tab.data());
  const PrefillMap m = prefill_map(*dims, T, n, nchunks);
  offsets[M2_WS_XN] = m.xn;
  offsets[M2_WS_ZX] = m.zx;
  offsets[M2_WS_U] = m.u;
  offsets[M2_WS_Y] = m.y;
  offsets[M2_WS_G] = m.g;
  offsets[M2_WS_UNSCALE] = m.unscale;
  if (kind == M2_WS_KIND_PREFILL_W8A8) {
    offsets[M2_WS_Q8] = m.q8;
    offsets[M2_WS_SQ] = m.sq;
  }
  return M2_OK;
}

int m2_set_wait_limit(int64_t cycles) {
  const long long v = cycles > 0 ? (long long)cycles : 4000000000LL;
  if (wait_limit_gemv(v) != cudaSuccess || wait_limit_gemv_mma(v) != cudaSuccess ||
      wait_limit_gemm_tc(v) != cudaSuccess || wait_limit_mixer(v) != cudaSuccess) {
    cudaGetLastError();
    return M2_ERR_DEVICE;
  }
  return M2_OK;
}

int m2_wait_check(const void* probe, void* out, cudaStream_t stream) {
  if (!probe || !out) return M2_ERR_ARG;
  if (!al16(probe) || !al16(out)) return M2_ERR_ALIGN;
  return launch_status(launch_wait_check(probe, out, stream));
}

int64_t m2_launch_count(void) { return g_launches.load(); }

int m2_trace_begin(int32_t capacity) {
  if (capacity <= 0) return M2_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  for (auto& t : g_trace) {
    cudaEventDestroy(t.a);
    cudaEventDestroy(t.b);
  }
  g_trace.assign(capacity, TraceSlot{});
  for (auto& t : g_trace) {
    if (cudaEventCreate(&t.a) != cudaSuccess || cudaEventCreate(&t.b) != cudaSuccess) return M2_ERR_LAUNCH;
  }
  g_trace_used = 0;
  g_trace_on = true;
  return M2_OK;
}

int m2_trace_end(double* ms, int32_t* launches, int32_t n_ids) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_on = false;
  if (ms && launches) {
    for (int i = 0; i < n_ids; ++i) {
      ms[i] = 0.0;
      launches[i] = 0;
    }
  }
  for (int i = 0; i < g_trace_used; ++i) {
    const TraceSlot& t = g_trace[i];
    if (cudaEventSynchronize(t.b) != cudaSuccess) return M2_ERR_LAUNCH;
    float v = 0.f;
    cudaEventElapsedTime(&v, t.a, t.b);
    if (ms && launches && t.id >= 0 && t.id < n_ids) {
      ms[t.id] += v;
      launches[t.id] += 1;
    }
  }
  for (auto& t : g_trace) {
    cudaEventDestroy(t.a);
    cudaEventDestroy(t.b);
  }
  g_trace.clear();
  const int used = g_trace_used;
  g_trace_used = 0;
  return used;
}

int m2_set_fused_decode(int enable) {
  const int prev = g_fused_decode;
  g_fused_decode = enable ? 1 : 0;
  return prev;
}

const char* m2_kernel_name(int32_t id) { return (id >= 0 && id < K_COUNT) ? kNames[id] : nullptr; }

int32_t m2_kernel_count(void) { return K_COUNT; }

}  // extern "C"
