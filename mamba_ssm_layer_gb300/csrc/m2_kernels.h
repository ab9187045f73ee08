// m2_kernels.h -- internal (not exported) launcher interface between the ABI
// layer (m2_abi.cu) and the kernel translation units.  Launchers enqueue on
// `stream`, do no argument validation (the ABI layer did it) and return a
// cudaError_t from the launch.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace m2 {

// Kernel ids for launch counting and tracing (names in m2_abi.cu).
enum KernelId : int32_t {
  K_PREP = 0,
  K_GEMV_FP8,        // + GemvEpi: store, conv (in_proj), resid (out_proj)
  K_GEMV_FP8_CONV,
  K_GEMV_FP8_RESID,
  K_GEMV_BF16,
  K_GEMV_BF16_CONV,
  K_GEMV_BF16_RESID,
  K_CONV_UPDATE,
  K_CONV_POS,
  K_SSM_STEP,
  K_CONV_PREFILL,
  K_SSM_SCAN_SEQ,
  K_GEMM_TC,
  K_SSD_CHUNK_STATE,
  K_SSD_STATE_PASS,
  K_SSD_CHUNK_OUT,
  K_GEMM_TC_REDUCE,
  K_CONV_RING,
  K_DECODE_FUSED,
  K_COPY,
  K_WAIT_CHECK,
  K_COUNT
};

// Called by every launcher around its launch (counting / tracing).
void trace_pre(int32_t id, cudaStream_t s);
void trace_post(int32_t id, cudaStream_t s);

// Host readers of each translation unit's device status word (0 or
// M2_ERR_TIMEOUT); clear != 0 resets it.
int status_gemv(int clear);
int status_gemv_mma(int clear);
int status_gemm_tc(int clear);
int status_mixer(int clear);
// Setters of each translation unit's pipeline wait limit (SM clock cycles).
cudaError_t wait_limit_gemv(long long cycles);
cudaError_t wait_limit_gemv_mma(long long cycles);
cudaError_t wait_limit_gemm_tc(long long cycles);
cudaError_t wait_limit_mixer(long long cycles);

// Number of SMs of the current device (cached).
int num_sms();

// Opt a kernel into large dynamic shared memory once per device.
cudaError_t set_smem_once(const void* func, int bytes, int* done_mask);

// ------------------------------------------------------------------ GEMV

enum GemvEpi : int32_t {
  EPI_STORE = 0,       // out[m*ldo+n] = bf16(acc)
  EPI_RESID = 1,       // out[m*ldo+n] = bf16(resid[m*ldr+n] + acc)   (resid may alias out)
  EPI_INPROJ_CONV = 2  // rows [xbc0, xbc0+d_xbc): conv update + SiLU; other rows: store
};

struct GemvArgs {
  const uint16_t* A;   // [M][lda] bf16
  int32_t lda;
  const void* W;       // [N][K] E4M3 or bf16
  const uint16_t* S;   // E4M3 scales [ceil(N/128)][ceil(K/128)] (unused for bf16)
  int32_t M, N, K;
  uint16_t* out;       // [M][ldo]
  int32_t ldo;
  int32_t epi;
  const uint16_t* resid;  // EPI_RESID
  int32_t ldr;
  // EPI_INPROJ_CONV: ring [M][dconv-1][d_xbc], pos [M], conv_w [d_xbc][dconv], conv_b [d_xbc]
  uint16_t* ring;
  const int32_t* pos;
  const uint16_t* conv_w;
  const uint16_t* conv_b;
  int32_t xbc0, d_xbc, dconv;
  int32_t evict_first;  // stream weights with the L2 evict-first policy
  // Activation input of the GEMV:
  int32_t act;          // GemvAct
  const float* unscale; // ACT_PREPARED: per batch row factor applied to the row totals
  // Launch as a programmatic dependent of the previous kernel.  Then only A and
  // unscale may be produced by that immediately preceding kernel; the
  // epilogue inputs (ring, pos, resid) must come from earlier launches, and
  // are read before the dependency wait.
  int32_t pdl;
  // tensor-core GEMM only: scratch for k-split partials (may be null: no split)
  float* part;
  size_t part_bytes;
  // Decode GEMV only: the activation rows are computed in the GEMV's prologue
  // from the norm's inputs instead of being read prepared (NORM_NONE).
  int32_t norm;             // GemvNorm
  const uint16_t* norm_w;   // [K] bf16 norm weight
  float norm_eps;
  const char* l2_ahead;     // optional: bytes for a later launch, pulled toward L2 once this
  size_t l2_ahead_bytes;    // launch's own weight ring is issued (16-byte aligned, multiple of 16)
  const float* gy;          // NORM_GATED: y [M][ldgy] fp32, z [M][ldgz] bf16 (whole-row span)
  int32_t ldgy;
  const uint16_t* gz;
  int32_t ldgz;
  // Tensor-core GEMM, W8A8 arm (E4M3 weights only): when q8 is set, the
  // activations are E4M3 codes [M][ldq] (A unused) with fp32 scales
  // [K/128][ldsq] (ldsq a multiple of 128), and the product is
  // sum_b S[n/128][b] * sq[b][m] * sum_{k in b} q8[m][k] W[n][k].
  const uint8_t* q8;
  int32_t ldq;
  const float* sq;
  int32_t ldsq;
};

enum GemvNorm : int32_t {
  NORM_NONE = 0,
  NORM_RMS = 1,    // A rows are the hidden rows x: activation = bf16(x * r * w)
  NORM_GATED = 2   // activation = bf16(y * r * w * silu(z)), r over the whole row
};

enum GemvAct : int32_t {
  ACT_PLAIN = 0,    // A is bf16; for E4M3 weights the kernel finds each row's f16 prescale
  ACT_PREPARED = 1  // A is already f16 (E4M3 weights: prescaled by 2^j, unscale = 2^-j) or bf16
};

// Activation preparation (one CTA per batch row): the norm that produces a
// GEMV's activation, rounded to bf16 at the layer's rounding point, then
// either stored as bf16 or, for an E4M3-weight GEMV, as f16 after an exact
// per-row power-of-two prescale 2^j that puts the row maximum in [2^14, 2^15)
// (unscale[m] = 2^-j).
enum PrepMode : int32_t {
  PREP_RMSNORM = 0,  // x * r * w, r = 1/sqrt(mean(x^2) + eps) (input RMSNorm)
  PREP_GATED = 1,    // y * r * w * silu(z), r over groups of `group` (gated RMSNorm)
  PREP_QUANT = 2     // x as is (bf16 rows), for the W8A8 quantization alone
};
struct PrepArgs {
  int32_t mode;
  const uint16_t* x;  // PREP_RMSNORM: [M][ldx] bf16
  int32_t ldx;
  const float* y;     // PREP_GATED: [M][ldy] fp32
  int32_t ldy;
  const uint16_t* z;  // PREP_GATED: [M][ldz] bf16
  int32_t ldz;
  const uint16_t* w;  // norm weight [K] bf16
  float eps;
  int32_t group;
  int32_t M, K;
  uint16_t* out;      // [M][ldo]
  int32_t ldo;
  int32_t f16;        // 1: prescaled f16 + unscale; 0: bf16
  float* unscale;     // [M] (f16 mode)
  int32_t pdl;
  // W8A8 arm (out may be null): E4M3 codes [M][ldq] and fp32 block scales
  // [ceil(K/128)][ldsq] of each row and 128-element block: amax = max |v|,
  // codes E4M3(v * (448 / amax)), scale amax / 448 (fp32; zero block: 0, 0).
  uint8_t* q8;
  int32_t ldq;
  float* sq;
  int32_t ldsq;
};
cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s);

// CUDA-core GEMV (fp32 accumulation) with bulk-copy weight streaming; any M
// (processed in groups of up to 4 rows, re-streaming the weights per group).
cudaError_t launch_gemv(const GemvArgs& a, bool fp8, cudaStream_t s);

// Launch helper: plain launch, or with programmatic stream serialisation (the
// kernel may start while the previous kernel in the stream is still running;
// it must execute griddepcontrol.wait before touching that kernel's outputs).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
}

// ------------------------------------------------------------------ mixer ops

// One-token conv update for B sequences (no pos advance; see launch_conv_pos).
cudaError_t launch_conv_update(uint16_t* ring, const int32_t* pos, const uint16_t* x, int32_t ldx,
                               const uint16_t* w, const uint16_t* b, uint16_t* out, int32_t ldo, int32_t B,
                               int32_t C, int32_t dconv, int32_t silu, cudaStream_t s);
cudaError_t launch_conv_pos(int32_t* pos, int32_t B, int32_t add, cudaStream_t s);
// n16 16-byte units from src to dst (both 16-byte aligned, device-accessible
// addresses), as a programmatic dependent of the previous kernel.
cudaError_t launch_copy16(const void* src, void* dst, size_t n16, cudaStream_t s);

struct SsmArgs {
  float* h;            // [B][H][P][N]
  const uint16_t* x;   // rows ld_in apart
  const uint16_t* Bm;
  const uint16_t* Cm;
  const uint16_t* dt;
  int32_t ld_in;
  const float* A_log;
  const float* D;
  const float* dt_bias;
  float* y;            // [B][ldy]
  int32_t ldy;
  int32_t B, H, P, N, G;
  int32_t* pos_inc;    // if non-null: pos_inc[b] += 1 (decode fusion)
  int32_t pdl;         // launch as a programmatic dependent of the previous kernel
  // Optional L2 prefetch issued at kernel start (the weights of the launch
  // after next): a byte range, 16-byte aligned, size a multiple of 16.
  const void* l2_prefetch;
  size_t l2_prefetch_bytes;
};
cudaError_t launch_ssm_step(const SsmArgs& a, cudaStream_t s);

// The whole decode step of one sequence in one cooperative launch
// (k_gemv_mma.cu): in = the in_proj GEMV (M = 1, NORM_RMS, EPI_INPROJ_CONV),
// ssm = the SSM step (B = 1, y written for the gated norm, pos_inc advanced),
// out = the out_proj GEMV (M = 1, NORM_GATED on ssm.y and z, EPI_RESID in
// place).  Both projections in the same format (fp8).  Calls on one device
// must not overlap: the grid barriers share one device-wide counter.
struct FusedStepArgs {
  GemvArgs in;
  SsmArgs ssm;
  GemvArgs out;
};
bool decode_fused_supported(const FusedStepArgs& fa, bool fp8);
cudaError_t launch_decode_fused(const FusedStepArgs& fa, bool fp8, cudaStream_t s);

// Largest batch row count one GEMV pass covers for a K-wide row.
int gemv_rows_per_pass(int K, bool fp8);

// tcgen05 GEMM (k_gemm_tc.cu) for M > 8 rows: bf16 activations (ACT_PLAIN).
bool gemm_tc_supported(int M, int N, int K, bool fp8);
// k-split factor the GEMM uses for this shape, and the partial scratch it needs
// (0 when it does not split).
int gemm_tc_ksplit(int M, int N, int K);
size_t gemm_tc_partial_bytes(int M, int N, int K);
cudaError_t launch_gemm_tc(const GemvArgs& a, bool fp8, cudaStream_t s);
// The timeout-path check of m2_wait_check (k_gemm_tc.cu): probe and out are
// 16-byte aligned device addresses of 16 bytes.
cudaError_t launch_wait_check(const void* probe, void* out, cudaStream_t s);

// Warp-MMA decode GEMV (k_gemv_mma.cu): M <= 8, K % 64 == 0, K <= 8192.
bool gemv_mma_supported(int M, int K);
cudaError_t launch_gemv_mma(const GemvArgs& a, bool fp8, cudaStream_t s);


// Prefill conv over a varlen batch: T token rows (xbc rows ldx apart -> u
// [T][ldu]), rows cu[i] .. cu[i+1]-1 of sequence i (cu: device, nseq+1
// entries); reads each sequence's ring [nseq][d_conv-1][C] for the first taps
// and leaves it holding the sequence's last tokens.  Does not advance pos.
cudaError_t launch_conv_prefill(uint16_t* ring, const int32_t* pos, const uint16_t* xbc, int32_t ldx,
                                const uint16_t* w, const uint16_t* b, uint16_t* u, int32_t ldu, int32_t T,
                                int32_t C, int32_t dconv, const int32_t* cu, int32_t nseq, cudaStream_t s);

// Sequential per-token scan of one sequence (T steps, state in registers).
struct ScanArgs {
  float* h;            // [H][P][N]
  const uint16_t* x;   // [T] rows ld_in apart
  const uint16_t* Bm;
  const uint16_t* Cm;
  const uint16_t* dt;  // [T] rows ld_dt apart
  int32_t ld_in, ld_dt;
  const float* A_log;
  const float* D;
  const float* dt_bias;
  float* y;            // [T][ldy]
  int32_t ldy;
  int32_t T, H, P, N, G;
  int32_t* pos_inc;    // pos_inc[0] += T if non-null
};
cudaError_t launch_ssm_scan_seq(const ScanArgs& a, cudaStream_t s);

// Chunked (state-space dual) scan of a varlen batch of sequences, chunk
// length 128 (k_ssd.cu): chunk states, a sequential pass over each sequence's
// chunk states, chunk outputs.  Sequence i owns token rows cu[i] .. cu[i+1]-1
// and chunks cprefix[i] .. cprefix[i+1]-1 (ceil(T_i / 128) of them).
struct SsdArgs {
  float* h;            // [nseq][H][P][N], updated in place
  const uint16_t* x;   // token rows ld_in apart
  const uint16_t* Bm;
  const uint16_t* Cm;
  const uint16_t* dt;  // token rows ld_dt apart
  int32_t ld_in, ld_dt;
  const float* A_log;
  const float* D;
  const float* dt_bias;
  float* y;            // [T][ldy]
  int32_t ldy;
  int32_t T, H, P, N, G;
  int32_t* pos_inc;    // pos_inc[i] += T_i if non-null
  float* dH;           // scratch [H][nchunks][P][N]
  float* decay;        // scratch [H][nchunks]
  int32_t nchunks;     // total chunks of all sequences
  int32_t nseq;
  const int32_t* cu;       // device [nseq + 1] token offsets
  const int32_t* cprefix;  // device [nseq + 1] chunk offsets
};
// Chunks of a varlen batch and the host tables (cu then cprefix, 2 * (nseq + 1) ints).
int32_t ssd_chunk_table(const int32_t* cu_host, int32_t nseq, int32_t* table_out);
bool ssd_supported(int H, int P, int N, int G);
size_t ssd_workspace_bytes(int nchunks, int H, int P, int N);  // dH then decay, each 256-aligned
cudaError_t launch_ssd(const SsdArgs& a, cudaStream_t s);

}  // namespace m2
