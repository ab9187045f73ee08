/*
 * mamba2.h -- C ABI of the GB300 (sm_103a) Mamba-2 layer forward library
 * (libmamba2_gb300.so).
 *
 * The layer is the Nemotron-H Mamba-2 mixer block as the source listing
 * "spark_model/layers/nemotron_mamba2.rs" describes it in its module header
 * ("Forward pass", steps 1-8):
 *   1 RMSNorm (weight * x)        2 in_proj GEMV -> [z, xBC, dt]
 *   3 conv1d update on xBC, with bias, fused SiLU
 *   4 split xBC -> x, B, C        5 Mamba-2 SSM state update and output
 *   6 gated RMSNorm: rms_norm(y, ssm_norm) * silu(z)
 *   7 out_proj GEMV               8 residual add
 * FP8 projections use the w8a16 block-scaled GEMV of the page "Struct
 * Qwen3SsmLayer" (`set_fp8_decode_weights`):
 *   out[n] = sum_k A[k] * E4M3(W[n,k]) * block_scale[n/128, k/128],
 * with the scale grid [ceil(N/128)][ceil(K/128)] in bf16 and the index
 * block_scale[n/128 * k_blocks + k/128] of "Struct NemotronMamba2Layer"
 * (`set_fp8_weights`).
 *
 * Conventions for every entry point below:
 *  - Every data pointer is a DEVICE pointer owned by the caller (m2_copy also
 *    takes page-locked host pointers).  The library allocates and frees no
 *    device memory; scratch comes from the caller's workspace (`ws`,
 *    `ws_bytes`), or from the built-in scratch of mamba2_layer_decode_noalloc.
 *  - bf16 values are passed as uint16_t bit patterns; E4M3 as uint8_t.
 *    Matrices are row-major with the last index contiguous.
 *  - Work is enqueued asynchronously on `stream` (0 = legacy default stream)
 *    of the current device; the call returns once it is enqueued.
 *  - Return value: M2_OK (0) or a negative M2_ERR_* code.  All arguments are
 *    checked on the host before anything is launched: on an argument error
 *    nothing is launched and no buffer is touched.  M2_ERR_LAUNCH reports a
 *    launch failure seen by cudaGetLastError after enqueueing.
 *  - Kernels never spin without a bound.  If a bounded wait inside a kernel
 *    gives up, the kernel records M2_ERR_TIMEOUT in a device status word that
 *    m2_device_status() returns.
 *  - Calls that share state or workspace must be ordered (same stream, or
 *    synchronised); concurrent calls on distinct buffers are independent,
 *    except mamba2_layer_decode_noalloc (one built-in scratch per device) and
 *    the single-launch batch-1 decode selected by m2_set_fused_decode(1) (one
 *    grid-barrier counter per device).
 */
#ifndef MAMBA2_GB300_H
#define MAMBA2_GB300_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status codes */
enum {
  M2_OK = 0,
  M2_ERR_ARG = -1,         /* null pointer, non-positive or inconsistent size */
  M2_ERR_FORMAT = -2,      /* weight format tag / scale grid inconsistent     */
  M2_ERR_WORKSPACE = -3,   /* workspace missing or smaller than required      */
  M2_ERR_LAUNCH = -4,      /* a CUDA launch or attribute call failed          */
  M2_ERR_UNSUPPORTED = -5, /* shape outside the supported range               */
  M2_ERR_ALIGN = -6,       /* pointer not 16-byte aligned where required      */
  M2_ERR_DEVICE = -7,      /* no device, or a device older than sm_103        */
  M2_ERR_TIMEOUT = -8,     /* a bounded in-kernel wait gave up                */
  M2_ERR_SCRATCH = -9      /* request larger than the built-in scratch of
                              mamba2_layer_decode_noalloc                     */
};

/* Weight formats.  FP8_BLOCK128: E4M3 bytes [n][k] plus bf16 scales
 * [ceil(n/128)][ceil(k/128)] ("Fp8BlockScaled").  BF16: bf16 [n][k], no scale
 * (the unquantised projections of a mixed-precision checkpoint, source listing
 * struct comment on native BF16 projections). */
enum { M2_W_FP8_BLOCK128 = 1, M2_W_BF16 = 2 };

/* Layer dimensions.  d_inner = nheads*head_dim; d_xbc = d_inner +
 * 2*n_groups*d_state; in_proj rows n_in = 2*d_inner + 2*n_groups*d_state +
 * nheads.  gnorm_group is the span of the gated RMSNorm (d_inner: the whole
 * row; a divisor of d_inner: group-wise).  Supported: hidden and d_inner
 * multiples of 16 and <= 16384; d_state in {16,32,64,128}; head_dim <= 256;
 * nheads % n_groups == 0; 2 <= d_conv <= 8. */
typedef struct m2_dims {
  int32_t hidden, nheads, head_dim, d_state, n_groups, d_conv;
  float eps_in;     /* input RMSNorm epsilon (1e-5) */
  float eps_gated;  /* gated RMSNorm epsilon (1e-5) */
  int32_t gnorm_group;
} m2_dims;

typedef struct m2_weight {
  const void* w;          /* [n][k]: uint8 E4M3 or uint16 bf16; 16-byte aligned */
  const uint16_t* scale;  /* FP8: bf16 [ceil(n/128)][ceil(k/128)]; BF16: NULL   */
  int32_t n, k;
  int32_t fmt;            /* M2_W_FP8_BLOCK128 or M2_W_BF16                    */
} m2_weight;

/* One layer's parameters (all device pointers; the caller keeps them alive). */
typedef struct m2_layer {
  const uint16_t* norm_w;  /* [hidden] bf16, input RMSNorm weight            */
  m2_weight in_proj;       /* n = n_in, k = hidden                           */
  const uint16_t* conv_w;  /* [d_xbc][d_conv] bf16 (tap d_conv-1 = current)  */
  const uint16_t* conv_b;  /* [d_xbc] bf16                                   */
  const float* A_log;      /* [nheads]; A = -exp(A_log)                      */
  const float* D;          /* [nheads]                                       */
  const float* dt_bias;    /* [nheads]                                       */
  const uint16_t* gnorm_w; /* [d_inner] bf16, gated RMSNorm weight           */
  m2_weight out_proj;      /* n = hidden, k = d_inner                        */
} m2_layer;

/* Human-readable text for a status code (static storage). */
const char* m2_strerror(int status);

/* Host-only check of dimensions and parameters (formats, scale grids, shapes,
 * alignment).  Launches nothing.  The layer entry points run it themselves. */
int m2_validate(const m2_dims* dims, const m2_layer* layer);

/* Bytes of workspace that mamba2_layer_decode with batch <= max_batch and
 * mamba2_layer_prefill with T <= max_tokens need (the larger of the two).
 * Returns 0 for invalid dims. */
size_t m2_workspace_bytes(const m2_dims* dims, int32_t max_batch, int32_t max_tokens);

/* One decode step of B independent sequences, one token each (page "Trait
 * TransformerLayer", `decode` / `decode_multi_seq`: weights are read once for
 * all B rows).
 *   hidden     [B][hidden] bf16, read and overwritten with the layer output
 *              hidden + out_proj(...)  (in place, as `decode` specifies).
 *   ssm_state  [B][nheads][head_dim][d_state] fp32, updated in place.
 *   conv_state [B][d_conv-1][d_xbc] bf16 ring: token t of a sequence lives in
 *              slot t mod (d_conv-1); zero-initialise for a new sequence.
 *   conv_pos   [B] int32, tokens seen so far per sequence; advanced by 1.
 *   ws         workspace of at least m2_workspace_bytes(dims, B, 0) bytes,
 *              256-byte aligned; its contents are scratch.
 * The step runs as a chain of three kernels (B <= 8) or five (tensor-core
 * projections, B > 8).  After m2_set_fused_decode(1), a B = 1 step (both
 * projections in one format, K <= 8192) runs as one cooperative launch with
 * two grid-wide barriers instead; such calls on one device must not overlap
 * in time (the barriers share one device-wide counter), so issue them on one
 * stream.  Both forms give bit-identical results. */
int mamba2_layer_decode(const m2_dims* dims, const m2_layer* layer, uint16_t* hidden, int32_t B,
                        float* ssm_state, uint16_t* conv_state, int32_t* conv_pos, void* ws,
                        size_t ws_bytes, cudaStream_t stream);

/* mamba2_layer_decode with a prefetch hint: the device byte range
 * [prefetch, prefetch + prefetch_bytes) -- typically the first weights the
 * NEXT call on this stream reads, e.g. the following layer's in_proj -- is
 * pulled toward L2 while this step's out_proj runs, when the memory system
 * has spare bandwidth (the out_proj reads its own weights from L2, where the
 * SSM kernel put them).  A hint only: results are bit-identical to
 * mamba2_layer_decode, and it applies to the batch <= 8 kernel chain (other
 * forms ignore it).  prefetch_bytes 0 (or a null prefetch) means no hint.
 * More is not better: the pulled bytes share the memory system with the
 * step's own traffic (measured on the 8B-like layer at batch 1: the first
 * 8 MB of the next layer's 76 MB in_proj gave the shortest step, the whole
 * matrix a longer one than no hint).
 * Errors, returned before anything is launched: M2_ERR_ALIGN if prefetch is
 * not 16-byte aligned; M2_ERR_ARG if the range is not inside one device
 * allocation or exceeds M2_PREFETCH_MAX_BYTES.  Other arguments and errors as
 * mamba2_layer_decode. */
#define M2_PREFETCH_MAX_BYTES (96ull << 20)
int mamba2_layer_decode_prefetch(const m2_dims* dims, const m2_layer* layer, uint16_t* hidden, int32_t B,
                                 float* ssm_state, uint16_t* conv_state, int32_t* conv_pos, void* ws,
                                 size_t ws_bytes, const void* prefetch, size_t prefetch_bytes, cudaStream_t stream);

/* Select the single-launch batch-1 decode step (enable != 0) or the kernel
 * chain (0, the default) for later mamba2_layer_decode calls in this process.
 * Host setting only; returns the previous setting. */
int m2_set_fused_decode(int enable);

/* Prefill of T tokens of ONE sequence (page "Trait TransformerLayer",
 * `prefill`: projections as GEMMs over the T tokens; the result equals T
 * sequential decode steps).  The recurrence runs as the chunked
 * state-space-dual scan with 128-token chunks (source listing kernel table,
 * "SSD chunked prefill scan"): only chunk states are carried serially.
 * hidden [T][hidden] bf16 in/out; ssm_state
 * [nheads][head_dim][d_state] fp32, conv_state [d_conv-1][d_xbc] bf16 and
 * conv_pos [1] int32 are the sequence's state before the block and are left
 * as the state after it (conv_pos += T).  ws: m2_workspace_bytes(dims, 0, T). */
int mamba2_layer_prefill(const m2_dims* dims, const m2_layer* layer, uint16_t* hidden, int32_t T,
                         float* ssm_state, uint16_t* conv_state, int32_t* conv_pos, void* ws,
                         size_t ws_bytes, cudaStream_t stream);

/* Prefill of a varlen batch of sequences in one call per kernel ("Trait
 * TransformerLayer": `decode_batched` runs K tokens of one sequence with
 * GEMM-batched projections, `decode_verify_multi` n sequences x k tokens in one
 * weight sweep, rows sequence-major; the same batching serves prompts of
 * different lengths).  Token rows cu_seqlens[i] .. cu_seqlens[i+1]-1 of hidden
 * belong to sequence i; each sequence's result equals its own prefill (and so
 * its T_i sequential decode steps).  K-token decode of n sequences is the case
 * cu_seqlens = {0, K, 2K, ...}.
 *   hidden      [T][hidden] bf16 in/out, T = cu_seqlens[nseq] >= 1.
 *   nseq        number of sequences (>= 1); sequences of length 0 are allowed
 *               and left untouched.
 *   cu_seqlens  HOST array of nseq + 1 int32 offsets: cu_seqlens[0] = 0,
 *               non-decreasing.  Read during the call only.
 *   ssm_state   [nseq][nheads][head_dim][d_state] fp32, conv_state
 *               [nseq][d_conv-1][d_xbc] bf16, conv_pos [nseq] int32: each
 *               sequence's state before its block, left as the state after it
 *               (conv_pos[i] += T_i).
 *   ws          m2_workspace_bytes_varlen(dims, nseq, T) bytes suffice.
 * The call enqueues one small host-to-device copy of the sequence tables into
 * the workspace ahead of the kernels. */
int mamba2_layer_prefill_varlen(const m2_dims* dims, const m2_layer* layer, uint16_t* hidden, int32_t nseq,
                                const int32_t* cu_seqlens, float* ssm_state, uint16_t* conv_state,
                                int32_t* conv_pos, void* ws, size_t ws_bytes, cudaStream_t stream);

/* The same prefill on the W8A8 arm: the inputs of the E4M3 projections are
 * quantized to E4M3 too, per token row and 128-element k block
 * (amax = max |v|, codes E4M3(v * (448 / amax)) rounded to nearest even and
 * saturated, scale amax / 448, both in fp32; an all-zero block has scale 0),
 * and the projections multiply E4M3 by E4M3 on the tensor cores:
 *   out[m][n] = sum_b S[n/128][b] * s_a[m][b] * sum_{k in b} E4M3(q[m][k]) * E4M3(W[n][k]).
 * The pages give FP8 x FP8 GEMMs and a bf16 -> FP8 activation conversion for
 * prefill, not their scaling; this is the block scaling of the weights applied
 * to the activations.  It changes the numbers (activation rounding of about
 * 2^-4 relative) and is selected explicitly.  BF16-weight projections keep
 * bf16 activations.  Needs more than 8 token rows (M2_ERR_UNSUPPORTED
 * otherwise); arguments as mamba2_layer_prefill_varlen. */
int mamba2_layer_prefill_varlen_w8a8(const m2_dims* dims, const m2_layer* layer, uint16_t* hidden, int32_t nseq,
                                     const int32_t* cu_seqlens, float* ssm_state, uint16_t* conv_state,
                                     int32_t* conv_pos, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Workspace bytes for mamba2_layer_prefill_varlen (and its W8A8 form) with at
 * most max_seqs sequences and max_total_tokens token rows.  Returns 0 for
 * invalid dims. */
size_t m2_workspace_bytes_varlen(const m2_dims* dims, int32_t max_seqs, int32_t max_total_tokens);

/* The w8a16 block-scaled GEMV/GEMM (page "Struct Qwen3SsmLayer",
 * `set_fp8_decode_weights`):
 *   out[m][n] = bf16( sum_k A[m][k] * E4M3(W[n][k]) * S[n/128][k/128] )
 * A [M][K] bf16, W [N][K] E4M3 (16-byte aligned, K % 16 == 0), S bf16
 * [ceil(N/128)][ceil(K/128)], out [M][N] bf16.  fp32 accumulation. */
int w8a16_gemv(const uint16_t* A, const uint8_t* W, const uint16_t* S, uint16_t* out, int32_t M,
               int32_t N, int32_t K, cudaStream_t stream);

/* The W8A8 arm's product as a unit (the FP8-activation counterpart of
 * w8a16_gemv): each row of A [M][K] bf16 is quantized to E4M3 per 128-element
 * k block as in mamba2_layer_prefill_varlen_w8a8, then
 *   out[m][n] = bf16( sum_b S[n/128][b] * s_a[m][b] * sum_{k in b} E4M3(q[m][k]) * E4M3(W[n][k]) )
 * on the tensor cores.  M > 8, K % 128 == 0.  ws: m2_w8a8_workspace_bytes(M,
 * K) bytes, 256-byte aligned; on return it holds the codes [M][rup16(K)]
 * (uint8) followed, at the next 256-byte boundary, by the scales
 * [K/128][rup128(M)] (fp32). */
size_t m2_w8a8_workspace_bytes(int32_t M, int32_t K);
int w8a8_gemm(const uint16_t* A, const uint8_t* W, const uint16_t* S, uint16_t* out, int32_t M, int32_t N, int32_t K,
              void* ws, size_t ws_bytes, cudaStream_t stream);

/* One-token causal depthwise conv update with bias and optional SiLU (source
 * listing, `conv1d_update_biased`) for B sequences of C channels:
 *   out[b][c] = act( bias[c] + sum_{j<d_conv-1} w[c][j] * ring[b][(pos_b+j) mod (d_conv-1)][c]
 *                    + w[c][d_conv-1] * x[b][c] )
 * then x[b][c] is stored into slot pos_b mod (d_conv-1) and conv_pos[b] += 1.
 * x rows are ld_x elements apart (so x can be a view into a wider row); out
 * is [B][C].  bias may be NULL (no bias).  act = SiLU if silu != 0. */
int conv1d_update(uint16_t* conv_state, int32_t* conv_pos, const uint16_t* x, int32_t ld_x,
                  const uint16_t* w, const uint16_t* bias, uint16_t* out, int32_t B, int32_t C,
                  int32_t d_conv, int32_t silu, cudaStream_t stream);

/* One Mamba-2 SSM decode step for B sequences (source listing, `ssm_decode`;
 * dt clamp [1e-9, 1e9] as passed there):
 *   dt = clamp(softplus(dt_raw[b][h] + dt_bias[h]), 1e-9, 1e9);  dA = exp(-dt*exp(A_log[h]))
 *   h[b][h][p][n] = dA*h + dt * x[b][h*P+p] * Bm[b][g*N+n],   g = h / (H/G)
 *   y[b][h*P+p]   = sum_n Cm[b][g*N+n] * h[b][h][p][n] + D[h] * x[b][h*P+p]
 * x, Bm, Cm, dt_raw are bf16 with rows ld_in elements apart (views into one
 * [B][ld_in] buffer are fine); h fp32 [B][H][P][N] in place; y fp32 [B][H*P]. */
int mamba2_ssm_step(float* h, const uint16_t* x, const uint16_t* Bm, const uint16_t* Cm,
                    const uint16_t* dt_raw, int32_t ld_in, const float* A_log, const float* D,
                    const float* dt_bias, float* y, int32_t B, int32_t H, int32_t P, int32_t N,
                    int32_t G, cudaStream_t stream);

/* Decode without any caller-provided or library-allocated workspace.  The
 * pages have no counterpart: this entry point exists for callers that cannot
 * allocate device memory on demand -- for example a plug-in running inside a
 * host application that reserved all device memory for its own pool up
 * front, or a latency-critical serving loop that must not call into the
 * allocator (cudaMalloc may synchronise the device and can fail once memory
 * is committed).  It behaves exactly like mamba2_layer_decode (same
 * arguments apart from the workspace, same kernels, same results), but its
 * scratch lives in one fixed array inside the library, M2_NOALLOC_SCRATCH_BYTES
 * (8 MiB) per device, which every GPU that loads the library holds until the
 * process exits.  It allocates nothing itself.
 *  - Requests whose decode workspace (m2_workspace_bytes(dims, B, 0)) exceeds
 *    M2_NOALLOC_SCRATCH_BYTES return M2_ERR_SCRATCH and launch nothing (for
 *    the hidden-4096 / 8192-inner layer that is B > 88).
 *  - The first call on a device looks up the array's device address for that
 *    device (cudaGetSymbolAddress, with that device current); make that first
 *    call before any stream capture on the device.
 *  - All calls share the one array and it keeps the previous call's
 *    contents; nothing in it needs to start at zero (the per-sequence state
 *    lives in the caller's buffers).  Calls whose work overlaps on the GPU --
 *    concurrent streams, or several host threads -- race on the array: order
 *    them on one stream or synchronise between them. */
#define M2_NOALLOC_SCRATCH_BYTES (8u << 20)
int mamba2_layer_decode_noalloc(const m2_dims* dims, const m2_layer* layer, uint16_t* hidden, int32_t B,
                                float* ssm_state, uint16_t* conv_state, int32_t* conv_pos, cudaStream_t stream);

/* Stream-ordered copy of `bytes` between device memory and/or page-locked host
 * memory (cudaHostAlloc / cudaHostRegister), done by a kernel launched as a
 * programmatic dependent of the previous kernel on `stream`.  A decode loop
 * that stages its hidden rows through host buffers then stays one chain of
 * kernels: a cudaMemcpyAsync between two launches keeps the next layer kernel
 * from starting its weight stream before the copy and the kernel before it
 * have finished.  dst and src 16-byte aligned, bytes a multiple of 16
 * (M2_ERR_ALIGN otherwise); pageable host memory, an unknown pointer, or a
 * range [p, p + bytes) that does not lie inside one allocation of dst or of
 * src: M2_ERR_ARG, nothing launched.  Both pointers are checked on the host
 * (cudaPointerGetAttributes, and the allocation's address range) before the
 * launch. */
int m2_copy(void* dst, const void* src, size_t bytes, cudaStream_t stream);

/* ------------------------------------------------------------ diagnostics */

/* Where a call keeps its intermediate values in the workspace, for reading
 * them back (tests, debugging).  kind: M2_WS_KIND_DECODE (n = batch rows,
 * cu_seqlens unused), M2_WS_KIND_PREFILL or M2_WS_KIND_PREFILL_W8A8 (n =
 * sequences, cu_seqlens their host offsets as for the varlen prefill; the
 * one-sequence prefill is n = 1, {0, T}).  offsets[n_offsets >= M2_WS_COUNT]
 * receives byte offsets from ws, SIZE_MAX for a region the call does not use:
 *   M2_WS_XN  input RMSNorm output [rows][hidden] (tensor-core paths)
 *   M2_WS_ZX  in_proj output [rows][rup8(n_in)] bf16: z | xBC | dt (decode:
 *             the xBC part holds the conv output; the raw xBC is in the ring)
 *   M2_WS_U   prefill conv output [T][d_xbc] bf16
 *   M2_WS_Y   SSM output y [rows][d_inner] fp32
 *   M2_WS_G   gated-norm output [rows][d_inner], when a separate kernel
 *             writes it (tensor-core projections): bf16 for an out_proj with
 *             bf16 weights; for E4M3 weights f16, row r prescaled by an exact
 *             power of two 2^j whose inverse is M2_WS_UNSCALE's entry rows + r
 *   M2_WS_UNSCALE  fp32 [2][rows]: the inverse prescale of each row of the
 *             in_proj input (first half) and of the out_proj input (second)
 *   M2_WS_Q8  W8A8: E4M3 codes [T][rup16(max(hidden, d_inner))] of the last
 *             projection's input; M2_WS_SQ: its fp32 block scales
 *             [d_inner/128][rup128(T)].
 * Contents are valid after the call completes and until the next call on the
 * same workspace.  Host only; returns M2_OK or M2_ERR_ARG. */
enum { M2_WS_KIND_DECODE = 0, M2_WS_KIND_PREFILL = 1, M2_WS_KIND_PREFILL_W8A8 = 2 };
enum { M2_WS_XN = 0, M2_WS_ZX, M2_WS_U, M2_WS_Y, M2_WS_G, M2_WS_Q8, M2_WS_SQ, M2_WS_UNSCALE, M2_WS_COUNT };
int m2_workspace_map(const m2_dims* dims, int32_t kind, int32_t n, const int32_t* cu_seqlens, size_t* offsets,
                     int32_t n_offsets);

/* Device status word: M2_OK, or the first M2_ERR_TIMEOUT a kernel recorded on
 * the current device.  Synchronises the device.  clear != 0 resets it. */
int m2_device_status(int clear);

/* Limit of the library's in-kernel pipeline waits on the current device, in
 * SM clock cycles (cycles <= 0 restores the default, 4e9: about 2 s at the
 * maximum clock).  A pipeline wait that reaches the limit gives up: the kernel
 * records M2_ERR_TIMEOUT (see m2_device_status), stops its own loop, waits for
 * the copies and tensor-core work it already issued (that wait always uses the
 * default limit), frees its tensor memory and returns; the outputs of that
 * call are undefined.  A limit shorter than a correct call needs therefore
 * turns every call into a timeout: it is meant for detecting a stalled
 * pipeline sooner and for testing the timeout path, not for tuning.  Affects
 * launches made after the call; returns M2_OK or M2_ERR_DEVICE. */
int m2_set_wait_limit(int64_t cycles);

/* Check of the timeout path on the current device: enqueues one small kernel
 * that holds tensor memory and has a bulk copy of the 16 bytes at `probe` into
 * shared memory in flight while it waits, with the pipeline wait limit, on a
 * barrier that nothing signals.  The wait gives up (the status word then holds
 * M2_ERR_TIMEOUT), the kernel waits for its own copy, writes the 16 bytes to
 * `out`, frees its tensor memory and returns, leaving the device usable.  probe
 * and out are 16-byte aligned device pointers (M2_ERR_ALIGN / M2_ERR_ARG
 * otherwise, nothing launched).  Lower the limit first (m2_set_wait_limit):
 * with the default the kernel runs for about two seconds.  Returns the launch
 * status, not the timeout (read that with m2_device_status). */
int m2_wait_check(const void* probe, void* out, cudaStream_t stream);

/* Number of kernels this library has launched in this process (all devices). */
int64_t m2_launch_count(void);

/* Per-kernel timing: m2_trace_begin(capacity) makes every later launch record
 * a CUDA event pair around itself on its stream (up to `capacity` launches);
 * m2_trace_end synchronises, writes per kernel id the summed milliseconds and
 * the launch count into ms[n_ids] / launches[n_ids], and stops tracing.
 * Events are host-side objects (cudaEventCreate); no device memory is used.
 * Tracing serialises kernels that could otherwise overlap. */
int m2_trace_begin(int32_t capacity);
int m2_trace_end(double* ms, int32_t* launches, int32_t n_ids);
/* Name of kernel id `id` (0 <= id < m2_kernel_count()), or NULL. */
const char* m2_kernel_name(int32_t id);
int32_t m2_kernel_count(void);

#ifdef __cplusplus
}
#endif
#endif /* MAMBA2_GB300_H */
