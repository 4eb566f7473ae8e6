/*
 * q4w.h -- C ABI of the q4_0 weight-only int4 decode kernels (GB300, sm_103a).
 *
 * One shared library, libq4w.so.  Plain pointers and sizes only; no C++ types
 * or exceptions cross this boundary.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.  Every array argument is DEVICE memory owned by the caller, unless
 *   the argument's comment says "host".  The library allocates nothing and
 *   frees nothing in any call; scratch space comes from the caller through a
 *   (workspace pointer, size) pair sized by q4_workspace_bytes().
 * Streams.  `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   Work is enqueued asynchronously; nothing is synchronised.  Results are
 *   ready when the stream reaches that point.
 * Device.  Calls run on the current CUDA device, which must be compute
 *   capability 10.3 (GB300); anything else returns Q4_ERR_ARCH.
 * Errors.  Each call returns a q4_status.  Argument checks happen before any
 *   launch, so a non-zero status from a check means nothing was enqueued.
 *   q4_last_error() returns a thread-local message naming the offending
 *   argument; q4_status_string() names the code.
 * Alignment.  Every device pointer must be 16-byte aligned (Q4_ERR_ALIGN).
 *
 * q4_0 weight layout ("the ggml q4_0 grid", per-block-32 symmetric int4; see
 * "visible-cx/gemma-4-E2B-CoreAI", Provenance, and "Gemma 4 E2B (text
 * decoder) - Core AI", QAT weights), planar, row-major, for a matrix of N
 * rows and K columns (K a multiple of 32):
 *   codes  uint8  [N][K/2]   byte j of a row holds column 2j in its low nibble
 *                            and column 2j+1 in its high nibble (low nibble
 *                            first, "Gemma-4 E2B mobile mixed-bit QAT weights",
 *                            the decode recipe);
 *   scales uint16 [N][K/32]  IEEE fp16 bit patterns, one per 32-column block.
 *   The weight value is scale * (code - 8): unsigned code minus midpoint
 *   ("Gemma-4 E2B mobile mixed-bit QAT weights", P6 DONE; the affine form
 *   scale*code - 8*scale of its receiving-end design).
 * Activations named *_f16 are uint16 arrays of IEEE fp16 bit patterns.
 */
#ifndef Q4W_H_
#define Q4W_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* q4_stream_t; /* same handle as cudaStream_t */

typedef enum q4_status {
  Q4_OK = 0,
  Q4_ERR_NULL = 1,        /* a required pointer is NULL */
  Q4_ERR_SHAPE = 2,       /* a size is out of range or inconsistent */
  Q4_ERR_ALIGN = 3,       /* a device pointer is not 16-byte aligned */
  Q4_ERR_WORKSPACE = 4,   /* workspace NULL or smaller than required */
  Q4_ERR_ARCH = 5,        /* the current device is not compute capability 10.3 */
  Q4_ERR_CUDA = 6,        /* a CUDA runtime call failed (message has the CUDA error) */
  Q4_ERR_TIMEOUT = 7,     /* a bounded device-side wait ran out */
  Q4_ERR_DEVICE = 8       /* a device-side check failed (see the entry point) */
} q4_status;

/* Operation ids for q4_workspace_bytes(). */
typedef enum q4_op {
  Q4_OP_GEMV = 0,
  Q4_OP_GEMM_CHUNK = 1,
  Q4_OP_PLE = 2,
  Q4_OP_LMHEAD = 3,
  Q4_OP_DECODE_PASS = 4
} q4_op;

/* ---------------------------------------------------------------------- */
/* Quantise (setup, not part of a decode step).                            */
/* ---------------------------------------------------------------------- */
/* q4_quantize: fp32 W [N][K] -> q4_0 codes [N][K/2] + fp16 scales [N][K/32].
 * Per 32-column block: m = the element of largest |w| (the first one in
 * column order on ties); d = m / -8 in fp32 (exact); code = clamp(round(w/d)
 * + 8, 0, 15) with an IEEE fp32 quotient and rounding half away from zero;
 * the stored scale is d rounded to fp16 (nearest-even).  An all-zero block
 * stores scale +0 and codes 8.  Source: "visible-cx/gemma-4-E2B-CoreAI",
 * Provenance (int4 per-block-32, q4_0 grid; rounding happens at export);
 * "Gemma 4 E2B (text decoder) - Core AI", QAT weights (per-block-32 absmax
 * symmetric int4; --lin-sym is the literal grid).
 *   N >= 1, K >= 32, K % 32 == 0.
 *   err: optional device int32; set to 1 if a block had a non-finite weight
 *   or a scale beyond the fp16 range (those blocks are stored as zero).  The
 *   word is only ever set, never cleared, by the kernel.              */
int q4_quantize(const float* W, int N, int K, uint8_t* codes, uint16_t* scales,
                int32_t* err, q4_stream_t stream);

/* q8_quantize: fp32 W [N][K] -> int8 per-block-32 codes [N][K] + fp16 scales
 * [N][K/32], the form of the PLE projection ("Gemma-4 E2B mobile mixed-bit
 * QAT weights", decode recipe: PLE gate/proj and the per-layer model
 * projection are INT8; official-checkpoint notes: genuinely signed int8, the
 * projection re-quantised to int8 per block of 32).  Per 32-column block:
 * a = max |w|; d = a / 127 in fp32; code = clamp(round(w/d), -127, 127) with
 * an IEEE fp32 quotient and rounding half away from zero; the stored scale
 * is d rounded to fp16 (nearest-even).  The weight value is scale * code
 * (two's-complement code, no midpoint).  A block whose d is zero stores
 * scale +0 and codes 0.
 *   N >= 1, K >= 32, K % 32 == 0.
 *   err: optional device int32; set to 1 if a block had a non-finite weight
 *   or a scale beyond the fp16 range (those blocks are stored as zero).    */
int q8_quantize(const float* W, int N, int K, int8_t* codes, uint16_t* scales,
                int32_t* err, q4_stream_t stream);

/* ---------------------------------------------------------------------- */
/* S=1 decode GEMV ("main", one token per call).                           */
/* ---------------------------------------------------------------------- */
/* q4_gemv: y[b][n] = sum_k scale[n][k/32] * (code[n][k] - 8) * x[b][k],
 * fp32 accumulation, for b < batch.  Source: "visible-cx/gemma-4-E2B-CoreAI",
 * Provenance (main = S=1 decode); "Gemma-4 E2B mobile mixed-bit QAT weights",
 * the S=4 verify ("weights read once for 4 rows") for batch > 1.
 *   codes/scales: q4_0 matrix [N][K]; x_f16: [batch][K]; y: f32 [batch][N].
 *   1 <= batch <= 8; N >= 1; K % 32 == 0, 32 <= K <= 32768.
 *   Deterministic: the same inputs give the same bits on every call.
 *   ws/ws_bytes: unused (may be NULL/0).                                    */
int q4_gemv(const uint8_t* codes, const uint16_t* scales, const uint16_t* x_f16,
            float* y, int N, int K, int batch, void* ws, size_t ws_bytes,
            q4_stream_t stream);

/* q4_gemv_weights_ro: q4_gemv with the caller's promise that the weights are
 * read-only for the call: no kernel issued earlier on the stream that may
 * still be running writes codes or scales (model weights written once at
 * load time, say).  The kernel then starts streaming its weight tiles
 * before the preceding kernel on the stream has finished (programmatic
 * dependent launch); it reads x, and writes y, only after that kernel's
 * results are visible, as q4_gemv does.  Same arguments, results and bits
 * as q4_gemv.  If the promise is broken the kernel may compute with weights
 * from before the earlier kernel's writes.  batch > 1 behaves as q4_gemv. */
int q4_gemv_weights_ro(const uint8_t* codes, const uint16_t* scales, const uint16_t* x_f16,
                       float* y, int N, int K, int batch, void* ws, size_t ws_bytes,
                       q4_stream_t stream);

/* q2_gemv: INT2 per-row symmetric GEMV (the mixed-bit recipe's FFN of
 * L15-L34 and tied head):  y[n] = scale[n] * sum_k (code[n][k] - 2) x[k],
 * fp32 accumulation, the row scale applied once after the row sum.
 * Source: "Gemma-4 E2B mobile mixed-bit QAT weights - extraction + Core AI
 * transplant", The decode recipe (Section 10: INT2, 4 codes per byte, first
 * code in bits[1:0], per-channel symmetric), P6 DONE (unsigned code minus the
 * midpoint 2), P3 DONE (scale after the reduction).
 *   codes: device [N][K/4] bytes; scales: device f32 [N]; x_f16: device [K];
 *   y: device f32 [N].  All 16-byte aligned.  N >= 1; K % 64 == 0,
 *   64 <= K <= 32768.  No workspace.  Asynchronous on `stream`.
 *   Errors: Q4_ERR_NULL / Q4_ERR_ALIGN / Q4_ERR_SHAPE before any launch.  */
int q2_gemv(const uint8_t* codes, const float* scales, const uint16_t* x_f16, float* y, int N, int K,
            q4_stream_t stream);

/* ---------------------------------------------------------------------- */
/* S=64 chunked-prefill GEMM ("prefill", static query width 64).           */
/* ---------------------------------------------------------------------- */
/* q4_gemm_chunk: Y[t][n] = sum_k bf16(scale*(code-8))[n][k] * bf16(x[t][k]),
 * fp32 accumulation on the tensor cores.  Both tiles are rounded to bf16
 * (nearest-even) before the products.  Source: "visible-cx/gemma-4-E2B-
 * CoreAI", Provenance and Performance (prefill serves full-width 64-token
 * chunks only; the remainder goes through main).
 *   X_f16: [M][K] with M == 64; Y: f32 [M][N]; codes/scales [N][K].
 *   N % 128 == 0, K % 64 == 0, 64 <= K <= 32768.
 *   ws: q4_workspace_bytes(Q4_OP_GEMM_CHUNK, N, K, 64) bytes (64 * K * 2,
 *   rounded up to 256), 16-byte aligned; it receives X rounded to bf16
 *   (by a conversion kernel launched on `stream` before the GEMM) and must
 *   not be shared by overlapping calls.  NULL or smaller: Q4_ERR_WORKSPACE. */
int q4_gemm_chunk(const uint8_t* codes, const uint16_t* scales, const uint16_t* X_f16,
                  float* Y, int M, int N, int K, void* ws, size_t ws_bytes,
                  q4_stream_t stream);

/* ---------------------------------------------------------------------- */
/* w4a8: int8 quantize/dequantize on the activations of a q4_0 linear.     */
/* ---------------------------------------------------------------------- */
/* The w4a8 bundle ("visible-cx/gemma-4-E2B-CoreAI", About the w4a8 bundle)
 * keeps the int4 per-block-32 weights and puts an int8 quantize/dequantize
 * pair, calibrated on 128 samples, on the input of every linear layer.
 * Readings (the pages name the pair, not its grid): per-tensor symmetric,
 * zero point 0, one fp32 scale s per linear input;
 *   q = clamp(rint(x / s), -128, 127)  (IEEE fp32 quotient, ties to even),
 *   x' = s * q,
 * and calibration by min-max: s = max |x| / 127 over the samples (fp32), 1
 * when every sample is zero.  The layer sees x'; since q is exact in fp16 and
 * bf16 the kernels multiply the weights by q and scale each output by s.
 * x must be finite (a NaN or infinity gives an undefined code).           */

/* q4_gemv_a8: y[n] = act_scale * sum_k scale[n][k/32] * (code[n][k] - 8) * q[k],
 * q the codes of x_f16 [K] under act_scale; fp32 accumulation (each block's
 * dot with integer q is exact in fp32).  codes/scales: q4_0 matrix [N][K];
 * y: f32 [N].  N >= 1; K % 32 == 0, 32 <= K <= 32768; act_scale finite and
 * > 0 (else Q4_ERR_SHAPE).  Deterministic.                                 */
int q4_gemv_a8(const uint8_t* codes, const uint16_t* scales, const uint16_t* x_f16,
               float act_scale, float* y, int N, int K, q4_stream_t stream);

/* q4_gemm_chunk_a8: q4_gemm_chunk on the activation codes:
 * Y[t][n] = act_scale * sum_k bf16(scale*(code-8))[n][k] * q[t][k], q the
 * codes of X_f16 under act_scale (exact in bf16).  Shapes, workspace and
 * errors as q4_gemm_chunk; act_scale finite and > 0 (else Q4_ERR_SHAPE).  */
int q4_gemm_chunk_a8(const uint8_t* codes, const uint16_t* scales, const uint16_t* X_f16,
                     float act_scale, float* Y, int M, int N, int K, void* ws,
                     size_t ws_bytes, q4_stream_t stream);

/* q4_act_calibrate_a8: *scale_out (device f32) = max |x| / 127 over the n fp16
 * values of x_f16 (all calibration samples, concatenated), or 1 when every
 * value is zero.  n >= 1.  One CTA reduces the values (a calibration step,
 * not a per-token one).                                                    */
int q4_act_calibrate_a8(const uint16_t* x_f16, long long n, float* scale_out,
                        q4_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Per-Layer-Embedding gather + projection.                                */
/* ---------------------------------------------------------------------- */
/* ple_gather_project: for each of S tokens t with id v = ids[t]:
 *   g[t][j]   = (float(table[v][j]) * row_scale[v]) * embed_scale   (fp32)
 *   p[t][j]   = sum_d proj[j][d] * float(hidden[t][d])             (fp32)
 *   n[t][c*ld+i] = p[t][c*ld+i] * rsqrt(mean_i p[t][c*ld+i]^2 + eps) * norm_w[i]
 *   out[t][j] = n[t][j] + g[t][j]                                  (f32)
 * for j < L*ld, chunks c < L.  Source: "visible-cx/gemma-4-E2B-CoreAI", The
 * PLE gather-table sidecar (int8 table [V][8960] + per-row f32 scale, x16.0,
 * proj.f32 [8960][1536], proj_norm.f32 [256]); "Gemma-4 E2B mobile mixed-bit
 * QAT weights", P2 DONE (35 layer-major blocks of 256 concatenated on axis 1).
 *   ids: int32 [S]; table: int8 [V][L*ld]; row_scale: f32 [V];
 *   proj: f32 [L*ld][D]; hidden_f16: [S][D]; norm_w: f32 [ld];
 *   out: f32 [S][L*ld]; gathered_opt: int8 [S][L*ld] copy of the table rows,
 *   or NULL.  1 <= S <= 4096; ld == 256; 1 <= L <= 256; D % 32 == 0,
 *   32 <= D <= 32768; V >= 1.  An id outside [0, V) writes zeros for that
 *   token and sets the optional device int32 *err to 1 (never cleared by
 *   the kernel).
 *   Arithmetic of p: each projection weight w is multiplied as two fp16
 *   pieces, p1 = fp16(w) and p2 = fp16((w - p1) * 2^11), both rounded to
 *   nearest even, so p1 + p2 * 2^-11 keeps 22 significant bits of w
 *   (relative error <= 2^-22 for |w| >= 2^-14, absolute <= 2^-36 below);
 *   the fp16 hidden is exact; products are exact and summed in fp32.
 *   Projection weights must be finite with |w| < 65520 (fp16 range); larger
 *   ones give an undefined result.                                        */
int ple_gather_project(const int32_t* ids, int S, const int8_t* table,
                       const float* row_scale, int V, int L, int ld, float embed_scale,
                       const float* proj, const uint16_t* hidden_f16, int D,
                       const float* norm_w, float eps, float* out, int8_t* gathered_opt,
                       int32_t* err, q4_stream_t stream);

/* ple_gather_project_q8: ple_gather_project with the projection in int8
 * per-block-32 form (the q8_quantize layout): proj[j][d] =
 * proj_scales[j][d/32] * proj_codes[j][d].  On the tensor cores every
 * projection weight enters as fp16(scale * code), rounded once to nearest
 * even (hidden fp16 is exact), with fp32 accumulation; the rest is the f32
 * form's arithmetic.  Source: "Gemma-4 E2B mobile mixed-bit QAT weights",
 * decode recipe (per_layer_model_projection [8960,1536] INT8) and
 * official-checkpoint notes (re-quantised to int8 per block of 32).
 *   proj_codes: int8 [L*ld][D]; proj_scales: fp16 bits [L*ld][D/32]; every
 *   scale * 127 must be finite in fp16 (|weights| <= 65504).  D % 128 == 0,
 *   128 <= D <= 2048; every other argument, limit and error as
 *   ple_gather_project.                                                    */
int ple_gather_project_q8(const int32_t* ids, int S, const int8_t* table,
                          const float* row_scale, int V, int L, int ld, float embed_scale,
                          const int8_t* proj_codes, const uint16_t* proj_scales,
                          const uint16_t* hidden_f16, int D, const float* norm_w, float eps,
                          float* out, int8_t* gathered_opt, int32_t* err, q4_stream_t stream);

/* ---------------------------------------------------------------------- */
/* LM head + softcap + argmax.                                             */
/* ---------------------------------------------------------------------- */
/* lmhead_softcap_argmax: for each batch row b:
 *   z[n] = sum_k scale[n][k/32]*(code[n][k]-8)*h[b][k]   (fp32)
 *   s[n] = tanh(z[n] / cap) * cap
 *   idx[b] = argmax_n s[n] (lowest index among equal z), top1[b] = s[idx],
 *   top2[b] = the largest s over the other rows.
 * The logits are not read back unless logits_opt is given.  Source: "Gemma 4
 * E2B (text decoder) - Core AI", Signature features (final logit softcap
 * tanh(z/30)*30) and What it took (fused head with a two-level in-kernel
 * argmax, no logit readback).
 *   h_f16: [b][K]; idx int32 [b]; top1, top2 f32 [b];
 *   logits_opt: f32 [b][V] softcapped logits, or NULL.
 *   1 <= b <= 8; V >= 2; K % 32 == 0, 32 <= K <= 32768; cap > 0.
 *   ws: q4_workspace_bytes(Q4_OP_LMHEAD, V, K, b) bytes; its contents on
 *   entry do not matter.  Calls that share one ws must not overlap.
 * Arithmetic: b = 1 sums exact products (fp32 accumulation).  For b >= 2
 * with V % 128 == 0, V >= 128 x (SM count), K % 64 == 0 and K <= 1984, z is
 * computed on the tensor cores with each weight rounded once to fp16,
 * fp16(d*(q-8)), and fp32 accumulation, and selected in the same kernel (z
 * is not written unless logits_opt is given; the workspace then also holds
 * the fp16 copy of h, 32 K bytes); other shapes sum exact products on the
 * CUDA cores, where every batch row's h is staged in shared memory: K <=
 * 25024 for b = 2..4 and K <= 12864 for b = 5..8 (larger: Q4_ERR_SHAPE).  Either way each row's sum has a fixed order: repeated calls
 * give the same bits.                                                       */
int lmhead_softcap_argmax(const uint8_t* codes, const uint16_t* scales,
                          const uint16_t* h_f16, int b, int V, int K, float cap,
                          int32_t* idx, float* top1, float* top2, float* logits_opt,
                          void* ws, size_t ws_bytes, q4_stream_t stream);

/* lmhead_softcap_argmax_noalloc: the same operation as lmhead_softcap_argmax
 * for callers that cannot allocate device memory (engines that fix every
 * device allocation at start-up, or C hosts that only own the buffers they
 * pass in; cudaMalloc would also synchronise the device inside a token loop).
 * The pages have no counterpart: this is a library convenience.  Its scratch
 * is a file-scope device array of 64 KiB that every GPU loading the library
 * holds until the process exits.  Every batch size (1..8) runs on the CUDA
 * cores with exact products, whose scratch is a 256-byte ticket block plus
 * one 16-byte top-two record per batch slot (8) for each of 2 x SMs CTAs:
 * 256 + 256 x SMs bytes (39,168 on a 152-SM GB300), independent of V, K and
 * b.  A device with more than 255 SMs gets Q4_ERR_WORKSPACE.  (The figure
 * q4_workspace_bytes(Q4_OP_LMHEAD, ...) reports is the workspace entry
 * point's need, which for b >= 2 on a large vocabulary includes the
 * tensor-core path's token operand; it is not this limit.)  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current, and caches it per device without a lock: host threads
 * whose first calls on one device coincide all store the same address.  Make
 * that first call before any stream capture.  All calls share the one array,
 * which keeps the last call's contents (the ticket word is cleared on the
 * stream before each kernel): calls whose kernels overlap on the GPU (other
 * streams, other host threads) race and must be serialised by the caller.
 * Arguments and results as in lmhead_softcap_argmax, without ws / ws_bytes;
 * nothing is allocated. */
int lmhead_softcap_argmax_noalloc(const uint8_t* codes, const uint16_t* scales,
                                  const uint16_t* h_f16, int b, int V, int K, float cap,
                                  int32_t* idx, float* top1, float* top2, float* logits_opt,
                                  q4_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Decode weight pass over a stack of layers (S=1).                        */
/* ---------------------------------------------------------------------- */
typedef struct q4_matrix {
  const uint8_t* codes;    /* device, [rows][cols/2] */
  const uint16_t* scales;  /* device, [rows][cols/32] */
} q4_matrix;

typedef struct q4_layer {
  int q_rows;      /* rows of W_q = cols of W_o (e.g. 2048 or 4096) */
  int kv_rows;     /* rows of W_k and W_v; 0 when the layer shares K/V */
  int mlp_rows;    /* rows of W_gate and W_up = cols of W_down */
  q4_matrix q, k, v, o, gate, up, down;   /* k, v ignored when kv_rows == 0 */
} q4_layer;

/* q4_decode_pass: the weight pass of one decode step over n_layers layers,
 * hidden size H.  Per layer, with RMSNorm(v) = v * rsqrt(mean(v^2) + eps):
 *   a = f16(RMSNorm(h));  q = W_q a;  k = W_k a;  v = W_v a;
 *   o = W_o f16(q);       b = f16(RMSNorm(o));
 *   g = W_gate b;  u = W_up b;  m = f16(gelu_tanh(g) * u);
 *   h' = f16(RMSNorm(W_down m))
 * with fp32 accumulation and fp32 gelu_tanh(x) = 0.5x(1+tanh(sqrt(2/pi)(x +
 * 0.044715x^3))).  k and v are computed (into the workspace) and not used.
 * Sources: "Gemma 4 E2B (text decoder) - Core AI", Signature features (35
 * layers, dual head_dim, KV-sharing, double-wide MLP, RMSNorm weight applied
 * directly); "Gemma-4 E2B mobile mixed-bit QAT weights", the decode recipe
 * and P2 progress (shapes) and Speed (fused gate/up with an fp32 tanh GELU).
 * The exact stage order is this library's synthetic weight-pass workload.
 *   layers: HOST array of n_layers descriptors (read during the call only);
 *   h0_f16, h_out_f16: device [H]; 1 <= n_layers <= 256; H % 32 == 0;
 *   q_rows, mlp_rows % 32 == 0 and in [32, 32768]; kv_rows >= 0.
 *   ws: q4_workspace_bytes(Q4_OP_DECODE_PASS, H, max(q_rows + 2 kv_rows),
 *   max(mlp_rows)) bytes; overlapping calls must not share it.
 *   When H <= 4096, n_layers <= 48 and H, every q_rows and every mlp_rows
 *   are multiples of 256 up to 12288, the whole pass is one persistent
 *   cooperative launch (one CTA per SM) preceded by two memsets on `stream`:
 *   each stage output word carries the index of the stage that wrote it,
 *   and the next stage polls its input (bounded; Q4_ERR_TIMEOUT via
 *   q4_device_status) until every word carries that index.  Otherwise
 *   every stage is one kernel launch (programmatic dependent launch between
 *   stages).  Either form can be captured into a CUDA graph.              */
int q4_decode_pass(const q4_layer* layers, int n_layers, int H, const uint16_t* h0_f16,
                   uint16_t* h_out_f16, float eps, void* ws, size_t ws_bytes,
                   q4_stream_t stream);

/* q4_decode_pass_launches: how many kernels one q4_decode_pass call with
 * these arguments launches: 1 (the persistent form) or 4 * n_layers + 1
 * (one per stage, then the closing RMSNorm).  Memsets are not counted.
 * Returns a negative Q4_ERR_* when layers is NULL or n_layers is out of
 * range; shapes are otherwise checked by q4_decode_pass itself. */
int q4_decode_pass_launches(const q4_layer* layers, int n_layers, int H);

/* Prologue of one decode-pass stage, exposed for stage tests. */
typedef enum q4_stage_in {
  Q4_IN_F16 = 0,          /* x = in (fp16) */
  Q4_IN_RMS_F16 = 1,      /* x = f16(RMSNorm(in fp16)) */
  Q4_IN_RMS_F32 = 2,      /* x = f16(RMSNorm(in f32)) */
  Q4_IN_RMS2_F32 = 3      /* x = f16(RMSNorm(f16(RMSNorm(in f32)))) */
} q4_stage_in;

/* q4_gemv_stage: one stage of q4_decode_pass as a standalone call, with the
 * same kernel and launch shape the pass uses.  Up to three q4 matrices with
 * the same K are applied to one input vector:
 *   x = prologue(in) per `in_mode`;  y_i = W_i x  (fp32).
 * pair == 0: matrix i writes out32[i] (f32 [rows_i], may be NULL) and
 *            out16[i] (fp16 [rows_i], may be NULL).
 * pair == 1: exactly two matrices (gate, up) with rows_0 == rows_1; writes
 *            m = f16(gelu_tanh(y_0) * y_1) to out16[0], and y_0 / y_1 to
 *            out32[0] / out32[1] when those are non-NULL.
 *   in: device [K] fp16 (Q4_IN_F16, Q4_IN_RMS_F16) or f32 (the others).
 *   1 <= nmat <= 3; rows_i >= 1; K % 32 == 0, 32 <= K <= 32768.
 *   Source: as q4_decode_pass.                                             */
int q4_gemv_stage(const q4_matrix* mats /* host [nmat] */, const int* rows /* host [nmat] */,
                  int nmat, int K, const void* in, int in_mode, float eps, int pair,
                  float* const* out32 /* host [nmat] */, uint16_t* const* out16 /* host [nmat] */,
                  q4_stream_t stream);

/* q4_rmsnorm_f16: out = f16(RMSNorm(in f32 [H])), the last step of the pass.
 * Source: "Gemma 4 E2B (text decoder) - Core AI", Signature features. */
int q4_rmsnorm_f16(const float* in, int H, float eps, uint16_t* out_f16, q4_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Helpers.                                                                */
/* ---------------------------------------------------------------------- */
/* Bytes of workspace an operation needs (0 = none).  Arguments per op:
 *   Q4_OP_GEMV (N, K, batch), Q4_OP_GEMM_CHUNK (N, K, 64), Q4_OP_PLE (S, D, L),
 *   Q4_OP_LMHEAD (V, K, b), Q4_OP_DECODE_PASS (H, max q+2kv rows, max mlp).
 * Depends on the current device's SM count for Q4_OP_LMHEAD; returns 0 when
 * the current device cannot be queried.                                   */
size_t q4_workspace_bytes(int op, int a, int b, int c);

const char* q4_status_string(int status);
const char* q4_last_error(void);   /* thread-local; "" when no error yet */

/* q4_device_status: waits for `stream` to finish, then reads and clears the
 * library's device error word.  Returns Q4_ERR_TIMEOUT if a bounded
 * device-side wait of a kernel (an mbarrier or inter-CTA wait) ran out since
 * the last check; such a kernel returned early and its outputs are invalid. */
int q4_device_status(q4_stream_t stream);

/* q4_set_wait_limit: clock-cycle budget of every bounded device-side wait in
 * kernels launched after the call (default 4e9, about 2 s; the environment
 * variable Q4W_WAIT_LIMIT_CYCLES sets the initial value).  Returns the
 * previous budget.  A budget of 0 makes any wait that is not already
 * satisfied give up at once (used to test the timeout path). */
long long q4_set_wait_limit(long long cycles);

/* q4_set_trace: diagnostic.  While `buf` (device memory) is set, every
 * persistent q4_decode_pass launch writes, per stage s and CTA c, eight
 * stamps to buf[(s * grid + c) * 8 + i] (grid = the SM count): i=0 the
 * globaltimer (ns) when the CTA entered the stage; the others SM clock
 * cycles since then: 1 input complete and staged, 2 x built, 3 x in
 * registers, 5 first weight tile landed (shifted left by one; bit 0 set when
 * it had landed before the consumers asked), 6 first tile usable by the
 * whole warp, 4 this CTA's rows written; 7 unused.  Needs
 * 4 * n_layers * grid * 8 * 8 bytes.
 * The other tensor-core kernels use the same buffer when it is large enough
 * for their layout (else they write nothing):
 *   ple_gather_project / _q8: CTA 0 writes row r < 256 of 8 words (SM
 *   cycles since its start) per stage r: 0 tile loads issued, 1 tiles seen
 *   by the converter warps, 2 operand converted (words 1-2: even stages
 *   only in the int8 form, whose two converter groups alternate), 3 MMAs
 *   started, 4 MMAs committed; the epilogue: row 255 word 5 accumulator
 *   ready, row 254 word 0 the cluster barrier passed, word 1 the partial
 *   sums sent or received, word 2 the sums of squares received, row 255
 *   word 6 RMS factors, word 7 and row 254 word 3 output written, row 254
 *   word 4 exit; then every CTA writes its start and end globaltimer (ns) as two
 *   words at 2048 + 2 * (blockIdx.y * gridDim.x + blockIdx.x).  Needs
 *   (2048 + 2 * 4 * L * ceil(S / 64)) * 8 bytes.
 *   q4_gemm_chunk and the batched LM head: CTA 0 writes 8 words (SM cycles)
 *   per 128-column chunk g < 256 of its work: 0 weight tile load issued,
 *   1 landed, 2 operand slot free, 3 operand converted, 4 MMAs started,
 *   5 committed, 6 accumulator ready, 7 written out (6 and 7 on an item's
 *   first chunk).  Needs 256 * 8 * 8 bytes.
 * NULL turns it off. */
int q4_set_trace(void* buf, size_t bytes);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int q4_version(void);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* Q4W_H_ */
