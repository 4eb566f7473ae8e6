// Internal declarations shared by the translation units of libq4w.so.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/q4w.h"

namespace q4w {

// ---------------------------------------------------------------- errors ---
// Records a thread-local message and returns the status (host side).
int fail(int status, const char* fmt, ...);
int cuda_fail(cudaError_t e, const char* what);
void clear_error();

// Device facts cached per device (queried once).
struct DeviceInfo {
  int ordinal;   // the CUDA device number
  int sms;
  int cc_major, cc_minor;
  size_t smem_optin;
};
// Returns Q4_OK and fills *info for the current device, or an error status.
int current_device(DeviceInfo* info);

// "Already done" flags of a one-time set-up step, one per device (a kernel's
// shared-memory attribute is a per-device setting).  Devices past the table
// redo the step on every call.  Two host threads may both find a flag clear
// and both do the step; that is harmless, as the step sets the same value.
struct PerDevice {
  bool done[64];
  bool get(int d) const { return d >= 0 && d < 64 && done[d]; }
  void set(int d) {
    if (d >= 0 && d < 64) done[d] = true;
  }
};

// Cycle budget of every bounded device-side wait (q4_set_wait_limit; the
// Q4W_WAIT_LIMIT_CYCLES environment variable sets the initial value).
long long wait_limit();
// Device address of the library's error word on the current device.
unsigned* device_error_word();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------- launch plumbing ---
// One matrix of a fused GEMV stage and where its rows go.
struct StageMat {
  const uint8_t* codes;
  const __half* scales;
  int rows;
  float* out32;
  __half* out16;
  int tagged;        // outputs carry the stage tag (persistent pass): out16 -> uint32
                     // (half | tag << 16), out32 -> uint64 (float | tag << 32)
};

struct StageArgs {
  StageMat mat[3];
  int nmat;
  int pair;          // 1: mat[0]=gate, mat[1]=up -> m16 = f16(gelu(g) * u) into mat[0].out16
  int K;
  const void* in;
  int in_mode;       // q4_stage_in
  float eps;
  int in_tag;        // > 0: `in` is tagged (as out16/out32 above); wait until every tag equals it
  int out_tag;       // tag written with tagged outputs
  int weights_early; // 1: the weights are not written by the preceding kernel, so with programmatic
                     // dependent launch they may be fetched before that kernel has finished
};

// Launches one fused stage (prologue + GEMV + epilogue).  `pdl` adds the
// programmatic-dependent-launch attribute.  Returns a q4_status.
int launch_stage(const StageArgs& a, const DeviceInfo& dev, cudaStream_t s, bool pdl);
int launch_gemv_batched(const uint8_t* codes, const __half* scales, const __half* x, float* y,
                        int N, int K, int batch, const DeviceInfo& dev, cudaStream_t s);
int launch_rmsnorm_f16(const float* in, int H, float eps, __half* out, cudaStream_t s, bool pdl);
int launch_quantize(const float* W, int N, int K, uint8_t* codes, __half* scales, int32_t* err,
                    const DeviceInfo& dev, cudaStream_t s);
// tensor_cores: batch rows 2..8 may use the tensor-core kernel (fp16 weight
// tiles; its workspace holds z [b][V]); false keeps every batch on the CUDA
// cores with the small workspace.
int launch_lmhead(const uint8_t* codes, const __half* scales, const __half* h, int b, int V, int K,
                  float cap, int32_t* idx, float* top1, float* top2, float* logits, void* ws,
                  const DeviceInfo& dev, cudaStream_t s, bool tensor_cores = true);
size_t lmhead_ws_bytes(int V, int K, int b, const DeviceInfo& dev, bool tensor_cores = true);
int launch_ple(const int32_t* ids, int S, const int8_t* table, const float* row_scale, int V, int L,
               int ld, float embed_scale, const float* proj, const __half* hidden, int D,
               const float* norm_w, float eps, float* out, int8_t* gathered, int32_t* err,
               const DeviceInfo& dev, cudaStream_t s);
// The same with the projection in int8 per-block-32 form (codes [L*ld][D], fp16
// scales [L*ld][D/32]); D % 128 == 0, D <= 2048.
int launch_ple_q8(const int32_t* ids, int S, const int8_t* table, const float* row_scale, int V, int L, int ld,
                  float embed_scale, const int8_t* proj_codes, const uint16_t* proj_scales, const __half* hidden,
                  int D, const float* norm_w, float eps, float* out, int8_t* gathered, int32_t* err,
                  const DeviceInfo& dev, cudaStream_t s);
int launch_quantize_q8(const float* W, int N, int K, int8_t* codes, __half* scales, int32_t* err,
                       const DeviceInfo& dev, cudaStream_t s);
// Streaming engine (bulk-copy ring; K % 256 == 0 and K <= 12288).
bool stream_eligible(int K);
int launch_stage_stream(const StageArgs& a, const DeviceInfo& dev, cudaStream_t s, bool pdl);
int launch_head_stream(const uint8_t* codes, const __half* scales, const __half* h, int V, int K, float cap,
                       int32_t* idx, float* top1, float* top2, float* logits, void* ws, const DeviceInfo& dev,
                       cudaStream_t s);
size_t decode_ctl_bytes();
// Diagnostic stamp buffer set by q4_set_trace (device memory), or nullptr.
void* trace_buffer(size_t* bytes);
int launch_decode_pass_stream(const q4_layer* layers, int n_layers, int H, const __half* h0, __half* h_out,
                              float eps, float* kv32, void* tagged, size_t tagged_bytes, int* ctl,
                              const DeviceInfo& dev, cudaStream_t s);
size_t head_batch_smem(int b, int K);
int launch_gemv_batch_decoded(const uint8_t* codes, const __half* scales, const __half* x, float* y, int N, int K,
                              int batch, const DeviceInfo& dev, cudaStream_t s);
// Tensor map of a 2-D row-major [rows][cols] array (esize-byte elements) with
// boxes of box_rows x box_cols; Q4_OK or an error status naming `what`.
int encode_tensor_2d(CUtensorMap* tm, const void* base, CUtensorMapDataType type, int esize, uint64_t cols,
                     uint64_t rows, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle,
                     const char* what);
size_t gemm_ws_bytes(int K);   // the bf16 copy of X [64][K]
// act_scale > 0: the w4a8 form -- the token operand is the activation codes
// q = clamp(rint(x / act_scale), -128, 127) and Y is scaled by act_scale.
int launch_gemm_chunk(const uint8_t* codes, const __half* scales, const __half* X, float* Y, int M,
                      int N, int K, void* ws, const DeviceInfo& dev, cudaStream_t s, float act_scale = 0.f);
// w4a8 (k_a8.cu): the single-vector q4_0 GEMV on the activation codes, y =
// act_scale * (W q); and the min-max calibration s = max |x| / 127 (1 when
// every x is zero) over n fp16 values into *s_out (device).
int launch_gemv_a8(const uint8_t* codes, const __half* scales, const __half* x, float act_scale, float* y, int N,
                   int K, const DeviceInfo& dev, cudaStream_t s);
int launch_a8_calibrate(const __half* x, long long n, float* s_out, cudaStream_t s);
// The LM head of ntok <= 8 vectors on the tensor cores: z[t][n] through the
// GEMM kernel with fp16 tiles (weights rounded once to fp16, tokens exact),
// one CTA per 128-row tile (no split of K, so every row is summed in one fixed
// order), the token operand resident in shared memory; z never reaches
// memory: the epilogue softcaps it into head.logits (when set) and keeps a
// running top two per token, and the CTA that finishes last merges the per-CTA
// records into idx/top1/top2.  N % 128 == 0, K % 64 == 0, head_mma_fits(K);
// ws: mma16_ws_bytes(K) bytes for the token operand; head.partials: one
// record per SM and kMaxBatch tokens; head.ticket zero.
bool head_mma_fits(int K);
struct Top2;
struct HeadOutputs {
  float cap;
  float* logits;
  Top2* partials;
  unsigned* ticket;
  int32_t* idx;
  float* top1;
  float* top2;
};
size_t mma16_ws_bytes(int K);
int launch_head_mma(const uint8_t* codes, const __half* scales, const __half* X, int ntok, int N, int K, void* ws,
                    const HeadOutputs& head, const DeviceInfo& dev, cudaStream_t s);

}  // namespace q4w
