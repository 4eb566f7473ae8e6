// q4_0 quantiser: one warp per 32-column block.
//
// Per block ("visible-cx/gemma-4-E2B-CoreAI", Provenance; "Gemma 4 E2B (text
// decoder) - Core AI", QAT weights): m = the element of largest magnitude
// (first in column order on ties), d = m / -8 in fp32, code = clamp(round(w/d)
// + 8, 0, 15) from the IEEE fp32 quotient with ties away from zero (roundf),
// scale = fp16(d) nearest-even.  An all-zero block stores +0 and codes 8.
#include "q4w_device.cuh"
#include "q4w_internal.cuh"

namespace q4w {

__global__ void __launch_bounds__(kThreads) quantize_kernel(const float* __restrict__ W, long nblocks,
                                                           uint8_t* __restrict__ codes,
                                                           __half* __restrict__ scales,
                                                           int32_t* __restrict__ err) {
  const int lane = threadIdx.x & 31;
  const long warps = (long)gridDim.x * kWarps;
  for (long blk = (long)blockIdx.x * kWarps + (threadIdx.x >> 5); blk < nblocks; blk += warps) {
    const float w = W[blk * 32 + lane];
    // arg-max of |w| with the lowest column on ties
    float best = fabsf(w);
    int bi = lane;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ob > best || (ob == best && oi < bi)) {
        best = ob;
        bi = oi;
      }
    }
    const bool finite = __all_sync(0xffffffffu, isfinite(w));
    const float m = __shfl_sync(0xffffffffu, w, bi);
    float d = m / -8.0f;
    const bool bad = !finite || fabsf(d) > 65504.0f;
    int code = 8;
    if (m == 0.0f || bad) {
      d = 0.0f;
    } else {
      const float q = roundf(__fdiv_rn(w, d)) + 8.0f;
      code = (int)fminf(fmaxf(q, 0.0f), 15.0f);
    }
    const int hi = __shfl_down_sync(0xffffffffu, code, 1);
    if ((lane & 1) == 0) codes[blk * 16 + (lane >> 1)] = (uint8_t)(code | (hi << 4));
    if (lane == 0) {
      scales[blk] = __float2half_rn(d);
      if (bad && err) atomicExch(err, 1);
    }
  }
}

int launch_quantize(const float* W, int N, int K, uint8_t* codes, __half* scales, int32_t* err,
                    const DeviceInfo& dev, cudaStream_t s) {
  const long nblocks = (long)N * (K >> 5);
  long grid = (nblocks + kWarps - 1) / kWarps;
  if (grid > (long)dev.sms * 8) grid = (long)dev.sms * 8;
  quantize_kernel<<<(unsigned)grid, kThreads, 0, s>>>(W, nblocks, codes, scales, err);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? Q4_OK : cuda_fail(e, "quantize launch");
}

// int8 per-block-32 quantiser, one warp per block ("Gemma-4 E2B mobile
// mixed-bit QAT weights", decode recipe and official-checkpoint notes: the
// PLE projection is int8 per block of 32, signed): a = max |w|, d = a / 127
// in fp32, code = clamp(round(w / d), -127, 127) from the IEEE fp32 quotient
// with ties away from zero, scale = fp16(d) nearest-even.  A block whose d is
// zero stores +0 and codes 0.
__global__ void __launch_bounds__(kThreads) quantize_q8_kernel(const float* __restrict__ W, long nblocks,
                                                              int8_t* __restrict__ codes,
                                                              __half* __restrict__ scales,
                                                              int32_t* __restrict__ err) {
  const int lane = threadIdx.x & 31;
  const long warps = (long)gridDim.x * kWarps;
  for (long blk = (long)blockIdx.x * kWarps + (threadIdx.x >> 5); blk < nblocks; blk += warps) {
    const float w = W[blk * 32 + lane];
    float a = fabsf(w);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const bool finite = __all_sync(0xffffffffu, isfinite(w));
    float d = __fdiv_rn(a, 127.0f);
    const bool bad = !finite || d > 65504.0f;
    int code = 0;
    if (d == 0.0f || bad) {
      d = 0.0f;
    } else {
      code = (int)fminf(fmaxf(roundf(__fdiv_rn(w, d)), -127.0f), 127.0f);
    }
    codes[blk * 32 + lane] = (int8_t)code;
    if (lane == 0) {
      scales[blk] = __float2half_rn(d);
      if (bad && err) atomicExch(err, 1);
    }
  }
}

int launch_quantize_q8(const float* W, int N, int K, int8_t* codes, __half* scales, int32_t* err,
                       const DeviceInfo& dev, cudaStream_t s) {
  const long nblocks = (long)N * (K >> 5);
  long grid = (nblocks + kWarps - 1) / kWarps;
  if (grid > (long)dev.sms * 8) grid = (long)dev.sms * 8;
  quantize_q8_kernel<<<(unsigned)grid, kThreads, 0, s>>>(W, nblocks, codes, scales, err);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? Q4_OK : cuda_fail(e, "quantize_q8 launch");
}

}  // namespace q4w
