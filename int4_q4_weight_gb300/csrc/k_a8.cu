// w4a8: an int8 quantize/dequantize pair on a linear layer's input in front
// of the q4_0 weights ("visible-cx/gemma-4-E2B-CoreAI", About the w4a8
// bundle: the same int4 per-block-32 weights and graph, an int8
// quantize/dequantize pair on the input of every linear layer, calibrated on
// 128 samples).
//
// Per-tensor symmetric int8, zero point 0, fp32 scale s: q = clamp(rint(x /
// s), -128, 127) from the IEEE fp32 quotient (half to even), x' = s q.  q is
// an integer of at most 8 bits, exact in fp16, so the GEMV multiplies the
// weights by q and scales each row sum by s once: y = s (W q).  With integer
// activations a block's dot product is exact in fp32 (products of 11 by 8
// bits, partial sums below 2^24), so the roundings left are the block scale
// multiplies, the fp32 sum over blocks and the final multiply by s.
//
// GEMV mapping: 16 lanes per row, 16 rows per CTA (256 threads); lane li
// takes the row's 32-column blocks li, li + 16, ..., four loads in flight at
// a time.  x is quantised while it is staged once per CTA, as q's half pairs
// (q[8i+j], q[8i+j+4]) and block biases in the q4_block_dot_h layout.
//
// Calibration (min-max): one CTA reduces max |x| over the samples, then
// s = max / 127 (IEEE fp32 quotient), or 1 when every sample is zero.
#include "q4w_device.cuh"
#include "q4w_internal.cuh"

namespace q4w {

namespace a8 {

constexpr int kThr = 256;
constexpr int kLPR = 16;                  // lanes per row
constexpr int kRowsPerCta = kThr / kLPR;  // 16
constexpr int kXw = 20;                   // words per staged block: 16 half pairs, the bias, 3 pad
                                          // (80 bytes: 8 lanes on 8 consecutive blocks hit 8 bank groups)
constexpr int kInFlight = 4;              // weight blocks a lane loads before using them
constexpr int kCalThr = 1024;

__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ float ld_cg_half(const __half* p) {
  unsigned short r;
  asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(r) : "l"(p));
  return __half2float(__ushort_as_half(r));
}
__device__ __forceinline__ uint32_t half_pair(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __launch_bounds__(kThr) gemv_a8_kernel(const uint8_t* __restrict__ codes,
                                                       const __half* __restrict__ scales, const __half* x, float s,
                                                       float* __restrict__ y, int N, int K) {
  extern __shared__ __align__(16) uint32_t xs[];   // [K / 32][kXw]
  const int tid = threadIdx.x, lane = tid & 31, li = lane & (kLPR - 1);
  const int row = blockIdx.x * kRowsPerCta + (tid >> 4);
  const int nb = K >> 5;
  // the next kernel may be scheduled now; x is read (and y written) only
  // after the previous kernel's results are visible
  pdl_trigger();
  pdl_wait();

  // chunk ch = columns 8 ch .. 8 ch + 7 (block ch / 4, quarter ch % 4); the
  // four chunks of a block sit on four consecutive lanes of one warp
  const int nch = 4 * nb;
  for (int base = 0; base < nch; base += kThr) {   // uniform: every lane takes part in the shuffles
    const int ch = base + tid;
    const bool v = ch < nch;
    const uint4 u = v ? ld_cg_v4(x + 8 * ch) : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    float q[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      q[2 * i] = a8_code(f.x, s);
      q[2 * i + 1] = a8_code(f.y, s);
    }
    // sums of q at the block's even and odd columns (exact: integers)
    float pe = (q[0] + q[2]) + (q[4] + q[6]), po = (q[1] + q[3]) + (q[5] + q[7]);
    pe += __shfl_xor_sync(0xffffffffu, pe, 1);
    po += __shfl_xor_sync(0xffffffffu, po, 1);
    pe += __shfl_xor_sync(0xffffffffu, pe, 2);
    po += __shfl_xor_sync(0xffffffffu, po, 2);
    if (v) {
      uint32_t* dst = xs + (ch >> 2) * kXw + 4 * (ch & 3);
      *reinterpret_cast<uint4*>(dst) =
          make_uint4(half_pair(q[0], q[4]), half_pair(q[1], q[5]), half_pair(q[2], q[6]), half_pair(q[3], q[7]));
      if ((ch & 3) == 0) xs[(ch >> 2) * kXw + 16] = __float_as_uint(kBiasEven * pe + kBiasOdd * po);
    }
  }
  __syncthreads();

  float acc = 0.f;
  if (row < N) {   // uniform over the row's 16 lanes
    const uint8_t* crow = codes + (size_t)row * (K >> 1);
    const __half* srow = scales + (size_t)row * nb;
    for (int b0 = li; b0 < nb; b0 += kInFlight * kLPR) {
      uint4 cw[kInFlight];
      float d[kInFlight];
#pragma unroll
      for (int j = 0; j < kInFlight; ++j) {
        const int blk = b0 + j * kLPR;
        if (blk < nb) {
          cw[j] = ld_cg_v4(crow + 16 * blk);
          d[j] = ld_cg_half(srow + blk);
        }
      }
#pragma unroll
      for (int j = 0; j < kInFlight; ++j) {
        const int blk = b0 + j * kLPR;
        if (blk < nb) {
          const uint4* p = reinterpret_cast<const uint4*>(xs + blk * kXw);
          uint32_t xr[16];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const uint4 e = p[t];
            xr[4 * t] = e.x;
            xr[4 * t + 1] = e.y;
            xr[4 * t + 2] = e.z;
            xr[4 * t + 3] = e.w;
          }
          acc = fmaf(d[j], q4_block_dot_h(cw[j], xr, __uint_as_float(xs[blk * kXw + 16])), acc);
        }
      }
    }
  }
#pragma unroll
  for (int o = kLPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (li == 0 && row < N) y[row] = acc * s;
}

__global__ void __launch_bounds__(kCalThr) calibrate_kernel(const __half* __restrict__ x, long long n,
                                                            float* __restrict__ s_out) {
  __shared__ float red[kCalThr / 32];
  float m = 0.f;
  const long long n8 = n >> 3;   // whole 16-byte groups, then the tail
  for (long long g = threadIdx.x; g < n8; g += kCalThr) {
    const uint4 u = ld_cg_v4(x + 8 * g);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
  for (long long i = 8 * n8 + threadIdx.x; i < n; i += kCalThr) m = fmaxf(m, fabsf(__half2float(x[i])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float amax = 0.f;
    for (int i = 0; i < kCalThr / 32; ++i) amax = fmaxf(amax, red[i]);
    *s_out = amax > 0.f ? __fdiv_rn(amax, 127.f) : 1.f;
  }
}

}  // namespace a8

int launch_gemv_a8(const uint8_t* codes, const __half* scales, const __half* x, float act_scale, float* y, int N,
                   int K, const DeviceInfo& dev, cudaStream_t s) {
  const size_t smem = (size_t)(K >> 5) * a8::kXw * sizeof(uint32_t);
  static PerDevice attr;
  if (!attr.get(dev.ordinal)) {
    const cudaError_t e =
        cudaFuncSetAttribute(a8::gemv_a8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    if (e != cudaSuccess) return cuda_fail(e, "w4a8 GEMV smem attribute");
    attr.set(dev.ordinal);
  }
  if (smem > 96 * 1024) return fail(Q4_ERR_SHAPE, "w4a8 GEMV: K=%d too large", K);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((N + a8::kRowsPerCta - 1) / a8::kRowsPerCta);
  cfg.blockDim = dim3(a8::kThr);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, a8::gemv_a8_kernel, codes, scales, x, act_scale, y, N, K);
  return e == cudaSuccess ? Q4_OK : cuda_fail(e, "w4a8 GEMV launch");
}

int launch_a8_calibrate(const __half* x, long long n, float* s_out, cudaStream_t s) {
  a8::calibrate_kernel<<<1, a8::kCalThr, 0, s>>>(x, n, s_out);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? Q4_OK : cuda_fail(e, "w4a8 calibration launch");
}

}  // namespace q4w
