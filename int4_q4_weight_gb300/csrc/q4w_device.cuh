// Device-side building blocks shared by the q4_0 GEMV-shaped kernels.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace q4w {

constexpr int kThreads = 256;          // threads per CTA of the GEMV-shaped kernels
constexpr int kWarps = kThreads / 32;
constexpr int kXStride = 36;           // floats per 32-column block of x in shared memory:
                                       // 32 values, the block bias, 3 pad (144 B keeps
                                       // 8 lanes reading 8 blocks free of bank conflicts)

// ------------------------------------------------------------ PDL hooks ---
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }

// --------------------------------------------------------------- loads ---
// 16-byte streaming load of weight codes: read once, keep out of L1.
__device__ __forceinline__ uint4 ld_stream16(const uint8_t* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ float ld_scale(const __half* p) {
  unsigned short u;
  asm("ld.global.nc.u16 %0, [%1];" : "=h"(u) : "l"(p));
  return __half2float(__ushort_as_half(u));
}

// ------------------------------------------------------ packed fp32 x2 ---
typedef unsigned long long f2_t;   // two fp32 lanes in one 64-bit register pair

__device__ __forceinline__ f2_t f2_pack(float lo, float hi) {
  f2_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(f2_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2_t f2_fma(f2_t a, f2_t b, f2_t c) {
  f2_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// ------------------------------------------------- nibble -> float trick ---
// A 4-bit code n placed in mantissa bits [15,19) of the fp32 pattern of 256.0
// reads as exactly 256 + n; placed in bits [19,23) of 16.0 it reads as 16 + n.
// One LOP3 per code, no integer-to-float conversion.  The constant parts
// (256 or 16, plus the -8 midpoint) are removed through a per-block bias
//   bias = -264 * sum(x at even columns) - 24 * sum(x at odd columns),
// so that bias + sum_k F_k x_k = sum_k (code_k - 8) x_k.
__device__ __forceinline__ float nib_even(uint32_t s) {  // bits [15,19) -> 256 + n
  return __uint_as_float((s & 0x00078000u) | 0x43800000u);
}
__device__ __forceinline__ float nib_odd(uint32_t s) {   // bits [19,23) -> 16 + n
  return __uint_as_float((s & 0x00780000u) | 0x41800000u);
}

__device__ __forceinline__ f2_t f2_add(f2_t a, f2_t b) {
  f2_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// sum_k (code_k - 8) * x_k over one 32-column block.
// c: the block's 16 code bytes (column 2j in the low nibble of byte j).
// xv: x of the block as 8 float4 (columns 4t..4t+3 in xv[t]).
// Four independent accumulators (one per 32-bit word of codes, eight FMAs
// deep) are summed pairwise at the end.
__device__ __forceinline__ float q4_block_dot(const uint4 c, const float4 (&xv)[8], float bias) {
  const uint32_t w4[4] = {c.x, c.y, c.z, c.w};
  float a[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w = w4[i];          // columns 8i .. 8i+7, nibble j = column 8i+j
    const uint32_t s0 = w << 15, s1 = w << 7, s2 = w >> 1, s3 = w >> 9;
    float t = i == 0 ? bias : 0.f;
    t = fmaf(nib_even(s0), xv[2 * i].x, t);
    t = fmaf(nib_odd(s0), xv[2 * i].y, t);
    t = fmaf(nib_even(s1), xv[2 * i].z, t);
    t = fmaf(nib_odd(s1), xv[2 * i].w, t);
    t = fmaf(nib_even(s2), xv[2 * i + 1].x, t);
    t = fmaf(nib_odd(s2), xv[2 * i + 1].y, t);
    t = fmaf(nib_even(s3), xv[2 * i + 1].z, t);
    t = fmaf(nib_odd(s3), xv[2 * i + 1].w, t);
    a[i] = t;
  }
  return (a[0] + a[1]) + (a[2] + a[3]);
}


// ---------------------------------------------- fp16-magic block dot (fast) ---
// Two codes per LOP3.  In a 32-bit word of codes (columns 8i..8i+7, byte b =
// columns 8i+2b (low nibble) and 8i+2b+1 (high nibble)) the low nibbles of
// bytes 0 and 2 sit in bits [0,4) and [16,20): OR-ed into two fp16 1024.0
// patterns they read as the half pair (1024 + n, 1024 + n') exactly (fp16
// spacing at 1024 is 1); the high nibbles sit in bits [4,8) and [20,24) and
// read as (64 + n, 64 + n') in two fp16 64.0 patterns (spacing 1/16, the
// nibble counted in sixteenths).  The word shifted by 8 gives bytes 1 and 3
// the same way: four LOP3 and one shift per word.  Each half is multiplied by
// the matching fp16 x with the mixed-precision fp32 FMA (fma.rn.f32.f16:
// exact product, one fp32 rounding).  x is held as half pairs
// xh[4i + j] = (x[8i+j], x[8i+j+4]); the bias
//   -1032 * sum(x at even columns) - 72 * sum(x at odd columns)
// removes the 1024 + 8 and 64 + 8 offsets, so bias + sum F_k x_k =
// sum (code_k - 8) x_k.
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t magic) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(magic));
  return d;
}
__device__ __forceinline__ uint32_t shl_u32(uint32_t a, uint32_t n) {
  uint32_t d;
  asm("shl.b32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(n));
  return d;
}
__device__ __forceinline__ uint32_t shr_u32(uint32_t a, uint32_t n) {
  uint32_t d;
  asm("shr.b32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(n));
  return d;
}
__device__ __forceinline__ void fhfma2(float& lo, float& hi, uint32_t a, uint32_t b) {
  asm("{\n .reg .f16 a0, a1, b0, b1;\n mov.b32 {a0, a1}, %2;\n mov.b32 {b0, b1}, %3;\n"
      " fma.rn.f32.f16 %0, a0, b0, %0;\n fma.rn.f32.f16 %1, a1, b1, %1;\n}"
      : "+f"(lo), "+f"(hi)
      : "r"(a), "r"(b));
}

constexpr uint32_t kH64Mask = 0x00F000F0u;
constexpr uint32_t kH64Magic = 0x54005400u;     // fp16 64.0 in both halves
constexpr uint32_t kH1024Mask = 0x000F000Fu;
constexpr uint32_t kH1024Magic = 0x64006400u;   // fp16 1024.0 in both halves
constexpr float kBiasEven = -1032.f, kBiasOdd = -72.f;

// Half pair j (j = 0..3) of a code word, as q4_block_dot_h uses it.
__device__ __forceinline__ void q4_word_pairs(uint32_t w, uint32_t (&p)[4]) {
  const uint32_t w8 = shr_u32(w, 8);
  p[0] = lop3_and_or(w, kH1024Mask, kH1024Magic);    // columns 8i+0, 8i+4
  p[1] = lop3_and_or(w, kH64Mask, kH64Magic);        // columns 8i+1, 8i+5
  p[2] = lop3_and_or(w8, kH1024Mask, kH1024Magic);   // columns 8i+2, 8i+6
  p[3] = lop3_and_or(w8, kH64Mask, kH64Magic);       // columns 8i+3, 8i+7
}

__device__ __forceinline__ float q4_block_dot_h(const uint4 c, const uint32_t (&xh)[16], float bias) {
  const uint32_t w4[4] = {c.x, c.y, c.z, c.w};
  float lo = bias, hi = 0.f;   // even/odd halves accumulate separately (two chains)
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t pr[4];
    q4_word_pairs(w4[i], pr);
#pragma unroll
    for (int j = 0; j < 4; ++j) fhfma2(lo, hi, pr[j], xh[4 * i + j]);
  }
  return lo + hi;
}

__device__ __forceinline__ void load_xblock(const float* xs, int blk, float4 (&xv)[8], float& bias) {
  const float4* p = reinterpret_cast<const float4*>(xs + blk * kXStride);
#pragma unroll
  for (int t = 0; t < 8; ++t) xv[t] = p[t];
  bias = xs[blk * kXStride + 32];
}

// ----------------------------------------------------------- reductions ---
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum over the CTA (kThreads threads); every thread gets the result.
__device__ __forceinline__ float block_sum(float v, float* red /* kWarps floats */) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) t += red[i];
  return t;
}

__device__ __forceinline__ float f16_round(float v) { return __half2float(__float2half_rn(v)); }

// w4a8 activation code ("visible-cx/gemma-4-E2B-CoreAI", About the w4a8
// bundle: an int8 quantize/dequantize pair on every linear input):
// q = clamp(rint(x / s), -128, 127), the quotient an IEEE fp32 division and
// rint rounding half to even; an integer of at most 8 bits, exact in fp16
// and bf16.  x must be finite.
__device__ __forceinline__ float a8_code(float x, float s) {
  return fminf(fmaxf(rintf(__fdiv_rn(x, s)), -128.f), 127.f);
}

// x into the padded shared layout, then the per-block biases.
__device__ __forceinline__ void xs_store(float* xs, int k, float v) {
  xs[(k >> 5) * kXStride + (k & 31)] = v;
}
__device__ __forceinline__ float xs_load(const float* xs, int k) {
  return xs[(k >> 5) * kXStride + (k & 31)];
}
__device__ __forceinline__ void xs_biases(float* xs, int nb) {
  for (int b = threadIdx.x; b < nb; b += blockDim.x) {
    const float* p = xs + b * kXStride;
    float se = 0.f, so = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      se += p[2 * i];
      so += p[2 * i + 1];
    }
    xs[b * kXStride + 32] = -264.f * se - 24.f * so;
  }
}

// gelu with the tanh form, in fp32 with the accurate tanhf.
__device__ __forceinline__ float gelu_tanh_f32(float x) {
  const float c = 0.7978845608028654f;   // sqrt(2/pi)
  return 0.5f * x * (1.f + tanhf(c * (x + 0.044715f * x * x * x)));
}

}  // namespace q4w
