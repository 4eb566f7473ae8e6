// INT2 per-row symmetric GEMV: y[n] = scale[n] * sum_k (code[n][k] - 2) x[k]
// ("Gemma-4 E2B mobile mixed-bit QAT weights - extraction + Core AI
// transplant": The decode recipe (Section 10) -- FFN of L15-L34 and the tied
// head are INT2, per-channel symmetric, 4 codes per byte with the first in
// bits[1:0]; P6 DONE -- unsigned code minus midpoint; P3 DONE -- the per-row
// scale multiplies the row sum once).
//
// Decode: two codes per LOP3, without shifts for the low bytes of a 16-bit
// half.  Bits [2j, 2j+2) of bytes 0 and 2 of a code word land in the
// mantissa of fp16 1024, 256, 64 or 16 (j = 0..3), where the fp16 spacing
// makes each pattern read exactly as M_j + code; the word shifted by 8 does
// bytes 1 and 3 the same way.  Each half pair is multiplied into two fp32
// accumulators by the mixed-precision FMA against the matching x half pair;
// the per-chunk bias -sum (M_j + 2) x removes the offsets.
//
// Layout: a lane group of P lanes serves one row, each lane 16-byte chunks
// (64 columns) c = lane, lane + P, ...; x is staged in shared memory as the
// half pairs of every chunk (plus its bias), read by the row groups of a warp
// together.  Two rows per group are in flight.
#include "q4w_device.cuh"
#include "q4w_internal.cuh"

namespace q4w {

namespace q2 {

constexpr int kThr = 256;
constexpr int kChunkWords = 36;   // 32 half pairs + bias + pad: 144 B, lanes of a group hit other banks

__device__ __forceinline__ uint32_t magic_pair(int j) {
  return j == 0 ? 0x64006400u : j == 1 ? 0x5C005C00u : j == 2 ? 0x54005400u : 0x4C004C00u;
}
__device__ __forceinline__ float magic_offset(int j) {   // M_j + 2
  return j == 0 ? 1026.f : j == 1 ? 258.f : j == 2 ? 66.f : 18.f;
}

// sum over one 64-column chunk of (code - 2) x, given the chunk's x half pairs
// (word i, pair 4h + j) = (x[16i + 4h + j], x[16i + 8 + 4h + j]) and its bias
__device__ __forceinline__ float chunk_dot(const uint4 c, const uint32_t* xp) {
  const uint32_t w4[4] = {c.x, c.y, c.z, c.w};
  float lo = __uint_as_float(xp[32]), hi = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w = w4[i], w8 = shr_u32(w, 8);
    uint32_t xq[8];
    const uint4 a = *reinterpret_cast<const uint4*>(xp + 8 * i);
    const uint4 b = *reinterpret_cast<const uint4*>(xp + 8 * i + 4);
    xq[0] = a.x; xq[1] = a.y; xq[2] = a.z; xq[3] = a.w;
    xq[4] = b.x; xq[5] = b.y; xq[6] = b.z; xq[7] = b.w;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t mask = 0x00030003u << (2 * j);
      fhfma2(lo, hi, lop3_and_or(w, mask, magic_pair(j)), xq[j]);
      fhfma2(lo, hi, lop3_and_or(w8, mask, magic_pair(j)), xq[4 + j]);
    }
  }
  return lo + hi;
}

__global__ void __launch_bounds__(kThr) q2_gemv_kernel(const uint8_t* __restrict__ codes,
                                                      const float* __restrict__ scales,
                                                      const __half* __restrict__ x, float* __restrict__ y, int N,
                                                      int K, int lgP) {
  extern __shared__ __align__(16) uint32_t q2_smem[];
  const int nc = K >> 6;
  // x half pairs per chunk: word i (16 columns), pair 4h + j.  A thread takes
  // 8 consecutive halves x[16i + 8u .. 16i + 8u + 7] of one word half u: the
  // low halves of pairs 4h + j (u = 0) or the high halves (u = 1).
  for (int e = threadIdx.x; e < nc * 8; e += kThr) {
    const int ch = e >> 3, i = (e >> 1) & 3, u = e & 1;
    const uint4 v = *reinterpret_cast<const uint4*>(x + 64 * ch + 16 * i + 8 * u);
    const uint32_t hv[4] = {v.x, v.y, v.z, v.w};
    uint16_t* dst = reinterpret_cast<uint16_t*>(q2_smem + ch * kChunkWords + 8 * i) + u;
#pragma unroll
    for (int q = 0; q < 4; ++q) {   // column 8u + c of the word -> half u of pair c
      dst[2 * (2 * q)] = (uint16_t)(hv[q] & 0xFFFFu);
      dst[2 * (2 * q + 1)] = (uint16_t)(hv[q] >> 16);
    }
  }
  __syncthreads();
  // per-chunk bias from the staged pairs: -sum over pairs of (M_j + 2)(lo + hi)
  for (int ch = threadIdx.x; ch < nc; ch += kThr) {
    const uint32_t* xp = q2_smem + ch * kChunkWords;
    float s = 0.f;
#pragma unroll
    for (int p = 0; p < 32; ++p) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(xp + p));
      s -= magic_offset(p & 3) * (f.x + f.y);
    }
    q2_smem[ch * kChunkWords + 32] = __float_as_uint(s);
  }
  __syncthreads();

  const int P = 1 << lgP;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int li = lane & (P - 1), gid = threadIdx.x >> lgP, ngroups = kThr >> lgP;
  const int wg0 = (warp * 32) >> lgP;                 // the warp's first group
  const int G = gridDim.x * ngroups;                  // row groups in the grid
  const size_t rowb = (size_t)(K >> 2);
  // each pass: rows r0 = base + (gid - wg0) and r1 = r0 + G, base uniform per warp
  for (int base = blockIdx.x * ngroups + wg0; base < N; base += 2 * G) {
    const int r0 = base + (gid - wg0);
    const int r1 = r0 + G;
    const bool v0 = r0 < N, v1 = r1 < N;
    const uint8_t* c0 = codes + (size_t)(v0 ? r0 : N - 1) * rowb;
    const uint8_t* c1 = codes + (size_t)(v1 ? r1 : N - 1) * rowb;
    float a0 = 0.f, a1 = 0.f;
    for (int ch = li; ch < nc; ch += P) {
      const uint4 w0 = ld_stream16(c0 + 16 * ch);
      const uint4 w1 = ld_stream16(c1 + 16 * ch);
      const uint32_t* xp = q2_smem + ch * kChunkWords;
      a0 += chunk_dot(w0, xp);
      a1 += chunk_dot(w1, xp);
    }
    for (int o = P >> 1; o > 0; o >>= 1) {
      a0 += __shfl_xor_sync(0xffffffffu, a0, o);
      a1 += __shfl_xor_sync(0xffffffffu, a1, o);
    }
    if (li == 0) {
      if (v0) y[r0] = scales[r0] * a0;
      if (v1) y[r1] = scales[r1] * a1;
    }
  }
}

}  // namespace q2

// K % 64 == 0; lanes per row: the largest power of two up to 32 dividing the chunk count.
int launch_q2_gemv(const uint8_t* codes, const float* scales, const __half* x, float* y, int N, int K,
                   const DeviceInfo& dev, cudaStream_t s) {
  const int nc = K >> 6;
  int lgP = 5;
  while (lgP > 0 && nc % (1 << lgP)) --lgP;
  const size_t smem = (size_t)nc * q2::kChunkWords * 4;
  static PerDevice attr;
  cudaError_t e;
  if (!attr.get(dev.ordinal)) {
    e = cudaFuncSetAttribute(q2::q2_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    if (e != cudaSuccess) return cuda_fail(e, "q2 smem attribute");
    attr.set(dev.ordinal);
  }
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, q2::q2_gemv_kernel, q2::kThr, smem);
  if (e != cudaSuccess) return cuda_fail(e, "q2 occupancy");
  if (per_sm < 1) per_sm = 1;
  const int ngroups = q2::kThr >> lgP;
  const int need = (N + 2 * ngroups - 1) / (2 * ngroups);
  int grid = dev.sms * per_sm;
  if (grid > need) grid = need;
  q2::q2_gemv_kernel<<<grid, q2::kThr, smem, s>>>(codes, scales, x, y, N, K, lgP);
  e = cudaGetLastError();
  return e == cudaSuccess ? Q4_OK : cuda_fail(e, "q2 gemv launch");
}

}  // namespace q4w

extern "C" int q2_gemv(const uint8_t* codes, const float* scales, const uint16_t* x_f16, float* y, int N, int K,
                       q4_stream_t stream) {
  using namespace q4w;
  clear_error();
  if (!codes || !scales || !x_f16 || !y) return fail(Q4_ERR_NULL, "codes, scales, x_f16 and y must be non-NULL");
  const void* ptrs[4] = {codes, scales, x_f16, y};
  for (int i = 0; i < 4; ++i)
    if (!aligned16(ptrs[i])) return fail(Q4_ERR_ALIGN, "argument %d is not 16-byte aligned", i);
  if (N < 1) return fail(Q4_ERR_SHAPE, "N=%d must be >= 1", N);
  if (K < 64 || K % 64 || K > 32768) return fail(Q4_ERR_SHAPE, "K=%d must be a multiple of 64 in [64, 32768]", K);
  DeviceInfo dev;
  const int st = current_device(&dev);
  if (st != Q4_OK) return st;
  return launch_q2_gemv(codes, scales, reinterpret_cast<const __half*>(x_f16), y, N, K, dev,
                        reinterpret_cast<cudaStream_t>(stream));
}
