// Per-Layer-Embedding gather fused with its f32 projection and per-chunk
// RMSNorm ("visible-cx/gemma-4-E2B-CoreAI", The PLE gather-table sidecar:
// int8 table [V][L*ld] + per-row f32 scale, dequant x16.0, proj.f32
// [L*ld][D], proj_norm.f32 [ld]; "Gemma-4 E2B mobile mixed-bit QAT weights",
// P2 DONE: 35 layer-major blocks of 256 on axis 1).
//
// One CTA per (layer chunk c, group of kTG tokens); thread j owns output
// column c*ld + j.  The projection rows of chunk c stream through shared
// memory in [ld][kKT] tiles; the hidden rows of the token group are
// broadcast from shared memory.  The chunk's RMSNorm needs only the CTA's
// own columns, and the gathered table term is added in the same epilogue.
#include "q4w_device.cuh"
#include "q4w_internal.cuh"

namespace q4w {

constexpr int kLd = 256;   // ld: one thread per column of a chunk
constexpr int kTG = 16;    // tokens per CTA
constexpr int kKT = 32;    // projection columns per shared tile

__global__ void __launch_bounds__(kLd) ple_kernel(const int32_t* __restrict__ ids, int S,
                                                 const int8_t* __restrict__ table,
                                                 const float* __restrict__ row_scale, int V, int L,
                                                 float embed_scale, const float* __restrict__ proj,
                                                 const __half* __restrict__ hidden, int D,
                                                 const float* __restrict__ norm_w, float eps,
                                                 float* __restrict__ out,
                                                 int8_t* __restrict__ gathered,
                                                 int32_t* __restrict__ err) {
  __shared__ float ps[kLd][kKT + 1];
  __shared__ __align__(16) float hs[kKT][kTG];
  __shared__ float red[kLd / 32][kTG];
  const int c = blockIdx.x;           // layer chunk
  const int t0 = blockIdx.y * kTG;    // first token of the group
  const int j = threadIdx.x;
  const int PLD = L * kLd;
  const int ntok = S - t0 < kTG ? S - t0 : kTG;

  float acc[kTG];
#pragma unroll
  for (int t = 0; t < kTG; ++t) acc[t] = 0.f;

  const float* prow = proj + (size_t)c * kLd * D;
  for (int k0 = 0; k0 < D; k0 += kKT) {
    // projection tile [kLd][kKT], coalesced along the row
#pragma unroll 4
    for (int e = j; e < kLd * kKT; e += kLd) {
      const int r = e / kKT, cc = e % kKT;
      ps[r][cc] = prow[(size_t)r * D + k0 + cc];
    }
    for (int e = j; e < kKT * kTG; e += kLd) {
      const int t = e / kKT, cc = e % kKT;
      hs[cc][t] = t < ntok ? __half2float(hidden[(size_t)(t0 + t) * D + k0 + cc]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kKT; ++kk) {
      const float pv = ps[j][kk];
      const float4* h4 = reinterpret_cast<const float4*>(hs[kk]);
#pragma unroll
      for (int q = 0; q < kTG / 4; ++q) {
        const float4 hv = h4[q];
        acc[4 * q + 0] = fmaf(pv, hv.x, acc[4 * q + 0]);
        acc[4 * q + 1] = fmaf(pv, hv.y, acc[4 * q + 1]);
        acc[4 * q + 2] = fmaf(pv, hv.z, acc[4 * q + 2]);
        acc[4 * q + 3] = fmaf(pv, hv.w, acc[4 * q + 3]);
      }
    }
    __syncthreads();
  }

  // per-token sum of squares over the chunk's kLd columns
  const int w = j >> 5, l = j & 31;
#pragma unroll
  for (int t = 0; t < kTG; ++t) {
    const float v = warp_sum(acc[t] * acc[t]);
    if (l == 0) red[w][t] = v;
  }
  __syncthreads();
  const float nw = norm_w[j];
#pragma unroll
  for (int t = 0; t < kTG; ++t) {
    if (t >= ntok) break;
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kLd / 32; ++i) ss += red[i][t];
    const float r = 1.f / sqrtf(ss / (float)kLd + eps);
    const int tok = t0 + t;
    const int id = ids[tok];
    const size_t o = (size_t)tok * PLD + (size_t)c * kLd + j;
    if (id < 0 || id >= V) {
      out[o] = 0.f;
      if (gathered) gathered[o] = 0;
      if (err && j == 0) atomicExch(err, 1);
      continue;
    }
    const int8_t q = table[(size_t)id * PLD + (size_t)c * kLd + j];
    const float g = __fmul_rn(__fmul_rn((float)q, row_scale[id]), embed_scale);
    out[o] = acc[t] * r * nw + g;
    if (gathered) gathered[o] = q;
  }
}

int launch_ple(const int32_t* ids, int S, const int8_t* table, const float* row_scale, int V, int L,
               int ld, float embed_scale, const float* proj, const __half* hidden, int D,
               const float* norm_w, float eps, float* out, int8_t* gathered, int32_t* err,
               const DeviceInfo& dev, cudaStream_t s) {
  (void)dev;
  if (ld != kLd) return fail(Q4_ERR_SHAPE, "ple_gather_project: ld must be %d", kLd);
  dim3 grid(L, (S + kTG - 1) / kTG);
  ple_kernel<<<grid, kLd, 0, s>>>(ids, S, table, row_scale, V, L, embed_scale, proj, hidden, D, norm_w,
                                  eps, out, gathered, err);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? Q4_OK : cuda_fail(e, "ple launch");
}

}  // namespace q4w
