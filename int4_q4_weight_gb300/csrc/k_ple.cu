// Per-Layer-Embedding gather fused with its f32 projection and per-chunk
// RMSNorm ("visible-cx/gemma-4-E2B-CoreAI", The PLE gather-table sidecar:
// int8 table [V][L*ld] + per-row f32 scale, dequant x16.0, proj.f32
// [L*ld][D], proj_norm.f32 [ld]; "Gemma-4 E2B mobile mixed-bit QAT weights",
// P2 DONE: 35 layer-major blocks of 256 on axis 1).
//
// One CTA per (layer chunk c of 256 projection rows, group of 16 tokens):
// the chunk's RMSNorm needs only the CTA's own rows, and the gathered table
// term is added in the same epilogue.  The projection is register-tiled:
// thread (rg, tg) holds 4 rows (rg, rg+64, rg+128, rg+192) x 4 tokens
// (4 tg .. 4 tg + 3) of fp32 accumulators, so every shared-memory read feeds
// four FMAs.  Projection tiles [256 rows][32 columns] (rows padded to 36
// floats: 8 consecutive rows read a 16-byte group from 8 different bank
// groups) and hidden tiles [16 tokens][32 fp16] stream through a 3-stage
// cp.async ring.
#include "q4w_device.cuh"
#include "q4w_internal.cuh"

namespace q4w {

constexpr int kLd = 256;                 // ld: rows of one layer chunk
constexpr int kTG = 16;                  // tokens per CTA
constexpr int kKT = 32;                  // projection columns per tile
constexpr int kPS = kKT + 4;             // padded row stride of a projection tile (floats)
constexpr int kPleStages = 3;
constexpr int kPleThreads = 256;
constexpr int kProjTileFloats = kLd * kPS;
constexpr int kHidTileHalves = kTG * kKT;
constexpr size_t kPleStageBytes = (size_t)kProjTileFloats * 4 + (size_t)kHidTileHalves * 2;
constexpr size_t kPleSmem = kPleStages * kPleStageBytes;

__device__ __forceinline__ void ple_cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}

__global__ void __launch_bounds__(kPleThreads) ple_kernel(const int32_t* __restrict__ ids, int S,
                                                         const int8_t* __restrict__ table,
                                                         const float* __restrict__ row_scale, int V, int L,
                                                         float embed_scale, const float* __restrict__ proj,
                                                         const __half* __restrict__ hidden, int D,
                                                         const float* __restrict__ norm_w, float eps,
                                                         float* __restrict__ out, int8_t* __restrict__ gathered,
                                                         int32_t* __restrict__ err) {
  extern __shared__ __align__(16) uint8_t ple_smem[];
  __shared__ float red[kPleThreads / 32][4];
  const int c = blockIdx.x;            // layer chunk
  const int t0 = blockIdx.y * kTG;     // first token of the group
  const int tid = threadIdx.x;
  const int rg = tid & 63, tg = tid >> 6;
  const int PLD = L * kLd;
  const int ntok = S - t0 < kTG ? S - t0 : kTG;
  const float* prow = proj + (size_t)c * kLd * D;
  const int nkt = D / kKT;

  auto stage_proj = [&](int st) { return reinterpret_cast<float*>(ple_smem + (size_t)st * kPleStageBytes); };
  auto stage_hid = [&](int st) {
    return reinterpret_cast<__half*>(ple_smem + (size_t)st * kPleStageBytes + (size_t)kProjTileFloats * 4);
  };
  // tile kt of the projection (256 rows x 32 columns, 8 x 16 B per row) and of
  // the hidden rows (16 tokens x 32 fp16, 4 x 16 B per token; tokens past S
  // read token t0's row)
  auto issue = [&](int kt) {
    if (kt < nkt) {
      float* ps = stage_proj(kt % kPleStages);
      __half* hs = stage_hid(kt % kPleStages);
      const int k0 = kt * kKT;
      for (int e = tid; e < kLd * 8; e += kPleThreads) {
        const int r = e >> 3, q = e & 7;
        ple_cp16(ps + r * kPS + 4 * q, prow + (size_t)r * D + k0 + 4 * q);
      }
      if (tid < kTG * 4) {
        const int t = tid >> 2, q = tid & 3;
        const int tok = t < ntok ? t0 + t : t0;
        ple_cp16(hs + t * kKT + 8 * q, hidden + (size_t)tok * D + k0 + 8 * q);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int t = 0; t < 4; ++t) acc[i][t] = 0.f;

  issue(0);
  issue(1);
  for (int kt = 0; kt < nkt; ++kt) {
    issue(kt + 2);
    asm volatile("cp.async.wait_group 2;" ::: "memory");   // tile kt (this thread's copies) landed
    __syncthreads();                                        // ... and everyone else's
    const float* ps = stage_proj(kt % kPleStages);
    const __half* hs = stage_hid(kt % kPleStages);
#pragma unroll
    for (int k = 0; k < kKT; k += 4) {
      float4 pv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pv[i] = *reinterpret_cast<const float4*>(ps + (rg + 64 * i) * kPS + k);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int tt = 4 * tg + t;
        const uint2 hh = *reinterpret_cast<const uint2*>(hs + tt * kKT + k);
        const float2 h01 = __half22float2(*reinterpret_cast<const __half2*>(&hh.x));
        const float2 h23 = __half22float2(*reinterpret_cast<const __half2*>(&hh.y));
        // tokens past S read token t0's row; their sums are never used
        const float x0 = h01.x, x1 = h01.y, x2 = h23.x, x3 = h23.y;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float a = acc[i][t];
          a = fmaf(pv[i].x, x0, a);
          a = fmaf(pv[i].y, x1, a);
          a = fmaf(pv[i].z, x2, a);
          a = fmaf(pv[i].w, x3, a);
          acc[i][t] = a;
        }
      }
    }
    __syncthreads();   // the stage is reused by the copies issued next iteration
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");

  // per-token sum of squares over the chunk's 256 rows: 4 rows here, the 32
  // row groups of this warp, then the two warps of this token group
  const int w = tid >> 5, l = tid & 31;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) ss += acc[i][t] * acc[i][t];
    ss = warp_sum(ss);
    if (l == 0) red[w][t] = ss;
  }
  __syncthreads();
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int tt = 4 * tg + t;
    if (tt >= ntok) break;
    const float ss = red[2 * tg][t] + red[2 * tg + 1][t];
    const float r = 1.f / sqrtf(ss / (float)kLd + eps);
    const int tok = t0 + tt;
    const int id = ids[tok];
    const bool bad = id < 0 || id >= V;
    if (bad && err && rg == 0) atomicExch(err, 1);
    const float sc = bad ? 0.f : row_scale[id];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = rg + 64 * i;
      const size_t o = (size_t)tok * PLD + (size_t)c * kLd + row;
      if (bad) {
        out[o] = 0.f;
        if (gathered) gathered[o] = 0;
        continue;
      }
      const int8_t q = table[(size_t)id * PLD + (size_t)c * kLd + row];
      const float g = __fmul_rn(__fmul_rn((float)q, sc), embed_scale);
      out[o] = acc[i][t] * r * norm_w[row] + g;
      if (gathered) gathered[o] = q;
    }
  }
}

int launch_ple(const int32_t* ids, int S, const int8_t* table, const float* row_scale, int V, int L,
               int ld, float embed_scale, const float* proj, const __half* hidden, int D,
               const float* norm_w, float eps, float* out, int8_t* gathered, int32_t* err,
               const DeviceInfo& dev, cudaStream_t s) {
  (void)dev;
  if (ld != kLd) return fail(Q4_ERR_SHAPE, "ple_gather_project: ld must be %d", kLd);
  static bool attr = false;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(ple_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPleSmem);
    if (e != cudaSuccess) return cuda_fail(e, "ple smem attribute");
    attr = true;
  }
  dim3 grid(L, (S + kTG - 1) / kTG);
  ple_kernel<<<grid, kPleThreads, kPleSmem, s>>>(ids, S, table, row_scale, V, L, embed_scale, proj, hidden, D,
                                                  norm_w, eps, out, gathered, err);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? Q4_OK : cuda_fail(e, "ple launch");
}

}  // namespace q4w
