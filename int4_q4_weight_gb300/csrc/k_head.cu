// LM head fused with the logit softcap and a two-level argmax.
//
// "Gemma 4 E2B (text decoder) - Core AI": the final logits are softcapped as
// tanh(z/30)*30 (Signature features) and the head is fused with a two-level
// in-kernel argmax so that no logits are read back (What it took).  tanh is
// increasing, so the argmax and the runner-up are selected on z and only the
// two winners are softcapped; the full softcapped logits are written only
// when the caller asks for them.
//
// Level 1: every lane group keeps the top two (z, row) of the rows it
// computes; the CTA merges them into one partial per batch row in the
// workspace.  Level 2: the CTA that takes the last ticket of an atomic
// counter merges all partials (no CTA waits for another).
#include <climits>

#include "q4w_device.cuh"
#include "q4w_internal.cuh"
#include "q4w_top2.cuh"

namespace q4w {

// b == 1: lane groups own R rows each, like the decode GEMV stages.
template <int LPR, int R>
__global__ void __launch_bounds__(kThreads) head_rows_kernel(const uint8_t* __restrict__ codes,
                                                            const __half* __restrict__ scales,
                                                            const __half* __restrict__ h, int V, int K,
                                                            float cap, float* __restrict__ logits,
                                                            Top2* partials, unsigned* ticket,
                                                            int32_t* idx, float* top1, float* top2,
                                                            int tasks) {
  extern __shared__ float4 dyn_smem4[];
  float* xs = reinterpret_cast<float*>(dyn_smem4);
  __shared__ Top2 st[kWarps];
  const int nb = K >> 5;
  for (int k = threadIdx.x; k < K; k += kThreads) xs_store(xs, k, __half2float(h[k]));
  __syncthreads();
  xs_biases(xs, nb);
  __syncthreads();

  constexpr int G = 32 / LPR;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane / LPR, li = lane % LPR;
  const size_t row_bytes = (size_t)(K >> 1);
  Top2 best;
  top2_init(best);

  for (int task = blockIdx.x * kWarps + warp; task < tasks; task += gridDim.x * kWarps) {
    const int rbase = (task * G + g) * R;
    float acc[R];
    bool ok[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      acc[r] = 0.f;
      ok[r] = rbase + r < V;
    }
#pragma unroll 2
    for (int j = li; j < nb; j += LPR) {
      uint4 c[R];
      float d[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (ok[r]) {
          c[r] = ld_stream16(codes + (size_t)(rbase + r) * row_bytes + 16 * j);
          d[r] = ld_scale(scales + (size_t)(rbase + r) * nb + j);
        } else {
          c[r] = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
          d[r] = 0.f;
        }
      }
      float4 xv[8];
      float bias;
      load_xblock(xs, j, xv, bias);
#pragma unroll
      for (int r = 0; r < R; ++r) acc[r] = fmaf(d[r], q4_block_dot(c[r], xv, bias), acc[r]);
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], o);
    if (li == 0) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (!ok[r]) continue;
        top2_insert(best, acc[r], rbase + r);
        if (logits) logits[rbase + r] = cap * tanhf(acc[r] / cap);
      }
    }
  }
  // the CTA's record (non-leaders hold the empty state): shuffle merges
  // within each warp, then across the warps
  {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) top2_shfl_xor_merge(best, o);
    if (lane == 0) st[warp] = best;
    __syncthreads();
    if (warp == 0) {
      Top2 t;
      if (lane < kWarps)
        t = st[lane];
      else
        top2_init(t);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) top2_shfl_xor_merge(t, o);
      if (lane == 0) partials[(size_t)blockIdx.x * kMaxBatch] = t;
    }
  }
  head_finish(partials, ticket, 1, cap, idx, top1, top2);
}

int launch_head_batch(const uint8_t* codes, const __half* scales, const __half* h, int b, int V, int K, float cap,
                      int32_t* idx, float* top1, float* top2, float* logits, Top2* partials, unsigned* ticket,
                      int grid, cudaStream_t s, float* ydirect = nullptr);

static int lpr_for(int nb) {
  int l = 32;
  while (l > 1 && nb % l) l >>= 1;
  return l;
}

static int head_grid(const DeviceInfo& dev) { return 2 * dev.sms; }   // >= the streaming head's grid

// Batch rows 2..8 go through the tensor-core kernel (fp16 weight tiles, one
// CTA per 128-row tile, the selection in its epilogue) when the vocabulary
// fills every SM with tiles.
static bool head_tc_eligible(int b, int V, int K, const DeviceInfo& dev) {
  return b >= 2 && V % 128 == 0 && V >= 128 * dev.sms && K % 64 == 0 && head_mma_fits(K);
}

static size_t up256(size_t n) { return (n + 255) & ~(size_t)255; }

size_t lmhead_ws_bytes(int V, int K, int b, const DeviceInfo& dev, bool tensor_cores) {
  size_t n = kTicketBytes + up256((size_t)head_grid(dev) * kMaxBatch * sizeof(Top2));
  if (tensor_cores && head_tc_eligible(b, V, K, dev)) n += mma16_ws_bytes(K);
  return n;
}

// b = 1 on the CUDA-core kernel (K not eligible for the streaming engine).
template <int LPR>
static cudaError_t launch_head_t(const uint8_t* codes, const __half* scales, const __half* h, int V, int K,
                                 float cap, int32_t* idx, float* top1, float* top2, float* logits, Top2* partials,
                                 unsigned* ticket, const DeviceInfo& dev, cudaStream_t s) {
  const int nb = K >> 5;
  int grid = head_grid(dev);
  constexpr int G = 32 / LPR;
  constexpr int R = 4;
  const int tasks = (V + G * R - 1) / (G * R);
  const int need = (tasks + kWarps - 1) / kWarps;
  if (grid > need) grid = need;
  const size_t smem = (size_t)nb * kXStride * sizeof(float);
  auto k = head_rows_kernel<LPR, R>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  k<<<grid, kThreads, smem, s>>>(codes, scales, h, V, K, cap, logits, partials, ticket, idx, top1, top2, tasks);
  return cudaGetLastError();
}

int launch_lmhead(const uint8_t* codes, const __half* scales, const __half* h, int b, int V, int K,
                  float cap, int32_t* idx, float* top1, float* top2, float* logits, void* ws,
                  const DeviceInfo& dev, cudaStream_t s, bool tensor_cores) {
  if (b == 1 && (size_t)(K >> 5) * kXStride * sizeof(float) > (size_t)200 * 1024)
    return fail(Q4_ERR_SHAPE, "lmhead: K %d does not fit in shared memory", K);
  if (b > 1 && !(tensor_cores && head_tc_eligible(b, V, K, dev)) && head_batch_smem(b, K) > (size_t)220 * 1024)
    return fail(Q4_ERR_SHAPE, "lmhead: batch %d x K %d does not fit in shared memory", b, K);
  if (b == 1 && stream_eligible(K))
    return launch_head_stream(codes, scales, h, V, K, cap, idx, top1, top2, logits, ws, dev, s);
  unsigned* ticket = reinterpret_cast<unsigned*>(ws);
  Top2* partials = reinterpret_cast<Top2*>(reinterpret_cast<char*>(ws) + kTicketBytes);
  cudaError_t e = cudaMemsetAsync(ticket, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return cuda_fail(e, "lmhead ticket reset");
  if (tensor_cores && head_tc_eligible(b, V, K, dev)) {
    // z = W h on the tensor cores; its epilogue softcaps and selects
    void* xws = reinterpret_cast<char*>(ws) + kTicketBytes + up256((size_t)head_grid(dev) * kMaxBatch * sizeof(Top2));
    const HeadOutputs out = {cap, logits, partials, ticket, idx, top1, top2};
    return launch_head_mma(codes, scales, h, b, V, K, xws, out, dev, s);
  }
  if (b > 1) {
    int grid = head_grid(dev);
    const int need = (V + 7) / 8;   // at least one row per group of the smallest grouping
    if (grid > need) grid = need;
    return launch_head_batch(codes, scales, h, b, V, K, cap, idx, top1, top2, logits, partials, ticket, grid, s);
  }
  switch (lpr_for(K >> 5)) {
    case 32: e = launch_head_t<32>(codes, scales, h, V, K, cap, idx, top1, top2, logits, partials, ticket, dev, s); break;
    case 16: e = launch_head_t<16>(codes, scales, h, V, K, cap, idx, top1, top2, logits, partials, ticket, dev, s); break;
    case 8: e = launch_head_t<8>(codes, scales, h, V, K, cap, idx, top1, top2, logits, partials, ticket, dev, s); break;
    case 4: e = launch_head_t<4>(codes, scales, h, V, K, cap, idx, top1, top2, logits, partials, ticket, dev, s); break;
    case 2: e = launch_head_t<2>(codes, scales, h, V, K, cap, idx, top1, top2, logits, partials, ticket, dev, s); break;
    default: e = launch_head_t<1>(codes, scales, h, V, K, cap, idx, top1, top2, logits, partials, ticket, dev, s); break;
  }
  return e == cudaSuccess ? Q4_OK : cuda_fail(e, "lmhead launch");
}

}  // namespace q4w
