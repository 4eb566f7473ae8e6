// S=1 q4_0 GEMV stages (prologue + dequant-GEMV + epilogue), the batched GEMV
// and the closing RMSNorm of the decode pass.
//
// Mapping: a warp owns G = 32/LPR lane groups of LPR lanes; a lane group owns
// R rows (R pairs of rows for the gate/up pair).  Lane li of a group walks
// the 32-column blocks li, li+LPR, ... of its rows: per block one 16-byte
// streaming load of codes per row plus one fp16 scale, x read from shared
// memory once and reused for all R rows, then a shuffle reduction over the
// group.  x lives in shared memory in a padded layout (kXStride floats per
// block, the last slots holding the block bias of the nibble trick).
#include "q4w_device.cuh"
#include "q4w_internal.cuh"

namespace q4w {

// ------------------------------------------------------------ prologue ---
__device__ __forceinline__ float load_in(const void* in, int mode, int k) {
  if (mode == Q4_IN_F16 || mode == Q4_IN_RMS_F16)
    return __half2float(reinterpret_cast<const __half*>(in)[k]);
  return reinterpret_cast<const float*>(in)[k];
}

// Fills xs with x = prologue(in) (fp32 copies of fp16 values) and the
// per-block biases.  Ends with a CTA barrier.
__device__ void stage_prologue(const void* in, int mode, int K, float eps, float* xs, float* red) {
  const int tid = threadIdx.x;
  if (mode == Q4_IN_F16) {
    for (int k = tid; k < K; k += kThreads) xs_store(xs, k, load_in(in, mode, k));
  } else {
    float ss = 0.f;
    for (int k = tid; k < K; k += kThreads) {
      const float v = load_in(in, mode, k);
      ss += v * v;
    }
    ss = block_sum(ss, red);
    const float r = 1.f / sqrtf(ss / (float)K + eps);
    if (mode != Q4_IN_RMS2_F32) {
      for (int k = tid; k < K; k += kThreads) xs_store(xs, k, f16_round(load_in(in, mode, k) * r));
    } else {
      float ss2 = 0.f;
      for (int k = tid; k < K; k += kThreads) {
        const float t = f16_round(load_in(in, mode, k) * r);
        xs_store(xs, k, t);
        ss2 += t * t;
      }
      ss2 = block_sum(ss2, red);
      const float r2 = 1.f / sqrtf(ss2 / (float)K + eps);
      for (int k = tid; k < K; k += kThreads) xs_store(xs, k, f16_round(xs_load(xs, k) * r2));
    }
  }
  __syncthreads();
  xs_biases(xs, K >> 5);
  __syncthreads();
}

// ------------------------------------------------------- fused stage ---
template <int LPR, int R, bool PAIR>
__global__ void __launch_bounds__(kThreads) stage_kernel(const StageArgs a, int total, int tasks) {
  extern __shared__ float4 dyn_smem4[];
  float* xs = reinterpret_cast<float*>(dyn_smem4);
  __shared__ float red[kWarps];

  pdl_trigger();
  pdl_wait();
  stage_prologue(a.in, a.in_mode, a.K, a.eps, xs, red);

  constexpr int G = 32 / LPR;
  constexpr int NM = PAIR ? 2 : 1;
  const int nb = a.K >> 5;
  const size_t row_bytes = (size_t)(a.K >> 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane / LPR, li = lane % LPR;

  for (int task = blockIdx.x * kWarps + warp; task < tasks; task += gridDim.x * kWarps) {
    const int rbase = (task * G + g) * R;
    const uint8_t* cp[R][NM];
    const __half* sp[R][NM];
    int mi[R], lr[R];
    bool ok[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int row = rbase + r;
      ok[r] = row < total;
      int m = 0, l = ok[r] ? row : 0;
      if (!PAIR) {
        if (l >= a.mat[0].rows) {
          l -= a.mat[0].rows;
          m = 1;
          if (l >= a.mat[1].rows) {
            l -= a.mat[1].rows;
            m = 2;
          }
        }
      }
      mi[r] = m;
      lr[r] = l;
#pragma unroll
      for (int t = 0; t < NM; ++t) {
        const StageMat& M = a.mat[PAIR ? t : m];
        cp[r][t] = M.codes + (size_t)l * row_bytes;
        sp[r][t] = M.scales + (size_t)l * nb;
      }
    }
    float acc[R][NM];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int t = 0; t < NM; ++t) acc[r][t] = 0.f;

#pragma unroll 2
    for (int j = li; j < nb; j += LPR) {
      uint4 c[R][NM];
      float d[R][NM];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int t = 0; t < NM; ++t) {
          if (ok[r]) {
            c[r][t] = ld_stream16(cp[r][t] + 16 * j);
            d[r][t] = ld_scale(sp[r][t] + j);
          } else {
            c[r][t] = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
            d[r][t] = 0.f;
          }
        }
      float4 xv[8];
      float bias;
      load_xblock(xs, j, xv, bias);
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int t = 0; t < NM; ++t) acc[r][t] = fmaf(d[r][t], q4_block_dot(c[r][t], xv, bias), acc[r][t]);
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int t = 0; t < NM; ++t)
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) acc[r][t] += __shfl_xor_sync(0xffffffffu, acc[r][t], o);

    if (li == 0) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (!ok[r]) continue;
        if (PAIR) {
          const float gv = acc[r][0], uv = acc[r][NM - 1];
          const int row = rbase + r;
          if (a.mat[0].out32) a.mat[0].out32[row] = gv;
          if (a.mat[1].out32) a.mat[1].out32[row] = uv;
          a.mat[0].out16[row] = __float2half_rn(gelu_tanh_f32(gv) * uv);
        } else {
          const StageMat& M = a.mat[mi[r]];
          if (M.out32) M.out32[lr[r]] = acc[r][0];
          if (M.out16) M.out16[lr[r]] = __float2half_rn(acc[r][0]);
        }
      }
    }
  }
}

// ----------------------------------------------------- batched GEMV ---
// One warp per row; lane group g handles batch rows g, g+G, ...  x of all
// batch rows sits in shared memory (batch-major, padded layout).
template <int LPR>
__global__ void __launch_bounds__(kThreads) gemv_batched_kernel(const uint8_t* __restrict__ codes,
                                                               const __half* __restrict__ scales,
                                                               const __half* __restrict__ x,
                                                               float* __restrict__ y, int N, int K,
                                                               int B) {
  extern __shared__ float4 dyn_smem4[];
  float* xs = reinterpret_cast<float*>(dyn_smem4);
  const int nb = K >> 5;
  const int xstride = nb * kXStride;
  for (int i = threadIdx.x; i < B * K; i += kThreads) {
    const int b = i / K, k = i - b * K;
    xs_store(xs + b * xstride, k, __half2float(x[i]));
  }
  __syncthreads();
  for (int b = 0; b < B; ++b) xs_biases(xs + b * xstride, nb);
  __syncthreads();

  constexpr int G = 32 / LPR;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane / LPR, li = lane % LPR;
  const size_t row_bytes = (size_t)(K >> 1);
  for (int row = blockIdx.x * kWarps + warp; row < N; row += gridDim.x * kWarps) {
    const uint8_t* cp = codes + (size_t)row * row_bytes;
    const __half* sp = scales + (size_t)row * nb;
    for (int b0 = 0; b0 < B; b0 += G) {
      const int b = b0 + g;
      const bool okb = b < B;
      float acc = 0.f;
      for (int j = li; j < nb; j += LPR) {
        const uint4 c = ld_stream16(cp + 16 * j);
        const float d = ld_scale(sp + j);
        float4 xv[8];
        float bias;
        load_xblock(xs + (okb ? b : 0) * xstride, j, xv, bias);
        acc = fmaf(d, q4_block_dot(c, xv, bias), acc);
      }
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (li == 0 && okb) y[(size_t)b * N + row] = acc;
    }
  }
}

// ------------------------------------------------------ closing norm ---
__global__ void __launch_bounds__(kThreads) rmsnorm_f16_kernel(const float* __restrict__ in, int H,
                                                              float eps, __half* __restrict__ out) {
  __shared__ float red[kWarps];
  pdl_trigger();
  pdl_wait();
  float ss = 0.f;
  for (int k = threadIdx.x; k < H; k += kThreads) ss += in[k] * in[k];
  ss = block_sum(ss, red);
  const float r = 1.f / sqrtf(ss / (float)H + eps);
  for (int k = threadIdx.x; k < H; k += kThreads) out[k] = __float2half_rn(in[k] * r);
}

// ------------------------------------------------------------- launch ---
template <typename... KArgs, typename... Args>
static cudaError_t launch_k(void (*k)(KArgs...), int grid, size_t smem, cudaStream_t s, bool pdl,
                            Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

static int lpr_for(int nb) {
  int l = 32;
  while (l > 1 && nb % l) l >>= 1;
  return l;
}

template <int LPR, int R, bool PAIR>
static cudaError_t launch_stage_t(const StageArgs& a, int total, const DeviceInfo& dev, cudaStream_t s,
                                  bool pdl) {
  constexpr int G = 32 / LPR;
  const int tasks = (total + G * R - 1) / (G * R);
  int grid = (tasks + kWarps - 1) / kWarps;
  if (grid > 2 * dev.sms) grid = 2 * dev.sms;
  const size_t smem = (size_t)(a.K >> 5) * kXStride * sizeof(float);
  auto k = stage_kernel<LPR, R, PAIR>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_k(k, grid, smem, s, pdl, a, total, tasks);
}

template <int LPR, bool PAIR>
static cudaError_t launch_stage_r(const StageArgs& a, int total, const DeviceInfo& dev, cudaStream_t s,
                                  bool pdl) {
  // Pick the rows-per-lane R that finishes in the fewest per-lane row steps
  // over the resident warps; larger R wins ties (more reuse of x).
  constexpr int G = 32 / LPR;
  const long warps = (long)dev.sms * 2 * kWarps;
  int best_r = 1;
  long best_cost = -1;
  for (int r = 4; r >= 1; r >>= 1) {
    const long tasks = (total + G * r - 1) / (G * r);
    const long cost = ((tasks + warps - 1) / warps) * r;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_r = r;
    }
  }
  if (best_r == 4) return launch_stage_t<LPR, 4, PAIR>(a, total, dev, s, pdl);
  if (best_r == 2) return launch_stage_t<LPR, 2, PAIR>(a, total, dev, s, pdl);
  return launch_stage_t<LPR, 1, PAIR>(a, total, dev, s, pdl);
}

template <bool PAIR>
static cudaError_t launch_stage_l(const StageArgs& a, int total, const DeviceInfo& dev, cudaStream_t s,
                                  bool pdl) {
  switch (lpr_for(a.K >> 5)) {
    case 32: return launch_stage_r<32, PAIR>(a, total, dev, s, pdl);
    case 16: return launch_stage_r<16, PAIR>(a, total, dev, s, pdl);
    case 8: return launch_stage_r<8, PAIR>(a, total, dev, s, pdl);
    case 4: return launch_stage_r<4, PAIR>(a, total, dev, s, pdl);
    case 2: return launch_stage_r<2, PAIR>(a, total, dev, s, pdl);
    default: return launch_stage_r<1, PAIR>(a, total, dev, s, pdl);
  }
}

int launch_stage(const StageArgs& a, const DeviceInfo& dev, cudaStream_t s, bool pdl) {
  if (stream_eligible(a.K)) return launch_stage_stream(a, dev, s, pdl);
  int total = 0;
  if (a.pair) {
    total = a.mat[0].rows;
  } else {
    for (int i = 0; i < a.nmat; ++i) total += a.mat[i].rows;
  }
  cudaError_t e = a.pair ? launch_stage_l<true>(a, total, dev, s, pdl)
                         : launch_stage_l<false>(a, total, dev, s, pdl);
  return e == cudaSuccess ? Q4_OK : cuda_fail(e, "stage launch");
}

template <int LPR>
static cudaError_t launch_batched_t(const uint8_t* codes, const __half* scales, const __half* x,
                                    float* y, int N, int K, int B, const DeviceInfo& dev,
                                    cudaStream_t s) {
  const size_t smem = (size_t)B * (K >> 5) * kXStride * sizeof(float);
  auto k = gemv_batched_kernel<LPR>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  int grid = (N + kWarps - 1) / kWarps;
  if (grid > 2 * dev.sms) grid = 2 * dev.sms;
  return launch_k(k, grid, smem, s, false, codes, scales, x, y, N, K, B);
}

int launch_gemv_batched(const uint8_t* codes, const __half* scales, const __half* x, float* y,
                        int N, int K, int batch, const DeviceInfo& dev, cudaStream_t s) {
  // Batch 2..8 with x staged whole: each weight block decoded once for all
  // batch rows (the batched head's kernel).
  if (batch >= 2 && batch <= 8 && head_batch_smem(batch, K) <= (size_t)220 * 1024)
    return launch_gemv_batch_decoded(codes, scales, x, y, N, K, batch, dev, s);
  // Otherwise split the batch into launches whose x fits in shared memory.
  const size_t per_row = (size_t)(K >> 5) * kXStride * sizeof(float);
  int chunk = (int)((size_t)200 * 1024 / per_row);
  if (chunk < 1) return fail(Q4_ERR_SHAPE, "K=%d too large for the batched GEMV", K);
  if (chunk > batch) chunk = batch;
  for (int b0 = 0; b0 < batch; b0 += chunk) {
    const int nbt = batch - b0 < chunk ? batch - b0 : chunk;
    const __half* xb = x + (size_t)b0 * K;
    float* yb = y + (size_t)b0 * N;
    cudaError_t e;
    switch (lpr_for(K >> 5)) {
      case 32: e = launch_batched_t<32>(codes, scales, xb, yb, N, K, nbt, dev, s); break;
      case 16: e = launch_batched_t<16>(codes, scales, xb, yb, N, K, nbt, dev, s); break;
      case 8: e = launch_batched_t<8>(codes, scales, xb, yb, N, K, nbt, dev, s); break;
      case 4: e = launch_batched_t<4>(codes, scales, xb, yb, N, K, nbt, dev, s); break;
      case 2: e = launch_batched_t<2>(codes, scales, xb, yb, N, K, nbt, dev, s); break;
      default: e = launch_batched_t<1>(codes, scales, xb, yb, N, K, nbt, dev, s); break;
    }
    if (e != cudaSuccess) return cuda_fail(e, "batched gemv launch");
  }
  return Q4_OK;
}

int launch_rmsnorm_f16(const float* in, int H, float eps, __half* out, cudaStream_t s, bool pdl) {
  cudaError_t e = launch_k(rmsnorm_f16_kernel, 1, 0, s, pdl, in, H, eps, out);
  return e == cudaSuccess ? Q4_OK : cuda_fail(e, "rmsnorm launch");
}

}  // namespace q4w
