// Per-Layer-Embedding gather fused with its f32 projection and per-chunk
// RMSNorm ("visible-cx/gemma-4-E2B-CoreAI", The PLE gather-table sidecar:
// int8 table [V][L*ld] + per-row f32 scale, dequant x16.0, proj.f32
// [L*ld][D], proj_norm.f32 [ld]; "Gemma-4 E2B mobile mixed-bit QAT weights",
// P2 DONE: 35 layer-major blocks of 256 on axis 1).
//
// The projection p[t] = proj . hidden[t] is a dense contraction (L*ld rows x
// D x S tokens), so it runs on the 5th-generation tensor cores in TF32:
// tcgen05.mma kind::tf32, M = 128 projection rows, N = the token group (up to
// 64, padded to a multiple of 16 with zero rows), fp32 accumulator in TMEM.
// The fp16 hidden values are exact in TF32; the f32 projection enters with a
// 10-bit mantissa (the tensor core reads the top 19 bits of each fp32 word).
//
// One CTA per (128-row half of a 256-row layer chunk, group of 64 tokens);
// the two halves of a chunk form a cluster of two and swap their per-token
// sums of squares through distributed shared memory, so each finishes the
// chunk's RMSNorm for its own rows and adds the gathered table term in the
// same epilogue.
//
// Warp roles (192 threads):
//   warp 0     one thread issuing the TMA loads: the projection tile [128
//              rows][32 fp32] (128-byte swizzle, the tensor core's K-major
//              layout) and the hidden tile [64 tokens][32 fp16]
//   warp 1     TMEM allocation and the single thread issuing the MMAs
//   warps 2-5  widen the hidden tile to fp32 in the 128-byte swizzle layout
//              (the B operand), then run the epilogue on their TMEM lane
//              quarters (warp w reads lanes 32 (w % 4) .. + 31)
// A ring of kStages stages (A 16 KB + B 8 KB + hidden 4 KB) is guarded by
// full (TMA bytes), bready (converter warps) and empty (MMA commit)
// mbarriers.  Every mbarrier wait is bounded; on expiry the CTA sets its
// abort flag and the device error word, every role leaves its loop, work in
// flight is drained, and both CTAs of the cluster still meet at the cluster
// barriers, so neither waits for a partner that has given up.
#include "q4w_device.cuh"
#include "q4w_internal.cuh"
#include "q4w_tc.cuh"

namespace q4w {

namespace ple {

constexpr int kLd = 256;                            // rows of one layer chunk
constexpr int kRows = 128;                          // rows per CTA (MMA M)
constexpr int kTok = 64;                            // tokens per CTA (MMA N <= 64)
constexpr int kKC = 32;                             // K columns per stage (128 B of fp32)
constexpr int kStages = 6;
constexpr int kABytes = kRows * kKC * 4;            // 16 KB
constexpr int kBBytes = kTok * kKC * 4;             // 8 KB
constexpr int kHBytes = kTok * kKC * 2;             // 4 KB
constexpr int kStageBytes = kABytes + kBBytes + kHBytes;   // 28 KB, a multiple of 1024
constexpr int kThreads = 192;
constexpr int kEpi0 = 2;                            // first converter / epilogue warp
constexpr int kTmemCols = 64;
constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes;
constexpr long long kDrainCycles = 2000000000LL;

// Instruction descriptor, kind::tf32: D f32, A and B tf32, both K-major,
// M = 128, N = n (a multiple of 16).
__device__ __forceinline__ uint32_t idesc_tf32(int n) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}

struct Params {
  CUtensorMap tm_proj;   // f32 [L*ld][D], box [128 rows][32], 128-byte swizzle
  CUtensorMap tm_hid;    // fp16 bits [S][D], box [64 rows][32]; rows past S read as zero
  const int32_t* ids;
  const int8_t* table;
  const float* row_scale;
  const float* norm_w;
  float* out;
  int8_t* gathered;
  int32_t* err;          // optional id-range flag
  unsigned* dev_err;     // the library's device error word (bounded waits)
  int S, V, L, D;
  float embed_scale, eps;
  long long wait_limit;
  unsigned long long* trace;   // optional: CTA 0 stamps [chunk][8], SM cycles since the start
};

constexpr int kTraceChunks = 256;

// Sum over the 32 lanes of v[0..15] for 16 tokens: a halving exchange leaves
// lanes 2i and 2i+1 with the total of token i (16 shuffles instead of 80).
__device__ __forceinline__ float lane_token_sums16(float (&v)[16], int lane) {
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1) {
    const int off = 2 * w;   // 16, 8, 4, 2
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float keep = up ? v[i + w] : v[i];
      const float give = up ? v[i] : v[i + w];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, give, off);
    }
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

__global__ void __launch_bounds__(kThreads, 1) ple_tc_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t bars[3 * kStages + 2];   // full, bready, empty, accfull, drain
  __shared__ uint32_t tmem_sh;
  __shared__ int abort_sh;
  __shared__ float red[4][kTok];     // per epilogue warp: per-token sums of squares over its 32 rows
  __shared__ float ssq_peer[kTok];   // written by the other half of the chunk
  __shared__ float rfac[kTok];       // per-token RMS factor
  __shared__ float tsc[kTok];        // per-token table scale (0 for a bad id)
  __shared__ int tid_sh[kTok];       // per-token id (-1: out of range)
  __shared__ long long t0_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = blockIdx.x & 1;                 // rank in the cluster of two
  const int chunk = blockIdx.x >> 1;
  const int row0 = chunk * kLd + half * kRows;     // first projection row of this CTA
  const int t0 = blockIdx.y * kTok;
  const int ntok = min(kTok, p.S - t0);
  const int npad = (ntok + 15) & ~15;
  const int nk = p.D / kKC;
  const int PLD = p.L * kLd;
  const uint32_t full0 = tc::smem_u32(bars), bready0 = full0 + 8 * kStages, empty0 = bready0 + 8 * kStages;
  const uint32_t accfull = empty0 + 8 * kStages, drain = accfull + 8;
  volatile int* abort_flag = &abort_sh;
  unsigned long long* const tr = (p.trace && blockIdx.x == 0 && blockIdx.y == 0) ? p.trace : nullptr;
  auto stamp = [&](int c, int k) {
    if (tr && c < kTraceChunks) tr[c * 8 + k] = (unsigned long long)(clock64() - t0_sh);
  };

  if (threadIdx.x == 0) {
    abort_sh = 0;
    t0_sh = clock64();
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(full0 + 8 * s, 1);
      tc::mbar_init(bready0 + 8 * s, 4);
      tc::mbar_init(empty0 + 8 * s, 1);
    }
    tc::mbar_init(accfull, 1);
    tc::mbar_init(drain, 1);
    tc::mbar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(tc::smem_u32(&tmem_sh), kTmemCols);
  if (threadIdx.x >= kEpi0 * 32 && threadIdx.x < kEpi0 * 32 + kTok) {
    const int t = threadIdx.x - kEpi0 * 32;
    int id = -1;
    float sc = 0.f;
    if (t < ntok) {
      const int v = p.ids[t0 + t];
      if (v >= 0 && v < p.V) {
        id = v;
        sc = p.row_scale[v];
      } else if (p.err) {
        atomicExch(p.err, 1);
      }
    }
    tid_sh[t] = id;
    tsc[t] = sc;
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  // the peer CTA has started before anyone stores into its shared memory
  // (this phase is waited for just before the exchange)
  tc::cluster_arrive_relaxed();
  const uint32_t tmem = tmem_sh;

  if (warp == 0) {
    // ------------------------------------------------------------- TMA loads
    if (lane == 0) {
      const uint64_t pol_once = tc::policy_evict_first(), pol_keep = tc::policy_evict_last();
      const uint32_t st0 = tc::smem_u32(smem);
      int c = 0;
      for (; c < nk; ++c) {
        const int s = c % kStages, round = c / kStages;
        if (!tc::mbar_wait(empty0 + 8 * s, (round & 1) ^ 1, p.wait_limit, abort_flag, p.dev_err)) break;
        const uint32_t A = st0 + s * kStageBytes, H = A + kABytes + kBBytes;
        stamp(c, 0);
        tc::mbar_expect_tx(full0 + 8 * s, kABytes + kHBytes);
        // x = 32 c fp32 (128 c bytes) and 32 c fp16 (64 c bytes): 16-byte aligned
        tc::tma_load_2d(A, &p.tm_proj, c * kKC, row0, full0 + 8 * s, pol_once);
        tc::tma_load_2d(H, &p.tm_hid, c * kKC, t0, full0 + 8 * s, pol_keep);
      }
      // every issued load lands before the CTA may exit
      for (int q = max(0, c - kStages); q < c; ++q)
        tc::mbar_drain(full0 + 8 * (q % kStages), (q / kStages) & 1, kDrainCycles, p.dev_err);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t st0 = tc::smem_u32(smem);
      const uint32_t idesc = idesc_tf32(npad);
      bool ok = true;
      for (int c = 0; c < nk && ok; ++c) {
        const int s = c % kStages, round = c / kStages;
        if (!tc::mbar_wait(full0 + 8 * s, round & 1, p.wait_limit, abort_flag, p.dev_err) ||
            !tc::mbar_wait(bready0 + 8 * s, round & 1, p.wait_limit, abort_flag, p.dev_err)) {
          ok = false;
          break;
        }
        tc::fence_after();
        stamp(c, 3);
        const uint32_t A = st0 + s * kStageBytes, B = A + kABytes;
#pragma unroll
        for (int k = 0; k < kKC / 8; ++k)   // K = 8 tf32 (32 bytes) per MMA
          mma_tf32(tmem, tc::desc_sw128(A + 32 * k), tc::desc_sw128(B + 32 * k), idesc, (c | k) ? 1u : 0u);
        tc::commit(empty0 + 8 * s);
        stamp(c, 4);
      }
      if (ok) tc::commit(accfull);
      // every tcgen05 operation issued here has finished before TMEM is freed
      tc::commit(drain);
      tc::mbar_drain(drain, 0, kDrainCycles, p.dev_err);
    }
    __syncwarp();
  } else {
    // ------------------------------------- B operand: fp16 hidden -> fp32 tile
    const int ct = threadIdx.x - kEpi0 * 32;   // 0..127
    bool ok = true;
    for (int c = 0; c < nk; ++c) {
      const int s = c % kStages, round = c / kStages;
      const bool landed = tc::mbar_wait(full0 + 8 * s, round & 1, p.wait_limit, abort_flag, p.dev_err);
      if (!__all_sync(0xffffffffu, landed)) {   // leave the loop as a whole warp
        ok = false;
        break;
      }
      if (ct == 0) stamp(c, 1);
      uint8_t* st = smem + (size_t)s * kStageBytes;
      uint8_t* B = st + kABytes;
      const uint8_t* H = B + kBBytes;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int idx = ct + 128 * i;      // (token t, 16-byte group j of its 128-byte row)
        const int t = idx >> 3, j = idx & 7;
        // tokens past S: zero rows (the tensor map already reads them as zero)
        const uint2 h = t < ntok ? *reinterpret_cast<const uint2*>(H + t * (kKC * 2) + j * 8) : make_uint2(0u, 0u);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&h.y));
        // 128-byte swizzle: group j of row t sits at group j ^ (t % 8) of its row
        *reinterpret_cast<float4*>(B + (t >> 3) * 1024 + (t & 7) * 128 + ((j ^ (t & 7)) << 4)) =
            make_float4(a.x, a.y, b.x, b.y);
      }
      tc::fence_proxy_async();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(bready0 + 8 * s);
      if (ct == 0) stamp(c, 2);
    }
    // ------------------------------------------------------------- epilogue
    const int q = warp & 3;                    // TMEM lane quarter
    const int row = 32 * q + lane;             // row of this CTA's tile
    const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16);
    if (ok) ok = tc::mbar_wait(accfull, 0, p.wait_limit, abort_flag, p.dev_err, 128);
    ok = __all_sync(0xffffffffu, ok);   // the TMEM loads below are warp-wide
    tc::fence_after();
    if (ct == 0) stamp(0, 5);
    if (ok) {
      for (int cb = 0; cb < npad / 16; ++cb) {
        float v[16];
        tc::tmem_ld16(taddr + cb * 16, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] *= v[j];
        const float s = lane_token_sums16(v, lane);
        if ((lane & 1) == 0) red[q][cb * 16 + (lane >> 1)] = s;
      }
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    // this half's sums (warp quarters added in row order), then the swap
    float own = 0.f;
    if (ct < kTok) own = ((red[0][ct] + red[1][ct]) + red[2][ct]) + red[3][ct];
    tc::cluster_wait();   // phase 1: the peer is running
    if (ct < kTok) tc::st_cluster_f32(&ssq_peer[ct], (uint32_t)(half ^ 1), own);
    tc::cluster_arrive_release();
    tc::cluster_wait();   // phase 2: both halves' sums are in place
    if (ct < kTok) {
      const float lo = half == 0 ? own : ssq_peer[ct], hi = half == 0 ? ssq_peer[ct] : own;
      rfac[ct] = 1.f / sqrtf((lo + hi) / (float)kLd + p.eps);
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (ct == 0) stamp(0, 6);
    if (ok) {
      const int j = row0 + row;                        // output column
      const float nw = p.norm_w[half * kRows + row];
      for (int cb = 0; cb < npad / 16; ++cb) {
        float v[16];
        tc::tmem_ld16(taddr + cb * 16, v);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int t = cb * 16 + u;
          if (t >= ntok) break;
          const size_t o = (size_t)(t0 + t) * PLD + j;
          const int id = tid_sh[t];
          if (id < 0) {
            p.out[o] = 0.f;
            if (p.gathered) p.gathered[o] = 0;
            continue;
          }
          const int8_t tq = p.table[(size_t)id * PLD + j];
          const float g = __fmul_rn(__fmul_rn((float)tq, tsc[t]), p.embed_scale);
          p.out[o] = v[u] * rfac[t] * nw + g;
          if (p.gathered) p.gathered[o] = tq;
        }
      }
    }
  }
  if (threadIdx.x == kEpi0 * 32) stamp(0, 7);
  if (warp < kEpi0) {   // the TMA and MMA warps take part in both cluster phases too
    tc::cluster_wait();
    tc::cluster_arrive_release();
    tc::cluster_wait();
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace ple

int launch_ple(const int32_t* ids, int S, const int8_t* table, const float* row_scale, int V, int L,
               int ld, float embed_scale, const float* proj, const __half* hidden, int D,
               const float* norm_w, float eps, float* out, int8_t* gathered, int32_t* err,
               const DeviceInfo& dev, cudaStream_t s) {
  (void)dev;
  if (ld != ple::kLd) return fail(Q4_ERR_SHAPE, "ple_gather_project: ld must be %d", ple::kLd);
  ple::Params p;
  memset(&p, 0, sizeof(p));
  int st = encode_tensor_2d(&p.tm_proj, proj, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)D, (uint64_t)L * ld,
                            ple::kKC, ple::kRows, CU_TENSOR_MAP_SWIZZLE_128B, "proj");
  if (st != Q4_OK) return st;
  st = encode_tensor_2d(&p.tm_hid, hidden, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, (uint64_t)D, (uint64_t)S, ple::kKC,
                        ple::kTok, CU_TENSOR_MAP_SWIZZLE_NONE, "hidden");
  if (st != Q4_OK) return st;
  p.ids = ids;
  p.table = table;
  p.row_scale = row_scale;
  p.norm_w = norm_w;
  p.out = out;
  p.gathered = gathered;
  p.err = err;
  p.dev_err = device_error_word();
  if (!p.dev_err) return fail(Q4_ERR_CUDA, "device error word unavailable");
  p.S = S;
  p.V = V;
  p.L = L;
  p.D = D;
  p.embed_scale = embed_scale;
  p.eps = eps;
  p.wait_limit = wait_limit();
  size_t tbytes = 0;
  void* tb = trace_buffer(&tbytes);
  p.trace = (tb && tbytes >= (size_t)ple::kTraceChunks * 8 * sizeof(unsigned long long))
                ? static_cast<unsigned long long*>(tb)
                : nullptr;
  static bool attr = false;
  cudaError_t e;
  if (!attr) {
    e = cudaFuncSetAttribute(ple::ple_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ple::kSmem);
    if (e != cudaSuccess) return cuda_fail(e, "ple smem attribute");
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * L, (S + ple::kTok - 1) / ple::kTok);
  cfg.blockDim = dim3(ple::kThreads);
  cfg.dynamicSmemBytes = ple::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, ple::ple_tc_kernel, p);
  return e == cudaSuccess ? Q4_OK : cuda_fail(e, "ple launch");
}

}  // namespace q4w
