// LM head for a batch of 2..8 hidden vectors (the S=4 / S=8 verify shapes):
// z[b][v] = sum_k W[v][k] h[b][k] with the same softcap and two-level top-two
// selection as the single-vector head ("Gemma 4 E2B (text decoder) - Core
// AI", Signature features and What it took).
//
// Each weight block is decoded once and applied to every batch vector: a
// lane turns its 16 code bytes into 16 fp16 half pairs (q4_word_pairs: one
// LOP3 each), then for each batch vector multiplies
// them into two fp32 accumulators with the mixed-precision FMA, against the
// vector's half pairs (x[8i+j], x[8i+j+4]) staged in shared memory.  Per
// vector the arithmetic is that of the single-vector head (the block bias of
// q4_block_dot_h, lo/hi accumulators, one fmaf with the scale
// per block, the lane-group reduction from P/2 down); only the order in
// which the block bias sums x differs.
#include "q4w_device.cuh"
#include "q4w_internal.cuh"
#include "q4w_top2.cuh"

namespace q4w {

namespace hb {

constexpr int kThr = 256;
constexpr int kWarpsHB = kThr / 32;
__device__ __forceinline__ void top2_shfl_merge(Top2& t, int o) {
  Top2 u;
  u.v1 = __shfl_xor_sync(0xffffffffu, t.v1, o);
  u.v2 = __shfl_xor_sync(0xffffffffu, t.v2, o);
  u.i1 = __shfl_xor_sync(0xffffffffu, t.i1, o);
  u.i2 = __shfl_xor_sync(0xffffffffu, t.i2, o);
  top2_merge(t, u);
}

// NBP: batch vectors computed (B rounded up to 4 or 8; the rest have x = 0).
// lgP: log2 of the lanes per row (P <= 32, P divides the block count).
template <int NBP>
__global__ void __launch_bounds__(kThr) head_batch_kernel(const uint8_t* __restrict__ codes,
                                                         const __half* __restrict__ scales,
                                                         const __half* __restrict__ h, int B, int V, int K,
                                                         int lgP, float cap, float* __restrict__ logits,
                                                         Top2* partials, unsigned* ticket, int32_t* idx,
                                                         float* top1, float* top2, float* __restrict__ ydirect) {
  extern __shared__ __align__(16) uint32_t hb_smem[];
  const int nb = K >> 5;
  const int xstride = 16 * NBP + 4;           // words per block (+4: lanes of a group hit other banks)
  uint32_t* xw = hb_smem;                     // [nb][16 pairs][NBP] half pairs
  float* xb = reinterpret_cast<float*>(hb_smem + (size_t)nb * xstride);   // [nb][NBP] biases
  __shared__ Top2 st[kWarpsHB][kMaxBatch];

  // the first kPre blocks of this lane's first row are fetched before x is
  // staged (they do not depend on x), so their latency overlaps the staging
  // (batch 2..4 only: with 8 vectors the registers would cut the occupancy)
  constexpr int kPre = NBP == 4 ? 4 : 0;
  uint4 pc[kPre > 0 ? kPre : 1];
  float pd[kPre > 0 ? kPre : 1];
  if constexpr (kPre > 0) {
    const int P = 1 << lgP, li = (threadIdx.x & 31) & (P - 1), gid = threadIdx.x >> lgP;
    const int wg0 = ((threadIdx.x >> 5) * 32) >> lgP;
    const int wrow0 = blockIdx.x * (kThr >> lgP) + wg0;
    if (wrow0 < V) {   // uniform per warp
      const int row0 = wrow0 + (gid - wg0);
      const int row = row0 < V ? row0 : V - 1;
#pragma unroll
      for (int t = 0; t < kPre; ++t) {
        if (t < (nb >> lgP)) {
          const int j = li + P * t;
          pc[t] = ld_stream16(codes + (size_t)row * (K >> 1) + 16 * j);
          pd[t] = ld_scale(scales + (size_t)row * nb + j);
        }
      }
    }
  }
  // stage the half pairs (x[32j+8i+jj], x[32j+8i+jj+4]) and the block biases:
  // one thread per (batch row b, block j, 8-column chunk i), one 16-byte load
  // giving the chunk's four pairs and its even / odd column sums; the four
  // chunks of a block sit in adjacent lanes and add by shuffles (the same
  // order as the single-vector engine).  Rows b >= B are zero.
  // Up to kLB 16-byte loads of a thread are issued before any is used, so
  // their L2 round trips overlap instead of following one another.
  const int nch = nb * 4;
  constexpr int kLB = 4;
  for (int e00 = 0; e00 < NBP * nch; e00 += kLB * kThr) {   // uniform trip counts: the shuffles use the full mask
    uint4 vv[kLB];
#pragma unroll
    for (int u = 0; u < kLB; ++u) {
      const int e = e00 + u * kThr + threadIdx.x;
      const int i = e & 3, j = (e >> 2) % nb, b = (e >> 2) / nb;
      vv[u] = make_uint4(0u, 0u, 0u, 0u);
      if (e < NBP * nch && b < B) vv[u] = __ldg(reinterpret_cast<const uint4*>(h + (size_t)b * K + 32 * j + 8 * i));
    }
#pragma unroll
    for (int u = 0; u < kLB; ++u) {
      const int e0 = e00 + u * kThr;
      if (e0 >= NBP * nch) break;   // uniform
      const int e = e0 + threadIdx.x;
      const bool in = e < NBP * nch;
      const int i = e & 3, j = (e >> 2) % nb, b = (e >> 2) / nb;
      const uint4 v = vv[u];
      float pe = 0.f, po = 0.f;
      const uint32_t hv[4] = {v.x, v.y, v.z, v.w};   // hv[q] = (x[8i+2q], x[8i+2q+1])
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hv[q]));
        pe += f.x;
        po += f.y;
      }
      pe += __shfl_xor_sync(0xffffffffu, pe, 1);
      po += __shfl_xor_sync(0xffffffffu, po, 1);
      pe += __shfl_xor_sync(0xffffffffu, pe, 2);
      po += __shfl_xor_sync(0xffffffffu, po, 2);
      if (in) {
        uint32_t* dst = xw + j * xstride + (4 * i) * NBP + b;
        dst[0 * NBP] = __byte_perm(hv[0], hv[2], 0x5410);   // (x[8i], x[8i+4])
        dst[1 * NBP] = __byte_perm(hv[0], hv[2], 0x7632);   // (x[8i+1], x[8i+5])
        dst[2 * NBP] = __byte_perm(hv[1], hv[3], 0x5410);   // (x[8i+2], x[8i+6])
        dst[3 * NBP] = __byte_perm(hv[1], hv[3], 0x7632);   // (x[8i+3], x[8i+7])
        if (i == 0) xb[j * NBP + b] = kBiasEven * pe + kBiasOdd * po;
      }
    }
  }
  __syncthreads();

  const int P = 1 << lgP;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int li = lane & (P - 1);
  const int gid = threadIdx.x >> lgP, ngroups = kThr >> lgP;
  const size_t K2 = (size_t)(K >> 1);
  const int wg0 = (warp * 32) >> lgP;                  // the warp's first group
  const int bpl = nb >> lgP;                           // blocks per lane (P divides nb)
  const int wrow0 = blockIdx.x * ngroups + wg0;        // the warp's first row block
  Top2 best[NBP];
#pragma unroll
  for (int b = 0; b < NBP; ++b) top2_init(best[b]);

  // Row groups of a warp advance together (the shuffles use the full mask);
  // a group past the last row recomputes row V - 1 and drops it.
  const int step = gridDim.x * ngroups;
  for (int wrow = wrow0; wrow < V; wrow += step) {   // uniform per warp
    const int row0 = wrow + (gid - wg0);
    const bool valid = row0 < V;
    const int row = valid ? row0 : V - 1;
    const uint8_t* cp = codes + (size_t)row * K2;
    const __half* sp = scales + (size_t)row * nb;
    float acc[NBP];
#pragma unroll
    for (int b = 0; b < NBP; ++b) acc[b] = 0.f;
    // block t of this lane: code word c and scale d, into acc
    auto block = [&](int t, const uint4 c, const float d) {
      const int j = li + P * t;
      uint32_t wq[16];
      const uint32_t w4[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t pr[4];
        q4_word_pairs(w4[i], pr);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) wq[4 * i + jj] = pr[jj];
      }
      float lo[NBP], hi[NBP];
#pragma unroll
      for (int b = 0; b < NBP; ++b) {
        lo[b] = xb[j * NBP + b];
        hi[b] = 0.f;
      }
      const uint32_t* xj = xw + j * xstride;
#pragma unroll
      for (int p = 0; p < 16; ++p) {
        uint32_t xq[NBP];
#pragma unroll
        for (int q = 0; q < NBP / 4; ++q) {
          const uint4 u = *reinterpret_cast<const uint4*>(xj + p * NBP + 4 * q);
          xq[4 * q] = u.x;
          xq[4 * q + 1] = u.y;
          xq[4 * q + 2] = u.z;
          xq[4 * q + 3] = u.w;
        }
#pragma unroll
        for (int b = 0; b < NBP; ++b) fhfma2(lo[b], hi[b], wq[p], xq[b]);
      }
#pragma unroll
      for (int b = 0; b < NBP; ++b) acc[b] = fmaf(d, lo[b] + hi[b], acc[b]);
    };
    if constexpr (kPre > 0) {
      const bool first = wrow == wrow0;
#pragma unroll
      for (int t = 0; t < kPre; ++t) {
        if (t < bpl) {
          const int j = li + P * t;
          if (first)
            block(t, pc[t], pd[t]);
          else
            block(t, ld_stream16(cp + 16 * j), ld_scale(sp + j));
        }
      }
    }
    for (int t = kPre; t < bpl; ++t) {
      const int j = li + P * t;
      block(t, ld_stream16(cp + 16 * j), ld_scale(sp + j));
    }
#pragma unroll
    for (int b = 0; b < NBP; ++b)
      for (int o = P >> 1; o > 0; o >>= 1) acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], o);
    if (li == 0 && valid) {
#pragma unroll
      for (int b = 0; b < NBP; ++b) {
        if (b < B) {
          if (ydirect) {   // batched GEMV: the raw row sums
            ydirect[(size_t)b * V + row] = acc[b];
          } else {
            top2_insert(best[b], acc[b], row);
            if (logits) logits[(size_t)b * V + row] = cap * tanhf(acc[b] / cap);
          }
        }
      }
    }
  }
  if (ydirect) return;   // uniform over the grid
  // groups of a warp -> lane 0, warps -> the CTA's partial per batch row
#pragma unroll
  for (int b = 0; b < NBP; ++b)
    for (int o = P; o < 32; o <<= 1) top2_shfl_merge(best[b], o);
  if (lane == 0) {
#pragma unroll
    for (int b = 0; b < NBP; ++b)
      if (b < B) st[warp][b] = best[b];
  }
  __syncthreads();
  if (threadIdx.x < B) {
    Top2 t;
    top2_init(t);
    for (int w = 0; w < kWarpsHB; ++w) top2_merge(t, st[w][threadIdx.x]);
    partials[(size_t)blockIdx.x * kMaxBatch + threadIdx.x] = t;
  }
  head_finish(partials, ticket, B, cap, idx, top1, top2);
}

}  // namespace hb

// Lanes per row: the largest power of two up to 32 that divides the block count.
static int head_batch_lgp(int nb) {
  int lg = 5;
  while (lg > 0 && nb % (1 << lg)) --lg;
  return lg;
}

// b in [2, 8]; K % 32 == 0: shared memory of the x staging.
size_t head_batch_smem(int b, int K) {
  const int NBP = b <= 4 ? 4 : 8;
  const int nb = K >> 5;
  size_t bytes = (size_t)nb * (16 * NBP + 4) * 4 + (size_t)nb * NBP * 4;
  return bytes;
}

// ydirect != nullptr: batched GEMV, ydirect[b][row] = the row sums (no
// softcap, no selection; partials, ticket, idx, top1, top2 unused).
int launch_head_batch(const uint8_t* codes, const __half* scales, const __half* h, int b, int V, int K, float cap,
                      int32_t* idx, float* top1, float* top2, float* logits, Top2* partials, unsigned* ticket,
                      int grid, cudaStream_t s, float* ydirect) {
  const int lgP = head_batch_lgp(K >> 5);
  const size_t smem = head_batch_smem(b, K);
  cudaError_t e;
  // one wave: the grid is capped at the CTAs that are resident at once
  int sms = 0, per_sm = 0;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "batched head device query");
  if (b <= 4) {
    e = cudaFuncSetAttribute(hb::head_batch_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, hb::head_batch_kernel<4>, hb::kThr, smem);
    if (e == cudaSuccess && per_sm > 0 && grid > sms * per_sm) grid = sms * per_sm;
    if (e == cudaSuccess)
      hb::head_batch_kernel<4><<<grid, hb::kThr, smem, s>>>(codes, scales, h, b, V, K, lgP, cap, logits, partials,
                                                           ticket, idx, top1, top2, ydirect);
  } else {
    e = cudaFuncSetAttribute(hb::head_batch_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, hb::head_batch_kernel<8>, hb::kThr, smem);
    if (e == cudaSuccess && per_sm > 0 && grid > sms * per_sm) grid = sms * per_sm;
    if (e == cudaSuccess)
      hb::head_batch_kernel<8><<<grid, hb::kThr, smem, s>>>(codes, scales, h, b, V, K, lgP, cap, logits, partials,
                                                           ticket, idx, top1, top2, ydirect);
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? Q4_OK : cuda_fail(e, "batched head launch");
}

// Batched GEMV (batch 2..8) through the same kernel: y[b][n] = sum_k W[n][k] x[b][k].
// Returns Q4_ERR_SHAPE when the x staging does not fit in shared memory.
int launch_gemv_batch_decoded(const uint8_t* codes, const __half* scales, const __half* x, float* y, int N, int K,
                              int batch, const DeviceInfo& dev, cudaStream_t s) {
  if (batch < 2 || batch > 8 || head_batch_smem(batch, K) > (size_t)220 * 1024)
    return fail(Q4_ERR_SHAPE, "batched GEMV: batch %d x K %d does not fit", batch, K);
  // one CTA per (kThr / P) rows: CTAs past the last row would only stage x
  int grid = 2 * dev.sms;
  const int rows_per_cta = hb::kThr >> head_batch_lgp(K >> 5);
  const int need = (N + rows_per_cta - 1) / rows_per_cta;
  if (grid > need) grid = need;
  return launch_head_batch(codes, scales, x, batch, N, K, 1.f, nullptr, nullptr, nullptr, nullptr, nullptr,
                           nullptr, grid, s, y);
}

}  // namespace q4w
