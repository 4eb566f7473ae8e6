// Top-two (value, index) selection shared by the LM-head kernels.
#pragma once

#include <climits>
#include <stdint.h>

namespace q4w {

struct Top2 {
  float v1, v2;
  int i1, i2;
};

__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
  return a > b || (a == b && ia < ib);
}
__device__ __forceinline__ void top2_init(Top2& t) {
  t.v1 = t.v2 = -INFINITY;
  t.i1 = t.i2 = INT_MAX;
}
__device__ __forceinline__ void top2_insert(Top2& t, float v, int i) {
  if (better(v, i, t.v1, t.i1)) {
    t.v2 = t.v1;
    t.i2 = t.i1;
    t.v1 = v;
    t.i1 = i;
  } else if (better(v, i, t.v2, t.i2)) {
    t.v2 = v;
    t.i2 = i;
  }
}
__device__ __forceinline__ void top2_merge(Top2& t, const Top2& o) {
  top2_insert(t, o.v1, o.i1);
  top2_insert(t, o.v2, o.i2);
}

constexpr int kMaxBatch = 8;
constexpr size_t kTicketBytes = 256;

static __device__ __forceinline__ Top2 load_cg(const Top2* p) {
  Top2 t;
  t.v1 = __ldcg(&p->v1);
  t.v2 = __ldcg(&p->v2);
  t.i1 = __ldcg(&p->i1);
  t.i2 = __ldcg(&p->i2);
  return t;
}

// Second level: runs in the CTA that finishes last.  Warp w merges the
// partials of batch rows w, w + warps, ...: its lanes stride over the CTAs'
// records with four independent loads in flight, then a shuffle merge.  The
// result does not depend on the merge order (the ordering of better() is
// total and the records of different CTAs hold different rows).
static __device__ __forceinline__ void top2_shfl_xor_merge(Top2& t, int o) {
  Top2 u;
  u.v1 = __shfl_xor_sync(0xffffffffu, t.v1, o);
  u.v2 = __shfl_xor_sync(0xffffffffu, t.v2, o);
  u.i1 = __shfl_xor_sync(0xffffffffu, t.i1, o);
  u.i2 = __shfl_xor_sync(0xffffffffu, t.i2, o);
  top2_merge(t, u);
}

static __device__ __noinline__ void head_finish(const Top2* partials, unsigned* ticket, int B, float cap, int32_t* idx,
                            float* top1, float* top2) {
  __shared__ bool last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = (int)(blockDim.x >> 5);
  const int n = (int)gridDim.x;
  for (int b = warp; b < B; b += nwarps) {
    Top2 t;
    top2_init(t);
    for (int c0 = lane; c0 < n; c0 += 128) {
      Top2 u[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = c0 + 32 * k;
        if (c < n)
          u[k] = load_cg(partials + (size_t)c * kMaxBatch + b);
        else
          top2_init(u[k]);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) top2_merge(t, u[k]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) top2_shfl_xor_merge(t, o);
    if (lane == 0) {
      idx[b] = t.i1;
      top1[b] = cap * tanhf(t.v1 / cap);
      top2[b] = cap * tanhf(t.v2 / cap);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) *ticket = 0u;
}

}  // namespace q4w
