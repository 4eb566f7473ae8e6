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

// Second level: runs in the CTA that finishes last.
static __device__ __noinline__ void head_finish(const Top2* partials, unsigned* ticket, int B, float cap, int32_t* idx,
                            float* top1, float* top2) {
  __shared__ bool last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (threadIdx.x < B) {
    const int b = threadIdx.x;
    Top2 t;
    top2_init(t);
    for (int c = 0; c < (int)gridDim.x; ++c) top2_merge(t, load_cg(partials + (size_t)c * kMaxBatch + b));
    idx[b] = t.i1;
    top1[b] = cap * tanhf(t.v1 / cap);
    top2[b] = cap * tanhf(t.v2 / cap);
  }
  __syncthreads();
  if (threadIdx.x == 0) *ticket = 0u;
}

}  // namespace q4w
