// Streaming q4_0 GEMV engine: the fast path of the S=1 decode GEMV, of every
// decode-pass stage, of the b=1 LM head, and the persistent decode-pass kernel.
//
// Weights stream through shared memory: one producer thread issues 1-D bulk
// copies (cp.async.bulk, completion on an mbarrier) of contiguous row tiles
// (codes, then scales) into a ring of kSlots slots, with an L2 evict-first
// hint; kCW = 12 consumer warps dequantise and dot against x held in
// registers.  A row group of P lanes covers all K/32 blocks of a row, each
// lane up to three blocks (x of those blocks, 96 values, stays in registers
// for the whole stage); Gc = kCT/P groups take the rows of a tile in turn;
// P <= 32 reduces with shuffles, P > 32 through shared memory.  The per-row
// arithmetic (block order, bias trick, reduction tree) depends only on K, so
// every entry point produces the same bits for the same row.
//
// The decode pass runs as one cooperative launch: every CTA walks the same
// stage list; the producer runs ahead across stage boundaries (weights do
// not depend on activations).  Every stage output word carries the index of
// the stage that wrote it (relaxed gpu-scope stores of half | tag << 16 or
// float | tag << 32); the consumers of the next stage re-read their input
// words until all carry that index (no counters, no fences), apply the stage
// prologue and compute.  All waits are bounded in clock cycles; on expiry the
// CTA raises an abort flag (and a grid-wide one), every role leaves its loop,
// in-flight bulk copies are drained (bounded) and the kernel returns with the
// device error word set.
#include "q4w_device.cuh"
#include "q4w_internal.cuh"
#include "q4w_tc.cuh"
#include "q4w_top2.cuh"

namespace q4w {

namespace eng {

constexpr int kCW = 12;                   // consumer warps
constexpr int kCT = kCW * 32;             // consumer threads
constexpr int kTS = kCT + 32;             // threads per CTA
constexpr int kSlots = 3;
constexpr int kSlotBytes = 42 * 1024;
constexpr int kMaxNb = 384;               // K <= 12288 on this path
constexpr int kBPL = 3;                   // blocks per lane (upper bound)
constexpr int kXhStride = 20;             // uint32 per block: 16 half pairs, bias, 3 pad (80 B:
                                          // 8 lanes reading 8 consecutive blocks hit 8 bank groups)
constexpr size_t kXsBytes = (size_t)kMaxNb * kXhStride * sizeof(uint32_t);
constexpr size_t kSmemBytes = 128 + (size_t)kSlots * kSlotBytes + kXsBytes +
                              64 * sizeof(float) + 2 * kSlots * sizeof(uint64_t) + 64;
constexpr long long kDrainCycles = 2000000000LL;   // in-flight copies always land well within this

// ----------------------------------------------------------- primitives ---
// mbarriers, bulk copies, timers and cache policies: the shared building blocks
using tc::mbar_arrive;
using tc::mbar_expect_tx;
using tc::mbar_init;
using tc::mbar_probe;
using tc::mbar_test;
using tc::smem_u32;
__device__ __forceinline__ void bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Named barrier that also ANDs a predicate over its threads (uniform result).
__device__ __forceinline__ bool bar_and(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

struct Ctl {
  volatile int* abort_cta;   // shared
  int* abort_grid;           // global (decode pass) or nullptr
  long long limit;
  unsigned* err;             // the library's device error word
  unsigned long long* tr;    // trace stamps of the current stage (thread 0), or nullptr
  long long tr_c0;           // clock64() when the current stage began (trace only)
  bool trace_on;             // uniform: stamps are being taken (adds a barrier for stamp 1)
};

__device__ __forceinline__ void raise_abort(const Ctl& c) {
  *c.abort_cta = 1;
  atomicOr(c.err, 1u);
  if (c.abort_grid) atomicExch(c.abort_grid, 1);
}

__device__ __forceinline__ bool aborting(const Ctl& c) {
  return *c.abort_cta || (c.abort_grid && *(volatile int*)c.abort_grid);
}

// Bounded mbarrier wait; false on expiry (raises the abort) or when aborting.
// A retry suspends the thread in try_wait (up to kRetrySuspendNs, woken when
// the phase completes), so waiting warps do not poll.  The shared abort flag
// is read every iteration; the grid-wide flag (a global load, about an L2
// round trip) and the clock on the first retry and then every 256 (so a zero
// budget gives up at once).
constexpr uint32_t kRetrySuspendNs = 20000;
__device__ __forceinline__ bool mbar_wait(uint32_t a, uint32_t parity, const Ctl& c) {
  if (mbar_probe(a, parity)) return true;
  const long long t0 = clock64();
  for (unsigned it = 1;; ++it) {
    if (tc::mbar_test_for(a, parity, kRetrySuspendNs)) return true;
    if (*c.abort_cta) return false;
    if ((it & 255u) == 1) {   // first failed retry, then every 256
      if (c.abort_grid && *(volatile int*)c.abort_grid) return false;
      if (clock64() - t0 > c.limit) {
        raise_abort(c);
        return false;
      }
    }
  }
}

// Trace stamp: SM cycles since the current stage began.
__device__ __forceinline__ unsigned long long stamp(const Ctl& c) {
  return (unsigned long long)(clock64() - c.tr_c0);
}

// ------------------------------------------------------------- geometry ---
struct Geo {
  int K2, nb, P, Gc, R, T, total, lo, hi;
};

__device__ __forceinline__ int lanes_per_row(int nb) {
  int P = 1;
  while (P * kBPL < nb) P <<= 1;
  return P;
}

// Rows in flight per row group (R) and rows per tile (T = Gc * R when it
// fits a slot): two rows when every group gets at least two rows per CTA,
// so a tile has no idle row slots except at the end of a CTA's range.
__device__ __forceinline__ Geo make_geo(const StageArgs& a, int NM) {
  Geo g;
  g.K2 = a.K >> 1;
  g.nb = a.K >> 5;
  g.P = lanes_per_row(g.nb);
  g.Gc = kCT / g.P;
  g.total = a.pair ? a.mat[0].rows : a.mat[0].rows + (a.nmat > 1 ? a.mat[1].rows : 0) +
                                         (a.nmat > 2 ? a.mat[2].rows : 0);
  const int rpc = (g.total + gridDim.x - 1) / gridDim.x;
  g.lo = min(g.total, (int)blockIdx.x * rpc);
  g.hi = min(g.total, g.lo + rpc);
  const int row_bytes = NM * (g.K2 + g.nb * 2);
  const int fit = kSlotBytes / row_bytes;
  g.R = (rpc >= 2 * g.Gc && fit >= 2 * g.Gc) ? 2 : 1;
  g.T = g.Gc * g.R <= fit ? g.Gc * g.R : (fit < 1 ? 1 : fit);
  return g;
}

// Walk over this CTA's rows [lo, hi) of a stage, tile by tile: the next tile
// [r0, r0 + n) of matrix m (pair: of both matrices), at most T rows and never
// across a matrix boundary.  The boundaries are held in registers.
struct TileIter {
  int pos, hi, T, e0, e1, first_end;
  __device__ __forceinline__ TileIter(const StageArgs& a, const Geo& g) {
    pos = g.lo;
    hi = g.hi;
    T = g.T;
    const int r0 = a.mat[0].rows, r1 = a.mat[1].rows;
    const int nm = a.pair ? 1 : a.nmat;
    e0 = nm > 1 ? r0 : g.total;
    e1 = nm > 2 ? r0 + r1 : g.total;
    first_end = -1;
  }
  __device__ __forceinline__ bool next(int& m, int& r0, int& n) {
    if (pos >= hi) return false;
    m = (pos >= e0 ? 1 : 0) + (pos >= e1 ? 1 : 0);
    const int base = m == 0 ? 0 : (m == 1 ? e0 : e1);
    const int end = min(hi, m == 0 ? e0 : (m == 1 ? e1 : hi));
    r0 = pos - base;
    n = min(T, end - pos);
    pos += n;
    if (first_end < 0) first_end = pos;
    return true;
  }
  __device__ __forceinline__ bool first() const { return pos == first_end; }
};

// ------------------------------------------------------------- producer ---
// Issues the bulk copies of one stage's tiles; false when aborting.
template <int NM>
__device__ bool produce_stage(const StageArgs& a, uint32_t& gcount, uint32_t slots0, uint32_t full0,
                              uint32_t empty0, uint64_t policy, const Ctl& c) {
  const Geo g = make_geo(a, NM);
  TileIter it(a, g);
  int m, r0, n;
  while (it.next(m, r0, n)) {
    const uint32_t s = gcount % kSlots, round = gcount / kSlots;
    if (!mbar_wait(empty0 + 8 * s, (round & 1) ^ 1, c)) return false;
    const uint32_t per = (uint32_t)n * (g.K2 + g.nb * 2);
    mbar_expect_tx(full0 + 8 * s, NM * per);
    uint32_t dst = slots0 + s * kSlotBytes;
#pragma unroll
    for (int t = 0; t < NM; ++t) {
      const StageMat& M = a.mat[NM == 2 ? t : m];
      tc::bulk_load(dst, M.codes + (size_t)r0 * g.K2, (uint32_t)n * g.K2, full0 + 8 * s, policy);
      tc::bulk_load(dst + (uint32_t)n * g.K2, M.scales + (size_t)r0 * g.nb, (uint32_t)n * g.nb * 2, full0 + 8 * s,
               policy);
      dst += per;
    }
    ++gcount;
  }
  return true;
}

// After the producer stops: every issued copy has landed before the CTA exits.
__device__ void producer_drain(uint32_t gcount, uint32_t full0, unsigned* err) {
  const uint32_t first = gcount > (uint32_t)kSlots ? gcount - kSlots : 0u;
  for (uint32_t g = first; g < gcount; ++g) {
    const uint32_t s = g % kSlots, round = g / kSlots;
    const long long t0 = clock64();
    while (!mbar_test(full0 + 8 * s, round & 1)) {
      if (clock64() - t0 > kDrainCycles) {
        atomicOr(err, 1u);
        break;
      }
    }
  }
}

// ------------------------------------------------------------ consumers ---
__device__ __forceinline__ float consumer_sum(float v, float* red8) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  bar_sync(1, kCT);
  if (l == 0) red8[w] = v;
  bar_sync(1, kCT);
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < kCW; ++i) t += red8[i];
  return t;
}

__device__ __forceinline__ float load_in_cg(const void* in, int mode, int k) {
  if (mode == Q4_IN_F16 || mode == Q4_IN_RMS_F16)
    return __half2float(__ldcg(reinterpret_cast<const __half*>(in) + k));
  return __ldcg(reinterpret_cast<const float*>(in) + k);
}

// Sum over the consumer threads through red[0 .. kCW); every consumer gets it.
// The prologue gives each of its reductions its own red range, so one barrier
// suffices (the barrier that closed the previous user of red orders it).
__device__ __forceinline__ float consumer_sum1(float v, float* red) {
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  bar_sync(1, kCT);
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < kCW; ++i) t += red[i];
  return t;
}

// An fp32 input is staged in shared memory when it fits after the x words.
__host__ __device__ constexpr bool staged_f32(int K) {
  return (size_t)(K >> 5) * kXhStride * 4 + (size_t)K * 4 <= kXsBytes;
}

// x = prologue(in), written per 32-column block as the half pairs
// (x[8i+j], x[8i+j+4]) plus the bias of q4_block_dot_h (kXhStride words).
//
// Staged path (every fp16 input here, fp32 inputs up to K = 4096): the input
// is copied to shared memory with 16-byte loads from L2 -- for a tagged input
// (persistent pass) each element is re-read until it carries the expected
// stage tag, which is how a stage learns that its input is complete -- then
// the RMS factors, and each thread turns its chunks of eight elements into
// fp16 x, half pairs and block biases.  The staging lives inside the x
// buffer: an fp16 chunk is staged exactly where its four pair words go (the
// thread that converts a chunk is the only one reading or writing it), an
// fp32 input after the x words of this K.  Otherwise x is computed per pair
// straight from global memory.
__device__ __forceinline__ uint4 ldcg_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// Bounded re-read of one 16-byte group of tagged words until all tags match.
// Reads of tagged words are relaxed gpu-scope loads (and their writes relaxed
// gpu-scope stores): a plain load in a polling loop is a weak access the
// compiler may merge with an earlier read of the same address.  Half words
// are 32-bit elements, float words 64-bit elements, each read whole.
__device__ __forceinline__ uint4 ld_tagged(const uint4* p, bool f16) {
  uint4 r;
  if (f16) {
    asm volatile("ld.relaxed.gpu.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p)
                 : "memory");
  } else {
    unsigned long long a, b;
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0,%1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
    r = make_uint4((uint32_t)a, (uint32_t)(a >> 32), (uint32_t)b, (uint32_t)(b >> 32));
  }
  return r;
}
__device__ __forceinline__ void st_tagged32(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_tagged64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ bool tags_ready(const uint4& v, bool f16, uint32_t tag) {
  return f16 ? ((v.x >> 16) == tag && (v.y >> 16) == tag && (v.z >> 16) == tag && (v.w >> 16) == tag)
             : (v.y == tag && v.w == tag);
}

// u holds a read of p whose tags were not all current.
__device__ __forceinline__ bool poll_tags(const uint4* p, uint4& u, bool f16, uint32_t tag, const Ctl& c) {
  const long long t0 = clock64();
  for (unsigned it = 0;; ++it) {
    u = ld_tagged(p, f16);
    if (tags_ready(u, f16, tag)) return true;
    if ((it & 63u) == 0) {
      if (aborting(c)) return false;
      if (clock64() - t0 > c.limit) {
        raise_abort(c);
        return false;
      }
    }
  }
}

struct InVec {   // plain (untagged) input read from global memory
  const void* g;
  const uint8_t* s;
  int mode;
  __device__ __forceinline__ float operator()(int k) const { return load_in_cg(g, mode, k); }
};

__device__ __forceinline__ float xform(float v, int mode, float r, float r2) {
  if (mode == Q4_IN_F16) return v;
  const float t = f16_round(v * r);
  return mode == Q4_IN_RMS2_F32 ? f16_round(t * r2) : t;
}

// false when aborting (uniform over the consumers).  kDirect: an untagged
// fp16 input with no normalisation may be read straight from global memory
// (single-stage kernels; the persistent pass never has such an input).
// One staged 8-byte group -- four fp16 values packed as two half pairs, or
// two floats -- added into a sum of squares in one fixed order.  The tagged
// and the untagged staging both stage 8-byte groups v = tid, tid + kCT, ...
// per thread and add them here, so the persistent pass and the stage-by-stage
// launches form the same sums while the input is read.
__device__ __forceinline__ float group_sq(uint2 p, bool f16, float acc) {
  if (f16) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&p.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&p.y));
    acc = fmaf(a.x, a.x, acc);
    acc = fmaf(a.y, a.y, acc);
    acc = fmaf(b.x, b.x, acc);
    acc = fmaf(b.y, b.y, acc);
  } else {
    const float a = __uint_as_float(p.x), b = __uint_as_float(p.y);
    acc = fmaf(a, a, acc);
    acc = fmaf(b, b, acc);
  }
  return acc;
}

template <bool kDirect>
__device__ bool eng_prologue(const StageArgs& a, uint32_t* xh, float* red8, const Ctl& c) {
  const int tid = threadIdx.x, K = a.K, mode = a.in_mode;
  const bool f16in = mode == Q4_IN_F16 || mode == Q4_IN_RMS_F16;
  const bool staged = f16in || staged_f32(K);
  // fp32 staging: after this K's x words (16-byte aligned: 80 bytes per block)
  float* const st32 = reinterpret_cast<float*>(xh + (K >> 5) * kXhStride);
  // an fp16 chunk's home: the four pair words of its quarter of its block
  auto home16 = [&](int ch) { return xh + (ch >> 2) * kXhStride + 4 * (ch & 3); };
  // an untagged fp16 input with no normalisation is read once, so each
  // thread takes its 8-element chunks straight from global memory
  const bool direct = kDirect && a.in_tag == 0 && mode == Q4_IN_F16;
  float r = 1.f, r2 = 1.f;
  float ssq = 0.f;   // this thread's share of the sum of squares, formed while staging
  if (staged) {
    bool ok = true;
    if (a.in_tag == 0) {
      if (!direct) {
        uint2* dst32 = reinterpret_cast<uint2*>(st32);
        if (mode == Q4_IN_F16) {   // no sum of squares needed: 16-byte loads
          const uint4* src = reinterpret_cast<const uint4*>(a.in);
          for (int v = tid; v < K / 8; v += kCT) *reinterpret_cast<uint4*>(home16(v)) = ldcg_v4(src + v);
        } else {
          // 8-byte groups, as the tagged staging takes them
          const uint2* src = reinterpret_cast<const uint2*>(a.in);
          const int nv = f16in ? K / 4 : K / 2;
          for (int v = tid; v < nv; v += kCT) {
            uint2 g;
            asm volatile("ld.global.cg.v2.u32 {%0,%1}, [%2];" : "=r"(g.x), "=r"(g.y) : "l"(src + v));
            if (f16in)
              *reinterpret_cast<uint2*>(home16(v >> 1) + 2 * (v & 1)) = g;
            else
              dst32[v] = g;
            ssq = group_sq(g, f16in, ssq);
          }
        }
      }
    } else {
      // Tagged words: half | tag << 16 (four per 16 bytes) or float | tag << 32
      // (two per 16 bytes).  A thread issues all of its 16-byte reads at once
      // (one L2 round trip), then re-reads only groups whose tags are stale.
      const uint4* src = reinterpret_cast<const uint4*>(a.in);
      uint2* dst32 = reinterpret_cast<uint2*>(st32);
      const int nv = f16in ? K / 4 : K / 2;
      const uint32_t tag = (uint32_t)a.in_tag;
      constexpr int kPB = 4;
      for (int v0 = tid; v0 < nv && ok; v0 += kPB * kCT) {
        uint4 u[kPB];
#pragma unroll
        for (int i = 0; i < kPB; ++i)
          if (v0 + i * kCT < nv) u[i] = ld_tagged(src + v0 + i * kCT, f16in);
#pragma unroll
        for (int i = 0; i < kPB; ++i) {
          const int v = v0 + i * kCT;
          if (v < nv && ok) {
            if (!tags_ready(u[i], f16in, tag)) ok = poll_tags(src + v, u[i], f16in, tag, c);
            // fp16: group v is half (v & 1) of chunk v >> 1
            const uint2 g = f16in ? make_uint2(__byte_perm(u[i].x, u[i].y, 0x5410), __byte_perm(u[i].z, u[i].w, 0x5410))
                                  : make_uint2(u[i].x, u[i].z);
            if (f16in)
              *reinterpret_cast<uint2*>(home16(v >> 1) + 2 * (v & 1)) = g;
            else
              dst32[v] = g;
            ssq = group_sq(g, f16in, ssq);
          }
        }
      }
    }
    if (!direct && !bar_and(1, kCT, ok)) return false;
    if (c.tr) c.tr[1] = stamp(c);   // input complete and staged
    // Each thread takes chunks of eight consecutive elements (four chunks per
    // 32-column block): sums of squares for the RMS factors, then x, whose
    // half pairs (x[8i+j], x[8i+j+4]) lie within one chunk; the bias sums the
    // block's four chunks across adjacent lanes.
    const int nch = K >> 3;
    auto load8 = [&](int ch, float (&v)[8]) {
      if (f16in) {
        const uint4 u = direct ? ldcg_v4(reinterpret_cast<const uint4*>(a.in) + ch)
                               : *reinterpret_cast<const uint4*>(home16(ch));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
          v[2 * i] = f.x;
          v[2 * i + 1] = f.y;
        }
      } else {
        const float4 f0 = *reinterpret_cast<const float4*>(st32 + 8 * ch);
        const float4 f1 = *reinterpret_cast<const float4*>(st32 + 8 * ch + 4);
        v[0] = f0.x;
        v[1] = f0.y;
        v[2] = f0.z;
        v[3] = f0.w;
        v[4] = f1.x;
        v[5] = f1.y;
        v[6] = f1.z;
        v[7] = f1.w;
      }
    };
    if (mode != Q4_IN_F16) {
      const float ss = consumer_sum1(ssq, red8);
      r = 1.f / sqrtf(ss / (float)K + a.eps);
      if (mode == Q4_IN_RMS2_F32) {
        float ss2 = 0.f;
        for (int ch = tid; ch < nch; ch += kCT) {
          float v[8];
          load8(ch, v);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float t = f16_round(v[e] * r);
            ss2 += t * t;
          }
        }
        ss2 = consumer_sum1(ss2, red8 + 16);
        r2 = 1.f / sqrtf(ss2 / (float)K + a.eps);
      }
    }
    // K % 256 == 0 here, so every pass of this loop keeps whole warps active
    for (int ch = tid; ch < nch; ch += kCT) {
      float v[8];
      load8(ch, v);
      uint32_t hx[8];
      float pe = 0.f, po = 0.f;   // sums over the chunk's even / odd columns
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const __half x = __float2half_rn(xform(v[e], mode, r, r2));
        hx[e] = __half_as_ushort(x);
        if (e & 1)
          po += __half2float(x);
        else
          pe += __half2float(x);
      }
      const int blk = ch >> 2, i = ch & 3;
      *reinterpret_cast<uint4*>(home16(ch)) =
          make_uint4(hx[0] | (hx[4] << 16), hx[1] | (hx[5] << 16), hx[2] | (hx[6] << 16), hx[3] | (hx[7] << 16));
      pe += __shfl_xor_sync(0xffffffffu, pe, 1);
      po += __shfl_xor_sync(0xffffffffu, po, 1);
      pe += __shfl_xor_sync(0xffffffffu, pe, 2);
      po += __shfl_xor_sync(0xffffffffu, po, 2);
      if (i == 0) xh[blk * kXhStride + 16] = __float_as_uint(kBiasEven * pe + kBiasOdd * po);
    }
    bar_sync(1, kCT);
    return true;
  }
  // unstaged (large fp32 input, untagged only): per pair from global memory
  InVec in{a.in, nullptr, mode};
  if (mode != Q4_IN_F16) {
    float ss = 0.f;
    for (int k = tid; k < K; k += kCT) {
      const float v = in(k);
      ss += v * v;
    }
    ss = consumer_sum(ss, red8);
    r = 1.f / sqrtf(ss / (float)K + a.eps);
    if (mode == Q4_IN_RMS2_F32) {
      float ss2 = 0.f;
      for (int k = tid; k < K; k += kCT) {
        const float t = f16_round(in(k) * r);
        ss2 += t * t;
      }
      ss2 = consumer_sum(ss2, red8);
      r2 = 1.f / sqrtf(ss2 / (float)K + a.eps);
    }
  }
  const int npairs = (K >> 5) * 16;
  for (int idx = tid; idx < npairs; idx += kCT) {
    const int b = idx >> 4, pr = idx & 15, i = pr >> 2, j = pr & 3;
    const int k = 32 * b + 8 * i + j;
    const __half va = __float2half_rn(xform(in(k), mode, r, r2));
    const __half vc = __float2half_rn(xform(in(k + 4), mode, r, r2));
    xh[b * kXhStride + pr] = (uint32_t)__half_as_ushort(va) | ((uint32_t)__half_as_ushort(vc) << 16);
    // columns 8i+j and 8i+j+4 share the parity of j
    const float sum = __half2float(va) + __half2float(vc);
    float se = (j & 1) ? 0.f : sum, so = (j & 1) ? sum : 0.f;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
      se += __shfl_xor_sync(0xffffffffu, se, o);
      so += __shfl_xor_sync(0xffffffffu, so, o);
    }
    if (pr == 0) xh[b * kXhStride + 16] = __float_as_uint(kBiasEven * se + kBiasOdd * so);
  }
  bar_sync(1, kCT);
  return true;
}

__device__ __forceinline__ void load_xh(const uint32_t* xh, int blk, uint32_t (&v)[16], float& bias) {
  const uint4* p = reinterpret_cast<const uint4*>(xh + blk * kXhStride);
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint4 u = p[t];
    v[4 * t] = u.x;
    v[4 * t + 1] = u.y;
    v[4 * t + 2] = u.z;
    v[4 * t + 3] = u.w;
  }
  bias = __uint_as_float(xh[blk * kXhStride + 16]);
}

struct StageEpi {
  const StageArgs* a;
  template <int NM>
  __device__ __forceinline__ void operator()(int m, int row, const float (&acc)[NM]) const {
    const uint32_t tag = (uint32_t)a->out_tag;
    if (NM == 2) {
      const float gv = acc[0], uv = acc[NM - 1];
      if (a->mat[0].out32) a->mat[0].out32[row] = gv;
      if (a->mat[1].out32) a->mat[1].out32[row] = uv;
      const __half mh = __float2half_rn(gelu_tanh_f32(gv) * uv);
      if (a->mat[0].tagged)
        st_tagged32(reinterpret_cast<uint32_t*>(a->mat[0].out16) + row, (uint32_t)__half_as_ushort(mh) | (tag << 16));
      else
        a->mat[0].out16[row] = mh;
    } else {
      const StageMat& M = a->mat[m];
      if (M.tagged) {
        if (M.out32)
          st_tagged64(reinterpret_cast<unsigned long long*>(M.out32) + row,
                      (unsigned long long)__float_as_uint(acc[0]) | ((unsigned long long)tag << 32));
        if (M.out16)
          st_tagged32(reinterpret_cast<uint32_t*>(M.out16) + row,
                      (uint32_t)__half_as_ushort(__float2half_rn(acc[0])) | (tag << 16));
      } else {
        if (M.out32) M.out32[row] = acc[0];
        if (M.out16) M.out16[row] = __float2half_rn(acc[0]);
      }
    }
  }
};

struct HeadEpi {
  Top2* best;
  float* logits;
  float cap;
  template <int NM>
  __device__ __forceinline__ void operator()(int m, int row, const float (&acc)[NM]) const {
    (void)m;
    top2_insert(*best, acc[0], row);
    if (logits) logits[row] = cap * tanhf(acc[0] / cap);
  }
};

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ float lds_half(const uint8_t* p) {
  return __half2float(*reinterpret_cast<const __half*>(p));
}

// Fast consumer: P lanes per row, BPL blocks per lane, nb == P * BPL exactly.
// Rows are taken two at a time (independent chains); for P <= 32 the row
// loop is uniform across the warp so shuffles use the full mask.  The tile
// handshake is per warp (P <= 32) or per row group (P > 32); the stage result
// is made uniform over all consumers at the end.
template <int NM, int P, int BPL, int R, class Epi>
__device__ bool consume_fast(const StageArgs& a, const Geo& g, uint32_t& gcount, const uint8_t* slots,
                             uint32_t full0, uint32_t empty0, const uint32_t* xs, float* red, const Ctl& c,
                             const Epi& epi) {
  constexpr int Gc = kCT / P;
  constexpr int GW = P <= 32 ? 32 / P : 1;       // groups per warp
  constexpr int WPG = P > 32 ? P / 32 : 1;       // warps per group
  const int ct = threadIdx.x, lane = ct & 31, warp = ct >> 5;
  const int gid = ct / P, li = ct % P;
  uint32_t xr[BPL][16];
  float bias[BPL];
#pragma unroll
  for (int b = 0; b < BPL; ++b) load_xh(xs, li + P * b, xr[b], bias[b]);
  const int K2 = g.K2, nb = g.nb;
  const int row_first = P <= 32 ? warp * GW + lane / P : gid;   // this lane's first row of a tile
  if (c.tr && ct == 0) c.tr[3] = stamp(c);   // x in registers
  bool ok = true;
  TileIter it(a, g);
  int m, r0, n;
  while (it.next(m, r0, n)) {
    const uint32_t s = gcount % kSlots, round = gcount / kSlots;
    const bool early = c.tr && mbar_probe(full0 + 8 * s, round & 1);
    const bool landed = mbar_wait(full0 + 8 * s, round & 1, c);
    // first tile landed; bit 0 set when it had landed before the consumers asked
    if (c.tr && ct == 0 && it.first()) c.tr[5] = (stamp(c) << 1) | (early ? 1ull : 0ull);
    // every later tile: stamp 7 ends as the last tile's landing (bit 0: it had landed already)
    if (c.tr && ct == 0 && !it.first()) c.tr[7] = (stamp(c) << 1) | (early ? 1ull : 0ull);
    const bool all = (P <= 32) ? (__all_sync(0xffffffffu, landed) != 0) : bar_and(2 + gid, P, landed);
    if (!all) {
      ok = false;
      break;
    }
    if (c.tr && ct == 0 && it.first()) c.tr[6] = stamp(c);
    const uint8_t* S = slots + (size_t)s * kSlotBytes;
    const int per = n * (K2 + nb * 2);
    const uint8_t* sc_base = S + n * K2;
    // rows row_first + q * Gc (q < R); a partial last tile computes a clamped
    // copy of its last row in the idle slots and drops the result
    int rr[R];
    bool vv[R];
#pragma unroll
    for (int q = 0; q < R; ++q) {
      const int r = row_first + q * Gc;
      vv[q] = r < n;
      rr[q] = vv[q] ? r : n - 1;
    }
    float acc[R][NM];
#pragma unroll
    for (int q = 0; q < R; ++q)
#pragma unroll
      for (int t = 0; t < NM; ++t) acc[q][t] = 0.f;
#pragma unroll
    for (int b = 0; b < BPL; ++b) {
      const int j = li + P * b;
#pragma unroll
      for (int t = 0; t < NM; ++t) {
        uint4 cw[R];
        float d[R];
#pragma unroll
        for (int q = 0; q < R; ++q) {
          cw[q] = lds128(S + t * per + rr[q] * K2 + 16 * j);
          d[q] = lds_half(sc_base + t * per + (rr[q] * nb + j) * 2);
        }
#pragma unroll
        for (int q = 0; q < R; ++q) acc[q][t] = fmaf(d[q], q4_block_dot_h(cw[q], xr[b], bias[b]), acc[q][t]);
      }
    }
    if (P <= 32) {
#pragma unroll
      for (int q = 0; q < R; ++q)
#pragma unroll
        for (int t = 0; t < NM; ++t)
#pragma unroll
          for (int o = P / 2; o > 0; o >>= 1) acc[q][t] += __shfl_xor_sync(0xffffffffu, acc[q][t], o);
    } else {
      const int wig = warp - gid * WPG;
#pragma unroll
      for (int q = 0; q < R; ++q)
#pragma unroll
        for (int t = 0; t < NM; ++t) {
          acc[q][t] = warp_sum(acc[q][t]);
          if (lane == 0) red[((gid * WPG + wig) * R + q) * NM + t] = acc[q][t];
        }
      bar_sync(2 + gid, P);
      if (li == 0) {
#pragma unroll
        for (int q = 0; q < R; ++q)
#pragma unroll
          for (int t = 0; t < NM; ++t) {
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < WPG; ++w) v += red[((gid * WPG + w) * R + q) * NM + t];
            acc[q][t] = v;
          }
      }
      bar_sync(2 + gid, P);
    }
    if (li == 0) {
#pragma unroll
      for (int q = 0; q < R; ++q)
        if (vv[q]) epi.template operator()<NM>(m, r0 + rr[q], acc[q]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
    ++gcount;
  }
  return bar_and(1, kCT, ok);
}

// Generic consumer for any K % 256 == 0 up to kMaxNb blocks: runtime P,
// up to kBPL blocks per lane with masking, one row at a time.
template <int NM, class Epi>
__device__ bool consume_generic(const StageArgs& a, const Geo& g, uint32_t& gcount, const uint8_t* slots,
                                uint32_t full0, uint32_t empty0, const uint32_t* xs, float* red, const Ctl& c,
                                const Epi& epi) {
  const int ct = threadIdx.x, lane = ct & 31, warp = ct >> 5;
  const int P = g.P, Gc = g.Gc;
  const int gid = ct / P, li = ct % P;
  uint32_t xr[kBPL][16];
  float bias[kBPL];
#pragma unroll
  for (int b = 0; b < kBPL; ++b) {
    const int j = li + P * b;
    if (j < g.nb) {
      load_xh(xs, j, xr[b], bias[b]);
    } else {
#pragma unroll
      for (int t = 0; t < 16; ++t) xr[b][t] = 0u;
      bias[b] = 0.f;
    }
  }
  const int GW = P <= 32 ? 32 / P : 1, WPG = P > 32 ? P / 32 : 1;
  const int row_first = P <= 32 ? warp * GW : gid;
  const int row_lane = P <= 32 ? lane / P : 0;
  if (c.tr && ct == 0) c.tr[3] = stamp(c);   // x in registers
  bool ok = true;
  TileIter it(a, g);
  int m, r0, n;
  while (it.next(m, r0, n)) {
    const uint32_t s = gcount % kSlots, round = gcount / kSlots;
    const bool early = c.tr && mbar_probe(full0 + 8 * s, round & 1);
    const bool landed = mbar_wait(full0 + 8 * s, round & 1, c);
    if (c.tr && ct == 0 && it.first()) c.tr[5] = (stamp(c) << 1) | (early ? 1ull : 0ull);
    // every later tile: stamp 7 ends as the last tile's landing (bit 0: it had landed already)
    if (c.tr && ct == 0 && !it.first()) c.tr[7] = (stamp(c) << 1) | (early ? 1ull : 0ull);
    const bool all = (P <= 32) ? (__all_sync(0xffffffffu, landed) != 0) : bar_and(2 + gid, P, landed);
    if (!all) {
      ok = false;
      break;
    }
    if (c.tr && ct == 0 && it.first()) c.tr[6] = stamp(c);
    const uint8_t* S = slots + (size_t)s * kSlotBytes;
    const int per = n * (g.K2 + g.nb * 2);
    for (int rb = row_first; rb < n; rb += Gc) {
      const int r = rb + row_lane;
      const bool v = r < n;
      float acc[NM];
#pragma unroll
      for (int t = 0; t < NM; ++t) acc[t] = 0.f;
#pragma unroll
      for (int b = 0; b < kBPL; ++b) {
        const int j = li + P * b;
        if (v && j < g.nb) {
#pragma unroll
          for (int t = 0; t < NM; ++t) {
            const uint8_t* base = S + t * per;
            const uint4 cw = lds128(base + r * g.K2 + 16 * j);
            const float d = lds_half(base + n * g.K2 + (r * g.nb + j) * 2);
            acc[t] = fmaf(d, q4_block_dot_h(cw, xr[b], bias[b]), acc[t]);
          }
        }
      }
      if (P <= 32) {
#pragma unroll
        for (int t = 0; t < NM; ++t)
          for (int o = P >> 1; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
      } else {
        const int wig = warp - gid * WPG;
#pragma unroll
        for (int t = 0; t < NM; ++t) {
          acc[t] = warp_sum(acc[t]);
          if (lane == 0) red[(gid * WPG + wig) * NM + t] = acc[t];
        }
        bar_sync(2 + gid, P);
        if (li == 0) {
#pragma unroll
          for (int t = 0; t < NM; ++t) {
            float vv = 0.f;
            for (int w = 0; w < WPG; ++w) vv += red[(gid * WPG + w) * NM + t];
            acc[t] = vv;
          }
        }
        bar_sync(2 + gid, P);
      }
      if (li == 0 && v) epi.template operator()<NM>(m, r0 + r, acc);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
    ++gcount;
  }
  return bar_and(1, kCT, ok);
}

// Processes one stage's tiles; false when aborting (uniform over consumers).
// kPass: the persistent pass, which instantiates the fast consumer only for
// the (K, rows in flight) pairs of the E2B layer shapes (hidden 1536; q/o
// 2048 or 4096; MLP 6144 or 12288) -- fewer code paths in one kernel keep its
// register allocation free of spills; any other shape takes the generic
// consumer, which computes the same bits.
template <int NM, bool kPass, class Epi>
__device__ bool consume_stage(const StageArgs& a, const Geo& g, uint32_t& gcount, const uint8_t* slots,
                              uint32_t full0, uint32_t empty0, const uint32_t* xs, float* red, const Ctl& c,
                              const Epi& epi) {
#define Q4W_FAST(P, BPL)                                                                              \
  return g.R == 2 ? consume_fast<NM, P, BPL, 2>(a, g, gcount, slots, full0, empty0, xs, red, c, epi)  \
                  : consume_fast<NM, P, BPL, 1>(a, g, gcount, slots, full0, empty0, xs, red, c, epi)
#define Q4W_FAST_R(P, BPL, R) return consume_fast<NM, P, BPL, R>(a, g, gcount, slots, full0, empty0, xs, red, c, epi)
  if (g.T == g.Gc * g.R) {
    if (kPass) {
      if (NM == 2) {
        if (a.K == 1536 && g.R == 1) Q4W_FAST_R(16, 3, 1);
      } else {
        if (g.R == 1) {
          switch (a.K) {
            case 1536: Q4W_FAST_R(16, 3, 1);
            case 2048: Q4W_FAST_R(32, 2, 1);
            case 4096: Q4W_FAST_R(64, 2, 1);
            case 6144: Q4W_FAST_R(64, 3, 1);
            default: break;
          }
        } else if (a.K == 12288) {
          Q4W_FAST_R(128, 3, 2);
        }
      }
    } else {
      switch (a.K) {
        case 1536: Q4W_FAST(16, 3);
        case 2048: Q4W_FAST(32, 2);
        case 4096: Q4W_FAST(64, 2);
        case 6144: Q4W_FAST(64, 3);
        case 12288: Q4W_FAST(128, 3);
        default: break;
      }
    }
  }
#undef Q4W_FAST
#undef Q4W_FAST_R
  return consume_generic<NM>(a, g, gcount, slots, full0, empty0, xs, red, c, epi);
}

// ---------------------------------------------------------- shared memory ---
struct Smem {
  uint8_t* slots;
  uint32_t* xs;   // half pairs + bias per block
  float* red;
  uint32_t slots0, full0, empty0;
};

// Carves the dynamic shared memory (declared 1024-byte aligned) by offsets so
// that the compiler keeps shared-space loads.
__device__ __forceinline__ Smem carve(uint8_t* raw) {
  Smem s;
  size_t off = 0;
  s.slots = raw + off;
  off += (size_t)kSlots * kSlotBytes;
  s.xs = reinterpret_cast<uint32_t*>(raw + off);
  off += kXsBytes;
  s.red = reinterpret_cast<float*>(raw + off);
  off += 64 * sizeof(float);
  uint64_t* bars = reinterpret_cast<uint64_t*>(raw + off);
  s.slots0 = smem_u32(s.slots);
  s.full0 = smem_u32(bars);
  s.empty0 = smem_u32(bars + kSlots);
  return s;
}

__device__ __forceinline__ void init_barriers(const Smem& S) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(S.full0 + 8 * i, 1);
      mbar_init(S.empty0 + 8 * i, kCW);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
}

// ------------------------------------------------------- single stage ---
template <int NM>
__global__ void __launch_bounds__(kTS, 1) stage_stream_kernel(const StageArgs a, long long limit, unsigned* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ int abort_sh;
  const Smem S = carve(smem_raw);
  if (threadIdx.x == 0) abort_sh = 0;
  init_barriers(S);
  __syncthreads();
  pdl_trigger();
  const Ctl c{&abort_sh, nullptr, limit, err, nullptr};
  uint32_t gcount = 0;
  if (threadIdx.x >= kCT) {
    if (threadIdx.x == kCT) {
      const uint64_t pol = tc::policy_evict_first();
      if (!a.weights_early) pdl_wait();
      produce_stage<NM>(a, gcount, S.slots0, S.full0, S.empty0, pol, c);
      producer_drain(gcount, S.full0, c.err);
    }
    __syncwarp();
  } else {
    pdl_wait();
    if (eng_prologue<true>(a, S.xs, S.red, c)) {
      StageEpi epi{&a};
      consume_stage<NM, false>(a, make_geo(a, NM), gcount, S.slots, S.full0, S.empty0, S.xs, S.red, c, epi);
    }
  }
  __syncthreads();
}

// ----------------------------------------------------------- LM head b=1 ---
__global__ void __launch_bounds__(kTS, 1) head_stream_kernel(const StageArgs a, float cap, float* logits,
                                                            Top2* partials, unsigned* ticket, int32_t* idx,
                                                            float* top1, float* top2, long long limit, unsigned* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ int abort_sh;
  __shared__ Top2 st[kTS / 32];
  const Smem S = carve(smem_raw);
  if (threadIdx.x == 0) abort_sh = 0;
  init_barriers(S);
  __syncthreads();
  const Ctl c{&abort_sh, nullptr, limit, err, nullptr};
  uint32_t gcount = 0;
  Top2 best;
  top2_init(best);
  if (threadIdx.x >= kCT) {
    if (threadIdx.x == kCT) {
      const uint64_t pol = tc::policy_evict_first();
      produce_stage<1>(a, gcount, S.slots0, S.full0, S.empty0, pol, c);
      producer_drain(gcount, S.full0, c.err);
    }
    __syncwarp();
  } else {
    if (eng_prologue<true>(a, S.xs, S.red, c)) {
      HeadEpi epi{&best, logits, cap};
      consume_stage<1, false>(a, make_geo(a, 1), gcount, S.slots, S.full0, S.empty0, S.xs, S.red, c, epi);
    }
  }
  // the CTA's record: shuffle merges within each warp, then across the warps
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) top2_shfl_xor_merge(best, o);
  if (lane == 0) st[warp] = best;
  __syncthreads();
  if (warp == 0) {
    Top2 t;
    if (lane < kTS / 32)
      t = st[lane];
    else
      top2_init(t);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) top2_shfl_xor_merge(t, o);
    if (lane == 0) partials[(size_t)blockIdx.x * kMaxBatch] = t;
  }
  head_finish(partials, ticket, 1, cap, idx, top1, top2);
}

// --------------------------------------------------------- decode pass ---
constexpr int kMaxMegaLayers = 48;

struct MegaLayer {
  const uint8_t* codes[7];      // q, k, v, o, gate, up, down
  const __half* scales[7];
  int q_rows, kv_rows, mlp_rows;
};

struct MegaArgs {
  MegaLayer L[kMaxMegaLayers];
  int n_layers, H;
  float eps;
  const __half* h0;
  __half* h_out;
  float* kv32;                  // k and v outputs (plain: nothing in the pass reads them)
  uint32_t* q16t;               // stage outputs, each word carrying its stage tag;
  unsigned long long* o32t;     // all zeroed before every launch
  uint32_t* m16t;
  unsigned long long* y32t;
  int* abort_grid;              // zeroed before the launch
  long long limit;
  unsigned* err;
  unsigned long long* trace;    // optional: [4 * n_layers][gridDim.x][8] globaltimer stamps
};

// Stage s of the pass as StageArgs (the same stages the launch path issues).
// Stage s tags its outputs s + 1; its input is complete once every element
// carries tag s (stage 0 reads the untagged h0).
__device__ __forceinline__ StageArgs mega_stage(const MegaArgs& A, const MegaLayer* Ls, int s) {
  const MegaLayer& L = Ls[s >> 2];
  StageArgs a = {};
  a.eps = A.eps;
  a.in_tag = s;
  a.out_tag = s + 1;
  switch (s & 3) {
    case 0:
      a.mat[0] = {L.codes[0], L.scales[0], L.q_rows, nullptr, reinterpret_cast<__half*>(A.q16t), 1};
      a.nmat = 1;
      if (L.kv_rows > 0) {
        a.mat[1] = {L.codes[1], L.scales[1], L.kv_rows, A.kv32, nullptr, 0};
        a.mat[2] = {L.codes[2], L.scales[2], L.kv_rows, A.kv32 + L.kv_rows, nullptr, 0};
        a.nmat = 3;
      }
      a.K = A.H;
      a.in = (s == 0) ? static_cast<const void*>(A.h0) : static_cast<const void*>(A.y32t);
      a.in_mode = (s == 0) ? Q4_IN_RMS_F16 : Q4_IN_RMS2_F32;
      break;
    case 1:
      a.mat[0] = {L.codes[3], L.scales[3], A.H, reinterpret_cast<float*>(A.o32t), nullptr, 1};
      a.nmat = 1;
      a.K = L.q_rows;
      a.in = A.q16t;
      a.in_mode = Q4_IN_F16;
      break;
    case 2:
      a.mat[0] = {L.codes[4], L.scales[4], L.mlp_rows, nullptr, reinterpret_cast<__half*>(A.m16t), 1};
      a.mat[1] = {L.codes[5], L.scales[5], L.mlp_rows, nullptr, nullptr, 0};
      a.nmat = 2;
      a.pair = 1;
      a.K = A.H;
      a.in = A.o32t;
      a.in_mode = Q4_IN_RMS_F32;
      break;
    default:
      a.mat[0] = {L.codes[6], L.scales[6], A.H, reinterpret_cast<float*>(A.y32t), nullptr, 1};
      a.nmat = 1;
      a.K = L.mlp_rows;
      a.in = A.m16t;
      a.in_mode = Q4_IN_F16;
      break;
  }
  return a;
}

__global__ void __launch_bounds__(kTS, 1) decode_pass_kernel(const __grid_constant__ MegaArgs A) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ int abort_sh;
  // layer descriptors copied once from the parameter space: a stage reads its
  // descriptor from shared memory instead of through the constant caches
  __shared__ __align__(16) MegaLayer Ls[kMaxMegaLayers];
  // Stage descriptors live in shared memory: as per-thread values they would
  // sit in local memory (the matrix array is indexed at run time), hundreds
  // of KB per CTA that the small L1 left beside the shared carve-out cannot
  // hold.  sa[s & 1] is stage s for the consumers (thread 0 fills the next
  // one while a stage runs); sp is the producer's.
  __shared__ __align__(16) StageArgs sa[2];
  __shared__ __align__(16) StageArgs sp;
  __shared__ Geo sg[2];   // the consumers' tile geometry of sa[0], sa[1]
  const Smem S = carve(smem_raw);
  if (threadIdx.x == 0) abort_sh = 0;
  init_barriers(S);
  {
    constexpr int kWords = (int)(sizeof(MegaLayer) / sizeof(uint32_t));
    const uint32_t* src = reinterpret_cast<const uint32_t*>(A.L);
    uint32_t* dst = reinterpret_cast<uint32_t*>(Ls);
    for (int i = threadIdx.x; i < A.n_layers * kWords; i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    sa[0] = mega_stage(A, Ls, 0);
    sg[0] = make_geo(sa[0], sa[0].pair ? 2 : 1);
  }
  __syncthreads();
  Ctl c{&abort_sh, A.abort_grid, A.limit, A.err, nullptr, 0, A.trace != nullptr};
  const int nst = 4 * A.n_layers;
  uint32_t gcount = 0;
  if (threadIdx.x >= kCT) {
    if (threadIdx.x == kCT) {
      const uint64_t pol = tc::policy_evict_first();
      for (int s = 0; s < nst; ++s) {
        sp = mega_stage(A, Ls, s);
        const StageArgs& a = sp;
        const bool ok = a.pair ? produce_stage<2>(a, gcount, S.slots0, S.full0, S.empty0, pol, c)
                               : produce_stage<1>(a, gcount, S.slots0, S.full0, S.empty0, pol, c);
        if (!ok) break;
      }
      producer_drain(gcount, S.full0, c.err);
    }
    __syncwarp();
  } else {
    bool ok = true;
    for (int s = 0; s < nst && ok; ++s) {
      unsigned long long* tr = nullptr;
      if (A.trace && threadIdx.x == 0) {
        tr = A.trace + ((size_t)s * gridDim.x + blockIdx.x) * 8;
        tr[0] = tc::globaltimer();
        c.tr_c0 = clock64();
      }
      c.tr = tr;
      // every consumer finished stage s - 1 (the barrier closing its rows), so
      // the slot of stage s + 1 is free; the barrier closing stage s publishes it
      if (threadIdx.x == 0 && s + 1 < nst) {
        StageArgs& nx = sa[(s + 1) & 1];
        nx = mega_stage(A, Ls, s + 1);
        sg[(s + 1) & 1] = make_geo(nx, nx.pair ? 2 : 1);
      }
      const StageArgs& a = sa[s & 1];
      if (tr) tr[7] = 0;
      // the prologue waits (bounded) until its whole input carries tag s
      ok = eng_prologue<false>(a, S.xs, S.red, c);
      if (!ok) break;
      if (tr) tr[2] = stamp(c);
      StageEpi epi{&a};
      const Geo& g = sg[s & 1];
      ok = a.pair ? consume_stage<2, true>(a, g, gcount, S.slots, S.full0, S.empty0, S.xs, S.red, c, epi)
                  : consume_stage<1, true>(a, g, gcount, S.slots, S.full0, S.empty0, S.xs, S.red, c, epi);
      if (tr) tr[4] = stamp(c);
    }
    // closing RMSNorm of the last down-projection output (tag nst), by CTA 0,
    // with the summation order of q4_rmsnorm_f16 (256 partial sums)
    if (ok && blockIdx.x == 0) {
      const int H = A.H;
      float* sf = reinterpret_cast<float*>(S.slots);   // the ring is idle once the last stage is done
      bool ok2 = true;
      for (int v = threadIdx.x; v < H / 2 && ok2; v += kCT) {
        const uint4* p = reinterpret_cast<const uint4*>(A.y32t) + v;
        uint4 u = ld_tagged(p, false);
        if (!tags_ready(u, false, (uint32_t)nst)) ok2 = poll_tags(p, u, false, (uint32_t)nst, c);
        sf[2 * v] = __uint_as_float(u.x);
        sf[2 * v + 1] = __uint_as_float(u.z);
      }
      if (bar_and(1, kCT, ok2)) {
        float ss = 0.f;
        for (int k = threadIdx.x; k < H; k += kCT) ss += sf[k] * sf[k];
        ss = consumer_sum(ss, S.red);
        const float r = 1.f / sqrtf(ss / (float)H + A.eps);
        for (int k = threadIdx.x; k < H; k += kCT) A.h_out[k] = __float2half_rn(sf[k] * r);
      }
    }
  }
  __syncthreads();
}

}  // namespace eng

// ------------------------------------------------------------- launchers ---
bool stream_eligible(int K) { return K % 256 == 0 && (K >> 5) <= eng::kMaxNb; }

static cudaError_t set_smem(const void* fn) {
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)eng::kSmemBytes);
}

int launch_stage_stream(const StageArgs& a, const DeviceInfo& dev, cudaStream_t s, bool pdl) {
  static PerDevice attr;
  cudaError_t e;
  if (!attr.get(dev.ordinal)) {
    if ((e = set_smem((const void*)eng::stage_stream_kernel<1>)) != cudaSuccess ||
        (e = set_smem((const void*)eng::stage_stream_kernel<2>)) != cudaSuccess)
      return cuda_fail(e, "stream stage smem attribute");
    attr.set(dev.ordinal);
  }
  int total = a.pair ? a.mat[0].rows : 0;
  if (!a.pair)
    for (int i = 0; i < a.nmat; ++i) total += a.mat[i].rows;
  const int K2 = a.K >> 1, nb = a.K >> 5;
  const int rows_per_tile = eng::kSlotBytes / ((a.pair ? 2 : 1) * (K2 + nb * 2));
  int grid = (total + rows_per_tile - 1) / rows_per_tile;
  if (grid < dev.sms) grid = total < dev.sms ? total : dev.sms;
  if (grid > dev.sms) grid = dev.sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(eng::kTS);
  cfg.dynamicSmemBytes = eng::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr1[1];
  attr1[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr1[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr1;
  cfg.numAttrs = pdl ? 1 : 0;
  const long long lim = wait_limit();
  unsigned* err = device_error_word();
  if (!err) return fail(Q4_ERR_CUDA, "device error word unavailable");
  e = a.pair ? cudaLaunchKernelEx(&cfg, eng::stage_stream_kernel<2>, a, lim, err)
             : cudaLaunchKernelEx(&cfg, eng::stage_stream_kernel<1>, a, lim, err);
  return e == cudaSuccess ? Q4_OK : cuda_fail(e, "stream stage launch");
}

int launch_head_stream(const uint8_t* codes, const __half* scales, const __half* h, int V, int K, float cap,
                       int32_t* idx, float* top1, float* top2, float* logits, void* ws, const DeviceInfo& dev,
                       cudaStream_t s) {
  static PerDevice attr;
  cudaError_t e;
  if (!attr.get(dev.ordinal)) {
    if ((e = set_smem((const void*)eng::head_stream_kernel)) != cudaSuccess)
      return cuda_fail(e, "stream head smem attribute");
    attr.set(dev.ordinal);
  }
  unsigned* ticket = reinterpret_cast<unsigned*>(ws);
  Top2* partials = reinterpret_cast<Top2*>(reinterpret_cast<char*>(ws) + kTicketBytes);
  e = cudaMemsetAsync(ticket, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return cuda_fail(e, "lmhead ticket reset");
  StageArgs a = {};
  a.mat[0] = {codes, scales, V, nullptr, nullptr};
  a.nmat = 1;
  a.K = K;
  a.in = h;
  a.in_mode = Q4_IN_F16;
  unsigned* err = device_error_word();
  if (!err) return fail(Q4_ERR_CUDA, "device error word unavailable");
  const int grid = V < dev.sms ? V : dev.sms;
  eng::head_stream_kernel<<<grid, eng::kTS, eng::kSmemBytes, s>>>(a, cap, logits, partials, ticket, idx, top1,
                                                                  top2, wait_limit(), err);
  e = cudaGetLastError();
  return e == cudaSuccess ? Q4_OK : cuda_fail(e, "stream head launch");
}

static void* g_trace_buf = nullptr;
static size_t g_trace_bytes = 0;

void* trace_buffer(size_t* bytes) {
  *bytes = g_trace_bytes;
  return g_trace_buf;
}

size_t decode_ctl_bytes() { return 256; }

int launch_decode_pass_stream(const q4_layer* layers, int n_layers, int H, const __half* h0, __half* h_out,
                              float eps, float* kv32, void* tagged, size_t tagged_bytes, int* ctl,
                              const DeviceInfo& dev, cudaStream_t s) {
  if (n_layers > eng::kMaxMegaLayers) return fail(Q4_ERR_SHAPE, "persistent pass holds at most %d layers",
                                                  eng::kMaxMegaLayers);
  static PerDevice attr;
  cudaError_t e;
  if (!attr.get(dev.ordinal)) {
    if ((e = set_smem((const void*)eng::decode_pass_kernel)) != cudaSuccess)
      return cuda_fail(e, "decode pass smem attribute");
    attr.set(dev.ordinal);
  }
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, eng::decode_pass_kernel, eng::kTS, eng::kSmemBytes);
  if (e != cudaSuccess) return cuda_fail(e, "decode pass occupancy");
  if (per_sm < 1) return fail(Q4_ERR_CUDA, "decode pass kernel does not fit on an SM");
  static eng::MegaArgs A;   // host staging of the kernel parameter
  memset(&A, 0, sizeof(A));
  int max_qkv = 0, max_mlp = 0;
  for (int l = 0; l < n_layers; ++l) {
    const q4_layer& L = layers[l];
    const q4_matrix* m[7] = {&L.q, &L.k, &L.v, &L.o, &L.gate, &L.up, &L.down};
    for (int i = 0; i < 7; ++i) {
      A.L[l].codes[i] = m[i]->codes;
      A.L[l].scales[i] = reinterpret_cast<const __half*>(m[i]->scales);
    }
    A.L[l].q_rows = L.q_rows;
    A.L[l].kv_rows = L.kv_rows;
    A.L[l].mlp_rows = L.mlp_rows;
    if (L.q_rows + 2 * L.kv_rows > max_qkv) max_qkv = L.q_rows + 2 * L.kv_rows;
    if (L.mlp_rows > max_mlp) max_mlp = L.mlp_rows;
  }
  // tagged regions, in this order: q [QKV] x 4 B, o [H] x 8 B, m [I] x 4 B, y [H] x 8 B
  auto up = [](size_t n) { return (n + 255) & ~(size_t)255; };
  char* p = static_cast<char*>(tagged);
  A.q16t = reinterpret_cast<uint32_t*>(p);
  p += up((size_t)max_qkv * 4);
  A.o32t = reinterpret_cast<unsigned long long*>(p);
  p += up((size_t)H * 8);
  A.m16t = reinterpret_cast<uint32_t*>(p);
  p += up((size_t)max_mlp * 4);
  A.y32t = reinterpret_cast<unsigned long long*>(p);
  p += up((size_t)H * 8);
  if ((size_t)(p - static_cast<char*>(tagged)) > tagged_bytes)
    return fail(Q4_ERR_WORKSPACE, "tagged stage buffers need %zu bytes", (size_t)(p - static_cast<char*>(tagged)));
  A.n_layers = n_layers;
  A.H = H;
  A.eps = eps;
  A.h0 = h0;
  A.h_out = h_out;
  A.kv32 = kv32;
  A.abort_grid = ctl;
  A.limit = wait_limit();
  A.trace = static_cast<unsigned long long*>(g_trace_buf);
  if (A.trace && g_trace_bytes < (size_t)4 * n_layers * dev.sms * 8 * sizeof(unsigned long long))
    return fail(Q4_ERR_WORKSPACE, "trace buffer too small for %d layers", n_layers);
  A.err = device_error_word();
  if (!A.err) return fail(Q4_ERR_CUDA, "device error word unavailable");
  // every tag (and the abort word) back to 0 before the pass
  e = cudaMemsetAsync(tagged, 0, tagged_bytes, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(ctl, 0, decode_ctl_bytes(), s);
  if (e != cudaSuccess) return cuda_fail(e, "decode pass tag reset");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(dev.sms);
  cfg.blockDim = dim3(eng::kTS);
  cfg.dynamicSmemBytes = eng::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, eng::decode_pass_kernel, A);
  return e == cudaSuccess ? Q4_OK : cuda_fail(e, "decode pass launch");
}

}  // namespace q4w

extern "C" int q4_set_trace(void* buf, size_t bytes) {
  q4w::g_trace_buf = buf;
  q4w::g_trace_bytes = buf ? bytes : 0;
  return Q4_OK;
}
