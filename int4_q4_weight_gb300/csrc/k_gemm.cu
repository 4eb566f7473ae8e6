// S=64 chunked-prefill dequant-GEMM on the 5th-generation tensor cores.
//
// "visible-cx/gemma-4-E2B-CoreAI", Provenance / Performance: the prefill
// entry point has a static query width of 64 and serves full-width chunks.
// Y[t][n] = sum_k bf16(scale*(code-8))[n][k] * bf16(x[t][k]), fp32 accumulate.
//
// Swap-AB: the weight tile is the M=128 operand (A, dequantised by the
// converter warps straight into tensor memory), the 64 tokens are the N=64
// operand (B, in shared memory), the accumulator D[128][64] (fp32) lives in
// tensor memory.  With A in tensor memory the shared-memory port carries only
// the raw codes and the token tiles.  One CTA per SM, persistent over work
// items (a 128-row tile and a range of 64-column K chunks; K is split across
// CTAs when there are fewer tiles than SMs, the splits then add into Y).
//
// Warp roles (768 threads):
//   warps 0-3   epilogue: tcgen05.ld of their TMEM lane quarter (both
//               issuers' accumulators, added), store to Y; in the LM-head
//               form (16 tokens, fp16 tiles) no Y: each thread keeps the best
//               two (z, row) per token over its rows, the warps merge them at
//               the end, and the CTA that finishes last merges every CTA's
//               record (tanh(z/cap)*cap written only when the caller asks for
//               the logits)
//   warps 4-19  converters, four groups of one warp per TMEM lane quarter
//               (the only lanes a warp's scheduler may access); consecutive
//               chunks go to consecutive groups.  Raw codes + scales from the
//               raw ring, nibble -> bf16 d*(q-8) rounded once (or fp16 for the
//               head form); a thread owns a tile row (TMEM lane) and writes
//               the chunk's 128 columns of it as two tcgen05.st of 32 columns
//   warps 20-21 MMA issuers (20 also allocates TMEM): one elected lane each
//               issues half of every chunk's 8 MMAs (A from tensor memory)
//               into its own accumulator, and commits.  An MMA takes ~65
//               cycles of its issuing thread, so one issuer alone capped the
//               kernel at ~0.5 us per chunk
//   warp 22     raw-ring TMA loads (one elected lane issues)
//   warp 23     token tile (B) of each operand stage: one bulk copy from the
//               bf16 copy of X, completing on the stage's full barrier
// X is rounded to bf16 once per call by a small kernel ahead of the GEMM (in
// the caller's workspace) instead of once per tile and chunk.  The raw ring
// (kRawStages x 256 K columns: codes 16 KB + scales 2 KB) keeps weight bytes
// in flight; the operand stages (kStages x (A: 64 TMEM columns, B: 16 KB of
// shared memory), 128 K columns each) feed the tensor cores.  full counts the
// chunk's converter group and the B loader (with its bytes), so an MMA issuer
// waits on one barrier per stage.
// Two items' accumulators (2 issuers x 2 x N columns) let the epilogue of
// one item overlap the MMAs of the next.  Every mbarrier wait is bounded in
// clock cycles; on expiry the CTA raises an abort flag, every role leaves its
// loop, each MMA issuer drains its own tcgen05 work (bounded again), TMEM is
// freed and the kernel returns with the device error word set.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "q4w_device.cuh"
#include "q4w_internal.cuh"
#include "q4w_tc.cuh"
#include "q4w_top2.cuh"

namespace q4w {

__device__ unsigned int g_device_error = 0;   // bit 0: a bounded wait ran out

// Device address of g_device_error for the current device (kernels in other
// translation units receive it as an argument).  Queried once per device.
unsigned* device_error_word() {
  static unsigned* cache[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<unsigned*>(p);
  }
  return cache[dev];
}

namespace gemm {

constexpr int kStages = 4;
constexpr int kRawStages = 8;
constexpr int kRawChunks = 2;          // operand chunks per raw stage (256 K columns)
constexpr int kTileM = 128;            // weight rows per tile (MMA M)
constexpr int kTok = 64;               // tokens of the prefill GEMM (MMA N)
constexpr int kChunk = 128;            // K columns per operand stage (8 MMAs of K = 16)
// A operand stages in tensor memory: 128 lanes (tile rows) x 64 columns (128
// 16-bit weights of a chunk, two per 32-bit column, K order)
constexpr int kACols = kChunk / 2;
// per token count N (the MMA N): token tile bytes per stage (the only operand
// in shared memory), the first TMEM column of the A stages (after two items'
// accumulators, one per MMA issuer) and the TMEM columns allocated (a power
// of two)
__host__ __device__ constexpr int b_bytes(int n) { return n * kChunk * 2; }
__host__ __device__ constexpr int stage_bytes(int n) { return b_bytes(n); }
__host__ __device__ constexpr int a_col0(int n) { return 4 * n < 32 ? 32 : 4 * n; }
__host__ __device__ constexpr int tmem_cols(int n) {
  return a_col0(n) + kStages * kACols <= 256 ? 256 : 512;
}
constexpr int kRawCodeBytes = kTileM * kChunk * kRawChunks / 2;   // 16 KB: [128 rows][128 B]
constexpr int kRawScaleBytes = kTileM * 16;                         // 2 KB: [128 rows][8 fp16]
constexpr int kRawBytes = kRawCodeBytes + kRawScaleBytes;
constexpr int kEpiWarps = 4, kProdWarps = 16;
// The converter warps form kGroups groups of one warp per lane quarter;
// consecutive chunks go to consecutive groups (chunk j of raw stage gr to
// group kRawChunks (gr % kStageSets) + j), so kGroups chunks are converted
// concurrently.
constexpr int kGroups = 4;
constexpr int kStageSets = kGroups / kRawChunks;       // raw stages per round of the groups
constexpr int kGroupWarps = kProdWarps / kGroups;      // 4: one per lane quarter
constexpr int kBPW = 16 / kGroupWarps;                 // 32-column blocks of a chunk per converter warp: 4
static_assert(kGroups % kRawChunks == 0 && kGroupWarps == 4, "one warp per lane quarter in a group");
constexpr int kIssuers = 2;                        // MMA-issuing warps, one accumulator each
constexpr int kMmaWarp = kEpiWarps + kProdWarps;   // 20, 21 (20 also allocates TMEM)
constexpr int kTmaWarp = kMmaWarp + kIssuers;      // 22
constexpr int kBWarp = kTmaWarp + 1;               // 23
constexpr int kThreadsG = (kBWarp + 1) * 32;       // 768
constexpr int kBars = 2 * kStages + 2 * kRawStages + 6;
static_assert(kBars <= 32, "one barrier per lane of warp 0");
// The LM-head form keeps the whole token operand (K / 8 column groups x 16
// tokens x 16 B = 32 K bytes) resident in shared memory, loaded once, instead
// of a ring of token tiles: no token-tile fetch sits between one chunk's MMAs
// and the next.
__host__ __device__ constexpr size_t xres_bytes(int K) { return ((size_t)K * 32 + 1023) & ~(size_t)1023; }
__host__ __device__ constexpr size_t operand_bytes(int n, bool head, int K) {
  return head ? xres_bytes(K) : (size_t)kStages * stage_bytes(n);
}
__host__ __device__ constexpr size_t smem_bytes(int n, bool head, int K) {   // dynamic shared memory
  return 1024 + operand_bytes(n, head, K) + (size_t)kRawStages * kRawBytes + kBars * 8;
}
// dynamic plus static shared memory (the LM-head records) within the 227 KB
// a CTA may hold
static_assert(smem_bytes(kTok, false, 0) + 1024 <= 232448, "shared memory");
constexpr size_t kSmemMax = 232448;   // dynamic plus static shared memory of a CTA
constexpr long long kDrainCycles = 2000000000LL;
constexpr long long kShortDrainCycles = 4000000LL;   // aborting: copies in flight land well within this

using tc::elect_one;

// Instruction descriptor, kind::f16: D f32, A and B bf16 (format 1) or fp16
// (format 0), both K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc(int n, bool f16) {
  return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(kTileM >> 4) << 24);
}

// Shared-memory matrix descriptor, no swizzle: 8x(16 B) core matrices;
// lbo = byte step between core matrices along K, sbo = along M/N.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
         ((uint64_t)(sbo >> 4) << 32) | (1ull << 46);
}

// The shared building blocks (q4w_tc.cuh) under the names this file uses;
// its bounded waits report to the library's device error word.
using tc::fence_proxy_async;
using tc::mbar_arrive;
using tc::mbar_expect_tx;
using tc::mbar_init;
using tc::mbar_test;
using tc::smem_u32;
using tc::tmem_ld16;
using tc::tmem_st32;

// Bounded wait.  Returns false when the wait ran out or the CTA is aborting.
// Waiting warps are suspended in the barrier wait (no polling), so the roles
// that wait most (MMA issuer, loaders, epilogue) take no issue slots from the
// converter warps on their schedulers.
__device__ __forceinline__ bool mbar_wait(uint32_t a, uint32_t parity, long long limit,
                                          volatile int* abort_flag) {
  return tc::mbar_wait(a, parity, limit, abort_flag, &g_device_error);
}
__device__ __forceinline__ void tc_fence_before() { tc::fence_before(); }
__device__ __forceinline__ void tc_fence_after() { tc::fence_after(); }
__device__ __forceinline__ void tc_commit(uint32_t mbar) { tc::commit(mbar); }
// D (+)= A . B with A in tensor memory (128 lanes x 8 columns per K = 16).
__device__ __forceinline__ void tc_mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t id,
                                          uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(id), "r"(accum)
      : "memory");
}

__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Column order inside every group of 8 K columns, both operands: slot s of
// the group holds column kSlotCol[s].  A 32-bit word of codes holds columns
// 0..7 as nibbles; one masked LOP3 takes the nibbles of columns c and c + 4
// (bits 4c and 4c + 16) into the two halves of a register, so the decoded
// pairs come out as (0,4), (1,5), (2,6), (3,7).  The token operand is laid
// out in the same order instead of permuting the weights back.
//   slot:    0 1 2 3 4 5 6 7
//   column:  0 4 1 5 2 6 3 7

// bf16x2 arithmetic (round to nearest even; fma rounds once)
__device__ __forceinline__ uint32_t bsub2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t bfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// The scale d (an fp16 value: 11 significant bits) as two bf16 pieces:
// hi = bf16(d), lo = d - hi (at most 3 significant bits, exact in bf16).
struct ScalePieces {
  uint32_t hi2, lo2;   // (hi, hi), (lo, lo)
};
__device__ __forceinline__ ScalePieces scale_pieces(float d) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(d);
  const __nv_bfloat16 lo = __float2bfloat16_rn(d - __bfloat162float(hi));   // exact
  const uint32_t h = __bfloat16_as_ushort(hi), l = __bfloat16_as_ushort(lo);
  return {h | (h << 16), l | (l << 16)};
}

// 8 columns as bf16(d (n - 8)), rounded once, in slot order.  Nibbles of
// columns 0 and 4 (and, from w >> 8, 2 and 6) land in mantissa bits 0-3 of
// bf16 128; those of columns 1 and 5 (3 and 7), shifted right by one, land
// in mantissa bits 3-6 of bf16 16.  Subtracting 136 or 24 gives the exact
// integers m = n - 8; m * lo is exact (at most 6 significant bits), and
// fma(m, hi, m * lo) is m * (hi + lo) = d (n - 8) rounded once to bf16.
__device__ __forceinline__ uint4 dequant_word(uint32_t w, const ScalePieces& sp) {
  const uint32_t w8 = w >> 8;
  const uint32_t v04 = lop3_and_or(w, 0x000F000Fu, 0x43004300u);        // 128 + n
  const uint32_t v15 = lop3_and_or(w >> 1, 0x00780078u, 0x41804180u);   // 16 + n
  const uint32_t v26 = lop3_and_or(w8, 0x000F000Fu, 0x43004300u);
  const uint32_t v37 = lop3_and_or(w8 >> 1, 0x00780078u, 0x41804180u);
  auto dq = [&](uint32_t v, uint32_t magic) {
    const uint32_t m = bsub2(v, magic);
    return bfma2(m, sp.hi2, bmul2(m, sp.lo2));
  };
  return make_uint4(dq(v04, 0x43084308u), dq(v15, 0x41C041C0u), dq(v26, 0x43084308u), dq(v37, 0x41C041C0u));
}

// The same 8 columns as fp16: fp16(d (n - 8)), rounded once, in slot order.
// A nibble lands in the mantissa of fp16 1024 (bits 0-3 of each half) or 64
// (bits 4-7): (1024 + n) - 1032 and (64 + n) - 72 are the exact small
// integers n - 8, and the half multiply by d rounds the exact product to
// nearest even.
__device__ __forceinline__ uint4 dequant_word_f16(uint32_t w, __half2 dd) {
  const uint32_t w8 = w >> 8;
  const __half2 m_even = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));   // 1032
  const __half2 m_odd = __halves2half2(__ushort_as_half(0x5480), __ushort_as_half(0x5480));    // 72
  const uint32_t p04 = lop3_and_or(w, 0x000F000Fu, 0x64006400u), p26 = lop3_and_or(w8, 0x000F000Fu, 0x64006400u);
  const uint32_t p15 = lop3_and_or(w, 0x00F000F0u, 0x54005400u), p37 = lop3_and_or(w8, 0x00F000F0u, 0x54005400u);
  auto dq = [&](uint32_t pv, __half2 m) {
    const __half2 v = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&pv), m), dd);
    return *reinterpret_cast<const uint32_t*>(&v);
  };
  return make_uint4(dq(p04, m_even), dq(p15, m_odd), dq(p26, m_even), dq(p37, m_odd));
}

__device__ __forceinline__ uint32_t h2_to_bf16x2(uint32_t h2) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
  return bf16x2(f.x, f.y);
}

struct Params {
  CUtensorMap tm_codes;   // codes [N][K/2] u8, box [128 rows][128 B]
  const uint8_t* xb;      // bf16 X as [K/8 column groups][64 tokens][8]: chunk c = bytes [8 KB c, 8 KB (c+1))
  CUtensorMap tm_sc;      // scales [N][K/32] fp16 (as u16), box [128 rows][8 scales]; K % 256 == 0
  const __half* scales;   // read directly when K % 256 != 0 (row stride not a multiple of 16 B)
  int sc_tma;
  float* Y;
  float out_scale;        // Y = out_scale * (the product): 1, or the w4a8 activation scale
  int N, K;
  int ntok;               // tokens written to Y (the rows of Y; the MMA N may be padded beyond)
  int tiles, splits, cps, nchunks, items;
  long long wait_limit;
  unsigned long long* trace;   // optional: CTA 0 stamps [chunk < kTraceChunks][8], SM cycles
  // LM-head form only (the kernel's HEAD instantiation, one CTA per tile):
  // the epilogue keeps a running top two per token instead of writing Y, and
  // the CTA that finishes last merges the per-CTA records
  float cap;           // softcap: logits = cap * tanh(z / cap)
  float* logits;       // optional softcapped logits [ntok][N]
  Top2* partials;      // [gridDim.x][kMaxBatch]
  unsigned* ticket;    // zero before the launch; zero again after it
  int32_t* idx;
  float* top1;
  float* top2;
};

constexpr int kTraceChunks = 256;

using tc::bulk_load;
using tc::tma_load_2d;

__device__ __forceinline__ void item_range(const Params& p, int item, int& tile, int& c0, int& c1) {
  tile = item / p.splits;
  const int sp = item - tile * p.splits;
  c0 = sp * p.cps;
  c1 = min(c0 + p.cps, p.nchunks);
}

// NT: the MMA N (token tile), F16: fp16 tiles (else bf16), HEAD: the LM-head
// epilogue (softcap and top two per token, no Y), A8: the w4a8 form (the
// token operand holds activation codes, Y is scaled by p.out_scale), its own
// instantiation so that the plain GEMM's epilogue carries no scaling.
template <int NT, bool F16, bool HEAD, bool A8 = false>
__global__ void __launch_bounds__(kThreadsG, 1) gemm_kernel(const __grid_constant__ Params p) {
  constexpr int kStageBytes = stage_bytes(NT);
  constexpr int kBBytes = b_bytes(NT);
  constexpr int kTmemCols = tmem_cols(NT);
  static_assert(a_col0(NT) + kStages * kACols <= 512, "tensor memory");
  static_assert(kIssuers == 2, "two accumulators per item");
  constexpr uint32_t kId = idesc(NT, F16);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* stage_base = smem;
  uint8_t* raw_base = smem + operand_bytes(NT, HEAD, p.K);
  uint64_t* bars = reinterpret_cast<uint64_t*>(raw_base + (size_t)kRawStages * kRawBytes);
  // bars: full[kStages], empty[kStages], accfull[2], accempty[2], drain,
  //       rawfull[kRawStages], rawempty[kRawStages], xfull (resident token operand)
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ long long t0_sh;
  __shared__ Top2 head_st[kEpiWarps][HEAD ? NT : 1];   // LM head: per epilogue warp and token
  __shared__ Top2 head_run[HEAD ? kMaxBatch : 1][HEAD ? kEpiWarps * 32 : 1];   // LM head: per token and row

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned long long* const tr = (p.trace && blockIdx.x == 0) ? p.trace : nullptr;
  auto stamp = [&](uint32_t chunk, int k) {
    if (tr && chunk < (uint32_t)kTraceChunks) tr[chunk * 8 + k] = (unsigned long long)(tc::clock_ordered() - t0_sh);
  };
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStages);
  const uint32_t accfull0 = smem_u32(bars + 2 * kStages), accempty0 = smem_u32(bars + 2 * kStages + 2);
  const uint32_t drain = smem_u32(bars + 2 * kStages + 4);
  const uint32_t rawfull0 = smem_u32(bars + 2 * kStages + 5), rawempty0 = rawfull0 + 8 * kRawStages;
  const uint32_t xfull = rawempty0 + 8 * kRawStages;
  volatile int* abort_flag = &abort_sh;

  if (warp == 0) {
    // lane i initialises barrier i (in the order of the layout above)
    if (lane == 0) {
      abort_sh = 0;
      t0_sh = tc::clock_ordered();
    }
    if (lane < kBars) {
      const int i = lane;
      unsigned count = 1;                                              // rawfull
      if (i < kStages) count = HEAD ? kGroupWarps : kGroupWarps + 1;   // full: the chunk's group (+ the B loader)
      else if (i < 2 * kStages + 2) count = 2;                         // empty, accfull: one commit per issuer
      else if (i < 2 * kStages + 4) count = kEpiWarps;                 // accempty
      else if (i == 2 * kStages + 4) count = 2;                        // drain: one commit per issuer
      else if (i >= 2 * kStages + 5 + kRawStages && i < kBars - 1)
        count = kRawChunks * kGroupWarps;                                  // rawempty: its readers
      // xfull (the last): the loader's bytes
      mbar_init(smem_u32(bars + i), count);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
  } else if (warp == kTmaWarp && lane == 0) {
    // the tensor maps' descriptors, fetched while the CTA sets up
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tm_codes)) : "memory");
    if (p.sc_tma) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tm_sc)) : "memory");
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_sh)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  if (warp == kTmaWarp) {
    // ------------------------------------------------------- raw tile loads
    // (the whole warp walks the loop, one elected lane issues)
    if (blockIdx.x < p.items) {
      uint64_t pol_stream;
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_stream));
      const uint32_t raw0 = smem_u32(raw_base);
      uint32_t g = 0, gc = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < p.items && ok; item += gridDim.x) {
        int tile, c0, c1;
        item_range(p, item, tile, c0, c1);
        for (int cs = c0; cs < c1; cs += kRawChunks, ++g) {
          const uint32_t s = g % kRawStages, round = g / kRawStages;
          const bool free_ = mbar_wait(rawempty0 + 8 * s, (round & 1) ^ 1, p.wait_limit, abort_flag);
          if (!__all_sync(0xffffffffu, free_)) {
            ok = false;
            break;
          }
          if (elect_one()) {
            const uint32_t dst = raw0 + s * kRawBytes;
            stamp(gc, 0);
            mbar_expect_tx(rawfull0 + 8 * s, p.sc_tma ? kRawBytes : kRawCodeBytes);
            tma_load_2d(dst, &p.tm_codes, cs * (kChunk / 2), tile * kTileM, rawfull0 + 8 * s, pol_stream);
            if (p.sc_tma)   // cs % kRawChunks == 0 here: the x coordinate is 16-byte aligned
              tma_load_2d(dst + kRawCodeBytes, &p.tm_sc, cs * (kChunk / 32), tile * kTileM, rawfull0 + 8 * s,
                          pol_stream);
          }
          __syncwarp();
          gc += min(cs + kRawChunks, c1) - cs;
        }
      }
      // every issued load lands before the CTA may exit
      const uint32_t first = g > (uint32_t)kRawStages ? g - kRawStages : 0u;
      for (uint32_t q = first; q < g; ++q) {
        const long long t0 = clock64();
        while (!mbar_test(rawfull0 + 8 * (q % kRawStages), (q / kRawStages) & 1)) {
          if (clock64() - t0 > kDrainCycles) {
            atomicOr(&g_device_error, 1u);
            break;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == kBWarp) {
    // ------------------------------------------- token tiles (B operand)
    uint64_t pol_keep;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_keep));
    pdl_wait();   // the bf16 copy of X is written by the kernel launched just before
    const uint32_t stage0 = smem_u32(stage_base);
    if constexpr (HEAD) {
      // the whole token operand, once: K * 32 bytes in pieces of at most 16 KB
      const uint32_t total = (uint32_t)p.K * 32u;
      if (elect_one()) {
        mbar_expect_tx(xfull, total);
        for (uint32_t off = 0; off < total; off += 16384u)
          bulk_load(stage0 + off, p.xb + off, min(16384u, total - off), xfull, pol_keep);
      }
      __syncwarp();
      const long long t0 = clock64();   // it lands before the CTA may exit
      while (!mbar_test(xfull, 0)) {
        if (clock64() - t0 > kDrainCycles) {
          atomicOr(&g_device_error, 1u);
          break;
        }
      }
      __syncwarp();
    }
    uint32_t g = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < p.items && ok && !HEAD; item += gridDim.x) {
      int tile, c0, c1;
      item_range(p, item, tile, c0, c1);
      for (int c = c0; c < c1; ++c, ++g) {
        const uint32_t s = g % kStages, round = g / kStages;
        const bool free_ = mbar_wait(empty0 + 8 * s, (round & 1) ^ 1, p.wait_limit, abort_flag);
        if (!__all_sync(0xffffffffu, free_)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          // [16 column groups][64 tokens][8]: core matrices 128 B apart along
          // the tokens, 1024 B apart along K; a last chunk of 64 columns is 8 KB
          const uint32_t bytes = (uint32_t)(min(kChunk, p.K - c * kChunk) / 64) * (kBBytes / 2);
          mbar_expect_tx(full0 + 8 * s, bytes);   // also this loader's arrival on full
          bulk_load(stage0 + s * kStageBytes, p.xb + (size_t)c * kBBytes, bytes, full0 + 8 * s, pol_keep);
        }
        __syncwarp();
      }
    }
    // every issued copy lands before the CTA may exit (full also waits for
    // the converters, which an aborting CTA may never bring, hence the
    // short bound then); none in the LM-head form
    const uint32_t first = g > (uint32_t)kStages ? g - kStages : 0u;
    for (uint32_t q = first; q < g; ++q) {
      const long long lim = *abort_flag ? kShortDrainCycles : kDrainCycles;
      const long long t0 = clock64();
      while (!mbar_test(full0 + 8 * (q % kStages), (q / kStages) & 1)) {
        if (clock64() - t0 > lim) {
          atomicOr(&g_device_error, 1u);
          break;
        }
      }
    }
    __syncwarp();
  } else if (warp >= kEpiWarps && warp < kMmaWarp) {
    // ----------------------------------------------------------- converters
    // Group cg (warps 4 + 4 cg .. 7 + 4 cg) converts chunk j of the raw stages
    // gr with kRawChunks (gr % kStageSets) + j == cg.  thread = tile row r
    // (TMEM lane r): warp w writes TMEM lanes 32 (w % 4) .. + 31 (the lane
    // quarter its scheduler may access), all four 32-column blocks of the
    // chunk for its rows, as two stores of 32 columns (two 16-bit weights per
    // column, slot order) into the stage's A columns
    const int wc = warp - kEpiWarps;                 // 0 .. kProdWarps - 1
    const int cg = wc / kGroupWarps;                 // chunk group
    const int r = 32 * (warp & 3) + lane;
    const uint32_t a_lane = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)a_col0(NT);
    uint32_t g0 = 0, gr = 0;   // first operand chunk of the raw stage, raw stages
    bool ok = true;
    for (int item = blockIdx.x; item < p.items && ok; item += gridDim.x) {
      int tile, c0, c1;
      item_range(p, item, tile, c0, c1);
      for (int cs = c0; cs < c1 && ok; cs += kRawChunks, ++gr) {
        const int j = cg - kRawChunks * (int)(gr % kStageSets);   // this group's chunk in the raw stage
        const uint32_t gs = g0;
        g0 += (uint32_t)(min(cs + kRawChunks, c1) - cs);
        if (j < 0 || j >= kRawChunks) continue;   // a raw stage of the other groups
        const uint32_t rs = gr % kRawStages, rround = gr / kRawStages;
        const bool landed = mbar_wait(rawfull0 + 8 * rs, rround & 1, p.wait_limit, abort_flag);
        if (!__all_sync(0xffffffffu, landed)) {
          ok = false;
          break;
        }
        const uint8_t* raw = raw_base + (size_t)rs * kRawBytes;
        const int c = cs + j;                  // this group's chunk
        const uint32_t g = gs + (uint32_t)j;
        const bool mine = c < c1;              // an item's last raw stage may hold one chunk
        if (wc == 0 && lane == 0) stamp(g, 1);
        const int nb = mine ? min(kChunk, p.K - c * kChunk) / 32 : 0;   // 32-column blocks: 4, or 2 at the end
        uint4 code[kBPW];
        float d[kBPW];
#pragma unroll
        for (int bb = 0; bb < kBPW; ++bb) {
          if (bb < nb) {
            // the codes tile arrives in the 128-byte swizzle: 16-byte group
            // i of row r sits at group i ^ (r % 8), so the 32 rows read by a
            // warp spread over the banks
            code[bb] = *reinterpret_cast<const uint4*>(raw + r * 128 + (((j * 4 + bb) ^ (r & 7)) << 4));
            d[bb] = p.sc_tma ? __half2float(*reinterpret_cast<const __half*>(raw + kRawCodeBytes + r * 16 +
                                                                              (j * 4 + bb) * 2))
                             : ld_scale(p.scales + ((size_t)tile * kTileM + r) * (p.K >> 5) + c * 4 + bb);
          }
        }
        __syncwarp();   // this warp has read its part of the raw stage
        if (lane == 0) mbar_arrive(rawempty0 + 8 * rs);
        if (!mine) continue;
        const uint32_t s = g % kStages, round = g / kStages;
        const bool free_ = mbar_wait(empty0 + 8 * s, (round & 1) ^ 1, p.wait_limit, abort_flag);
        if (!__all_sync(0xffffffffu, free_)) {
          ok = false;
          break;
        }
        tc_fence_after();   // the MMAs that read this A stage have completed
        if (wc == 0 && lane == 0) stamp(g, 2);
#pragma unroll
        for (int pp = 0; pp < kBPW / 2; ++pp) {
          if (2 * pp >= nb) break;   // warp-uniform: a last chunk of 64 columns has no blocks 2, 3
          uint32_t v[32];
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int bb = 2 * pp + i;
            const uint32_t w4[4] = {code[bb].x, code[bb].y, code[bb].z, code[bb].w};
            uint4 o[4];
            if (F16) {
              const __half2 dd = __float2half2_rn(d[bb]);   // d is an fp16 value: exact
#pragma unroll
              for (int q = 0; q < 4; ++q) o[q] = dequant_word_f16(w4[q], dd);
            } else {
              const ScalePieces sp = scale_pieces(d[bb]);
#pragma unroll
              for (int q = 0; q < 4; ++q) o[q] = dequant_word(w4[q], sp);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              v[16 * i + 4 * q] = o[q].x;
              v[16 * i + 4 * q + 1] = o[q].y;
              v[16 * i + 4 * q + 2] = o[q].z;
              v[16 * i + 4 * q + 3] = o[q].w;
            }
          }
          tmem_st32(a_lane + (uint32_t)(kACols * s + 32 * pp), v);
        }
        tc_fence_before();   // this warp's TMEM stores, before the MMA issuer reads them
        __syncwarp();
        if (lane == 0) mbar_arrive(full0 + 8 * s);
        if (wc == 0 && lane == 0) stamp(g, 3);
      }
    }
  } else if (warp >= kMmaWarp && warp < kMmaWarp + kIssuers) {
    // -------------------------------------------------------- MMA issuers
    // Issuer m takes the second or first half of each chunk's K steps into
    // its own accumulator (each accumulator's MMAs come from one thread, in
    // order); both commit to the stage's empty barrier.  (Each warp walks
    // the loop and waits together, one elected lane issues.)
    const int m = warp - kMmaWarp;
    uint32_t g = 0;
    int it = 0;
    bool ok = true;
    const uint32_t stage0 = smem_u32(stage_base);
    if constexpr (HEAD) ok = __all_sync(0xffffffffu, mbar_wait(xfull, 0, p.wait_limit, abort_flag));
    for (int item = blockIdx.x; item < p.items && ok; item += gridDim.x, ++it) {
      int tile, c0, c1;
      item_range(p, item, tile, c0, c1);
      const int a = it & 1;
      const bool acc_free = mbar_wait(accempty0 + 8 * a, ((it >> 1) & 1) ^ 1, p.wait_limit, abort_flag);
      if (!__all_sync(0xffffffffu, acc_free)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem + (uint32_t)((kIssuers * a + m) * NT);
      for (int c = c0; c < c1; ++c, ++g) {
        const uint32_t s = g % kStages, round = g / kStages;
        // full: the converter warps' A tile and the B loader's token tile
        const bool landed = mbar_wait(full0 + 8 * s, round & 1, p.wait_limit, abort_flag);
        if (!__all_sync(0xffffffffu, landed)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (elect_one()) {
          if (m == 0) stamp(g, 4);
          const int half = min(kChunk, p.K - c * kChunk) / 32;   // K steps per issuer: 4, or 2 at the end
          const int ks0 = m * half;
          // B: [16 column groups][NT tokens][8]: groups NT * 16 B apart;
          // K step ks starts NT * 32 bytes further (2 NT in the descriptor's
          // address field, which no step carries out of)
          const uint32_t bbase = HEAD ? stage0 + (uint32_t)c * kBBytes : stage0 + s * kStageBytes;
          const uint64_t bd0 = smem_desc(bbase + ks0 * NT * 32, NT * 16, 128);
          const uint32_t A = tmem + (uint32_t)(a_col0(NT) + kACols * s + 8 * ks0);   // lane 0
#pragma unroll
          for (int kk = 0; kk < kChunk / 32; ++kk) {
            if (kk < half) tc_mma_ta(d_tmem, A + 8 * kk, bd0 + (uint64_t)(kk * NT * 2), kId, (c > c0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(empty0 + 8 * s);
          if (m == 0) stamp(g, 5);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (elect_one()) tc_commit(accfull0 + 8 * a);
      __syncwarp();
    }
    // drain: every tcgen05 op issued here has finished before TMEM is freed
    if (elect_one()) tc_commit(drain);
    __syncwarp();
    const long long t0 = clock64();
    while (!mbar_test(drain, 0)) {
      if (clock64() - t0 > kDrainCycles) {   // independent of the (possibly zero) wait budget
        atomicOr(&g_device_error, 1u);
        break;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int row = warp * 32 + lane;          // TMEM lane = tile row
    if (p.splits > 1) pdl_wait();              // Y is cleared by the kernel launched just before
    // LM head: the best two (z, row) per token over the rows this thread
    // reads, kept in shared memory (token-major: a warp's records of one token
    // are 512 contiguous bytes)
    if constexpr (HEAD) {
#pragma unroll
      for (int t = 0; t < kMaxBatch; ++t) top2_init(head_run[t][row]);
    }
    int it = 0;
    uint32_t ge = 0;   // this item's first chunk in the CTA's sequence (trace only)
    for (int item = blockIdx.x; item < p.items; item += gridDim.x, ++it) {
      int tile, c0, c1;
      item_range(p, item, tile, c0, c1);
      const int a = it & 1;
      if (!mbar_wait(accfull0 + 8 * a, (it >> 1) & 1, p.wait_limit, abort_flag)) break;
      if (threadIdx.x == 0) stamp(ge, 6);
      tc_fence_after();
      const int n = tile * kTileM + row;   // output row (vocabulary index for the head)
#pragma unroll
      for (int cb = 0; cb < NT / 16; ++cb) {
        float v[16];
        const uint32_t t_acc = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(kIssuers * a * NT + cb * 16);
        tmem_ld16(t_acc, v);
        {   // the second issuer's accumulator, added in a fixed order
          float u[16];
          tmem_ld16(t_acc + (uint32_t)NT, u);
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] += u[j];
        }
        if constexpr (A8) {   // w4a8: Y = s * (W q)
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] *= p.out_scale;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int t = cb * 16 + j;
          if (t >= p.ntok) break;
          if constexpr (HEAD) {
            Top2 b = head_run[t][row];
            top2_insert(b, v[j], n);
            head_run[t][row] = b;
            if (p.logits) p.logits[(size_t)t * p.N + n] = p.cap * tanhf(v[j] / p.cap);
          } else {
            float* dst = p.Y + (size_t)t * p.N + n;
            if (p.splits == 1)
              *dst = v[j];
            else
              atomicAdd(dst, v[j]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(accempty0 + 8 * a);
      if (threadIdx.x == 0) stamp(ge, 7);
      ge += c1 - c0;
    }
    if constexpr (HEAD) {
      __syncwarp();
      for (int t = 0; t < p.ntok; ++t) {
        Top2 b = head_run[t][row];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) top2_shfl_xor_merge(b, o);
        if (lane == 0) head_st[warp][t] = b;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
  if constexpr (HEAD) {
    // this CTA's record per token (its epilogue warps' four), then the merge
    // over all CTAs' records in the CTA that finishes last
    if (threadIdx.x < p.ntok) {
      Top2 t;
      top2_init(t);
#pragma unroll
      for (int w = 0; w < kEpiWarps; ++w) top2_merge(t, head_st[w][threadIdx.x]);
      p.partials[(size_t)blockIdx.x * kMaxBatch + threadIdx.x] = t;
    }
    head_finish(p.partials, p.ticket, p.ntok, p.cap, p.idx, p.top1, p.top2);
  }
}

// X fp16 [ntok][K] -> the token operand as [K/8 column groups][NT tokens][8
// slots] (slot s holds column kSlotCol[s] of its group, the weights' order):
// bf16 (nearest even) for bf16 tiles, the fp16 bits unchanged for fp16 tiles;
// tokens ntok .. NT-1 are zero.  Each 128-column chunk is one contiguous
// NT * 256-byte token tile in the core-matrix layout.  One thread per
// (group, token).
template <int NT, bool F16>
__global__ void __launch_bounds__(256) x_layout_kernel(const __half* __restrict__ X, uint8_t* __restrict__ xb,
                                                       int K, int ntok, float4* __restrict__ yclear, int n4,
                                                       float act_s) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;   // = group * NT + token
  // the output the split-K GEMM adds into, cleared (n4 float4s; 0 if none)
  for (int k = i; k < n4; k += gridDim.x * blockDim.x) yclear[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (i < (K >> 3) * NT) {
    const int grp = i / NT, tok = i - grp * NT;
    uint4 o = make_uint4(0u, 0u, 0u, 0u);
    if (tok < ntok) {
      uint4 v = *reinterpret_cast<const uint4*>(X + (size_t)tok * K + grp * 8);
      if (act_s > 0.f) {   // w4a8: the token operand is the activation codes q (the GEMM scales Y by s)
        uint32_t* w = &v.x;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
          const __half2 h = __floats2half2_rn(a8_code(f.x, act_s), a8_code(f.y, act_s));
          w[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
      }
      // slot order 0 4 1 5 2 6 3 7 (the weights' decoded pairs)
      const uint4 q = make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632),
                                 __byte_perm(v.y, v.w, 0x5410), __byte_perm(v.y, v.w, 0x7632));
      o = F16 ? q : make_uint4(h2_to_bf16x2(q.x), h2_to_bf16x2(q.y), h2_to_bf16x2(q.z), h2_to_bf16x2(q.w));
    }
    *reinterpret_cast<uint4*>(xb + (size_t)i * 16) = o;
  }
  pdl_trigger();
}

}  // namespace gemm

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (the library does not link the driver library itself).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2-D row-major tensor [rows][cols] of esize-byte elements, one box per load.
int encode_tensor_2d(CUtensorMap* tm, const void* base, CUtensorMapDataType type, int esize, uint64_t cols,
                     uint64_t rows, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle,
                     const char* what) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return fail(Q4_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * (uint64_t)esize};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(tm, type, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(Q4_ERR_CUDA, "tensor map for %s: driver error %d", what, (int)r);
  return Q4_OK;
}

size_t gemm_ws_bytes(int K) { return ((size_t)gemm::kTok * K * 2 + 255) & ~(size_t)255; }
size_t mma16_ws_bytes(int K) { return ((size_t)16 * K * 2 + 255) & ~(size_t)255; }

// Y[t][n] (t < ntok) = the dequantised weights times X through gemm_kernel<NT, F16, HEAD>.
// allow_split: K may be split across CTAs (the splits add into Y with fp32
// atomics, so the summation order is not fixed); else one CTA per tile.
// HEAD: Y is not written; head->* receive the softcapped top two per token
// (and the softcapped logits when head->logits is set).
template <int NT, bool F16, bool HEAD, bool A8 = false>
static int launch_mma(const uint8_t* codes, const __half* scales, const __half* X, int ntok, float* Y, int N,
                      int K, void* ws, bool allow_split, const HeadOutputs* head, const DeviceInfo& dev,
                      cudaStream_t s, float act_scale = 0.f) {
  if (HEAD && (head == nullptr || allow_split)) return fail(Q4_ERR_SHAPE, "head GEMM: outputs missing or split K");
  gemm::Params p;
  memset(&p, 0, sizeof(p));
  if (HEAD) {
    p.cap = head->cap;
    p.logits = head->logits;
    p.partials = head->partials;
    p.ticket = head->ticket;
    p.idx = head->idx;
    p.top1 = head->top1;
    p.top2 = head->top2;
  }
  int st = encode_tensor_2d(&p.tm_codes, codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)K / 2, (uint64_t)N,
                            gemm::kChunk * gemm::kRawChunks / 2, gemm::kTileM, CU_TENSOR_MAP_SWIZZLE_128B, "codes");
  if (st != Q4_OK) return st;
  p.xb = static_cast<const uint8_t*>(ws);
  p.scales = scales;
  p.sc_tma = K % 256 == 0;
  if (p.sc_tma) {
    st = encode_tensor_2d(&p.tm_sc, scales, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, (uint64_t)K / 32, (uint64_t)N, 8,
                          gemm::kTileM, CU_TENSOR_MAP_SWIZZLE_NONE, "scales");
    if (st != Q4_OK) return st;
  }
  p.Y = Y;
  p.out_scale = act_scale > 0.f ? act_scale : 1.f;
  p.N = N;
  p.K = K;
  p.ntok = ntok;
  p.tiles = N / gemm::kTileM;
  p.nchunks = (K + gemm::kChunk - 1) / gemm::kChunk;
  int splits = allow_split ? (dev.sms + p.tiles - 1) / p.tiles : 1;
  if (splits > p.nchunks) splits = p.nchunks;
  if (splits < 1) splits = 1;
  p.cps = (p.nchunks + splits - 1) / splits;
  p.cps = (p.cps + gemm::kRawChunks - 1) / gemm::kRawChunks * gemm::kRawChunks;   // raw stages start aligned
  p.splits = (p.nchunks + p.cps - 1) / p.cps;
  p.items = p.tiles * p.splits;
  p.wait_limit = wait_limit();
  size_t tbytes = 0;
  void* tb = trace_buffer(&tbytes);
  p.trace = (tb && tbytes >= (size_t)gemm::kTraceChunks * 8 * sizeof(unsigned long long))
                ? static_cast<unsigned long long*>(tb)
                : nullptr;
  cudaError_t e;
  // dynamic shared memory up to what the CTA's static part leaves (set once
  // per instantiation and device)
  static PerDevice attr_set;
  static size_t dyn_max[64] = {0};
  if (!attr_set.get(dev.ordinal)) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, gemm::gemm_kernel<NT, F16, HEAD, A8>);
    if (e != cudaSuccess) return cuda_fail(e, "gemm attributes");
    dyn_max[dev.ordinal] = gemm::kSmemMax - fa.sharedSizeBytes;
    e = cudaFuncSetAttribute(gemm::gemm_kernel<NT, F16, HEAD, A8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)dyn_max[dev.ordinal]);
    if (e != cudaSuccess) return cuda_fail(e, "gemm smem attribute");
    attr_set.set(dev.ordinal);
  }
  const size_t dyn = gemm::smem_bytes(NT, HEAD, K);
  if (dyn > dyn_max[dev.ordinal]) return fail(Q4_ERR_SHAPE, "K=%d: the token operand does not fit", K);
  const int nx = (K >> 3) * NT;
  // split K: the token-layout kernel also clears Y, which the GEMM's
  // epilogue adds into only after waiting for that kernel
  const int n4 = p.splits > 1 ? (int)((size_t)ntok * N / 4) : 0;
  gemm::x_layout_kernel<NT, F16><<<(nx + 255) / 256, 256, 0, s>>>(X, static_cast<uint8_t*>(ws), K, ntok,
                                                                  reinterpret_cast<float4*>(Y), n4, act_scale);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "gemm token layout launch");
  // the GEMM starts while the token layout is written; only its B loader waits for it
  const int grid = p.items < dev.sms ? p.items : dev.sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(gemm::kThreadsG);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, gemm::gemm_kernel<NT, F16, HEAD, A8>, p);
  return e == cudaSuccess ? Q4_OK : cuda_fail(e, "gemm launch");
}

int launch_gemm_chunk(const uint8_t* codes, const __half* scales, const __half* X, float* Y, int M,
                      int N, int K, void* ws, const DeviceInfo& dev, cudaStream_t s, float act_scale) {
  (void)M;
  if (act_scale > 0.f)
    return launch_mma<gemm::kTok, false, false, true>(codes, scales, X, gemm::kTok, Y, N, K, ws, true, nullptr, dev,
                                                      s, act_scale);
  return launch_mma<gemm::kTok, false, false>(codes, scales, X, gemm::kTok, Y, N, K, ws, true, nullptr, dev, s);
}

bool head_mma_fits(int K) {
  // the resident token operand, the raw ring and the barriers, next to the
  // head form's static records (per-token top-two records: under 18 KB)
  return K >= 64 && gemm::smem_bytes(16, true, K) + 18 * 1024 <= gemm::kSmemMax;
}

int launch_head_mma(const uint8_t* codes, const __half* scales, const __half* X, int ntok, int N, int K, void* ws,
                    const HeadOutputs& head, const DeviceInfo& dev, cudaStream_t s) {
  if (ntok < 1 || ntok > kMaxBatch) return fail(Q4_ERR_SHAPE, "token count %d must be in [1, %d]", ntok, kMaxBatch);
  return launch_mma<16, true, true>(codes, scales, X, ntok, nullptr, N, K, ws, false, &head, dev, s);
}

}  // namespace q4w

extern "C" int q4_device_status(q4_stream_t stream) {
  using namespace q4w;
  clear_error();
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "q4_device_status: stream");
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "q4_device_status: read");
  if (v) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e, "q4_device_status: clear");
    return fail(Q4_ERR_TIMEOUT, "a bounded device-side wait ran out (error word 0x%x)", v);
  }
  return Q4_OK;
}
