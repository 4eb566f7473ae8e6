// Per-Layer-Embedding gather fused with its f32 projection and per-chunk
// RMSNorm ("visible-cx/gemma-4-E2B-CoreAI", The PLE gather-table sidecar:
// int8 table [V][L*ld] + per-row f32 scale, dequant x16.0, proj.f32
// [L*ld][D], proj_norm.f32 [ld]; "Gemma-4 E2B mobile mixed-bit QAT weights",
// P2 DONE: 35 layer-major blocks of 256 on axis 1).
//
// The projection p[t] = proj . hidden[t] is a dense contraction (L*ld rows x
// D x S tokens), so it runs on the 5th-generation tensor cores with f32-class
// arithmetic: each f32 weight w is split into two fp16 pieces,
// p1 = fp16(w) and p2 = fp16((w - p1) * 2^11), which keep 22 of its 24
// significant bits (|w - p1 - p2 2^-11| <= 2^-22 |w| in the normal range);
// the fp16 hidden values are exact, so tcgen05.mma kind::f16 forms exact
// products, accumulated in fp32 into two TMEM accumulators D1 = P1 . h and
// D2 = P2 . h, and p = D1 + D2 * 2^-11.  M = 128 projection rows, N = the
// token group (up to 64, padded to a multiple of 16 with zero rows).
//
// A 256-row layer chunk and a group of up to 64 tokens belong to a cluster of
// four CTAs: rank r = m + 2 kh takes the 128-row half m of the chunk over the
// K half kh of the hidden width.  The two K halves of a row half swap the
// partial sums of the rows the other one finishes (64 rows each) through
// distributed shared memory and add them in a fixed order; then every CTA
// sends its per-token sum of squares over its 64 finished rows to the three
// others, so each finishes the chunk's RMSNorm for its own rows, adds the gathered
// table term, and writes its [64 tokens][64 columns] output tile (and the
// gathered bytes) from shared memory with tensor stores.  Both exchanges are
// stores into the peers' shared memory that count their bytes on an mbarrier
// of the receiving CTA (st.async), so after the one cluster barrier at the
// start (every peer running) a CTA waits only for the data it needs.  The
// table bytes of those columns are fetched at the start by one 64-byte bulk
// copy per token.
//
// Warp roles (320 threads):
//   warp 0     TMA loads (one elected lane): per stage of 64 K columns the
//              raw projection tile as two boxes [128 rows][32 fp32]
//              (128-byte swizzle) and the hidden tile [64 tokens][64 fp16]
//              (128-byte swizzle: the B operand as loaded)
//   warp 1     TMEM allocation; the warp runs the MMA loop together and one
//              elected lane issues the MMAs (8 per stage: 4 per piece) and
//              the commits
//   warps 2-9  converters: split the raw tile in place into the pieces P1
//              and P2 (thread = projection row and raw box: the box's
//              128-byte row becomes 64 bytes of P1 and 64 of P2, in the
//              128-byte swizzle of a K-major fp16 operand); eight warps so
//              that each scheduler has two to switch between
//   warps 2-5  also issue the table copies and run the epilogue: each
//              reads the accumulator rows of its TMEM lane quarter (warp w
//              reads lanes 32 (w % 4) .. + 31) for the exchanges, and the
//              four then form the output tile in place (one token and four
//              columns per thread)
// A ring of kFStages stages (raw / pieces 32 KB + hidden 8 KB) is guarded by
// full (TMA bytes), bready (converter warps, which arrive only after seeing
// full) and empty (MMA commit) mbarriers; the MMA warp waits on bready alone.
// The int8 form (ple_tc_kernel<true>; "Gemma-4 E2B mobile mixed-bit QAT
// weights", decode recipe and official-checkpoint notes: the model projection
// is int8 per block of 32) keeps the clusters and the epilogue.  A stage is
// 128 K columns: the code tile [128 rows][128 int8] (128-byte swizzle) and two
// hidden tiles [64 tokens][64 fp16] (128-byte swizzle, the B operand as
// loaded) come from TMA into one of six 32 KB slots, so a K half of D = 1536
// is in flight at once; two groups of four converter warps (2-5, 6-9) take
// alternate stages and widen the codes to fp16(scale * code) straight into
// one of four 64-column A stages in tensor memory (thread = projection row =
// TMEM lane), and 8 MMAs of kind::f16 with A in tensor memory follow (each
// converter thread loads the block scales of its row for its group's stages
// at the start and reads them back from shared memory itself).  A slot is free again
// once its group has read the codes and the MMAs have read the hidden tile;
// an A stage once its MMAs have completed.  The K halves of a cluster take
// alternate 128-column units.
//
// In both forms the token ids, table copies and table scales are handled by
// warps 2-5 while the first tiles load, and the epilogue reads each row's 64
// accumulator columns with one TMEM load.
// The kernel is launched with programmatic dependent launch: its set-up
// overlaps the previous kernel, its first reads of inputs come after
// griddepcontrol.wait.  Every mbarrier wait is bounded; on expiry the CTA
// sets its abort flag and the device error word, every role leaves its loop,
// work in flight is drained, and every CTA still sends its partial sums and
// sums of squares, so each receiver's byte count is met; a CTA drains its
// receive barriers before it leaves, so no peer stores into a CTA that has
// gone.
#include "q4w_device.cuh"
#include "q4w_internal.cuh"
#include "q4w_tc.cuh"

namespace q4w {

namespace ple {

constexpr int kLd = 256;                            // rows of one layer chunk
constexpr int kRows = 128;                          // rows per CTA (MMA M)
constexpr int kTok = 64;                            // tokens per CTA (MMA N <= 64)
// f32 projection: one stage is 64 K columns
constexpr int kFC = 64;                             // K columns per stage
constexpr int kFStages = 4;
constexpr int kFBox = kRows * 32 * 4;               // 16 KB: raw box [128 rows][32 fp32]; then a piece
constexpr int kFRawBytes = 2 * kFBox;               // 32 KB: raw tile, then P1 (first half) and P2
constexpr int kFHBytes = kTok * kFC * 2;            // 8 KB: hidden tile [64 tokens][64 fp16]
constexpr int kFStageBytes = kFRawBytes + kFHBytes;   // 40 KB, a multiple of 1024
constexpr int kRecvBytes = kTok * 64 * 4;           // partner's partial sums of 64 rows
constexpr int kGtabBytes = kTok * 64;               // table bytes of the 64 finished rows per token
constexpr int kEpi0 = 2;                            // first converter / epilogue warp
constexpr int kConvWarps = 8;                       // converter warps: 2-5 (also the epilogue) and 6-9
constexpr int kThreads = (kEpi0 + kConvWarps) * 32;   // 320
constexpr int kCluster = 4;
constexpr long long kDrainCycles = 2000000000LL;

// int8 projection (per-block-32 codes + fp16 scales): one stage is 128 K
// columns, so that every code row of the tile is one full 128-byte line; the
// operands are two 64-column halves, each a 128-byte row of fp16 per operand
// row in the 128-byte swizzle.
constexpr int kQC = 128;                            // K columns per stage
constexpr int kQR = 6;                              // raw slots (a K half of D = 1536 stays resident)
constexpr int kQA = 4;                              // A stages in tensor memory
constexpr int kQBHalf = kTok * 64 * 2;              // 8 KB: fp16 hidden of 64 columns (tensor load)
constexpr int kQBBytes = 2 * kQBHalf;
constexpr int kQRawBytes = kRows * kQC;             // 16 KB int8 codes [128 rows][128], 128-byte swizzle
constexpr int kQSlotBytes = kQBBytes + kQRawBytes;  // 32 KB, a multiple of 1024
constexpr int kQACol0 = 64;                         // TMEM: the accumulator, then kQA A stages of 64 columns
constexpr int kQMaxStages = 8;                      // stages per K half: D <= 2048
constexpr int kQScBytes = kQMaxStages * kRows * 8;  // per (stage, row): the stage's four fp16 scales

template <bool Q8>
constexpr size_t ring_bytes() {
  return Q8 ? (size_t)kQR * kQSlotBytes : (size_t)kFStages * kFStageBytes;
}
// TMEM columns: two 64-column accumulators (f32 pieces), or one plus the A
// stages (int8 form: 64 + 4 x 64)
template <bool Q8>
constexpr int tmem_cols() {
  return Q8 ? 512 : 128;
}
template <bool Q8>
constexpr size_t smem_bytes() {
  return 1024 + ring_bytes<Q8>() + kRecvBytes + kGtabBytes + (Q8 ? kQScBytes : 0);
}

// Instruction descriptor, kind::f16: D f32, A and B fp16, both K-major.
__device__ __forceinline__ uint32_t idesc_f16(int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}

// D (+)= A . B with A in tensor memory (128 lanes x 8 columns per K = 16).
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}

// Eight int8 codes (two words, column order) -> the fp16 values fp16(code * d)
// in column order.  Each byte, offset to code + 128, becomes the low byte of
// the fp16 number 1024 + (code + 128) (the byte lands in the mantissa);
// subtracting 1152 leaves the exact integer code, and the half multiply
// rounds code * d once, to nearest even.
__device__ __forceinline__ uint4 dequant_i8_f16(uint2 c, __half2 dd) {
  const __half2 off = __half2half2(__ushort_as_half(0x6480));   // 1152
  auto two = [&](uint32_t u, uint32_t sel) {
    const uint32_t h = __byte_perm(u, 0x64646464u, sel);
    const __half2 v = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&h), off), dd);
    return *reinterpret_cast<const uint32_t*>(&v);
  };
  const uint32_t u0 = c.x ^ 0x80808080u, u1 = c.y ^ 0x80808080u;
  return make_uint4(two(u0, 0x4140u), two(u0, 0x4342u), two(u1, 0x4140u), two(u1, 0x4342u));
}

// Eight f32 weights -> their fp16 pieces (column order): p1 = fp16(w) and
// p2 = fp16((w - p1) * 2^11), both rounded to nearest even; w - p1 is exact
// in fp32 and the scaling by 2^11 is exact, so p1 + p2 2^-11 differs from w
// by at most 2^-22 |w| (fp16 normal range) or 2^-36 (below it).
__device__ __forceinline__ void split_f32_f16(const float (&w)[8], uint4& p1, uint4& p2) {
  uint32_t a[4], b[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    // two columns at a time: one packed conversion per piece, packed fp32
    // subtract and scale (both exact)
    const __half2 h = __floats2half2_rn(w[2 * e], w[2 * e + 1]);
    const float2 hf = __half22float2(h);
    unsigned long long d;
    asm("{\n .reg .b64 v, q;\n mov.b64 v, {%1, %2};\n mov.b64 q, {%3, %4};\n"
        " sub.rn.f32x2 v, v, q;\n mul.rn.f32x2 %0, v, %5;\n}"
        : "=l"(d)
        : "f"(w[2 * e]), "f"(w[2 * e + 1]), "f"(hf.x), "f"(hf.y), "l"(0x4500000045000000ull));   // 2048, 2048
    float r0, r1;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r0), "=f"(r1) : "l"(d));
    const __half2 l = __floats2half2_rn(r0, r1);
    a[e] = *reinterpret_cast<const uint32_t*>(&h);
    b[e] = *reinterpret_cast<const uint32_t*>(&l);
  }
  p1 = make_uint4(a[0], a[1], a[2], a[3]);
  p2 = make_uint4(b[0], b[1], b[2], b[3]);
}

struct Params {
  CUtensorMap tm_proj;   // f32 [L*ld][D], box [128 rows][32], 128-byte swizzle;
                         // int8 form: codes [L*ld][D], box [128 rows][128], 128-byte swizzle
  CUtensorMap tm_hid;    // fp16 bits [S][D], box [64 rows][64], 128-byte swizzle; rows past S
                         // and columns past D read as zero
  CUtensorMap tm_out;    // f32 out [S][L*ld], box [64 tokens][64 columns]; rows past S not written
  CUtensorMap tm_gat;    // int8 gathered [S][L*ld], box [64 tokens][64 columns] (when gathered != NULL)
  const uint2* proj_sc;      // int8 form: fp16 scales [L*ld][D/32] read as quads [L*ld][D/128]
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
  unsigned long long* trace;   // optional: CTA 0 stamps [stage][8], SM cycles since the start
};

constexpr int kTraceRows = 256;

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

using tc::elect_one;

// Q8: the projection is int8 per-block-32 (codes + fp16 scales), widened to
// fp16 tiles by the converter warps and multiplied on kind::f16 (the hidden
// tile then goes to the tensor core straight from its tensor load).
template <bool Q8>
__global__ void __launch_bounds__(kThreads, 1) ple_tc_kernel(const __grid_constant__ Params p) {
  constexpr int kSt = Q8 ? kQR : kFStages;                 // ring slots
  constexpr int kStB = Q8 ? kQSlotBytes : kFStageBytes;    // bytes per slot
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  // partner's partial sums, [token / 4][64 rows][4 tokens]
  float* recv = reinterpret_cast<float*>(smem + ring_bytes<Q8>());
  // table bytes of this CTA's 64 finished rows, [token][64]
  int8_t* gtab = reinterpret_cast<int8_t*>(smem + ring_bytes<Q8>() + kRecvBytes);
  // Q8: per (stage, row) the stage's four block scales, [stage][128 rows]
  uint2* scs = reinterpret_cast<uint2*>(smem + ring_bytes<Q8>() + kRecvBytes + kGtabBytes);
  // f32: full, bready, empty [kSt each]; int8: full, rempty [kQR each], aready,
  // aempty [kQA each]; then accfull, drain, gbar, xbar (the partner's partial
  // sums), sbar (the four sums of squares)
  constexpr int kNB = Q8 ? 2 * kQR + 2 * kQA + 5 : 3 * kSt + 5;
  __shared__ __align__(8) uint64_t bars[kNB];
  __shared__ uint32_t tmem_sh;
  __shared__ int abort_sh;
  __shared__ long long t0_sh;
  __shared__ float red[2][kTok];            // per finishing warp: per-token sums of squares over 32 rows
  __shared__ float ssq_in[kCluster][kTok];  // per cluster rank: sums over its 64 finished rows
  __shared__ __align__(16) float rfac[kTok];   // per-token RMS factor
  __shared__ __align__(16) float tsc[kTok];    // per-token table scale (0 for a bad id)
  __shared__ __align__(16) int tid_sh[kTok];   // per-token id (-1: out of range)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = blockIdx.x & (kCluster - 1);
  const int m = rank & 1, kh = rank >> 1;          // row half, K half
  const int chunk = blockIdx.x / kCluster;
  const int row0 = chunk * kLd + m * kRows;        // first projection row of this CTA
  const int t0 = blockIdx.y * kTok;
  const int ntok = min(kTok, p.S - t0);
  const int npad = (ntok + 15) & ~15;
  // K units: 64-column stages (f32; the last may be half past D, read as
  // zero), a contiguous half per K half; or 128-column stages (int8),
  // interleaved: stage st of K half kh is unit 2 st + kh
  const int nsub = Q8 ? p.D / kQC : (p.D + kFC - 1) / kFC;
  const int sb = kh == 0 ? 0 : (nsub + 1) / 2, se = kh == 0 ? (nsub + 1) / 2 : nsub;   // f32: my units
  const int ns = Q8 ? (nsub + 1 - kh) / 2 : se - sb;   // my stages (0 only when D has one unit)
  const int PLD = p.L * kLd;
  const uint32_t full0 = tc::smem_u32(bars), bready0 = full0 + 8 * kSt, empty0 = bready0 + 8 * kSt;
  const uint32_t rempty0 = bready0;                       // int8: raw slot read (converters + MMA)
  const uint32_t aready0 = full0 + 16 * kQR, aempty0 = aready0 + 8 * kQA;   // int8: A stages
  const uint32_t accfull = full0 + 8 * (kNB - 5), drain = accfull + 8, gbar = drain + 8;
  const uint32_t xbar = gbar + 8, sbar = xbar + 8;
  volatile int* abort_flag = &abort_sh;
  unsigned long long* const tr = (p.trace && blockIdx.x == 0 && blockIdx.y == 0) ? p.trace : nullptr;
  // with a trace: every CTA's start and end (globaltimer ns) after the stage stamps
  unsigned long long* const trc =
      p.trace ? p.trace + kTraceRows * 8 + 2 * ((size_t)blockIdx.y * gridDim.x + blockIdx.x) : nullptr;
  auto stamp = [&](int r, int k) {
    if (tr && r < kTraceRows) tr[r * 8 + k] = (unsigned long long)(tc::clock_ordered() - t0_sh);
  };

  if (threadIdx.x == 0) {
    abort_sh = 0;
    t0_sh = tc::clock_ordered();
    if (trc) trc[0] = tc::globaltimer();
    if constexpr (Q8) {
      for (int s = 0; s < kQR; ++s) {
        tc::mbar_init(full0 + 8 * s, 1);
        tc::mbar_init(rempty0 + 8 * s, 4 + 1);   // the stage's converter group, then the MMA commit
      }
      for (int s = 0; s < kQA; ++s) {
        tc::mbar_init(aready0 + 8 * s, 4);
        tc::mbar_init(aempty0 + 8 * s, 1);
      }
    } else {
      for (int s = 0; s < kSt; ++s) {
        tc::mbar_init(full0 + 8 * s, 1);
        tc::mbar_init(bready0 + 8 * s, kConvWarps);
        tc::mbar_init(empty0 + 8 * s, 1);
      }
    }
    tc::mbar_init(accfull, 1);
    tc::mbar_init(drain, 1);
    tc::mbar_init(gbar, kTok);   // one arrival per token slot
    tc::mbar_init(xbar, 1);
    tc::mbar_init(sbar, 1);
    // the bytes the peers will store here: the partner's partial sums of the
    // 64 rows finished here (npad tokens), and 64 sums of squares from each
    // of the three other CTAs
    tc::mbar_expect_tx(xbar, (uint32_t)(64 * 4 * npad));
    tc::mbar_expect_tx(sbar, (uint32_t)((kCluster - 1) * kTok * 4));
    tc::mbar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(tc::smem_u32(&tmem_sh), tmem_cols<Q8>());
  // programmatic dependent launch: the next kernel in the stream may be
  // scheduled now; this one reads its inputs only after the previous
  // kernel's results are visible
  pdl_trigger();
  pdl_wait();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  // cluster phase 1: every CTA of the cluster has started before anyone
  // stores into a peer's shared memory (waited for just before the first store)
  tc::cluster_arrive_relaxed();
  const uint32_t tmem = tmem_sh;

  if (warp == 0) {
    // ------------------------------------------------------------- TMA loads
    const uint64_t pol_once = tc::policy_evict_first(), pol_keep = tc::policy_evict_last();
    const uint32_t st0 = tc::smem_u32(smem);
    int st = 0;
    for (; st < ns; ++st) {
      const int s = st % kSt, round = st / kSt;
      const bool free_ =
          tc::mbar_wait((Q8 ? rempty0 : empty0) + 8 * s, (round & 1) ^ 1, p.wait_limit, abort_flag, p.dev_err);
      if (!__all_sync(0xffffffffu, free_)) break;
      if constexpr (Q8) {
        if (elect_one()) {
          const uint32_t B = st0 + s * kStB;
          stamp(st, 0);
          tc::mbar_expect_tx(full0 + 8 * s, (uint32_t)(kQRawBytes + kQBBytes));
          // x = 128 (2 st + kh) int8 code bytes / fp16 hidden columns (+ 64): 16-byte aligned
          const int x = (2 * st + kh) * kQC;
          tc::tma_load_2d(B + kQBBytes, &p.tm_proj, x, row0, full0 + 8 * s, pol_once);
          tc::tma_load_2d(B, &p.tm_hid, x, t0, full0 + 8 * s, pol_keep);
          tc::tma_load_2d(B + kQBHalf, &p.tm_hid, x + 64, t0, full0 + 8 * s, pol_keep);
        }
      } else if (elect_one()) {
        const uint32_t A = st0 + s * kFStageBytes;
        stamp(st, 0);
        // x = 64 (sb + st) fp32 / fp16 columns, and + 32: 16-byte aligned (a
        // box wholly past D reads as zeros and still delivers its bytes)
        const int x = (sb + st) * kFC;
        tc::mbar_expect_tx(full0 + 8 * s, (uint32_t)(kFRawBytes + kFHBytes));
        tc::tma_load_2d(A, &p.tm_proj, x, row0, full0 + 8 * s, pol_once);
        tc::tma_load_2d(A + kFBox, &p.tm_proj, x + 32, row0, full0 + 8 * s, pol_once);
        tc::tma_load_2d(A + kFRawBytes, &p.tm_hid, x, t0, full0 + 8 * s, pol_keep);
      }
      __syncwarp();
    }
    // every issued load lands before the CTA may exit
    for (int q = max(0, st - kSt); q < st; ++q)
      tc::mbar_drain(full0 + 8 * (q % kSt), (q / kSt) & 1, kDrainCycles, p.dev_err);
    tc::mbar_drain(gbar, 0, kDrainCycles, p.dev_err);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t st0 = tc::smem_u32(smem);
    const uint32_t idesc = idesc_f16(npad);
    bool ok = true;
    for (int st = 0; st < ns; ++st) {
      const int s = st % kSt, round = st / kSt;
      const int a = st % kQA;   // int8: the A stage in tensor memory
      // bready (aready) completes only after the converter warps have seen
      // this stage's TMA bytes land (full), so it orders the tiles too
      if constexpr (Q8)
        ok = tc::mbar_wait(aready0 + 8 * a, (st / kQA) & 1, p.wait_limit, abort_flag, p.dev_err);
      else
        ok = tc::mbar_wait(bready0 + 8 * s, round & 1, p.wait_limit, abort_flag, p.dev_err);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc::fence_after();
      if (elect_one()) {
        stamp(st, 3);
        if constexpr (Q8) {
          // K step k (16 columns): A columns 8k .. 8k + 7 of stage a; B half
          // k / 4 at byte 32 (k % 4) of each 128-byte row
          const uint32_t B = st0 + s * kStB, A = tmem + kQACol0 + 64 * a;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_f16_ta(tmem, A + 8 * k, tc::desc_sw128(B + (k >> 2) * kQBHalf + 32 * (k & 3)), idesc,
                       (st | k) ? 1u : 0u);
          tc::commit(aempty0 + 8 * a);
          tc::commit(rempty0 + 8 * s);
        } else {
          // D1 (columns 0-63) += P1 . h, D2 (columns 64-127) += P2 . h; K
          // step k (16 columns) of piece h sits in box k / 2 at byte
          // 64 h + 32 (k % 2) of each 128-byte row
          const uint32_t A = st0 + s * kStB, H = A + kFRawBytes;
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int k = 0; k < 4; ++k)   // K = 16 fp16 (32 bytes) per MMA
              mma_f16(tmem + 64 * h, tc::desc_sw128(A + (k >> 1) * kFBox + 64 * h + 32 * (k & 1)),
                      tc::desc_sw128(H + 32 * k), idesc, (st | k) ? 1u : 0u);
          tc::commit(empty0 + 8 * s);
        }
        stamp(st, 4);
      }
      __syncwarp();
    }
    if (elect_one()) {
      if (ok && ns > 0) tc::commit(accfull);
      // every tcgen05 operation issued here has finished before TMEM is freed
      tc::commit(drain);
    }
    __syncwarp();
    tc::mbar_drain(drain, 0, kDrainCycles, p.dev_err);
  } else {
    // ------------------------------------- converters (warps 2-9), epilogue (2-5)
    const int cv = threadIdx.x - kEpi0 * 32;   // converter thread 0..255
    const int ct = cv;                         // epilogue thread 0..127 (warps 2-5)
    const bool epi = cv < 128;
    // token ct's id; the table bytes of the finished rows: one 64-byte copy
    // per valid token, issued by that token's thread (column row0 + 64 kh and
    // the row width L * 256 are multiples of 16 bytes) after it has posted
    // the 64 bytes on gbar; every token slot arrives once, so no thread has to
    // count the valid ids.  The token's table scale is only needed by the
    // epilogue: its load stays in flight through the stage loop.
    int my_id = -1;
    float my_sc = 0.f;
    // the norm weights of the four output columns this epilogue thread
    // finishes (4 (ct % 16) .. + 3 of the 64 finished here), in flight
    // through the stage loop
    float my_nw[4] = {0.f, 0.f, 0.f, 0.f};
    if (epi) {
#pragma unroll
      for (int j = 0; j < 4; ++j) my_nw[j] = p.norm_w[m * kRows + 64 * kh + 4 * (ct & 15) + j];
    }
    if (epi && ct < ntok) {
      const int v = p.ids[t0 + ct];
      if (v >= 0 && v < p.V)
        my_id = v;
      else if (p.err)
        atomicExch(p.err, 1);
    }
    if (epi && ct < kTok) {
      tid_sh[ct] = my_id;
      if (my_id >= 0) {
        tc::mbar_expect_tx(gbar, 64u);
        tc::bulk_load(tc::smem_u32(gtab + ct * 64), p.table + (size_t)my_id * PLD + (size_t)row0 + 64 * kh, 64,
                      gbar, tc::policy_evict_first());
        my_sc = p.row_scale[my_id];
      } else {   // no copy: the gathered bytes are zero
        for (int e = 0; e < 64; e += 16) *reinterpret_cast<uint4*>(gtab + ct * 64 + e) = make_uint4(0u, 0u, 0u, 0u);
        tc::mbar_arrive(gbar);
      }
    }
    if constexpr (Q8) {
      // the block scales of the row this thread converts, for the stages of
      // its group (row stride D/128 quads), all loads in flight together;
      // the thread reads back only what it wrote, so no barrier is needed
      const int grp = (warp - kEpi0) >> 2, r = 32 * (warp & 3) + lane;
      const uint2* src = p.proj_sc + (size_t)(row0 + r) * (p.D / kQC) + kh;
      uint2 v[kQMaxStages / 2];
#pragma unroll
      for (int u = 0; u < kQMaxStages / 2; ++u)
        v[u] = grp + 2 * u < ns ? __ldg(src + 2 * (grp + 2 * u)) : make_uint2(0u, 0u);
#pragma unroll
      for (int u = 0; u < kQMaxStages / 2; ++u)
        if (grp + 2 * u < ns) scs[(grp + 2 * u) * kRows + r] = v[u];
    }
    bool ok = true;
    if constexpr (Q8) {
      // ------------------------ A operand: int8 codes -> fp16 tensor memory
      // two groups of four warps take alternate stages; thread = projection
      // row r (its warp's TMEM lane quarter): it reads the row's 128 codes
      // (8 swizzled 16-byte groups: a quarter-warp of eight consecutive rows
      // hits eight distinct bank groups), releases the raw slot, and writes
      // the 64 columns of fp16 pairs of its lane in the stage's A columns
      const int grp = (warp - kEpi0) >> 2;
      const int r = 32 * (warp & 3) + lane, r8 = r & 7;
      const uint32_t a_lane = tmem + kQACol0 + ((uint32_t)(32 * (warp & 3)) << 16);
      for (int st = grp; st < ns; st += 2) {
        const int s = st % kSt, round = st / kSt, a = st % kQA;
        const bool landed = tc::mbar_wait(full0 + 8 * s, round & 1, p.wait_limit, abort_flag, p.dev_err);
        if (!__all_sync(0xffffffffu, landed)) {   // leave the loop as a whole warp
          ok = false;
          break;
        }
        if (ct == 0) stamp(st, 1);
        const uint8_t* raw = smem + (size_t)s * kStB + kQBBytes + r * kQC;
        uint4 c[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) c[g] = *reinterpret_cast<const uint4*>(raw + ((g ^ r8) << 4));
        const uint2 s4 = scs[st * kRows + r];   // scales of columns 0-31, 32-63 (x), 64-95, 96-127 (y)
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(rempty0 + 8 * s);
        const bool freed = tc::mbar_wait(aempty0 + 8 * a, ((st / kQA) & 1) ^ 1, p.wait_limit, abort_flag, p.dev_err);
        if (!__all_sync(0xffffffffu, freed)) {
          ok = false;
          break;
        }
        tc::fence_after();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {   // columns 64 hh .. 64 hh + 63: blocks 2 hh, 2 hh + 1
          const uint32_t sw = hh ? s4.y : s4.x;
          uint32_t v[32];
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const __half2 dd = __half2half2(__ushort_as_half((uint16_t)(g < 2 ? sw & 0xFFFFu : sw >> 16)));
            const uint4 cc = c[4 * hh + g];
            const uint4 lo = dequant_i8_f16(make_uint2(cc.x, cc.y), dd);
            const uint4 hi = dequant_i8_f16(make_uint2(cc.z, cc.w), dd);
            v[8 * g + 0] = lo.x;
            v[8 * g + 1] = lo.y;
            v[8 * g + 2] = lo.z;
            v[8 * g + 3] = lo.w;
            v[8 * g + 4] = hi.x;
            v[8 * g + 5] = hi.y;
            v[8 * g + 6] = hi.z;
            v[8 * g + 7] = hi.w;
          }
          tc::tmem_st32(a_lane + 64 * a + 32 * hh, v);
        }
        tc::fence_before();   // this warp's TMEM stores, before the MMA issuer reads them
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(aready0 + 8 * a);
        if (ct == 0) stamp(st, 2);
      }
    } else {
      // ------------------------- A operands: raw f32 tile -> pieces P1, P2
      // thread cv = (projection row r, box hc): its 128-byte row of raw box
      // hc (columns 32 hc .. 32 hc + 31) becomes, in place, 64 bytes of P1
      // (16-byte groups 0-3: those columns of P1) followed by 64 bytes of P2
      // (groups 4-7), so a thread overwrites only what it read itself.  Both
      // layouts put 16-byte group g of row r at group g ^ (r % 8) of its row,
      // so a quarter-warp (eight consecutive rows) touches eight distinct banks
      const int r = cv & 127, hc = cv >> 7, r8 = r & 7;
      for (int st = 0; st < ns; ++st) {
        const int s = st % kSt, round = st / kSt;
        const bool landed = tc::mbar_wait(full0 + 8 * s, round & 1, p.wait_limit, abort_flag, p.dev_err);
        if (!__all_sync(0xffffffffu, landed)) {   // leave the loop as a whole warp
          ok = false;
          break;
        }
        if (ct == 0) stamp(st, 1);
        uint8_t* row_p = smem + (size_t)s * kFStageBytes + (r >> 3) * 1024 + r8 * 128;
        float w[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {   // floats 4c .. 4c+3 of box hc
          const float4 f = *reinterpret_cast<const float4*>(row_p + hc * kFBox + ((c ^ r8) << 4));
          w[4 * c] = f.x;
          w[4 * c + 1] = f.y;
          w[4 * c + 2] = f.z;
          w[4 * c + 3] = f.w;
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) {     // columns 32 hc + 8 g .. + 7
          float v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = w[8 * g + e];
          uint4 p1, p2;
          split_f32_f16(v, p1, p2);
          *reinterpret_cast<uint4*>(row_p + hc * kFBox + ((g ^ r8) << 4)) = p1;
          *reinterpret_cast<uint4*>(row_p + hc * kFBox + (((4 + g) ^ r8) << 4)) = p2;
        }
        tc::fence_proxy_async();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bready0 + 8 * s);
        if (ct == 0) stamp(st, 2);
      }
    }
    if (!epi) {
      tc::cluster_wait();   // conversion-only warps: the one cluster phase, like the TMA and MMA warps
    } else {
      // ----------------------------------------------------------- epilogue
      if (ct < kTok) tsc[ct] = my_sc;            // read after the barriers below
      const int q = warp & 3;                    // TMEM lane quarter
      const int row = 32 * q + lane;             // row of this CTA's tile
      const bool mine = (q >> 1) == kh;          // rows 64 kh .. 64 kh + 63 are finished here
      const int r64 = row & 63;
      const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16);
      const bool has = ns > 0;                   // without K work the partial sums are zero
      if (ok && has) ok = tc::mbar_wait(accfull, 0, p.wait_limit, abort_flag, p.dev_err);
      ok = __all_sync(0xffffffffu, ok);          // the TMEM loads below are warp-wide
      tc::fence_after();
      if (ct == 0) stamp(kTraceRows - 1, 5);
      // this row's accumulator columns (one per token): one load and one wait
      float acc[kTok];
      if (ok && has) {
        tc::tmem_ld64(taddr, acc);
        if constexpr (!Q8) {   // p = D1 + D2 * 2^-11 (the scaling is exact: one rounding)
          float acc2[kTok];
          tc::tmem_ld64(taddr + 64, acc2);
  #pragma unroll
          for (int u = 0; u < kTok; ++u) acc[u] = fmaf(acc2[u], 0x1p-11f, acc[u]);
        }
      } else {
  #pragma unroll
        for (int u = 0; u < kTok; ++u) acc[u] = 0.f;
      }
      tc::cluster_wait();                        // every peer is running (its barriers initialised)
      if (ct == 0) stamp(kTraceRows - 2, 0);
      // Partial sums and sums of squares go to the peers as stores that count
      // their bytes on the receiver's xbar / sbar; they are sent even after a
      // failed wait (with whatever values), so every receiver's byte count is
      // met and no CTA leaves while a peer may still store into it.
      if (!mine) {                               // the partner finishes these rows
        const uint32_t peer = tc::cluster_addr(recv, (uint32_t)(rank ^ 2));
        const uint32_t peer_bar = tc::cluster_addr(&bars[kNB - 2], (uint32_t)(rank ^ 2));
  #pragma unroll
        for (int cb = 0; cb < kTok / 16; ++cb) {
          if (cb < npad / 16) {
  #pragma unroll
            for (int g = 0; g < 4; ++g) {   // tokens 16 cb + 4 g .. + 3 of this row
              const int u = 16 * cb + 4 * g;
              tc::st_async_v4(peer + (uint32_t)((((cb * 4 + g) * 64) + r64) * 16), acc[u], acc[u + 1], acc[u + 2],
                              acc[u + 3], peer_bar);
            }
          }
        }
      } else {                                   // the partner's partial sums of these rows
        const bool g = tc::mbar_wait(xbar, 0, p.wait_limit, abort_flag, p.dev_err);
        ok = __all_sync(0xffffffffu, ok && g);
      }
      if (ct == 0) stamp(kTraceRows - 2, 1);
      // p = (K half 0) + (K half 1), the same order in both CTAs; the four token
      // groups' reductions are independent of one another
      float pv[kTok];   // this row's projection sums
  #pragma unroll
      for (int cb = 0; cb < kTok / 16; ++cb) {
        if (mine && cb < npad / 16) {   // warp-uniform
  #pragma unroll
          for (int g = 0; g < 4; ++g) {
            const float4 o4 = *reinterpret_cast<const float4*>(recv + (((cb * 4 + g) * 64) + r64) * 4);
            const float other[4] = {o4.x, o4.y, o4.z, o4.w};
  #pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int u = 16 * cb + 4 * g + e;
              pv[u] = kh == 0 ? acc[u] + other[e] : other[e] + acc[u];
            }
          }
        } else {
  #pragma unroll
          for (int u = 0; u < 16; ++u) pv[cb * 16 + u] = 0.f;
        }
      }
  #pragma unroll
      for (int cb = 0; cb < kTok / 16; ++cb) {
        if (mine && cb < npad / 16) {
          float v[16];
  #pragma unroll
          for (int u = 0; u < 16; ++u) v[u] = pv[cb * 16 + u] * pv[cb * 16 + u];
          const float s2 = lane_token_sums16(v, lane);
          if ((lane & 1) == 0) red[q & 1][cb * 16 + (lane >> 1)] = s2;
        }
      }
      // every read of the partner's partial sums is done (recv becomes the
      // output tile), and the per-warp sums of squares are in red
      asm volatile("bar.sync 1, 128;" ::: "memory");
      float* tile = recv;   // [64 tokens][64 columns] f32
      if (ct < kTok) {   // warps 2 and 3: this CTA's sums to the three peers
        const float own = red[0][ct] + red[1][ct];   // rows in order within this CTA's 64
        ssq_in[rank][ct] = own;   // read back by this thread only
  #pragma unroll
        for (int d = 1; d < kCluster; ++d) {
          const uint32_t r = (uint32_t)((rank + d) & (kCluster - 1));
          tc::st_async_f32(tc::cluster_addr(&ssq_in[rank][ct], r), own, tc::cluster_addr(&bars[kNB - 1], r));
        }
      }
      if (mine) {   // the finished sums into the tile while the peers' sums travel
  #pragma unroll
        for (int cb = 0; cb < kTok / 16; ++cb)
          if (cb < npad / 16) {
  #pragma unroll
            for (int u = 0; u < 16; ++u) tile[(cb * 16 + u) * 64 + r64] = pv[cb * 16 + u];
          }
      }
      if (ct < kTok) {
        // all four row quarters' sums are here
        const bool g = tc::mbar_wait(sbar, 0, p.wait_limit, abort_flag, p.dev_err);
        if (!__all_sync(0xffffffffu, g)) ok = false;
        if (ct == 0) stamp(kTraceRows - 2, 2);
        rfac[ct] = 1.f / sqrtf((((ssq_in[0][ct] + ssq_in[1][ct]) + ssq_in[2][ct]) + ssq_in[3][ct]) / (float)kLd +
                               p.eps);
      }
      {   // the gathered table bytes
        const bool g = ok && tc::mbar_wait(gbar, 0, p.wait_limit, abort_flag, p.dev_err);
        ok = __all_sync(0xffffffffu, g);
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (*abort_flag) ok = false;   // a wait of another epilogue warp gave up
      if (ct == 0) stamp(kTraceRows - 1, 6);
      if (ok) {
        // out = p * rfac * norm_w + (q * s) * 16 in place, thread = (token
        // t = ct / 16 + 8 k, columns 4 (ct % 16) .. + 3); padding tokens are
        // outside the tensor and not written; a bad id gives zeros
        const int cg = ct & 15;
        const float es = p.embed_scale;
  #pragma unroll
        for (int k = 0; k < kTok / 8; ++k) {
          const int t = (ct >> 4) + 8 * k;
          float4 v = *reinterpret_cast<const float4*>(tile + t * 64 + 4 * cg);
          const uint32_t tq = *reinterpret_cast<const uint32_t*>(gtab + t * 64 + 4 * cg);
          const float rf = rfac[t], sc = tsc[t];
          const bool good = tid_sh[t] >= 0;
          float* e = &v.x;
  #pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float g = __fmul_rn(__fmul_rn((float)(int8_t)(tq >> (8 * j)), sc), es);
            e[j] = good ? e[j] * rf * my_nw[j] + g : 0.f;
          }
          *reinterpret_cast<float4*>(tile + t * 64 + 4 * cg) = v;
        }
      }
      tc::fence_proxy_async();   // the tile (and the zeroed table rows) before the tensor stores read them
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (ct == 0 && ok) {
        const int x = row0 + 64 * kh;   // 64 f32 = 256 bytes, 64 int8: 16-byte aligned
        tc::tma_store_2d(&p.tm_out, x, t0, tc::smem_u32(recv));
        if (p.gathered) tc::tma_store_2d(&p.tm_gat, x, t0, tc::smem_u32(gtab));
        tc::bulk_commit();
        tc::bulk_wait_read_all();   // the tile has been read; the writes complete with the grid
      }
      if (mine && (q & 1) == 0 && lane == 0) stamp(kTraceRows - 2, 3);
      if (ct == 0) stamp(kTraceRows - 1, 7);
    }
  }
  if (warp < kEpi0) tc::cluster_wait();   // the TMA and MMA warps take part in the cluster phase too
  if (warp == kEpi0) {
    // every store a peer makes into this CTA has landed before it leaves
    // (already so unless a wait above gave up)
    tc::mbar_drain(xbar, 0, kDrainCycles, p.dev_err);
    tc::mbar_drain(sbar, 0, kDrainCycles, p.dev_err);
  }
  tc::fence_before();
  __syncthreads();
  if (trc && threadIdx.x == 0) trc[1] = tc::globaltimer();
  if (threadIdx.x == 0) stamp(kTraceRows - 2, 4);
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, tmem_cols<Q8>());
  }
}

}  // namespace ple

// proj: f32 [L*ld][D], or (Q8) int8 codes [L*ld][D] with fp16 scales proj_sc [L*ld][D/32].
template <bool Q8>
static int launch_ple_t(const int32_t* ids, int S, const int8_t* table, const float* row_scale, int V, int L,
                        int ld, float embed_scale, const void* proj, const uint16_t* proj_sc, const __half* hidden,
                        int D, const float* norm_w, float eps, float* out, int8_t* gathered, int32_t* err,
                        const DeviceInfo& dev, cudaStream_t s) {
  if (ld != ple::kLd) return fail(Q4_ERR_SHAPE, "ple_gather_project: ld must be %d", ple::kLd);
  ple::Params p;
  memset(&p, 0, sizeof(p));
  int st;
  if (Q8) {
    st = encode_tensor_2d(&p.tm_proj, proj, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)D, (uint64_t)L * ld, ple::kQC,
                          ple::kRows, CU_TENSOR_MAP_SWIZZLE_128B, "proj_codes");
    if (st != Q4_OK) return st;
    st = encode_tensor_2d(&p.tm_hid, hidden, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, (uint64_t)D, (uint64_t)S, 64,
                          ple::kTok, CU_TENSOR_MAP_SWIZZLE_128B, "hidden");
    if (st != Q4_OK) return st;
    p.proj_sc = reinterpret_cast<const uint2*>(proj_sc);
  } else {
    st = encode_tensor_2d(&p.tm_proj, proj, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)D, (uint64_t)L * ld, 32,
                          ple::kRows, CU_TENSOR_MAP_SWIZZLE_128B, "proj");
    if (st != Q4_OK) return st;
    st = encode_tensor_2d(&p.tm_hid, hidden, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, (uint64_t)D, (uint64_t)S, ple::kFC,
                          ple::kTok, CU_TENSOR_MAP_SWIZZLE_128B, "hidden");
    if (st != Q4_OK) return st;
  }
  st = encode_tensor_2d(&p.tm_out, out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)L * ld, (uint64_t)S, 64,
                        ple::kTok, CU_TENSOR_MAP_SWIZZLE_NONE, "out");
  if (st != Q4_OK) return st;
  if (gathered) {
    st = encode_tensor_2d(&p.tm_gat, gathered, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)L * ld, (uint64_t)S, 64,
                          ple::kTok, CU_TENSOR_MAP_SWIZZLE_NONE, "gathered");
    if (st != Q4_OK) return st;
  }
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
  const size_t trace_words =
      (size_t)ple::kTraceRows * 8 + 2 * (size_t)ple::kCluster * L * ((S + ple::kTok - 1) / ple::kTok);
  p.trace = (tb && tbytes >= trace_words * sizeof(unsigned long long))
                ? static_cast<unsigned long long*>(tb)
                : nullptr;
  constexpr size_t smem = ple::smem_bytes<Q8>();
  static PerDevice attr;
  cudaError_t e;
  if (!attr.get(dev.ordinal)) {
    e = cudaFuncSetAttribute(ple::ple_tc_kernel<Q8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "ple smem attribute");
    attr.set(dev.ordinal);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ple::kCluster * L, (S + ple::kTok - 1) / ple::kTok);
  cfg.blockDim = dim3(ple::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = ple::kCluster;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, ple::ple_tc_kernel<Q8>, p);
  return e == cudaSuccess ? Q4_OK : cuda_fail(e, "ple launch");
}

int launch_ple(const int32_t* ids, int S, const int8_t* table, const float* row_scale, int V, int L,
               int ld, float embed_scale, const float* proj, const __half* hidden, int D,
               const float* norm_w, float eps, float* out, int8_t* gathered, int32_t* err,
               const DeviceInfo& dev, cudaStream_t s) {
  return launch_ple_t<false>(ids, S, table, row_scale, V, L, ld, embed_scale, proj, nullptr, hidden, D, norm_w, eps,
                             out, gathered, err, dev, s);
}

int launch_ple_q8(const int32_t* ids, int S, const int8_t* table, const float* row_scale, int V, int L, int ld,
                  float embed_scale, const int8_t* proj_codes, const uint16_t* proj_scales, const __half* hidden,
                  int D, const float* norm_w, float eps, float* out, int8_t* gathered, int32_t* err,
                  const DeviceInfo& dev, cudaStream_t s) {
  if (D % ple::kQC != 0 || D > 2 * ple::kQMaxStages * ple::kQC)
    return fail(Q4_ERR_SHAPE, "ple_gather_project_q8: D=%d must be a multiple of %d up to %d", D, ple::kQC,
                2 * ple::kQMaxStages * ple::kQC);
  return launch_ple_t<true>(ids, S, table, row_scale, V, L, ld, embed_scale, proj_codes, proj_scales, hidden, D,
                            norm_w, eps, out, gathered, err, dev, s);
}

}  // namespace q4w
