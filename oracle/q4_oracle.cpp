// CPU oracle of the q4_0 weight-only int4 decode path, in plain C++17.
//
// TEST INFRASTRUCTURE ONLY: the test-suite, the package smoke check and the
// benchmark's CPU baseline / reference arm load it (through oracle/cpp_oracle.py);
// nothing on the product path does.  It shares no code with the CUDA library
// and includes none of its headers.
//
// Plain and slow on purpose: one loop per definition, sums in fp64 in index
// order, no blocking, vectors or fused multiply-adds (built with
// -ffp-contract=off -fno-fast-math).  Rows of a contraction may be split over
// std::thread; each row is summed by one thread in one fixed order, so the
// thread count never changes a result bit.  Number-format conversions are
// written from the IEEE-754 binary16 / bfloat16 definitions.
//
// Sources (page title, section) -- the same passages the numpy oracle follows:
//   "visible-cx/gemma-4-E2B-CoreAI": Provenance (q4_0 per-block-32 grid; S=1
//     main and S=64 prefill exports); The PLE gather-table sidecar (V 262144,
//     L 35, ld 256, embed scale 16.0 = sqrt(256), f32 projection, [256] norm).
//   "Gemma 4 E2B (text decoder) - Core AI": Signature features (35 layers,
//     dual head_dim, KV-sharing, double-wide MLP, tanh(z/30)*30 softcap,
//     RMSNorm weight applied directly); QAT weights (absmax symmetric int4);
//     What it took (head with in-kernel argmax).
//   "Gemma-4 E2B mobile mixed-bit QAT weights": P6 (unsigned code minus 8);
//     decode recipe (layer shapes, low nibble first); Speed (gate/up matvecs +
//     fp32 precise-tanh GELU + mul).
// Readings where the pages are silent (identical to the numpy oracle's):
//   R1 quantiser rounds the IEEE fp32 quotient w / d32 half away from zero,
//      d32 = m / -8 in fp32, scale stored as fp16 (nearest even);
//   R2 m = first element of largest |w| in k order; R3 zero block: d = +0,
//      codes 8; R4 RMSNorm eps 1e-6 (passed in), chain weight 1;
//   R5 PLE gathered term (float(q) * scale) * 16 in fp32, proj [L*ld][D];
//   R6 head ties -> lowest index, top-2 over the other rows, softcapped units;
//   R7 S=64 tiles rounded to bf16 (nearest even) before an exact sum;
//   R8 per layer: a = f16(RMSNorm(h)); q,k,v = W a; o = W_o f16(q);
//      b = f16(RMSNorm(o)); g,u = W b; m = f16(gelu_tanh(g) * u);
//      h' = f16(RMSNorm(W_d m)); k, v produced and not consumed.
// The "next" rows, with the numpy oracles' readings:
//   Q2 ("Gemma-4 E2B mobile mixed-bit QAT weights", decode recipe, P3, P6):
//      4 codes per byte, the first in bits [1:0], value code - 2, one f32
//      scale per row applied to the finished row sum;
//   Q8 (same page, decode recipe and official-checkpoint notes): per block
//      of 32, d = max |w| / 127 (fp32), code = clamp(round(w / d), -127,
//      127) from the fp32 quotient, half away from zero, scale fp16(d); a
//      zero block stores +0 and codes 0; the PLE on it is the f32 PLE on
//      w' = fp16(d) * code;
//   A8 ("visible-cx/gemma-4-E2B-CoreAI", About the w4a8 bundle): per-tensor
//      symmetric, zero point 0, fp32 scale s; q = clamp(rint(x / s), -128,
//      127) from the fp32 quotient, ties to even; x' = s q; min-max
//      calibration s = max |x| / 127 (fp32), 1 when every x is zero.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ------------------------------------------------------------ formats ---
// binary16 bits -> value (exact in double).
double f16_value(uint16_t h) {
  const int sign = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0)
    v = std::ldexp((double)m, -24);               // subnormal: m * 2^-24
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = std::ldexp((double)(m | 1024), e - 25);   // 1.m * 2^(e-15)
  return sign ? -v : v;
}

// double -> nearest binary16 (ties to even), one rounding from the exact value.
uint16_t f16_bits(double x) {
  if (std::isnan(x)) return 0x7e00;
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  const double a = std::fabs(x);
  if (a >= 65520.0) return sign | 0x7c00;   // at or past 65504 + half a step: infinity
  if (a < std::ldexp(1.0, -14)) {            // subnormal range: multiples of 2^-24
    const double r = std::nearbyint(std::ldexp(a, 24));   // 1024 reads as the smallest normal
    return sign | (uint16_t)r;
  }
  int e = 0;
  std::frexp(a, &e);                          // a in [2^(e-1), 2^e)
  const double r = std::nearbyint(std::ldexp(a, 11 - e));   // 11 significant bits
  int E = e - 1 + 15;
  uint32_t mant = (uint32_t)r;
  if (mant == 2048) {                         // rounded up to the next binade
    mant = 1024;
    E += 1;
  }
  if (E >= 31) return sign | 0x7c00;
  return sign | (uint16_t)(E << 10) | (uint16_t)(mant - 1024);
}

// float -> nearest bfloat16 (ties to even), kept as a float (finite inputs).
float bf16_round(float v) {
  uint32_t u;
  std::memcpy(&u, &v, 4);
  const uint64_t w = u;
  const uint64_t r = (w + 0x7fffu + ((w >> 16) & 1u)) >> 16;
  const uint32_t o = (uint32_t)(r << 16);
  float f;
  std::memcpy(&f, &o, 4);
  return f;
}

// ------------------------------------------------------------ threads ---
template <class F>
void parallel_rows(int n, int threads, F f) {
  if (threads <= 1 || n < 2) {
    f(0, n);
    return;
  }
  if (threads > n) threads = n;
  std::vector<std::thread> ts;
  for (int t = 0; t < threads; ++t) {
    const int lo = (int)((long long)n * t / threads), hi = (int)((long long)n * (t + 1) / threads);
    ts.emplace_back(f, lo, hi);
  }
  for (auto& t : ts) t.join();
}

// code of weight (n, k): byte k/2 of the row, low nibble for even k
inline int code_at(const uint8_t* codes, int K, int n, int k) {
  const uint8_t b = codes[(size_t)n * (K / 2) + k / 2];
  return (k & 1) ? (b >> 4) : (b & 15);
}

// w'[n][k] = d * (code - 8), exact in double
inline double weight_at(const uint8_t* codes, const uint16_t* scales, int K, int n, int k) {
  return f16_value(scales[(size_t)n * (K / 32) + k / 32]) * (double)(code_at(codes, K, n, k) - 8);
}

double rms_factor(const double* v, int n, double eps) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += v[i] * v[i];
  return 1.0 / std::sqrt(ss / n + eps);
}

double gelu_tanh_value(double x) {
  const double c = std::sqrt(2.0 / M_PI);
  return 0.5 * x * (1.0 + std::tanh(c * (x + 0.044715 * x * x * x)));
}

}  // namespace

extern "C" {

int q4o_version(void) { return 1; }

// ---------------------------------------------------------- conversions ---
void q4o_f16_from_f64(const double* x, uint16_t* bits, long long n) {
  for (long long i = 0; i < n; ++i) bits[i] = f16_bits(x[i]);
}

void q4o_f64_from_f16(const uint16_t* bits, double* x, long long n) {
  for (long long i = 0; i < n; ++i) x[i] = f16_value(bits[i]);
}

void q4o_bf16_rne(const float* in, float* out, long long n) {
  for (long long i = 0; i < n; ++i) out[i] = bf16_round(in[i]);
}

// -------------------------------------------------------- a1 quantise ---
// W fp32 [N][K] -> codes [N][K/2], fp16 scale bits [N][K/32].
// 0 ok; 1 K not a multiple of 32; 2 a non-finite weight; 3 a scale beyond fp16.
// Rows may be split over threads (each row is quantised by one thread).
int q4o_quantize(const float* W, int N, int K, uint8_t* codes, uint16_t* scales, int threads) {
  if (N < 0 || K <= 0 || K % 32) return 1;
  for (long long i = 0; i < (long long)N * K; ++i)
    if (!std::isfinite(W[i])) return 2;
  const int nb = K / 32;
  // a scale beyond fp16 is an error for the whole matrix, checked first
  for (long long i = 0; i < (long long)N * nb; ++i) {
    const float* blk = W + i * 32;
    float m = blk[0];
    for (int t = 1; t < 32; ++t)
      if (std::fabs(blk[t]) > std::fabs(m)) m = blk[t];
    if (std::fabs(m / -8.0f) > 65504.0f) return 3;
  }
  parallel_rows(N, threads, [&](int lo, int hi) {
  for (int n = lo; n < hi; ++n) {
    for (int j = 0; j < nb; ++j) {
      const float* blk = W + (size_t)n * K + 32 * j;
      float m = blk[0];
      for (int i = 1; i < 32; ++i)
        if (std::fabs(blk[i]) > std::fabs(m)) m = blk[i];   // first of the largest
      float d32 = m / -8.0f;                                 // exact
      if (m == 0.0f) d32 = 0.0f;                             // +0 (R3)
      scales[(size_t)n * nb + j] = f16_bits((double)d32);
      uint8_t q[32];
      for (int i = 0; i < 32; ++i) {
        if (d32 == 0.0f) {
          q[i] = 8;
          continue;
        }
        const float ratio = blk[i] / d32;                    // IEEE fp32 quotient
        double c = (double)std::round(ratio) + 8.0;          // half away from zero (R1)
        if (c < 0.0) c = 0.0;
        if (c > 15.0) c = 15.0;
        q[i] = (uint8_t)c;
      }
      for (int b = 0; b < 16; ++b) codes[(size_t)n * (K / 2) + 16 * j + b] = (uint8_t)(q[2 * b] | (q[2 * b + 1] << 4));
    }
  }
  });
  return 0;
}

// w' = d * (code - 8) for every weight, in double.
void q4o_dequantize(const uint8_t* codes, const uint16_t* scales, int N, int K, double* Wd) {
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) Wd[(size_t)n * K + k] = weight_at(codes, scales, K, n, k);
}

// ------------------------------------------------------------ a2 GEMV ---
// y[b][n] = sum_k w'[n][k] * x[b][k], fp64 in k order.  x: fp16 bits [B][K].
void q4o_gemv(const uint8_t* codes, const uint16_t* scales, const uint16_t* x, int N, int K, int B, double* y,
              int threads) {
  std::vector<double> xv((size_t)B * K);
  for (size_t i = 0; i < xv.size(); ++i) xv[i] = f16_value(x[i]);
  parallel_rows(N, threads, [&](int lo, int hi) {
    for (int n = lo; n < hi; ++n)
      for (int b = 0; b < B; ++b) {
        double acc = 0.0;
        for (int k = 0; k < K; ++k) acc += weight_at(codes, scales, K, n, k) * xv[(size_t)b * K + k];
        y[(size_t)b * N + n] = acc;
      }
  });
}

// ------------------------------------------------------- a6 S=64 GEMM ---
// Y[t][n] = sum_k bf16(w'[n][k]) * bf16(x[t][k]), fp64 in k order (R7).
void q4o_gemm_chunk(const uint8_t* codes, const uint16_t* scales, const uint16_t* X, int M, int N, int K, double* Y,
                    int threads) {
  std::vector<double> xt((size_t)M * K);
  for (size_t i = 0; i < xt.size(); ++i) xt[i] = (double)bf16_round((float)f16_value(X[i]));
  parallel_rows(N, threads, [&](int lo, int hi) {
    std::vector<double> wt(K);
    for (int n = lo; n < hi; ++n) {
      for (int k = 0; k < K; ++k) wt[k] = (double)bf16_round((float)weight_at(codes, scales, K, n, k));
      for (int t = 0; t < M; ++t) {
        double acc = 0.0;
        for (int k = 0; k < K; ++k) acc += wt[k] * xt[(size_t)t * K + k];
        Y[(size_t)t * N + n] = acc;
      }
    }
  });
}

// ------------------------------------------------------------ a5 head ---
void q4o_softcap(const double* z, double* s, long long n, double cap) {
  for (long long i = 0; i < n; ++i) s[i] = std::tanh(z[i] / cap) * cap;
}

// Per row b of h: z = W' h (fp64), s = tanh(z / cap) * cap; idx = first
// argmax of s, top1 = s[idx], top2 = largest s over the other rows (-inf when
// V == 1).  s_out [B][V] is optional.
void q4o_lmhead(const uint8_t* codes, const uint16_t* scales, const uint16_t* h, int B, int V, int K, double cap,
                int32_t* idx, double* top1, double* top2, double* s_out, int threads) {
  std::vector<double> z((size_t)B * V);
  q4o_gemv(codes, scales, h, V, K, B, z.data(), threads);
  for (int b = 0; b < B; ++b) {
    std::vector<double> s(V);
    for (int v = 0; v < V; ++v) s[v] = std::tanh(z[(size_t)v + (size_t)b * V] / cap) * cap;
    int best = 0;
    for (int v = 1; v < V; ++v)
      if (s[v] > s[best]) best = v;
    double second = -INFINITY;
    for (int v = 0; v < V; ++v)
      if (v != best && s[v] > second) second = s[v];
    idx[b] = best;
    top1[b] = s[best];
    top2[b] = second;
    if (s_out)
      for (int v = 0; v < V; ++v) s_out[(size_t)b * V + v] = s[v];
  }
}

// ------------------------------------------------------ norms, GELU ---
// out = (v * rsqrt(mean(v^2) + eps)) * w over each row of n values; w optional.
void q4o_rmsnorm(const double* v, const double* w, double eps, long long rows, int n, double* out) {
  for (long long r = 0; r < rows; ++r) {
    const double* x = v + r * n;
    const double f = rms_factor(x, n, eps);
    for (int i = 0; i < n; ++i) {
      const double t = x[i] * f;
      out[r * n + i] = w ? t * w[i] : t;
    }
  }
}

void q4o_gelu_tanh(const double* x, double* y, long long n) {
  for (long long i = 0; i < n; ++i) y[i] = gelu_tanh_value(x[i]);
}

// ------------------------------------------------------------- a4 PLE ---
double q4o_ple_embed_scale(void) { return 16.0; }   // sqrt(256): the sidecar's embed_scale_pl

// out[s][c] = RMSNorm_chunk(p)[s][c] * norm_w[c % ld] + g[s][c] with
//   g = (float(table[id][c]) * row_scale[id]) * embed_scale in fp32 and
//   p[s][r] = sum_d proj[r][d] * hidden[s][d] in fp64, chunks of ld values.
// gathered [S][L*ld] (optional) = the table rows.  0 ok; 1 an id out of range.
int q4o_ple(const int32_t* ids, int S, const int8_t* table, const float* row_scale, int V, int L, int ld,
            float embed_scale, const float* proj, const uint16_t* hidden, int D, const float* norm_w, double eps,
            double* out, int8_t* gathered, int threads) {
  for (int s = 0; s < S; ++s)
    if (ids[s] < 0 || ids[s] >= V) return 1;
  const int R = L * ld;
  std::vector<double> hid((size_t)S * D);
  for (size_t i = 0; i < hid.size(); ++i) hid[i] = f16_value(hidden[i]);
  std::vector<double> p((size_t)S * R);
  parallel_rows(R, threads, [&](int lo, int hi) {
    for (int r = lo; r < hi; ++r)
      for (int s = 0; s < S; ++s) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += (double)proj[(size_t)r * D + d] * hid[(size_t)s * D + d];
        p[(size_t)s * R + r] = acc;
      }
  });
  for (int s = 0; s < S; ++s) {
    const int id = ids[s];
    for (int l = 0; l < L; ++l) {
      const double* chunk = p.data() + (size_t)s * R + (size_t)l * ld;
      const double f = rms_factor(chunk, ld, eps);
      for (int i = 0; i < ld; ++i) {
        const int c = l * ld + i;
        const int8_t q = table[(size_t)id * R + c];
        const float g = ((float)q * row_scale[id]) * embed_scale;
        out[(size_t)s * R + c] = (chunk[i] * f) * (double)norm_w[i] + (double)g;
        if (gathered) gathered[(size_t)s * R + c] = q;
      }
    }
  }
  return 0;
}

// ------------------------------------------------ a3 synthetic E2B pass ---
void q4o_e2b_layer_dims(int layer, int* q, int* kv, int* mlp) {
  const bool full = layer % 5 == 4;            // L4, L9, ..., L34: 8 heads x 512
  const int head_dim = full ? 512 : 256;
  *q = 8 * head_dim;
  *kv = layer < 15 ? head_dim : 0;             // L15-L34 share K/V
  *mlp = layer < 15 ? 6144 : 12288;            // double-wide MLP on the shared layers
}

struct q4o_matrix {
  const uint8_t* codes;
  const uint16_t* scales;
};

// One layer (R8).  mats: q, k, v, o, gate, up, down (k and v may hold NULLs
// when KV == 0).  Stage outputs: fp16 bits for a, b, m, h_out; fp32 for the
// GEMV outputs (fp64 sums rounded to fp32, as the GEMV returns them).
void q4o_e2b_layer(const uint16_t* h, int H, const q4o_matrix* mats, int Q, int KV, int I, double eps,
                   uint16_t* a, float* q, float* k, float* v, float* o, uint16_t* b, float* g, float* u, uint16_t* m,
                   float* y, uint16_t* h_out, int threads) {
  int most = H;
  for (int n : {Q, KV, I})
    if (n > most) most = n;
  std::vector<double> t(H), y64(most);
  auto rms_to_f16 = [&](const double* in, int n, uint16_t* out) {
    const double f = rms_factor(in, n, eps);
    for (int i = 0; i < n; ++i) out[i] = f16_bits(in[i] * f);
  };
  auto gemv32 = [&](const q4o_matrix& W, const uint16_t* x, int rows, int cols, float* out) {
    q4o_gemv(W.codes, W.scales, x, rows, cols, 1, y64.data(), threads);
    for (int i = 0; i < rows; ++i) out[i] = (float)y64[i];
  };
  for (int i = 0; i < H; ++i) t[i] = f16_value(h[i]);
  rms_to_f16(t.data(), H, a);
  gemv32(mats[0], a, Q, H, q);
  if (KV > 0) {
    gemv32(mats[1], a, KV, H, k);
    gemv32(mats[2], a, KV, H, v);
  }
  std::vector<uint16_t> q16(Q);
  for (int i = 0; i < Q; ++i) q16[i] = f16_bits((double)q[i]);
  gemv32(mats[3], q16.data(), H, Q, o);
  for (int i = 0; i < H; ++i) t[i] = (double)o[i];
  rms_to_f16(t.data(), H, b);
  gemv32(mats[4], b, I, H, g);
  gemv32(mats[5], b, I, H, u);
  for (int i = 0; i < I; ++i) m[i] = f16_bits(gelu_tanh_value((double)g[i]) * (double)u[i]);
  gemv32(mats[6], m, H, I, y);
  for (int i = 0; i < H; ++i) t[i] = (double)y[i];
  rms_to_f16(t.data(), H, h_out);
}

// The chain over n_layers layers (7 matrices each, in the order above) from
// h0 to h_out; the stage buffers are the caller's scratch of the largest
// layer's sizes.  Used to time the oracle on the full pass.
void q4o_e2b_pass(const uint16_t* h0, int H, const q4o_matrix* mats, const int* dims /* [n][3]: Q, KV, I */,
                  int n_layers, double eps, uint16_t* h_out, int threads) {
  int maxQ = 0, maxKV = 0, maxI = 0;
  for (int l = 0; l < n_layers; ++l) {
    if (dims[3 * l] > maxQ) maxQ = dims[3 * l];
    if (dims[3 * l + 1] > maxKV) maxKV = dims[3 * l + 1];
    if (dims[3 * l + 2] > maxI) maxI = dims[3 * l + 2];
  }
  std::vector<uint16_t> h(h0, h0 + H), a(H), b(H), m(maxI), hn(H);
  std::vector<float> q(maxQ), k(maxKV > 0 ? maxKV : 1), v(maxKV > 0 ? maxKV : 1), o(H), g(maxI), u(maxI), y(H);
  for (int l = 0; l < n_layers; ++l) {
    q4o_e2b_layer(h.data(), H, mats + 7 * l, dims[3 * l], dims[3 * l + 1], dims[3 * l + 2], eps, a.data(), q.data(),
                  k.data(), v.data(), o.data(), b.data(), g.data(), u.data(), m.data(), y.data(), hn.data(), threads);
    h = hn;
  }
  std::memcpy(h_out, h.data(), sizeof(uint16_t) * H);
}

// --------------------------------------------------- NEXT-2 INT2 GEMV ---
// codes [N][K/4], scales f32 [N], x fp16 bits [B][K]:
// y[b][n] = scale[n] * sum_k (code - 2) * x[b][k], the sum in fp64, k order.
void q4o_q2_gemv(const uint8_t* codes, const float* scales, const uint16_t* x, int N, int K, int B, double* y,
                 int threads) {
  std::vector<double> xv((size_t)B * K);
  for (size_t i = 0; i < xv.size(); ++i) xv[i] = f16_value(x[i]);
  parallel_rows(N, threads, [&](int lo, int hi) {
    for (int n = lo; n < hi; ++n)
      for (int b = 0; b < B; ++b) {
        double acc = 0.0;
        for (int k = 0; k < K; ++k) {
          const int c = (codes[(size_t)n * (K / 4) + k / 4] >> (2 * (k % 4))) & 3;
          acc += (double)(c - 2) * xv[(size_t)b * K + k];
        }
        y[(size_t)b * N + n] = (double)scales[n] * acc;
      }
  });
}

// ---------------------------------------- NEXT-4 int8 per-block-32 weights ---
// W fp32 [N][K] -> codes int8 [N][K], fp16 scale bits [N][K/32].
// 0 ok; 1 K not a multiple of 32; 2 a non-finite weight; 3 a scale beyond fp16.
int q4o_q8_quantize(const float* W, int N, int K, int8_t* codes, uint16_t* scales) {
  if (N < 0 || K <= 0 || K % 32) return 1;
  for (long long i = 0; i < (long long)N * K; ++i)
    if (!std::isfinite(W[i])) return 2;
  const int nb = K / 32;
  for (long long i = 0; i < (long long)N * nb; ++i) {
    float a = 0.0f;
    for (int t = 0; t < 32; ++t) a = std::fmax(a, std::fabs(W[i * 32 + t]));
    if (a / 127.0f > 65504.0f) return 3;
  }
  for (int n = 0; n < N; ++n)
    for (int j = 0; j < nb; ++j) {
      const float* blk = W + (size_t)n * K + 32 * j;
      float a = 0.0f;
      for (int i = 0; i < 32; ++i) a = std::fmax(a, std::fabs(blk[i]));
      const float d32 = a / 127.0f;                     // IEEE fp32 quotient
      scales[(size_t)n * nb + j] = f16_bits((double)d32);
      for (int i = 0; i < 32; ++i) {
        double c = 0.0;
        if (d32 != 0.0f) {
          const float ratio = blk[i] / d32;             // IEEE fp32 quotient
          c = std::round((double)ratio);                // half away from zero
          if (c < -127.0) c = -127.0;
          if (c > 127.0) c = 127.0;
        }
        codes[(size_t)n * K + 32 * j + i] = (int8_t)c;
      }
    }
  return 0;
}

// w' = fp16(d) * code, exact in double.
void q4o_q8_dequantize(const int8_t* codes, const uint16_t* scales, int N, int K, double* Wd) {
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k)
      Wd[(size_t)n * K + k] = f16_value(scales[(size_t)n * (K / 32) + k / 32]) * (double)codes[(size_t)n * K + k];
}

// The PLE with the int8 projection: the f32 PLE on w' (exact in fp32: an
// 11-bit scale times an 8-bit code).
int q4o_ple_q8(const int32_t* ids, int S, const int8_t* table, const float* row_scale, int V, int L, int ld,
               float embed_scale, const int8_t* codes, const uint16_t* scales, const uint16_t* hidden, int D,
               const float* norm_w, double eps, double* out, int8_t* gathered, int threads) {
  const int R = L * ld;
  std::vector<double> wd((size_t)R * D);
  q4o_q8_dequantize(codes, scales, R, D, wd.data());
  std::vector<float> proj(wd.size());
  for (size_t i = 0; i < wd.size(); ++i) proj[i] = (float)wd[i];
  return q4o_ple(ids, S, table, row_scale, V, L, ld, embed_scale, proj.data(), hidden, D, norm_w, eps, out, gathered,
                 threads);
}

// ------------------------------------------------ NEXT-4 w4a8 activations ---
// Min-max calibration over n fp16 values.
float q4o_a8_calibrate(const uint16_t* x, long long n) {
  float amax = 0.0f;
  for (long long i = 0; i < n; ++i) amax = std::fmax(amax, (float)std::fabs(f16_value(x[i])));
  return amax > 0.0f ? amax / 127.0f : 1.0f;
}

// q[i] = clamp(rint(x[i] / s), -128, 127), the quotient in fp32, ties to even.
void q4o_a8_quantize(const uint16_t* x, long long n, float s, int32_t* q) {
  for (long long i = 0; i < n; ++i) {
    const float r = (float)f16_value(x[i]) / s;
    double c = std::nearbyint((double)r);               // round to nearest, ties to even
    if (c < -128.0) c = -128.0;
    if (c > 127.0) c = 127.0;
    q[i] = (int32_t)c;
  }
}

// y[n] = sum_k w'[n][k] * x'[k], x' = s q, fp64 in k order.
void q4o_gemv_a8(const uint8_t* codes, const uint16_t* scales, const uint16_t* x, int N, int K, float s, double* y,
                 int threads) {
  std::vector<int32_t> q(K);
  q4o_a8_quantize(x, K, s, q.data());
  std::vector<double> xd(K);
  for (int k = 0; k < K; ++k) xd[k] = (double)q[k] * (double)s;
  parallel_rows(N, threads, [&](int lo, int hi) {
    for (int n = lo; n < hi; ++n) {
      double acc = 0.0;
      for (int k = 0; k < K; ++k) acc += weight_at(codes, scales, K, n, k) * xd[k];
      y[n] = acc;
    }
  });
}

// Y[t][n] = sum_k bf16(w'[n][k]) * x'[t][k], x' = s q, fp64 in k order.
void q4o_gemm_chunk_a8(const uint8_t* codes, const uint16_t* scales, const uint16_t* X, int M, int N, int K, float s,
                       double* Y, int threads) {
  std::vector<int32_t> q((size_t)M * K);
  q4o_a8_quantize(X, (long long)M * K, s, q.data());
  std::vector<double> xd(q.size());
  for (size_t i = 0; i < q.size(); ++i) xd[i] = (double)q[i] * (double)s;
  parallel_rows(N, threads, [&](int lo, int hi) {
    std::vector<double> wt(K);
    for (int n = lo; n < hi; ++n) {
      for (int k = 0; k < K; ++k) {
        const float w32 = (float)weight_at(codes, scales, K, n, k);   // exact: 11 by 4 bits
        wt[k] = (double)bf16_round(w32);
      }
      for (int t = 0; t < M; ++t) {
        double acc = 0.0;
        for (int k = 0; k < K; ++k) acc += wt[k] * xd[(size_t)t * K + k];
        Y[(size_t)t * N + n] = acc;
      }
    }
  });
}

}  // extern "C"
