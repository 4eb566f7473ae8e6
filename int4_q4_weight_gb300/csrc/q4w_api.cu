// C ABI of libq4w.so: argument checks, status codes, dispatch to launchers.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "q4w_internal.cuh"

#define Q4W_VERSION 100   // 0.1.0

namespace q4w {

static thread_local char g_err[512] = "";

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(Q4_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

void clear_error() { g_err[0] = '\0'; }

static long long g_wait_limit = -1;

long long wait_limit() {
  if (g_wait_limit < 0) {
    const char* e = getenv("Q4W_WAIT_LIMIT_CYCLES");
    long long v = e ? atoll(e) : 4000000000LL;   // about 2 s at 2 GHz
    g_wait_limit = v < 0 ? 0 : v;
  }
  return g_wait_limit;
}

int current_device(DeviceInfo* info) {
  static DeviceInfo cache[64];
  static bool have[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev >= 0 && dev < 64 && have[dev]) {
    *info = cache[dev];
    return Q4_OK;
  }
  DeviceInfo d = {};
  d.ordinal = dev;
  int smem = 0;
  if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute");
  d.smem_optin = (size_t)smem;
  if (d.cc_major != 10 || d.cc_minor != 3)
    return fail(Q4_ERR_ARCH, "device %d is compute capability %d.%d; this library is built for 10.3 (sm_103a)",
                dev, d.cc_major, d.cc_minor);
  if (dev >= 0 && dev < 64) {
    cache[dev] = d;
    have[dev] = true;
  }
  *info = d;
  return Q4_OK;
}

}  // namespace q4w

using namespace q4w;

#define CHECK_NULL(p)                                              \
  do {                                                             \
    if ((p) == nullptr) return fail(Q4_ERR_NULL, "%s is NULL", #p); \
  } while (0)
#define CHECK_ALIGN(p)                                                                   \
  do {                                                                                   \
    if ((p) != nullptr && !aligned16(p))                                                 \
      return fail(Q4_ERR_ALIGN, "%s (%p) is not 16-byte aligned", #p, (const void*)(p)); \
  } while (0)
#define CHECK(cond, ...)                                 \
  do {                                                   \
    if (!(cond)) return fail(Q4_ERR_SHAPE, __VA_ARGS__); \
  } while (0)
#define DEVICE_OR_RETURN(dev)       \
  DeviceInfo dev;                   \
  do {                              \
    int st_ = current_device(&dev); \
    if (st_ != Q4_OK) return st_;   \
  } while (0)

static const int kMaxK = 32768;

extern "C" {

int q4_version(void) { return Q4W_VERSION; }

const char* q4_status_string(int status) {
  switch (status) {
    case Q4_OK: return "Q4_OK";
    case Q4_ERR_NULL: return "Q4_ERR_NULL";
    case Q4_ERR_SHAPE: return "Q4_ERR_SHAPE";
    case Q4_ERR_ALIGN: return "Q4_ERR_ALIGN";
    case Q4_ERR_WORKSPACE: return "Q4_ERR_WORKSPACE";
    case Q4_ERR_ARCH: return "Q4_ERR_ARCH";
    case Q4_ERR_CUDA: return "Q4_ERR_CUDA";
    case Q4_ERR_TIMEOUT: return "Q4_ERR_TIMEOUT";
    case Q4_ERR_DEVICE: return "Q4_ERR_DEVICE";
    default: return "Q4_ERR_UNKNOWN";
  }
}

const char* q4_last_error(void) { return g_err; }

long long q4_set_wait_limit(long long cycles) {
  const long long old = wait_limit();
  g_wait_limit = cycles < 0 ? 0 : cycles;
  return old;
}

// Decode-pass workspace, each region 256-byte aligned: k/v outputs [QKV] f32,
// then the four stage buffers sized for their tagged form (q [QKV] x 4 B,
// o [H] x 8 B, m [I] x 4 B, y [H] x 8 B; the launch-per-stage path uses the
// same regions untagged), then a 256-byte control block.
static size_t up256(size_t n) { return (n + 255) & ~(size_t)255; }
static size_t decode_tagged_bytes(size_t H, size_t QKV, size_t I) {
  return up256(QKV * 4) + up256(H * 8) + up256(I * 4) + up256(H * 8);
}
// One persistent cooperative launch when every stage fits the streaming
// engine and every stage input fits its shared staging area (H <= 4096).
static bool decode_persistent(const q4_layer* layers, int n_layers, int H) {
  bool ok = stream_eligible(H) && H <= 4096 && n_layers <= 48;
  for (int l = 0; l < n_layers && ok; ++l) ok = stream_eligible(layers[l].q_rows) && stream_eligible(layers[l].mlp_rows);
  return ok;
}

static size_t decode_ws_bytes(size_t H, size_t QKV, size_t I) {
  return up256(QKV * 4) + decode_tagged_bytes(H, QKV, I) + up256(decode_ctl_bytes());
}

size_t q4_workspace_bytes(int op, int a, int b, int c) {
  switch (op) {
    case Q4_OP_GEMV: return 0;
    case Q4_OP_GEMM_CHUNK: return (b >= 64 && b % 64 == 0) ? gemm_ws_bytes(b) : 0;
    case Q4_OP_PLE: return 0;
    case Q4_OP_LMHEAD: {
      DeviceInfo dev;
      if (current_device(&dev) != Q4_OK) return 0;
      return lmhead_ws_bytes(a, b, c, dev);
    }
    case Q4_OP_DECODE_PASS:
      if (a < 0 || b < 0 || c < 0) return 0;
      return decode_ws_bytes((size_t)a, (size_t)b, (size_t)c);
    default: return 0;
  }
}

int q4_quantize(const float* W, int N, int K, uint8_t* codes, uint16_t* scales, int32_t* err,
                q4_stream_t stream) {
  clear_error();
  CHECK_NULL(W);
  CHECK_NULL(codes);
  CHECK_NULL(scales);
  CHECK_ALIGN(W);
  CHECK_ALIGN(codes);
  CHECK_ALIGN(scales);
  CHECK_ALIGN(err);
  CHECK(N >= 1, "N=%d must be >= 1", N);
  CHECK(K >= 32 && K % 32 == 0, "K=%d must be a positive multiple of 32", K);
  DEVICE_OR_RETURN(dev);
  return launch_quantize(W, N, K, codes, reinterpret_cast<__half*>(scales), err, dev,
                         reinterpret_cast<cudaStream_t>(stream));
}

int q8_quantize(const float* W, int N, int K, int8_t* codes, uint16_t* scales, int32_t* err,
                q4_stream_t stream) {
  clear_error();
  CHECK_NULL(W);
  CHECK_NULL(codes);
  CHECK_NULL(scales);
  CHECK_ALIGN(W);
  CHECK_ALIGN(codes);
  CHECK_ALIGN(scales);
  CHECK_ALIGN(err);
  CHECK(N >= 1, "N=%d must be >= 1", N);
  CHECK(K >= 32 && K % 32 == 0, "K=%d must be a positive multiple of 32", K);
  DEVICE_OR_RETURN(dev);
  return launch_quantize_q8(W, N, K, codes, reinterpret_cast<__half*>(scales), err, dev,
                            reinterpret_cast<cudaStream_t>(stream));
}

static int gemv_impl(const uint8_t* codes, const uint16_t* scales, const uint16_t* x_f16, float* y, int N, int K,
                     int batch, q4_stream_t stream, bool weights_ro) {
  clear_error();
  CHECK_NULL(codes);
  CHECK_NULL(scales);
  CHECK_NULL(x_f16);
  CHECK_NULL(y);
  CHECK_ALIGN(codes);
  CHECK_ALIGN(scales);
  CHECK_ALIGN(x_f16);
  CHECK_ALIGN(y);
  CHECK(N >= 1, "N=%d must be >= 1", N);
  CHECK(K >= 32 && K % 32 == 0 && K <= kMaxK, "K=%d must be a multiple of 32 in [32, %d]", K, kMaxK);
  CHECK(batch >= 1 && batch <= 8, "batch=%d must be in [1, 8]", batch);
  DEVICE_OR_RETURN(dev);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (batch == 1) {
    StageArgs a = {};
    a.mat[0] = {codes, reinterpret_cast<const __half*>(scales), N, y, nullptr};
    a.nmat = 1;
    a.pair = 0;
    a.K = K;
    a.in = x_f16;
    a.in_mode = Q4_IN_F16;
    a.eps = 0.f;
    a.weights_early = weights_ro ? 1 : 0;
    return launch_stage(a, dev, s, true);
  }
  return launch_gemv_batched(codes, reinterpret_cast<const __half*>(scales),
                             reinterpret_cast<const __half*>(x_f16), y, N, K, batch, dev, s);
}

int q4_gemv(const uint8_t* codes, const uint16_t* scales, const uint16_t* x_f16, float* y, int N,
            int K, int batch, void* ws, size_t ws_bytes, q4_stream_t stream) {
  (void)ws;
  (void)ws_bytes;
  return gemv_impl(codes, scales, x_f16, y, N, K, batch, stream, false);
}

int q4_gemv_weights_ro(const uint8_t* codes, const uint16_t* scales, const uint16_t* x_f16, float* y, int N,
                       int K, int batch, void* ws, size_t ws_bytes, q4_stream_t stream) {
  (void)ws;
  (void)ws_bytes;
  return gemv_impl(codes, scales, x_f16, y, N, K, batch, stream, true);
}

int q4_gemv_stage(const q4_matrix* mats, const int* rows, int nmat, int K, const void* in,
                  int in_mode, float eps, int pair, float* const* out32, uint16_t* const* out16,
                  q4_stream_t stream) {
  clear_error();
  CHECK_NULL(mats);
  CHECK_NULL(rows);
  CHECK_NULL(in);
  CHECK_NULL(out32);
  CHECK_NULL(out16);
  CHECK_ALIGN(in);
  CHECK(nmat >= 1 && nmat <= 3, "nmat=%d must be in [1, 3]", nmat);
  CHECK(K >= 32 && K % 32 == 0 && K <= kMaxK, "K=%d must be a multiple of 32 in [32, %d]", K, kMaxK);
  CHECK(in_mode >= Q4_IN_F16 && in_mode <= Q4_IN_RMS2_F32, "in_mode=%d unknown", in_mode);
  CHECK(pair == 0 || pair == 1, "pair=%d must be 0 or 1", pair);
  CHECK(!pair || (nmat == 2 && rows[0] == rows[1]), "pair mode needs two matrices of equal rows");
  CHECK(!(eps < 0.f), "eps must be >= 0");
  StageArgs a = {};
  for (int i = 0; i < nmat; ++i) {
    if (mats[i].codes == nullptr || mats[i].scales == nullptr)
      return fail(Q4_ERR_NULL, "mats[%d] codes/scales is NULL", i);
    if (!aligned16(mats[i].codes) || !aligned16(mats[i].scales))
      return fail(Q4_ERR_ALIGN, "mats[%d] codes/scales not 16-byte aligned", i);
    if (rows[i] < 1) return fail(Q4_ERR_SHAPE, "rows[%d]=%d must be >= 1", i, rows[i]);
    if (!aligned16(out32[i]) || !aligned16(out16[i]))
      return fail(Q4_ERR_ALIGN, "out32[%d]/out16[%d] not 16-byte aligned", i, i);
    a.mat[i] = {mats[i].codes, reinterpret_cast<const __half*>(mats[i].scales), rows[i], out32[i],
                reinterpret_cast<__half*>(out16[i])};
  }
  if (pair && out16[0] == nullptr) return fail(Q4_ERR_NULL, "pair mode needs out16[0] for m");
  a.nmat = nmat;
  a.pair = pair;
  a.K = K;
  a.in = in;
  a.in_mode = in_mode;
  a.eps = eps;
  DEVICE_OR_RETURN(dev);
  return launch_stage(a, dev, reinterpret_cast<cudaStream_t>(stream), true);
}

int q4_rmsnorm_f16(const float* in, int H, float eps, uint16_t* out_f16, q4_stream_t stream) {
  clear_error();
  CHECK_NULL(in);
  CHECK_NULL(out_f16);
  CHECK_ALIGN(in);
  CHECK_ALIGN(out_f16);
  CHECK(H >= 1 && H <= (1 << 20), "H=%d out of range", H);
  CHECK(!(eps < 0.f), "eps must be >= 0");
  DEVICE_OR_RETURN(dev);
  return launch_rmsnorm_f16(in, H, eps, reinterpret_cast<__half*>(out_f16),
                            reinterpret_cast<cudaStream_t>(stream), false);
}

int q4_decode_pass_launches(const q4_layer* layers, int n_layers, int H) {
  clear_error();
  if (!layers) return -fail(Q4_ERR_NULL, "layers is NULL");
  if (n_layers < 1 || n_layers > 256) return -fail(Q4_ERR_SHAPE, "n_layers=%d must be in [1, 256]", n_layers);
  return decode_persistent(layers, n_layers, H) ? 1 : 4 * n_layers + 1;
}

int q4_decode_pass(const q4_layer* layers, int n_layers, int H, const uint16_t* h0_f16,
                   uint16_t* h_out_f16, float eps, void* ws, size_t ws_bytes, q4_stream_t stream) {
  clear_error();
  CHECK_NULL(layers);
  CHECK_NULL(h0_f16);
  CHECK_NULL(h_out_f16);
  CHECK_ALIGN(h0_f16);
  CHECK_ALIGN(h_out_f16);
  CHECK_ALIGN(ws);
  CHECK(n_layers >= 1 && n_layers <= 256, "n_layers=%d must be in [1, 256]", n_layers);
  CHECK(H >= 32 && H % 32 == 0 && H <= kMaxK, "H=%d must be a multiple of 32 in [32, %d]", H, kMaxK);
  CHECK(!(eps < 0.f), "eps must be >= 0");
  int max_qkv = 0, max_mlp = 0;
  for (int l = 0; l < n_layers; ++l) {
    const q4_layer& L = layers[l];
    if (L.q_rows < 32 || L.q_rows % 32 || L.q_rows > kMaxK)
      return fail(Q4_ERR_SHAPE, "layers[%d].q_rows=%d must be a multiple of 32 in [32, %d]", l, L.q_rows, kMaxK);
    if (L.mlp_rows < 32 || L.mlp_rows % 32 || L.mlp_rows > kMaxK)
      return fail(Q4_ERR_SHAPE, "layers[%d].mlp_rows=%d must be a multiple of 32 in [32, %d]", l, L.mlp_rows, kMaxK);
    if (L.kv_rows < 0 || L.kv_rows > kMaxK)
      return fail(Q4_ERR_SHAPE, "layers[%d].kv_rows=%d out of range", l, L.kv_rows);
    const q4_matrix* req[7] = {&L.q, &L.o, &L.gate, &L.up, &L.down, &L.k, &L.v};
    const char* nm[7] = {"q", "o", "gate", "up", "down", "k", "v"};
    const int nreq = L.kv_rows > 0 ? 7 : 5;
    for (int i = 0; i < nreq; ++i) {
      if (!req[i]->codes || !req[i]->scales)
        return fail(Q4_ERR_NULL, "layers[%d].%s codes/scales is NULL", l, nm[i]);
      if (!aligned16(req[i]->codes) || !aligned16(req[i]->scales))
        return fail(Q4_ERR_ALIGN, "layers[%d].%s codes/scales not 16-byte aligned", l, nm[i]);
    }
    const int qkv = L.q_rows + 2 * L.kv_rows;
    if (qkv > max_qkv) max_qkv = qkv;
    if (L.mlp_rows > max_mlp) max_mlp = L.mlp_rows;
  }
  const size_t need = decode_ws_bytes((size_t)H, (size_t)max_qkv, (size_t)max_mlp);
  if (ws == nullptr || ws_bytes < need)
    return fail(Q4_ERR_WORKSPACE, "ws must hold %zu bytes (got %zu)", need, ws ? ws_bytes : (size_t)0);
  DEVICE_OR_RETURN(dev);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  char* p = reinterpret_cast<char*>(ws);
  float* kv32 = reinterpret_cast<float*>(p);
  p += up256((size_t)max_qkv * 4);
  char* tagged = p;
  const size_t tagged_bytes = decode_tagged_bytes((size_t)H, (size_t)max_qkv, (size_t)max_mlp);
  __half* q16 = reinterpret_cast<__half*>(p);
  p += up256((size_t)max_qkv * 4);
  float* o32 = reinterpret_cast<float*>(p);
  p += up256((size_t)H * 8);
  __half* m16 = reinterpret_cast<__half*>(p);
  p += up256((size_t)max_mlp * 4);
  float* y32 = reinterpret_cast<float*>(p);
  p += up256((size_t)H * 8);
  int* ctl = reinterpret_cast<int*>(p);

  if (decode_persistent(layers, n_layers, H))
    return launch_decode_pass_stream(layers, n_layers, H, reinterpret_cast<const __half*>(h0_f16),
                                     reinterpret_cast<__half*>(h_out_f16), eps, kv32, tagged, tagged_bytes, ctl, dev,
                                     s);

  for (int l = 0; l < n_layers; ++l) {
    const q4_layer& L = layers[l];
    const bool first = l == 0;
    // [q|k|v] = W a,  a = f16(RMSNorm(h)); h = h0 (fp16) on the first layer,
    // else h = f16(RMSNorm(y of the previous layer)).
    StageArgs a = {};
    a.mat[0] = {L.q.codes, reinterpret_cast<const __half*>(L.q.scales), L.q_rows, nullptr, q16};
    a.nmat = 1;
    if (L.kv_rows > 0) {
      a.mat[1] = {L.k.codes, reinterpret_cast<const __half*>(L.k.scales), L.kv_rows, kv32, nullptr};
      a.mat[2] = {L.v.codes, reinterpret_cast<const __half*>(L.v.scales), L.kv_rows, kv32 + L.kv_rows, nullptr};
      a.nmat = 3;
    }
    a.K = H;
    a.in = first ? static_cast<const void*>(h0_f16) : static_cast<const void*>(y32);
    a.in_mode = first ? Q4_IN_RMS_F16 : Q4_IN_RMS2_F32;
    a.eps = eps;
    a.weights_early = !first;   // after the first launch the preceding kernel is one of ours
    int st = launch_stage(a, dev, s, !first);
    if (st != Q4_OK) return st;
    // o = W_o f16(q)
    StageArgs b = {};
    b.mat[0] = {L.o.codes, reinterpret_cast<const __half*>(L.o.scales), H, o32, nullptr};
    b.nmat = 1;
    b.K = L.q_rows;
    b.in = q16;
    b.in_mode = Q4_IN_F16;
    b.eps = eps;
    b.weights_early = 1;
    if ((st = launch_stage(b, dev, s, true)) != Q4_OK) return st;
    // m = f16(gelu(W_g b) * W_u b),  b = f16(RMSNorm(o))
    StageArgs c = {};
    c.mat[0] = {L.gate.codes, reinterpret_cast<const __half*>(L.gate.scales), L.mlp_rows, nullptr, m16};
    c.mat[1] = {L.up.codes, reinterpret_cast<const __half*>(L.up.scales), L.mlp_rows, nullptr, nullptr};
    c.nmat = 2;
    c.pair = 1;
    c.K = H;
    c.in = o32;
    c.in_mode = Q4_IN_RMS_F32;
    c.eps = eps;
    c.weights_early = 1;
    if ((st = launch_stage(c, dev, s, true)) != Q4_OK) return st;
    // y = W_down m
    StageArgs d = {};
    d.mat[0] = {L.down.codes, reinterpret_cast<const __half*>(L.down.scales), H, y32, nullptr};
    d.nmat = 1;
    d.K = L.mlp_rows;
    d.in = m16;
    d.in_mode = Q4_IN_F16;
    d.eps = eps;
    d.weights_early = 1;
    if ((st = launch_stage(d, dev, s, true)) != Q4_OK) return st;
  }
  return launch_rmsnorm_f16(y32, H, eps, reinterpret_cast<__half*>(h_out_f16), s, true);
}

int lmhead_softcap_argmax(const uint8_t* codes, const uint16_t* scales, const uint16_t* h_f16, int b,
                          int V, int K, float cap, int32_t* idx, float* top1, float* top2,
                          float* logits_opt, void* ws, size_t ws_bytes, q4_stream_t stream) {
  clear_error();
  CHECK_NULL(codes);
  CHECK_NULL(scales);
  CHECK_NULL(h_f16);
  CHECK_NULL(idx);
  CHECK_NULL(top1);
  CHECK_NULL(top2);
  CHECK_ALIGN(codes);
  CHECK_ALIGN(scales);
  CHECK_ALIGN(h_f16);
  CHECK_ALIGN(idx);
  CHECK_ALIGN(top1);
  CHECK_ALIGN(top2);
  CHECK_ALIGN(logits_opt);
  CHECK_ALIGN(ws);
  CHECK(b >= 1 && b <= 8, "b=%d must be in [1, 8]", b);
  CHECK(V >= 2, "V=%d must be >= 2", V);
  CHECK(K >= 32 && K % 32 == 0 && K <= kMaxK, "K=%d must be a multiple of 32 in [32, %d]", K, kMaxK);
  CHECK(cap > 0.f, "cap must be > 0");
  DEVICE_OR_RETURN(dev);
  const size_t need = lmhead_ws_bytes(V, K, b, dev);
  if (ws == nullptr || ws_bytes < need)
    return fail(Q4_ERR_WORKSPACE, "ws must hold %zu bytes (got %zu)", need, ws ? ws_bytes : (size_t)0);
  return launch_lmhead(codes, reinterpret_cast<const __half*>(scales),
                       reinterpret_cast<const __half*>(h_f16), b, V, K, cap, idx, top1, top2,
                       logits_opt, ws, dev, reinterpret_cast<cudaStream_t>(stream));
}

int ple_gather_project(const int32_t* ids, int S, const int8_t* table, const float* row_scale, int V,
                       int L, int ld, float embed_scale, const float* proj, const uint16_t* hidden_f16,
                       int D, const float* norm_w, float eps, float* out, int8_t* gathered_opt,
                       int32_t* err, q4_stream_t stream) {
  clear_error();
  CHECK_NULL(ids);
  CHECK_NULL(table);
  CHECK_NULL(row_scale);
  CHECK_NULL(proj);
  CHECK_NULL(hidden_f16);
  CHECK_NULL(norm_w);
  CHECK_NULL(out);
  CHECK_ALIGN(ids);
  CHECK_ALIGN(table);
  CHECK_ALIGN(row_scale);
  CHECK_ALIGN(proj);
  CHECK_ALIGN(hidden_f16);
  CHECK_ALIGN(norm_w);
  CHECK_ALIGN(out);
  CHECK_ALIGN(gathered_opt);
  CHECK_ALIGN(err);
  CHECK(S >= 1 && S <= 4096, "S=%d must be in [1, 4096]", S);
  CHECK(ld == 256, "ld=%d must be 256", ld);
  CHECK(L >= 1 && L <= 256, "L=%d must be in [1, 256]", L);
  CHECK(D >= 32 && D % 32 == 0 && D <= kMaxK, "D=%d must be a multiple of 32 in [32, %d]", D, kMaxK);
  CHECK(V >= 1, "V=%d must be >= 1", V);
  CHECK(!(eps < 0.f), "eps must be >= 0");
  DEVICE_OR_RETURN(dev);
  return launch_ple(ids, S, table, row_scale, V, L, ld, embed_scale, proj,
                    reinterpret_cast<const __half*>(hidden_f16), D, norm_w, eps, out, gathered_opt, err,
                    dev, reinterpret_cast<cudaStream_t>(stream));
}

int ple_gather_project_q8(const int32_t* ids, int S, const int8_t* table, const float* row_scale, int V, int L,
                          int ld, float embed_scale, const int8_t* proj_codes, const uint16_t* proj_scales,
                          const uint16_t* hidden_f16, int D, const float* norm_w, float eps, float* out,
                          int8_t* gathered_opt, int32_t* err, q4_stream_t stream) {
  clear_error();
  CHECK_NULL(ids);
  CHECK_NULL(table);
  CHECK_NULL(row_scale);
  CHECK_NULL(proj_codes);
  CHECK_NULL(proj_scales);
  CHECK_NULL(hidden_f16);
  CHECK_NULL(norm_w);
  CHECK_NULL(out);
  CHECK_ALIGN(ids);
  CHECK_ALIGN(table);
  CHECK_ALIGN(row_scale);
  CHECK_ALIGN(proj_codes);
  CHECK_ALIGN(proj_scales);
  CHECK_ALIGN(hidden_f16);
  CHECK_ALIGN(norm_w);
  CHECK_ALIGN(out);
  CHECK_ALIGN(gathered_opt);
  CHECK_ALIGN(err);
  CHECK(S >= 1 && S <= 4096, "S=%d must be in [1, 4096]", S);
  CHECK(ld == 256, "ld=%d must be 256", ld);
  CHECK(L >= 1 && L <= 256, "L=%d must be in [1, 256]", L);
  CHECK(D >= 128 && D % 128 == 0 && D <= 2048, "D=%d must be a multiple of 128 in [128, 2048]", D);
  CHECK(V >= 1, "V=%d must be >= 1", V);
  CHECK(!(eps < 0.f), "eps must be >= 0");
  DEVICE_OR_RETURN(dev);
  return launch_ple_q8(ids, S, table, row_scale, V, L, ld, embed_scale, proj_codes, proj_scales,
                       reinterpret_cast<const __half*>(hidden_f16), D, norm_w, eps, out, gathered_opt, err, dev,
                       reinterpret_cast<cudaStream_t>(stream));
}

static int gemm_chunk_impl(const uint8_t* codes, const uint16_t* scales, const uint16_t* X_f16, float* Y, int M,
                           int N, int K, void* ws, size_t ws_bytes, q4_stream_t stream, float act_scale) {
  clear_error();
  CHECK_NULL(codes);
  CHECK_NULL(scales);
  CHECK_NULL(X_f16);
  CHECK_NULL(Y);
  CHECK_ALIGN(codes);
  CHECK_ALIGN(scales);
  CHECK_ALIGN(X_f16);
  CHECK_ALIGN(Y);
  CHECK(M == 64, "M=%d must be 64 (the static prefill width)", M);
  CHECK(N >= 128 && N % 128 == 0, "N=%d must be a positive multiple of 128", N);
  CHECK(K >= 64 && K % 64 == 0 && K <= kMaxK, "K=%d must be a multiple of 64 in [64, %d]", K, kMaxK);
  CHECK_ALIGN(ws);
  if (ws == nullptr || ws_bytes < gemm_ws_bytes(K))
    return fail(Q4_ERR_WORKSPACE, "ws must hold %zu bytes (got %zu)", gemm_ws_bytes(K), ws ? ws_bytes : (size_t)0);
  DEVICE_OR_RETURN(dev);
  return launch_gemm_chunk(codes, reinterpret_cast<const __half*>(scales),
                           reinterpret_cast<const __half*>(X_f16), Y, M, N, K, ws, dev,
                           reinterpret_cast<cudaStream_t>(stream), act_scale);
}

int q4_gemm_chunk(const uint8_t* codes, const uint16_t* scales, const uint16_t* X_f16, float* Y, int M,
                  int N, int K, void* ws, size_t ws_bytes, q4_stream_t stream) {
  return gemm_chunk_impl(codes, scales, X_f16, Y, M, N, K, ws, ws_bytes, stream, 0.f);
}

static bool act_scale_ok(float s) { return s > 0.f && s <= 3.4e38f; }   // finite and positive (false for NaN)

int q4_gemm_chunk_a8(const uint8_t* codes, const uint16_t* scales, const uint16_t* X_f16, float act_scale,
                     float* Y, int M, int N, int K, void* ws, size_t ws_bytes, q4_stream_t stream) {
  if (!act_scale_ok(act_scale)) {
    clear_error();
    return fail(Q4_ERR_SHAPE, "act_scale=%g must be finite and > 0", (double)act_scale);
  }
  return gemm_chunk_impl(codes, scales, X_f16, Y, M, N, K, ws, ws_bytes, stream, act_scale);
}

int q4_gemv_a8(const uint8_t* codes, const uint16_t* scales, const uint16_t* x_f16, float act_scale, float* y,
               int N, int K, q4_stream_t stream) {
  clear_error();
  CHECK_NULL(codes);
  CHECK_NULL(scales);
  CHECK_NULL(x_f16);
  CHECK_NULL(y);
  CHECK_ALIGN(codes);
  CHECK_ALIGN(scales);
  CHECK_ALIGN(x_f16);
  CHECK_ALIGN(y);
  CHECK(N >= 1, "N=%d must be >= 1", N);
  CHECK(K >= 32 && K % 32 == 0 && K <= kMaxK, "K=%d must be a multiple of 32 in [32, %d]", K, kMaxK);
  CHECK(act_scale_ok(act_scale), "act_scale=%g must be finite and > 0", (double)act_scale);
  DEVICE_OR_RETURN(dev);
  return launch_gemv_a8(codes, reinterpret_cast<const __half*>(scales), reinterpret_cast<const __half*>(x_f16),
                        act_scale, y, N, K, dev, reinterpret_cast<cudaStream_t>(stream));
}

int q4_act_calibrate_a8(const uint16_t* x_f16, long long n, float* scale_out, q4_stream_t stream) {
  clear_error();
  CHECK_NULL(x_f16);
  CHECK_NULL(scale_out);
  CHECK_ALIGN(x_f16);
  CHECK(n >= 1, "n=%lld must be >= 1", n);
  DEVICE_OR_RETURN(dev);
  (void)dev;
  return launch_a8_calibrate(reinterpret_cast<const __half*>(x_f16), n, scale_out,
                             reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
