// lmhead_softcap_argmax_noalloc: the LM head entry point for callers that
// cannot allocate device memory.
//
// Some callers of a decode step cannot hand the library a workspace: a serving
// loop that plans every byte of device memory at start-up and forbids any
// allocation afterwards, or a C host that only owns the weight, activation and
// output buffers it was given (cudaMalloc also synchronises the device, which a
// latency-bound token loop cannot afford).  This entry point needs no
// workspace: the head's scratch (one ticket word and the per-CTA partial
// top-two records) lives in a file-scope device array of fixed size that every
// GPU loading the library holds until the process exits.
#include "q4w_internal.cuh"

namespace q4w {

constexpr size_t kHeadStaticScratchBytes = 64 * 1024;

// Scratch of the no-allocation head: ticket word, then the partial records.
static __device__ __align__(256) unsigned char g_head_scratch[kHeadStaticScratchBytes];

// Device address of g_head_scratch on the current device, looked up once per
// device with that device current.  In host code the array's name is only a
// host-side stand-in, never a device address.  The per-device cache is filled
// without a lock: host threads whose first calls on one device coincide each
// look the address up and store the same value.
static void* head_scratch_address(int* status) {
  static void* cache[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *status = cuda_fail(e, "cudaGetDevice");
    return nullptr;
  }
  if (dev < 0 || dev >= 64) {
    *status = fail(Q4_ERR_CUDA, "device index %d out of range", dev);
    return nullptr;
  }
  if (!cache[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_head_scratch);
    if (e != cudaSuccess) {
      *status = cuda_fail(e, "cudaGetSymbolAddress(head scratch)");
      return nullptr;
    }
    cache[dev] = p;
  }
  *status = Q4_OK;
  return cache[dev];
}

}  // namespace q4w

extern "C" int lmhead_softcap_argmax_noalloc(const uint8_t* codes, const uint16_t* scales,
                                             const uint16_t* h_f16, int b, int V, int K, float cap,
                                             int32_t* idx, float* top1, float* top2, float* logits_opt,
                                             q4_stream_t stream) {
  using namespace q4w;
  clear_error();
  if (!codes || !scales || !h_f16 || !idx || !top1 || !top2)
    return fail(Q4_ERR_NULL, "codes, scales, h_f16, idx, top1 and top2 must be non-NULL");
  const void* ptrs[7] = {codes, scales, h_f16, idx, top1, top2, logits_opt};
  for (int i = 0; i < 7; ++i)
    if (ptrs[i] && !aligned16(ptrs[i])) return fail(Q4_ERR_ALIGN, "argument %d is not 16-byte aligned", i);
  if (b < 1 || b > 8) return fail(Q4_ERR_SHAPE, "b=%d must be in [1, 8]", b);
  if (V < 2) return fail(Q4_ERR_SHAPE, "V=%d must be >= 2", V);
  if (K < 32 || K % 32 || K > 32768) return fail(Q4_ERR_SHAPE, "K=%d must be a multiple of 32 in [32, 32768]", K);
  if (!(cap > 0.f)) return fail(Q4_ERR_SHAPE, "cap must be > 0");
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != Q4_OK) return st;
  const size_t need = lmhead_ws_bytes(V, K, b, dev, false);
  if (need > kHeadStaticScratchBytes)
    return fail(Q4_ERR_WORKSPACE,
                "this device needs %zu bytes of head scratch, above the %zu-byte static maximum; use "
                "lmhead_softcap_argmax with a caller workspace",
                need, kHeadStaticScratchBytes);
  void* ws = head_scratch_address(&st);
  if (!ws) return st;
  // The launcher clears the ticket word on the stream before the kernel; the
  // partial records are fully rewritten by every call.
  return launch_lmhead(codes, reinterpret_cast<const __half*>(scales), reinterpret_cast<const __half*>(h_f16), b,
                       V, K, cap, idx, top1, top2, logits_opt, ws, dev, reinterpret_cast<cudaStream_t>(stream), false);
}
