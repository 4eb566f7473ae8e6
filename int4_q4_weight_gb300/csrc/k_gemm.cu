// S=64 chunked-prefill dequant-GEMM on the tcgen05 tensor cores (in progress).
#include "q4w_internal.cuh"

namespace q4w {

int launch_gemm_chunk(const uint8_t* codes, const __half* scales, const __half* X, float* Y, int M,
                      int N, int K, const DeviceInfo& dev, cudaStream_t s) {
  (void)codes; (void)scales; (void)X; (void)Y; (void)M; (void)N; (void)K; (void)dev; (void)s;
  return fail(Q4_ERR_SHAPE, "q4_gemm_chunk: tensor-core kernel not built yet");
}

}  // namespace q4w
