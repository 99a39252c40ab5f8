// prefill.cu -- token-permuted grouped SwiGLU expert GEMM (placeholder entry
// until the tcgen05 kernel lands).
#include "ft_common.cuh"

namespace ft {

size_t experts_prefill_workspace(int32_t T, int32_t k, int32_t H, int32_t I, int32_t E) {
  (void)H;
  (void)E;
  return (static_cast<size_t>(T) * k * I * 2 + 255) & ~static_cast<size_t>(255);
}

ft_status experts_prefill(const ft_bank*, const ft_bank*, int32_t, int32_t, const uint16_t*, int32_t,
                          int32_t, const int32_t*, const int32_t*, uint16_t*, void*, size_t,
                          int32_t*, cudaStream_t) {
  return fail(FT_ERR_UNSUPPORTED, "experts prefill: not built yet");
}

}  // namespace ft
