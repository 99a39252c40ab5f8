// noalloc.cu -- decode experts with library-owned scratch, for callers that
// must not allocate device memory.
//
// Some callers cannot hand the library a workspace: code that runs while a
// CUDA stream is being captured (cudaMalloc is not stream-ordered, so it
// cannot be recorded into the graph), hosts whose device memory is managed by
// another framework's pool (a side allocation would bypass its accounting
// and may fail once the pool has claimed the GPU), and latency-critical loops
// where an allocation's implicit device synchronisation is not acceptable.
// For them this file keeps the decode workspace (h, one fp32 row of the
// expert intermediate per (token, rank) pair) in a fixed array in device
// memory that the library owns.
//
// Cost and rules:
//   * the array is kStaticScratchBytes (1 MiB); every GPU on which the
//     library is loaded holds it until the process exits;
//   * calls whose decode workspace (T * k * I * 4 bytes, rounded up) exceeds
//     it are rejected (FT_ERR_INVALID);
//   * all calls share the one array: calls that may overlap on the GPU (two
//     streams, or two threads' streams) race on it and must be serialised by
//     the caller;
//   * the first call on each device looks the array's address up, once, with
//     that device current; make that first call before any stream capture;
//     the address is kept until the process exits, so the entry point must
//     not be used on a device after a reset of its primary context
//     (cudaDeviceReset) in the same process;
//   * the kernels write every scratch element they read within a call, so
//     nothing is cleared between calls.
#include <mutex>

#include "ft_common.cuh"

namespace ft {
namespace {

constexpr size_t kStaticScratchBytes = 1u << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

ft_status scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FT_ERR_CUDA, "experts decode (static scratch): %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return fail(FT_ERR_UNSUPPORTED, "experts decode (static scratch): device %d beyond %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr)
      return fail(FT_ERR_CUDA, "experts decode (static scratch): symbol address: %s", cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FT_OK;
}

}  // namespace
}  // namespace ft

extern "C" {

ft_status ft_moe_experts_decode_static(const ft_bank* cache_host, const ft_bank* pool_host, int32_t layer,
                                       int32_t E, const uint16_t* x, int32_t T, const int32_t* slot_ids,
                                       const int32_t* raw_ids, const float* topk_w, int32_t k, void* out,
                                       int32_t out_dtype, int32_t* dev_status, void* stream) {
  FT_REQUIRE(cache_host != nullptr, "experts decode (static scratch): cache bank is NULL");
  FT_REQUIRE(T >= 0 && k >= 1, "experts decode (static scratch): T=%d k=%d", T, k);
  const size_t need = ft_moe_experts_workspace(FT_DECODE, T, k, cache_host->H, cache_host->I, E);
  FT_REQUIRE(need <= ft::kStaticScratchBytes,
             "experts decode (static scratch): the workspace (%zu bytes) exceeds the %zu-byte static scratch",
             need, ft::kStaticScratchBytes);
  void* ws = nullptr;
  ft_status st = ft::scratch_for_current_device(&ws);
  if (st != FT_OK) return st;
  return ft_moe_experts_fwd(cache_host, pool_host, layer, E, x, nullptr, T, slot_ids, raw_ids, topk_w, k,
                            FT_DECODE, nullptr, out, out_dtype, ws, ft::kStaticScratchBytes, dev_status,
                            stream);
}

}  // extern "C"
