// abi.cu -- library-wide entry points: version, error strings, the expert
// block layout, and the device status read-back.
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "ft_common.cuh"

namespace ft {

static thread_local char g_err[512] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
}

ft_status fail(ft_status code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

struct SmemAttr {
  const void* kernel;
  int device;
  int bytes;
};
std::mutex g_attr_mu;
std::vector<SmemAttr> g_attrs;
}  // namespace

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) dev = 0;
  if (dev >= kMaxDevices) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
  }
  int n = g_sm_count[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
    g_sm_count[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

int device_smem_optin() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) dev = 0;
  int n = dev < kMaxDevices ? cache[dev].load(std::memory_order_relaxed) : 0;
  if (n <= 0) {
    cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (n <= 0) n = 48 * 1024;
    if (dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

ft_status ensure_dyn_smem(const void* kernel, int bytes, const char* what) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  std::lock_guard<std::mutex> lock(g_attr_mu);
  for (const SmemAttr& a : g_attrs)
    if (a.kernel == kernel && a.device == dev && a.bytes >= bytes) return FT_OK;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return fail(FT_ERR_CUDA, "%s: shared memory limit %d: %s", what, bytes, cudaGetErrorString(e));
  for (SmemAttr& a : g_attrs)
    if (a.kernel == kernel && a.device == dev) {
      a.bytes = bytes;
      return FT_OK;
    }
  g_attrs.push_back({kernel, dev, bytes});
  return FT_OK;
}

ft_status launch_check(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(FT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return FT_OK;
}

// One expert block: gate [I,H] | up [I,H] | down [H,I] as packed 4-bit codes,
// then gate/up/down scales ([rows, K/block] fp16 for int4, E4M3 bytes for
// NVFP4), the order of the NVMe-streaming post's engine step 1.
bool layout(int32_t fmt, int32_t H, int32_t I, int32_t group, Layout* L) {
  if (H <= 0 || I <= 0 || H % 32 || I % 32) return false;
  int32_t blk;
  uint64_t sb;
  if (fmt == FT_INT4) {
    if (group != 32 && group != 64 && group != 128) return false;
    if (H % group || I % group) return false;
    blk = group;
    sb = 2;
  } else if (fmt == FT_NVFP4) {
    if (group != 16) return false;
    blk = 16;
    sb = 1;
  } else {
    return false;
  }
  const uint64_t gate = static_cast<uint64_t>(I) * H / 2;
  const uint64_t down = static_cast<uint64_t>(H) * I / 2;
  const uint64_t gs = static_cast<uint64_t>(I) * (H / blk) * sb;
  const uint64_t ds = static_cast<uint64_t>(H) * (I / blk) * sb;
  L->off[0] = 0;
  L->off[1] = gate;
  L->off[2] = 2 * gate;
  L->off[3] = 2 * gate + down;
  L->off[4] = L->off[3] + gs;
  L->off[5] = L->off[4] + gs;
  L->total = L->off[5] + ds;
  L->block = blk;
  for (int i = 0; i < 6; ++i)
    if (L->off[i] % 16) return false;
  return L->total % 16 == 0;
}

ft_status check_bank(const ft_bank* b, const char* name, Layout* L) {
  FT_REQUIRE(b != nullptr, "%s: bank descriptor is NULL", name);
  if (!layout(b->fmt, b->H, b->I, b->group, L))
    return fail(FT_ERR_UNSUPPORTED, "%s: unsupported format %d H=%d I=%d group=%d", name, b->fmt,
                b->H, b->I, b->group);
  FT_REQUIRE(b->base != nullptr, "%s: base is NULL", name);
  FT_REQUIRE(reinterpret_cast<uintptr_t>(b->base) % 16 == 0, "%s: base not 16-byte aligned", name);
  FT_REQUIRE(b->stride >= L->total && b->stride % 16 == 0,
             "%s: stride %llu must be >= %llu and a multiple of 16", name,
             static_cast<unsigned long long>(b->stride), static_cast<unsigned long long>(L->total));
  FT_REQUIRE(b->n_blocks > 0 && b->n_blocks < (1ll << 31), "%s: n_blocks %lld", name,
             static_cast<long long>(b->n_blocks));
  FT_REQUIRE(b->fmt != FT_NVFP4 || b->tensor_scale != nullptr,
             "%s: NVFP4 bank needs tensor_scale", name);
  return FT_OK;
}

}  // namespace ft

extern "C" {

const char* ft_version(void) { return "ft_moe 0.1 (sm_103a)"; }

const char* ft_status_string(ft_status s) {
  switch (s) {
    case FT_OK: return "ok";
    case FT_ERR_INVALID: return "invalid argument";
    case FT_ERR_UNSUPPORTED: return "unsupported format or shape";
    case FT_ERR_CUDA: return "CUDA launch error";
    case FT_ERR_TIMEOUT: return "device wait timed out";
    case FT_ERR_BAD_ID: return "expert id out of range";
    case FT_ERR_RANGE: return "intermediate outside the f16 range";
    case FT_ERR_REJECTED: return "cache rebuild rejected";
    default: return "unknown status";
  }
}

const char* ft_last_error(void) { return ft::g_err; }

uint64_t ft_block_bytes(int32_t fmt, int32_t H, int32_t I, int32_t group, uint64_t* off6_host) {
  ft::Layout L;
  if (!ft::layout(fmt, H, I, group, &L)) return 0;
  if (off6_host)
    for (int i = 0; i < 6; ++i) off6_host[i] = L.off[i];
  return L.total;
}

ft_status ft_moe_get_status(const int32_t* dev_status, int32_t* out_host) {
  FT_REQUIRE(dev_status != nullptr && out_host != nullptr, "get_status: NULL pointer");
  cudaError_t e = cudaMemcpy(out_host, dev_status, sizeof(int32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return ft::fail(FT_ERR_CUDA, "get_status: %s", cudaGetErrorString(e));
  return FT_OK;
}

}  // extern "C"
