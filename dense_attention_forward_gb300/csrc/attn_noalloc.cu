// attn_noalloc.cu -- attn_fwd_host_noalloc: the host-to-host attention call for callers that
// cannot allocate device memory.
//
// attn_fwd_host needs five device buffers from its caller (the staging copies of q, k, v and
// the device-side o and lse). Some callers have no way to make them: code that must not call
// cudaMalloc because a framework or a pool allocator owns all device memory of the process, a
// plug-in that may only use the CUDA runtime without allocating, or a path whose allocations
// are forbidden after start-up. This entry point takes the same host buffers and stages them
// in one fixed array that the library itself holds in device memory, so the call allocates
// nothing.
//
// The array is a file-scope __device__ variable of ATTN_NOALLOC_MAX_ROWS rows: 4 x 8 MiB of
// BF16 rows (q, k, v, o) plus 128 KiB of fp32 lse. Every GPU on which this library's device
// code is loaded holds it until the process exits. Host code cannot use the array's name as a
// device address, so the address is looked up once per device with cudaGetSymbolAddress.
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <mutex>

#include "attn.h"

namespace gb300 {
namespace {

constexpr long long kMaxRows = ATTN_NOALLOC_MAX_ROWS;
constexpr size_t kRowBytes = 128 * 2;                        // one BF16 row of head dimension 128
constexpr size_t kTensorBytes = kMaxRows * kRowBytes;        // 8 MiB per tensor
constexpr size_t kStagingBytes = 4 * kTensorBytes + kMaxRows * 4;
static_assert(kTensorBytes % 256 == 0, "every region starts 256-byte aligned (TMA needs 16)");

// q | k | v | o | lse, each region sized for kMaxRows rows.
static __device__ __align__(256) unsigned char g_noalloc_staging[kStagingBytes];

constexpr int kMaxDevices = 64;
std::atomic<unsigned char*> g_staging_addr[kMaxDevices];
std::mutex g_setup_mutex;

// The device address of the staging array on the current device. Set-up, once per device with
// that device current: check that it is an sm_103 device, then cudaGetSymbolAddress (which may
// load this file's device code onto the device, so it belongs outside any stream capture).
int staging_address(unsigned char** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return ATTN_ERR_UNSUPPORTED_DEVICE;
  }
  if (dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED_DEVICE;
  unsigned char* p = g_staging_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    p = g_staging_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
      int major = 0, minor = 0;
      if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
          major != 10 || minor != 3) {
        cudaGetLastError();
        return ATTN_ERR_UNSUPPORTED_DEVICE;
      }
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_noalloc_staging) != cudaSuccess || addr == nullptr) {
        cudaGetLastError();
        return ATTN_ERR_LAUNCH;
      }
      p = static_cast<unsigned char*>(addr);
      g_staging_addr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return ATTN_OK;
}

}  // namespace
}  // namespace gb300

extern "C" int attn_fwd_host_noalloc(const void* q_h, const void* k_h, const void* v_h, void* o_h,
                                     float* lse_h, int B, int H, int S, int D, float scale, int causal,
                                     void* stream) {
  using namespace gb300;
  if (B <= 0 || H <= 0 || S <= 0) return ATTN_ERR_INVALID_ARG;
  if (D != 128) return ATTN_ERR_UNSUPPORTED_DIM;
  if (static_cast<long long>(B) * H * S > kMaxRows) return ATTN_ERR_INVALID_ARG;  // beyond the array
  unsigned char* base = nullptr;
  const int r = staging_address(&base);
  if (r != ATTN_OK) return r;
  // Fixed regions of the array serve as attn_fwd_host's device buffers. Nothing in them needs
  // clearing: the copies overwrite every input byte the kernel reads and the kernel writes every
  // output byte that is copied back, so the previous call's contents never show.
  float* lse_d = lse_h ? reinterpret_cast<float*>(base + 4 * kTensorBytes) : nullptr;
  return attn_fwd_host(q_h, k_h, v_h, o_h, lse_h, base, base + kTensorBytes, base + 2 * kTensorBytes,
                       base + 3 * kTensorBytes, lse_d, B, H, S, D, scale, causal, stream);
}
