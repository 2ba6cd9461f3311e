// selftest.cu -- single-tile tcgen05 GEMMs that exercise, in isolation, the three operand
// forms the attention kernel uses (test support; built as libattn_selftest.so):
//   mode 0: C = A B^T, A and B K-major SW128 in shared memory        (the S = Q K^T form)
//   mode 1: C = A B,   A K-major SW128, B MN-major SW128              (V as the B operand)
//   mode 2: C = A B,   A packed BF16 in tensor memory, B MN-major     (the O += P V form)
// A is [128 x 128] row-major BF16 (M x K); B is [128 N x 128 K] (mode 0) or [128 K x 128 N]
// (modes 1, 2) row-major BF16; C is [128 x 128] row-major fp32. One CTA of 128 threads.
// attn_selftest_elementwise runs the softmax's per-element helpers (MUFU exp2, BF16 packing
// and unpacking, three-input max) on arrays, for comparison with exact host values.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "ptx.cuh"

namespace gb300 {
namespace {

constexpr int kN = 128;
constexpr int kTile = kN * kN * 2;
constexpr int kSlice = kN * 128;

__global__ void __launch_bounds__(128, 1)
    selftest_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                         const uint32_t* __restrict__ a_rows, float* __restrict__ c, int mode) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sa = base, sb = base + kTile;
  const uint32_t bar_load = base + 2 * kTile, bar_mma = bar_load + 8;
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + 2 * kTile + 16);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0) {
    tmem_alloc(base + 2 * kTile + 16, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;

  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar_load, mode == 2 ? kTile : 2 * kTile);
    if (mode != 2) {
      tma_load_3d(sa, &tm_a, bar_load, 0, 0, 0);
      tma_load_3d(sa + kSlice, &tm_a, bar_load, 64, 0, 0);
    }
    tma_load_3d(sb, &tm_b, bar_load, 0, 0, 0);
    tma_load_3d(sb + kSlice, &tm_b, bar_load, 64, 0, 0);
  }
  if (mode == 2) {
    // Row r of A -> TMEM lane r, columns [128, 192): 16 BF16 K values per 8 columns.
    const int r = warp * 32 + lane;
    uint32_t v[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) v[j] = a_rows[r * 64 + j];
    tmem_st32_x64(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 128u, v);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (threadIdx.x == 0) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar_load, 0)) {
      if (global_timer_ns() - t0 > 1000000000ull) break;  // bounded: 1 s
    }
    tc_fence_after();
    const uint32_t idesc = idesc_bf16_f32(128, 128, 0, mode == 0 ? 0 : 1);
    const uint64_t da = smem_desc_sw128(sa, 16, 1024);
    const uint64_t db = mode == 0 ? smem_desc_sw128(sb, 16, 1024) : smem_desc_sw128(sb, kSlice, 1024);
    for (int kk = 0; kk < 8; ++kk) {
      const uint64_t koff = static_cast<uint64_t>(((kk >> 2) * kSlice + (kk & 3) * 32) >> 4);
      if (mode == 0) {
        mma_bf16_ss(tmem, da + koff, db + koff, idesc, kk > 0);
      } else if (mode == 1) {
        mma_bf16_ss(tmem, da + koff, db + static_cast<uint64_t>(kk * (2048 >> 4)), idesc, kk > 0);
      } else {
        mma_bf16_ts(tmem, tmem + 128u + kk * 8, db + static_cast<uint64_t>(kk * (2048 >> 4)), idesc,
                    kk > 0);
      }
    }
    mma_commit(bar_mma);
  }
  {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar_mma, 0)) {
      if (global_timer_ns() - t0 > 1000000000ull) break;  // bounded: 1 s
    }
  }
  tc_fence_after();
  const int r = warp * 32 + lane;
#pragma unroll 1
  for (int cc = 0; cc < 4; ++cc) {
    uint32_t v[32];
    tmem_ld32_x32_sync(tmem + (static_cast<uint32_t>(warp * 32) << 16) + cc * 32, v);
#pragma unroll
    for (int j = 0; j < 32; ++j) c[r * 128 + cc * 32 + j] = __uint_as_float(v[j]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_tile(CUtensorMap* m, const void* p) {
  const cuuint64_t dims[3] = {128, 128, 1};
  const cuuint64_t strides[2] = {256, 256 * 128};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return get_encode()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p), dims, strides, box, es,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per element i: f[4i] = 2^x[i] (MUFU, ftz), u[i] = BF16x2 of (x[i], y[i]) (round to
// nearest even, x in the low half), f[4i+1], f[4i+2] = that pair widened back to fp32,
// f[4i+3] = max(x[i], y[i], -x[i]).
__global__ void selftest_elementwise_kernel(const float* __restrict__ x, const float* __restrict__ y,
                                           uint32_t* __restrict__ u, float* __restrict__ f, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const uint32_t pk = pack_bf16x2(x[i], y[i]);
    float lo, hi;
    bf16x2_to_f32x2(pk, lo, hi);
    u[i] = pk;
    f[4 * i + 0] = ex2_ftz(x[i]);
    f[4 * i + 1] = lo;
    f[4 * i + 2] = hi;
    f[4 * i + 3] = max3(x[i], y[i], -x[i]);
  }
}

}  // namespace
}  // namespace gb300

extern "C" int attn_selftest_elementwise(const float* x, const float* y, unsigned int* u, float* f, int n,
                                         void* stream) {
  using namespace gb300;
  if (!x || !y || !u || !f || n <= 0) return 1;
  selftest_elementwise_kernel<<<(n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024, 256, 0,
                                static_cast<cudaStream_t>(stream)>>>(x, y, u, f, n);
  return cudaGetLastError() == cudaSuccess ? 0 : 5;
}

extern "C" int attn_selftest_gemm(const void* a, const void* b, float* c, int mode, void* stream) {
  using namespace gb300;
  if (!a || !b || !c || mode < 0 || mode > 2) return 1;
  if (!get_encode()) return 5;
  CUtensorMap ta, tb;
  if (!encode_tile(&ta, a) || !encode_tile(&tb, b)) return 5;
  const int smem = 2 * kTile + 64 + 1024;
  if (cudaFuncSetAttribute(selftest_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return 5;
  selftest_gemm_kernel<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(
      ta, tb, static_cast<const uint32_t*>(a), c, mode);
  return cudaGetLastError() == cudaSuccess ? 0 : 5;
}
