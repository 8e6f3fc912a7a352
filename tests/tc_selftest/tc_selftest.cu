// Operand-layout self-test of the tensor-core scan (test support, not part of
// libsss): one [128][128] bf16 product A B^T through every tcgen05
// shared-memory / tensor-memory operand form the scan kernels use, each
// written to its own fp32 block of `out` so a test can compare it with a plain
// matmul.  Built into tests/tc_selftest/_build/libsss_selftest.so from the
// library's own PTX wrappers.
#include <cudaTypedefs.h>

#include "../../selective_ssm_scan_gb300/csrc/common.cuh"
#include "../../selective_ssm_scan_gb300/csrc/scan_tc_util.cuh"
#include "../../selective_ssm_scan_gb300/csrc/tc_ptx.cuh"

namespace sss {
namespace selftest {
using namespace tc;
using namespace tcs;

// the single-head scan kernel's instruction descriptors
constexpr uint32_t kIdG = idesc_bf16(128, 128, 0, 0);   // K-major x K-major
constexpr uint32_t kIdS = idesc_bf16(128, 64, 1, 1);    // MN-major x MN-major, N = 64
constexpr uint32_t kIdYo = idesc_bf16(128, 64, 0, 1);   // K-major x MN-major, N = 64
constexpr uint32_t kIdYd = idesc_bf16(128, 128, 0, 1);  // (TMEM) x MN-major, N = 128

// ---------------------------------------------------------------------------
// the descriptor forms of the scan on one tile
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128, 1)
tc_selftest_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __nv_bfloat16* __restrict__ Am, const __nv_bfloat16* __restrict__ Bm,
                   float* __restrict__ out, int* status) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived from the shared array itself so that the
  // compiler keeps every access in the shared address space
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(sm);
  // every MN-major operand keeps valid memory one LBO (16 KB) past its start:
  // the hardware may read there even when N = 64 needs a single 64-wide block
  constexpr uint32_t oA = 0, oB = 32768, oAt = 65536, oBt = 98304, oMisc = 131072;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + oMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + oMisc + 16);
  const uint32_t bar_tma = smem_u32(&bars[0]), bar_mma = smem_u32(&bars[1]);
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;
  const uint32_t tl = tm + (uint32_t(warp * 32) << 16);
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_tma, 4u * 16384u);
    tma_load_2d(sb + oA, &tmA, 0, 0, bar_tma);
    tma_load_2d(sb + oA + 16384, &tmA, 64, 0, bar_tma);
    tma_load_2d(sb + oB, &tmB, 0, 0, bar_tma);
    tma_load_2d(sb + oB + 16384, &tmB, 64, 0, bar_tma);
  }
  const uint16_t* A16 = reinterpret_cast<const uint16_t*>(Am);
  const uint16_t* B16 = reinterpret_cast<const uint16_t*>(Bm);
  // MN-major A: row k = tid, 64-element m blocks 16 KB apart
  for (int j = 0; j < 2; ++j)
    for (int c = 0; c < 8; ++c) {
      uint32_t w[4];
      for (int e = 0; e < 4; ++e)
        w[e] = pack2(A16[(64 * j + 8 * c + 2 * e) * 128 + tid], A16[(64 * j + 8 * c + 2 * e + 1) * 128 + tid]);
      *reinterpret_cast<uint4*>(sm + oAt + j * 16384 + sw128(tid, c)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  // MN-major B (n < 64): row k = tid
  for (int c = 0; c < 8; ++c) {
    uint32_t w[4];
    for (int e = 0; e < 4; ++e)
      w[e] = pack2(B16[(8 * c + 2 * e) * 128 + tid], B16[(8 * c + 2 * e + 1) * 128 + tid]);
    *reinterpret_cast<uint4*>(sm + oBt + sw128(tid, c)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  // A row m = tid into TMEM as bf16 pairs (columns 448..511)
  for (int j = 0; j < 4; ++j) {
    uint32_t w[16];
    for (int i = 0; i < 16; ++i) w[i] = pack2(A16[tid * 128 + 32 * j + 2 * i], A16[tid * 128 + 32 * j + 2 * i + 1]);
    tmem_st_x16(tl + 448u + 16u * j, w);
  }
  tmem_st_wait();
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  bool ok = mbar_wait(bar_tma, 0, kWaitNs);
  if (!__syncthreads_or(!ok)) {
    if (tid == 0) {
      tc_fence_after();
      for (int kk = 0; kk < 8; ++kk)  // [0] K-major A, K-major B, N = 128
        mma_ss(tm + 0, kdesc(sb + oA, kk, 16384), kdesc(sb + oB, kk, 16384), kIdG, kk);
      for (int kk = 0; kk < 8; ++kk)  // [1] MN-major A, K-major B
        mma_ss(tm + 128, sdesc_sw128(sb + oAt + kk * 2048, 16384, 1024), kdesc(sb + oB, kk, 16384),
               idesc_bf16(128, 64, 1, 0), kk);
      for (int kk = 0; kk < 8; ++kk)  // [2] K-major A, MN-major B
        mma_ss(tm + 192, kdesc(sb + oA, kk, 16384), mndesc(sb + oBt, kk), kIdYo, kk);
      for (int kk = 0; kk < 8; ++kk)  // [3] A from TMEM, K-major B
        mma_ts(tm + 256, tm + 448u + 8u * kk, kdesc(sb + oB, kk, 16384), idesc_bf16(128, 64, 0, 0), kk);
      for (int kk = 0; kk < 8; ++kk)  // [4] A from TMEM, MN-major B
        mma_ts(tm + 320, tm + 448u + 8u * kk, mndesc(sb + oBt, kk), kIdYd, kk);
      for (int kk = 0; kk < 8; ++kk)  // [5] MN-major A, MN-major B
        mma_ss(tm + 384, sdesc_sw128(sb + oAt + kk * 2048, 16384, 1024), mndesc(sb + oBt, kk), kIdS, kk);
      mma_commit(bar_mma);
    }
    ok = mbar_wait(bar_mma, 0, kWaitNs);
    if (!__syncthreads_or(!ok)) {
      tc_fence_after();
      uint32_t r[32];
      for (int j = 0; j < 4; ++j) {
        tmem_ld_x32(tl + 32u * j, r);
        for (int i = 0; i < 32; ++i) out[tid * 128 + 32 * j + i] = __uint_as_float(r[i]);
      }
      for (int t = 1; t < 6; ++t)
        for (int j = 0; j < 2; ++j) {
          tmem_ld_x32(tl + 128u + 64u * (t - 1) + 32u * j, r);
          for (int i = 0; i < 32; ++i) out[t * 16384 + tid * 128 + 32 * j + i] = __uint_as_float(r[i]);
        }
    } else if (tid == 0) {
      raise_status(status, SSS_ERR_TIMEOUT);
    }
  } else if (tid == 0) {
    raise_status(status, SSS_ERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tm, 512);
}

// The N = 128 forms: the B operand is two 64-wide MN-major blocks 16 KB
// apart (as the hi and lo tiles of the scan are).  out[6..8]:
// [6] K-major A, [7] A from tensor memory, [8] MN-major A.
__global__ void __launch_bounds__(128, 1)
tc_selftest2_kernel(const __grid_constant__ CUtensorMap tmA, const __nv_bfloat16* __restrict__ Am,
                    const __nv_bfloat16* __restrict__ Bm, float* __restrict__ out, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(sm);
  constexpr uint32_t oA = 0, oAt = 32768, oBt = 65536, oMisc = 98304;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + oMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + oMisc + 16);
  const uint32_t bar_tma = smem_u32(&bars[0]), bar_mma = smem_u32(&bars[1]);
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;
  const uint32_t tl = tm + (uint32_t(warp * 32) << 16);
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_tma, 2u * 16384u);
    tma_load_2d(sb + oA, &tmA, 0, 0, bar_tma);
    tma_load_2d(sb + oA + 16384, &tmA, 64, 0, bar_tma);
  }
  const uint16_t* A16 = reinterpret_cast<const uint16_t*>(Am);
  const uint16_t* B16 = reinterpret_cast<const uint16_t*>(Bm);
  for (int j = 0; j < 2; ++j)
    for (int c = 0; c < 8; ++c) {
      uint32_t wa[4], wb[4];
      for (int e = 0; e < 4; ++e) {
        const int m = 64 * j + 8 * c + 2 * e;
        wa[e] = pack2(A16[m * 128 + tid], A16[(m + 1) * 128 + tid]);
        wb[e] = pack2(B16[m * 128 + tid], B16[(m + 1) * 128 + tid]);
      }
      *reinterpret_cast<uint4*>(sm + oAt + j * 16384 + sw128(tid, c)) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
      *reinterpret_cast<uint4*>(sm + oBt + j * 16384 + sw128(tid, c)) = make_uint4(wb[0], wb[1], wb[2], wb[3]);
    }
  for (int j = 0; j < 4; ++j) {
    uint32_t w[16];
    for (int i = 0; i < 16; ++i) w[i] = pack2(A16[tid * 128 + 32 * j + 2 * i], A16[tid * 128 + 32 * j + 2 * i + 1]);
    tmem_st_x16(tl + 384u + 16u * j, w);
  }
  tmem_st_wait();
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  bool ok = mbar_wait(bar_tma, 0, kWaitNs);
  if (!__syncthreads_or(!ok)) {
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id_k = idesc_bf16(128, 128, 0, 1), id_mn = idesc_bf16(128, 128, 1, 1);
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tm + 0, kdesc(sb + oA, kk, 16384), sdesc_sw128(sb + oBt + kk * 2048, 16384, 1024), id_k, kk);
      for (int kk = 0; kk < 8; ++kk)
        mma_ts(tm + 128, tm + 384u + 8u * kk, sdesc_sw128(sb + oBt + kk * 2048, 16384, 1024), id_k, kk);
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tm + 256, sdesc_sw128(sb + oAt + kk * 2048, 16384, 1024),
               sdesc_sw128(sb + oBt + kk * 2048, 16384, 1024), id_mn, kk);
      mma_commit(bar_mma);
    }
    ok = mbar_wait(bar_mma, 0, kWaitNs);
    if (!__syncthreads_or(!ok)) {
      tc_fence_after();
      uint32_t r[32];
      for (int t = 0; t < 3; ++t)
        for (int j = 0; j < 4; ++j) {
          tmem_ld_x32(tl + 128u * t + 32u * j, r);
          for (int i = 0; i < 32; ++i) out[(6 + t) * 16384 + tid * 128 + 32 * j + i] = __uint_as_float(r[i]);
        }
    } else if (tid == 0) {
      raise_status(status, SSS_ERR_TIMEOUT);
    }
  } else if (tid == 0) {
    raise_status(status, SSS_ERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tm, 512);
}


namespace {
bool make_tile_map(CUtensorMap* m, const void* ptr) {  // [128][128] bf16
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {128, 128};
  const cuuint64_t strides[1] = {256};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t tc_selftest_launch(const void* A, const void* B, float* out, int* status,
                               cudaStream_t st) {
  CUtensorMap mA, mB;
  if (!make_tile_map(&mA, A) || !make_tile_map(&mB, B)) return cudaErrorInvalidValue;
  const uint32_t smem = 131072 + 64 + 1024;
  cudaError_t e = cudaFuncSetAttribute(tc_selftest_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  tc_selftest_kernel<<<1, 128, smem, st>>>(mA, mB, static_cast<const __nv_bfloat16*>(A),
                                           static_cast<const __nv_bfloat16*>(B), out, status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const uint32_t smem2 = 98304 + 64 + 1024;
  e = cudaFuncSetAttribute(tc_selftest2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(smem2));
  if (e != cudaSuccess) return e;
  tc_selftest2_kernel<<<1, 128, smem2, st>>>(mA, static_cast<const __nv_bfloat16*>(A),
                                             static_cast<const __nv_bfloat16*>(B), out, status);
  return cudaGetLastError();
}

}  // namespace selftest
}  // namespace sss

// A, B: [128][128] bf16 row-major device matrices (16-byte aligned); out: 9
// fp32 [128][128] blocks (device); status: a device int the kernels OR
// SSS_ERR_TIMEOUT into.  Returns the CUDA error code of the launches.
extern "C" int sss_test_tcgen05_layouts(const void* A, const void* B, float* out, int* status,
                                        void* stream) {
  if (!A || !B || !out || !status) return int(cudaErrorInvalidValue);
  return int(sss::selftest::tc_selftest_launch(A, B, out, status,
                                               reinterpret_cast<cudaStream_t>(stream)));
}
