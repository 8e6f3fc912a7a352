// Helpers shared by the tensor-core scan kernels: bf16 hi/lo splitting,
// shared-memory operand descriptors of the chunk tiles, the bounded mbarrier
// wait with its abort flag, row stores of y, and the host-side tensor maps.
#pragma once

#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace sss {
namespace tcs {
using namespace tc;

// every mbarrier wait of the scan kernels gives up after this long
constexpr uint64_t kWaitNs = 2000000000ull;
// chunks whose log-decay range exceeds this are not factored as
// exp(Lam_t - R) exp(R - Lam_s) (the factors could leave the fp32 range)
constexpr float kFactorRange = 100.0f;

__device__ __forceinline__ uint16_t bf16_bits(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}
__device__ __forceinline__ uint32_t pack2(uint16_t lo_elem, uint16_t hi_elem) {
  return uint32_t(lo_elem) | (uint32_t(hi_elem) << 16);
}
// (a, b) -> packed hi pair and lo pair: v == hi + lo to ~2^-16 relative
// (one paired conversion for each half)
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h2 = __floats2bfloat162_rn(a, b);
  hi = *reinterpret_cast<const uint32_t*>(&h2);
  const __nv_bfloat162 l2 =
      __floats2bfloat162_rn(a - __uint_as_float(hi << 16), b - __uint_as_float(hi & 0xFFFF0000u));
  lo = *reinterpret_cast<const uint32_t*>(&l2);
}

// K-major descriptor of a [rows][128-element K] tile stored as two 64-wide K
// blocks `blk` bytes apart; K step kk covers K elements [16 kk, 16 kk + 16).
__device__ __forceinline__ uint64_t kdesc(uint32_t base, int kk, uint32_t blk) {
  return sdesc_sw128(base + uint32_t(kk >> 2) * blk + uint32_t(kk & 3) * 32u, 16, 1024);
}
// MN-major descriptor of [K rows][64 MN] tiles (128-byte rows), a second
// 64-wide MN block 16 KB further (used when N = 128): K step kk starts 16
// rows further.  The hardware may read up to 16 KB past the start even when
// N = 64, so every such tile keeps valid shared memory there.
__device__ __forceinline__ uint64_t mndesc(uint32_t base, int kk) {
  return sdesc_sw128(base + uint32_t(kk) * 2048u, 16384, 1024);
}

// The same K steps as additions to a base descriptor (start address in
// 16-byte units in the low 14 bits; shared addresses stay below 256 KB, so the
// sum never carries into the next field).  With the step a compile-time
// constant the issuing thread spends one 64-bit add per MMA instead of
// rebuilding the descriptor, which otherwise costs more than the MMA itself.
__host__ __device__ constexpr uint64_t kstep(int kk, uint32_t blk) {
  return uint64_t((uint32_t(kk >> 2) * blk + uint32_t(kk & 3) * 32u) >> 4);
}
__host__ __device__ constexpr uint64_t mnstep(int kk) { return uint64_t(kk) * 128u; }

// Row `r` (64 fp32 values, times `scale`) -> hi and lo bf16 rows of two
// MN-major tiles.
__device__ __forceinline__ void write_split_row(uint8_t* hi_tile, uint8_t* lo_tile, int r,
                                                const float* v, float scale = 1.0f) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      split2(scale * v[8 * c + 2 * k], scale * v[8 * c + 2 * k + 1], hw[k], lw[k]);
    *reinterpret_cast<uint4*>(hi_tile + sw128(r, c)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(lo_tile + sw128(r, c)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
}

struct Ctl {
  uint32_t bars;              // smem address of barrier 0
  volatile int* abort;
  int* status;
  __device__ uint32_t bar(int i) const { return bars + 8u * uint32_t(i); }
  // bounded wait; false when the CTA is aborting
  __device__ bool wait(int i, uint32_t parity) const {
    const uint32_t b = bar(i);
    if (mbar_try_wait(b, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    // sleep in the wait (woken by the phase completing) rather than spin
    while (!mbar_try_wait_sleep(b, parity, 20000u)) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > kWaitNs) {
        *abort = 1;
        raise_status(status, SSS_ERR_TIMEOUT);
        return false;
      }
    }
    return true;
  }
};

template <typename TY>
__device__ __forceinline__ void store_row16(TY* row, const float* v);
template <>
__device__ __forceinline__ void store_row16<float>(float* row, const float* v) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    reinterpret_cast<float4*>(row)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}
template <>
__device__ __forceinline__ void store_row16<__nv_bfloat16>(__nv_bfloat16* row, const float* v) {
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = pack2(bf16_bits(v[8 * q + 2 * k]), bf16_bits(v[8 * q + 2 * k + 1]));
    reinterpret_cast<uint4*>(row)[q] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ---- host: tensor maps ------------------------------------------------------
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [Bz][L][G*N] bf16 viewed as a 3-D tensor; boxes of 64 (n) x 128 (t) x 1.
inline bool make_bc_map(CUtensorMap* m, const void* ptr, int64_t Bz, int64_t L, int G, int N) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {cuuint64_t(G) * N, cuuint64_t(L), cuuint64_t(Bz)};
  const cuuint64_t strides[2] = {cuuint64_t(G) * N * 2, cuuint64_t(L) * G * N * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// raw input [Bz][L][D] bf16 as a 3-D tensor; boxes of 64 channels x `rows` x 1
inline bool make_x_map(CUtensorMap* m, const void* ptr, int64_t Bz, int64_t L, int64_t D,
                       uint32_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(L), cuuint64_t(Bz)};
  const cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(L) * D * 2};
  const cuuint32_t box[3] = {64, rows, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tcs
}  // namespace sss
