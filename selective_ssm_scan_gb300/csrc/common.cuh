// Shared device helpers of libsss: storage-type conversion, SiLU, the
// device status word.  Arithmetic of the method lives in the kernel files.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sss.h"

namespace sss {

// log-decay given to a token that starts a new packed sample: exp(-200) is
// 0 in fp32, so the state carried into it (and every product that weighs
// earlier tokens through the decay) is exactly zero
constexpr float kSampleStartLog = -200.0f;
// whether token t of row b starts a new sample (seq_idx [Bz, L], NULL: never)
__device__ __forceinline__ bool sample_start(const int32_t* seq_idx, int64_t b, int64_t L,
                                             int64_t t) {
  return seq_idx && t > 0 && seq_idx[b * L + t] != seq_idx[b * L + t - 1];
}

// Kernels OR status bits into a device status word (they never trap).  The
// word lives in api.cu; its device address is passed to every kernel.
__device__ __forceinline__ void raise_status(int* status, int bits) {
  if (status) atomicOr(status, bits);
}

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z)), with CUDA's fast __expf and
// __fdividef (a few ulp; the argument of the exp is capped at 80 so that the
// divisor stays finite: for z < -80 the result is ~1e-33 either way).
__device__ __forceinline__ float silu(float z) {
  return __fdividef(z, 1.0f + __expf(fminf(-z, 80.0f)));
}

// Wait until the kernel this one was launched as a programmatic dependent of
// has finished and its memory is visible (a no-op in an ordinary launch).
__device__ __forceinline__ void dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---- packed fp32 pairs: one instruction operates on two floats (f32x2) ------
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Host helpers implemented in api.cu.
int sm_count();        // SMs of the current device (cached per device)
int* status_word();    // device address of the status word (current device)

// Launch `kern` on `st`; with `dependent` as a programmatic dependent of the
// kernel before it on the stream (its blocks may start while that kernel's
// last blocks run; the kernel must execute griddepcontrol.wait, dep_wait()
// below, before it touches memory the earlier kernel writes or reads).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dep(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, bool dependent, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = dependent ? attr : nullptr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

inline size_t dtype_size(sss_dtype t) { return t == SSS_BF16 ? 2 : 4; }
inline bool dtype_ok(int t) { return t == SSS_F32 || t == SSS_BF16; }

}  // namespace sss

namespace sss {

// ---- vector load / store of VEC elements as floats -------------------------
template <typename T, int VEC>
__device__ __forceinline__ void ld_vec(const T* __restrict__ p, float* v) {
  constexpr int BYTES = int(sizeof(T)) * VEC;
  if constexpr (BYTES % 16 == 0) {
#pragma unroll
    for (int c = 0; c < BYTES / 16; ++c) {
      union { uint4 r; T e[16 / sizeof(T)]; } u;
      u.r = __ldg(reinterpret_cast<const uint4*>(p) + c);
#pragma unroll
      for (int i = 0; i < int(16 / sizeof(T)); ++i) v[c * int(16 / sizeof(T)) + i] = to_f32(u.e[i]);
    }
  } else if constexpr (BYTES == 8) {
    union { uint2 r; T e[8 / sizeof(T)]; } u;
    u.r = __ldg(reinterpret_cast<const uint2*>(p));
#pragma unroll
    for (int i = 0; i < VEC; ++i) v[i] = to_f32(u.e[i]);
  } else if constexpr (BYTES == 4 && VEC == 2) {
    union { uint32_t r; T e[2]; } u;
    u.r = __ldg(reinterpret_cast<const unsigned int*>(p));
    v[0] = to_f32(u.e[0]);
    v[1] = to_f32(u.e[1]);
  } else {
#pragma unroll
    for (int i = 0; i < VEC; ++i) v[i] = to_f32(p[i]);
  }
}

template <typename T, int VEC>
__device__ __forceinline__ void st_vec(T* __restrict__ p, const float* v) {
  constexpr int BYTES = int(sizeof(T)) * VEC;
  if constexpr (BYTES % 16 == 0) {
#pragma unroll
    for (int c = 0; c < BYTES / 16; ++c) {
      union { uint4 r; T e[16 / sizeof(T)]; } u;
#pragma unroll
      for (int i = 0; i < int(16 / sizeof(T)); ++i) u.e[i] = from_f32<T>(v[c * int(16 / sizeof(T)) + i]);
      reinterpret_cast<uint4*>(p)[c] = u.r;
    }
  } else if constexpr (BYTES == 8) {
    union { uint2 r; T e[8 / sizeof(T)]; } u;
#pragma unroll
    for (int i = 0; i < VEC; ++i) u.e[i] = from_f32<T>(v[i]);
    *reinterpret_cast<uint2*>(p) = u.r;
  } else if constexpr (BYTES == 4 && VEC == 2) {
    union { uint32_t r; T e[2]; } u;
    u.e[0] = from_f32<T>(v[0]);
    u.e[1] = from_f32<T>(v[1]);
    *reinterpret_cast<uint32_t*>(p) = u.r;
  } else {
#pragma unroll
    for (int i = 0; i < VEC; ++i) p[i] = from_f32<T>(v[i]);
  }
}

}  // namespace sss
