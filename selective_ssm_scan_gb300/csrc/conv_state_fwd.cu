// Causal depthwise conv1d with an explicit (K-1)-sample conv state, SiLU
// fused, final state written in the same pass.
//
// Follows "Chapter 7: state, chunking and incremental inference" (causal-conv1d
// tutorial), section "define the state with the extended sequence":
// u = [S_0..S_{K-2}, x_0..x_{L-1}], z_t = bias + sum_k w_k u_{t+k},
// F = u[L : L+K-1].
//
// GB300 mapping (HBM-bound: read x once, write u once; the kernel is
// latency-bound unless each SM keeps enough loads in flight):
//  * a work item is VEC adjacent channels (4 bytes of x: a bf16 pair or one
//    fp32) by TILE consecutive tokens of one sequence; a warp covers
//    32*VEC adjacent channels of a token, so each load is one fully used
//    128-byte line and the stores are 256 (fp32 u) or 128 (bf16 u) bytes;
//  * the TILE inputs of an item are loaded, still packed, into TILE
//    registers before any arithmetic: a thread holds ~40 registers, so an SM
//    runs 1500+ threads with TILE independent loads each in flight;
//  * the K-1 samples before the tile come from x (L2 hits: the previous
//    tile's tail) or, for tile 0, from the conv state;
//  * a 2-D grid (channel vectors x token tiles x sequences) gives every item
//    its coordinates without any division; ~46 registers let five
//    256-thread CTAs share an SM;
//  * the thread of tile 0 is the only one that reads S for its channels and
//    the only one that writes F, so state_out may alias state_in.
#include "common.cuh"

namespace sss {

constexpr int kConvMaxK = 8;
constexpr int kConvThreads = 256;

template <typename T, int VEC>
struct __align__(sizeof(T) * VEC) Pack {
  T e[VEC];
};

// One work item: VEC channels from d0 by the tokens [t0, t0 + nt) of
// sequence b (xp = &x[b][t0][d0], up = &u[b][t0][d0]).  FULL: nt == TILE,
// no per-token predicates.
template <typename TX, typename TU, int VEC, int TILE, int KT, bool SILU, bool FULL>
__device__ __forceinline__ void conv_item(const TX* __restrict__ xp, const float* __restrict__ w,
                                          const float* __restrict__ bias, const TX* s_in,
                                          TU* __restrict__ up, int64_t b, int d0, int tile,
                                          int nt, int D, int K) {
  constexpr int MK = KT > 0 ? KT : kConvMaxK;  // register window capacity
  constexpr int MW = MK - 1 > 0 ? MK - 1 : 1;
  using PX = Pack<TX, VEC>;
  // the tile's inputs, packed, all issued before any arithmetic
  PX xr[TILE];
  {
    const TX* q = xp;
#pragma unroll
    for (int i = 0; i < TILE; ++i) {
      if (FULL || i < nt) xr[i] = *reinterpret_cast<const PX*>(q);
      q += D;
    }
  }

  // window: the K-1 extended-sequence samples before token t0, oldest
  // first.  Tile 0 reads them from the conv state S; later tiles read the
  // previous tile's tail of x (TILE >= K-1).
  float win[MW][VEC];
#pragma unroll
  for (int j = 0; j < MW; ++j) {
#pragma unroll
    for (int v = 0; v < VEC; ++v) win[j][v] = 0.0f;  // unused entries stay 0
    if (j < K - 1) {
      if (tile == 0) {
        if (s_in) {
#pragma unroll
          for (int v = 0; v < VEC; ++v)
            win[j][v] = to_f32(s_in[(int64_t(b) * D + d0 + v) * (K - 1) + j]);
        }
      } else {
        const PX q = *reinterpret_cast<const PX*>(xp - int64_t(K - 1 - j) * D);
#pragma unroll
        for (int v = 0; v < VEC; ++v) win[j][v] = to_f32(q.e[v]);
      }
    }
  }

  // weights: wk[k] multiplies window sample k, wx the current input
  float wk[MW][VEC];
  float wx[VEC], bs[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) {
    bs[v] = bias ? bias[d0 + v] : 0.0f;
    if constexpr (KT == 4) {
      // one 16-byte load per channel (the host checks w's alignment)
      const float4 q = __ldg(reinterpret_cast<const float4*>(w) + (d0 + v));
      wk[0][v] = q.x;
      wk[1][v] = q.y;
      wk[2][v] = q.z;
      wx[v] = q.w;
    } else {
      wx[v] = w[(d0 + v) * K + (K - 1)];
#pragma unroll
      for (int k = 0; k < MW; ++k) wk[k][v] = (k < K - 1) ? w[(d0 + v) * K + k] : 0.0f;
    }
  }

#pragma unroll
  for (int i = 0; i < TILE; ++i, up += D) {
    if (FULL || i < nt) {
      float xv[VEC], z[VEC];
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        xv[v] = to_f32(xr[i].e[v]);
        float acc = bs[v];
#pragma unroll
        for (int k = 0; k < MW; ++k) acc = fmaf(wk[k][v], win[k][v], acc);
        acc = fmaf(wx[v], xv[v], acc);
        z[v] = SILU ? silu(acc) : acc;  // compile-time: no branch in the loop
      }
      st_vec<TU, VEC>(up, z);
      // slide the window by one sample (entries k >= K-1 stay unused: wk = 0)
#pragma unroll
      for (int k = 0; k < MW - 1; ++k)
#pragma unroll
        for (int v = 0; v < VEC; ++v) win[k][v] = (k < K - 2) ? win[k + 1][v] : win[k][v];
#pragma unroll
      for (int k = 0; k < MW; ++k)
        if (k == K - 2) {
#pragma unroll
          for (int v = 0; v < VEC; ++v) win[k][v] = xv[v];
        }
    }
  }

}

template <typename TX, typename TU, int VEC, int TILE, int KT, bool SILU>
__global__ void __launch_bounds__(kConvThreads)
conv_state_fwd_kernel(const TX* __restrict__ x, const float* __restrict__ w,
                      const float* __restrict__ bias, const TX* s_in, TX* s_out,
                      TU* __restrict__ u, int L, int D, int K_rt, int n_dvec, int tile_base) {
  const int K = KT > 0 ? KT : K_rt;
  // grid: x = channel vectors, y = token tiles (from tile_base), z = sequences
  const int dvec = blockIdx.x * blockDim.x + threadIdx.x;
  if (dvec >= n_dvec) return;
  const int tile = tile_base + int(blockIdx.y);
  const int64_t b = blockIdx.z;
  const int d0 = dvec * VEC;
  const int t0 = tile * TILE;
  const int nt = (L - t0) < TILE ? (L - t0) : TILE;
  const int64_t off = (b * L + t0) * D + d0;
  if (nt == TILE)
    conv_item<TX, TU, VEC, TILE, KT, SILU, true>(x + off, w, bias, s_in, u + off, b, d0, tile,
                                                 nt, D, K);
  else
    conv_item<TX, TU, VEC, TILE, KT, SILU, false>(x + off, w, bias, s_in, u + off, b, d0, tile,
                                                  nt, D, K);

  // final state F_j = ext[L + j].  Only tile 0 reads S for these channels
  // and it writes F last, in increasing j: when L + j < K-1 it reads
  // S[L + j], an entry it has not written yet (L + j >= j), so state_out
  // may alias state_in.
  if (tile == 0 && s_out) {
    const int64_t sb = (b * D + d0) * (K - 1);
    for (int j = 0; j < K - 1; ++j) {
      const int e = L + j;
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        TX fv;
        if (e < K - 1)
          fv = s_in ? s_in[sb + v * (K - 1) + e] : from_f32<TX>(0.0f);
        else
          fv = x[(b * L + (e - (K - 1))) * D + d0 + v];
        s_out[sb + v * (K - 1) + j] = fv;
      }
    }
  }
}

template <typename TX, typename TU, int VEC, int TILE>
static cudaError_t launch_conv(const void* x, const float* w, const float* bias,
                               const void* s_in, void* s_out, void* u, int64_t Bz,
                               int64_t L, int64_t D, int K, int silu_on,
                               cudaStream_t st) {
  const int64_t n_dvec = D / VEC;
  const int64_t n_tiles = L > 0 ? (L + TILE - 1) / TILE : 1;
  if (Bz == 0 || n_dvec == 0) return cudaSuccess;
  if (L > 0x7fffffffLL - TILE || D > 0x7fffffffLL) return cudaErrorInvalidValue;
  constexpr int64_t kMaxYZ = 65535;  // grid y and z limits: larger shapes take several launches
  auto args = [&](auto kern) -> cudaError_t {
    const unsigned gx = unsigned((n_dvec + kConvThreads - 1) / kConvThreads);
    for (int64_t b0 = 0; b0 < Bz; b0 += kMaxYZ) {
      const int64_t nb = (Bz - b0) < kMaxYZ ? (Bz - b0) : kMaxYZ;
      const TX* xb = static_cast<const TX*>(x) + b0 * L * D;
      const TX* sib = s_in ? static_cast<const TX*>(s_in) + b0 * D * (K - 1) : nullptr;
      TX* sob = s_out ? static_cast<TX*>(s_out) + b0 * D * (K - 1) : nullptr;
      TU* ub = static_cast<TU*>(u) + b0 * L * D;
      for (int64_t tb = 0; tb < n_tiles; tb += kMaxYZ) {
        const int64_t ny = (n_tiles - tb) < kMaxYZ ? (n_tiles - tb) : kMaxYZ;
        kern<<<dim3(gx, unsigned(ny), unsigned(nb)), kConvThreads, 0, st>>>(
            xb, w, bias, sib, sob, ub, int(L), int(D), K, int(n_dvec), int(tb));
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
      }
    }
    return cudaSuccess;
  };
  if (!silu_on) return args(conv_state_fwd_kernel<TX, TU, VEC, TILE, 0, false>);
  if (K == 4 && reinterpret_cast<uintptr_t>(w) % 16 == 0)
    return args(conv_state_fwd_kernel<TX, TU, VEC, TILE, 4, true>);
  if (K == 3) return args(conv_state_fwd_kernel<TX, TU, VEC, TILE, 3, true>);
  if (K == 2) return args(conv_state_fwd_kernel<TX, TU, VEC, TILE, 2, true>);
  return args(conv_state_fwd_kernel<TX, TU, VEC, TILE, 0, true>);
}

template <typename TX, typename TU>
static cudaError_t conv_dispatch_u(const void* x, const float* w, const float* bias,
                                   const void* s_in, void* s_out, void* u, int64_t Bz,
                                   int64_t L, int64_t D, int K, int silu_on,
                                   cudaStream_t st) {
  // a bf16 pair (4 bytes) per thread when the channel count and the
  // pointers allow it; one channel otherwise
  constexpr int VEC = sizeof(TX) == 2 ? 2 : 1;
  const bool aligned = (D % VEC == 0) &&
                       (reinterpret_cast<uintptr_t>(x) % (sizeof(TX) * VEC) == 0) &&
                       (reinterpret_cast<uintptr_t>(u) % (sizeof(TU) * VEC) == 0);
  if (aligned)
    return launch_conv<TX, TU, VEC, 16>(x, w, bias, s_in, s_out, u, Bz, L, D, K, silu_on, st);
  return launch_conv<TX, TU, 1, 16>(x, w, bias, s_in, s_out, u, Bz, L, D, K, silu_on, st);
}

cudaError_t conv_state_fwd_launch(const void* x, sss_dtype xt, const float* w,
                                  const float* bias, const void* s_in, void* s_out,
                                  void* u, sss_dtype ut, int64_t Bz, int64_t L,
                                  int64_t D, int K, int silu_on, cudaStream_t st) {
  if (xt == SSS_BF16 && ut == SSS_F32)
    return conv_dispatch_u<__nv_bfloat16, float>(x, w, bias, s_in, s_out, u, Bz, L, D, K, silu_on, st);
  if (xt == SSS_BF16 && ut == SSS_BF16)
    return conv_dispatch_u<__nv_bfloat16, __nv_bfloat16>(x, w, bias, s_in, s_out, u, Bz, L, D, K, silu_on, st);
  if (xt == SSS_F32 && ut == SSS_F32)
    return conv_dispatch_u<float, float>(x, w, bias, s_in, s_out, u, Bz, L, D, K, silu_on, st);
  return conv_dispatch_u<float, __nv_bfloat16>(x, w, bias, s_in, s_out, u, Bz, L, D, K, silu_on, st);
}


// ---- packed samples -----------------------------------------------------------
// The conv over rows that pack several samples ("Chapter 7: state, chunking
// and incremental inference", section "packed sequence boundaries"): tap k of
// token t reads u_{t+k} only when its sequence id equals token t's (identity
// equality); state entries (positions < 0) carry token 0's id.  F is the
// row's last K-1 inputs, as without ids.  One thread per (sequence, channel,
// tile of kPackTile tokens) walks its tile with a register window of inputs
// and ids; the thread of tile 0 writes F (state_out may alias state_in).
namespace {
constexpr int kPackTile = 16;

template <typename TX, typename TU, bool SILU>
__global__ void __launch_bounds__(kConvThreads)
conv_packed_kernel(const TX* __restrict__ x, const float* __restrict__ w,
                   const float* __restrict__ bias, const TX* s_in, TX* s_out,
                   const int32_t* __restrict__ seq_idx, TU* __restrict__ u, int64_t L, int64_t D,
                   int K) {
  const int64_t d = blockIdx.x * int64_t(kConvThreads) + threadIdx.x;
  if (d >= D) return;
  const int64_t b = blockIdx.z;
  const int64_t t0 = int64_t(blockIdx.y) * kPackTile;
  const int32_t* ids = seq_idx + b * L;
  const int32_t id0 = L > 0 ? ids[0] : 0;
  float win[kConvMaxK];   // u_{t-K+1} .. u_{t-1}, oldest first
  int32_t wid[kConvMaxK];
  float wk[kConvMaxK];
  for (int k = 0; k < K; ++k) wk[k] = w[d * K + k];
  const float bsd = bias ? bias[d] : 0.0f;
  for (int j = 0; j < K - 1; ++j) {
    const int64_t pos = t0 - (K - 1) + j;
    if (pos < 0) {
      const int64_t e = K - 1 + pos;  // extended index into S
      win[j] = s_in ? to_f32(s_in[(b * D + d) * (K - 1) + e]) : 0.0f;
      wid[j] = id0;
    } else {
      win[j] = to_f32(x[(b * L + pos) * D + d]);
      wid[j] = ids[pos];
    }
  }
  for (int64_t t = t0; t < t0 + kPackTile && t < L; ++t) {
    const float xv = to_f32(x[(b * L + t) * D + d]);
    const int32_t it = ids[t];
    float z = fmaf(wk[K - 1], xv, bsd);
    for (int j = 0; j < K - 1; ++j)
      if (wid[j] == it) z = fmaf(wk[j], win[j], z);
    u[(b * L + t) * D + d] = from_f32<TU>(SILU ? silu(z) : z);
    for (int j = 0; j + 1 < K - 1; ++j) {
      win[j] = win[j + 1];
      wid[j] = wid[j + 1];
    }
    if (K > 1) {
      win[K - 2] = xv;
      wid[K - 2] = it;
    }
  }
  if (blockIdx.y == 0 && s_out) {  // F_j = u[L + j], read in increasing j before it is written
    const int64_t sb = (b * D + d) * (K - 1);
    for (int j = 0; j < K - 1; ++j) {
      const int64_t e = L + j;
      s_out[sb + j] = e < K - 1 ? (s_in ? s_in[sb + e] : from_f32<TX>(0.0f))
                                : x[(b * L + (e - (K - 1))) * D + d];
    }
  }
}

template <typename TX, typename TU>
cudaError_t launch_packed(const void* x, const float* w, const float* bias, const void* s_in,
                          void* s_out, const int32_t* seq_idx, void* u, int64_t Bz, int64_t L,
                          int64_t D, int K, int silu_on, cudaStream_t st) {
  const int64_t tiles = L > 0 ? (L + kPackTile - 1) / kPackTile : 1;
  if (Bz == 0 || D == 0) return cudaSuccess;
  if (Bz > 65535 || tiles > 65535) return cudaErrorInvalidValue;
  const dim3 g(unsigned((D + kConvThreads - 1) / kConvThreads), unsigned(tiles), unsigned(Bz));
  if (silu_on)
    conv_packed_kernel<TX, TU, true><<<g, kConvThreads, 0, st>>>(
        static_cast<const TX*>(x), w, bias, static_cast<const TX*>(s_in), static_cast<TX*>(s_out),
        seq_idx, static_cast<TU*>(u), L, D, K);
  else
    conv_packed_kernel<TX, TU, false><<<g, kConvThreads, 0, st>>>(
        static_cast<const TX*>(x), w, bias, static_cast<const TX*>(s_in), static_cast<TX*>(s_out),
        seq_idx, static_cast<TU*>(u), L, D, K);
  return cudaGetLastError();
}
}  // namespace

cudaError_t conv_packed_launch(const void* x, sss_dtype xt, const float* w, const float* bias,
                               const void* s_in, void* s_out, const int32_t* seq_idx, void* u,
                               sss_dtype ut, int64_t Bz, int64_t L, int64_t D, int K, int silu_on,
                               cudaStream_t st) {
  if (xt == SSS_BF16 && ut == SSS_F32)
    return launch_packed<__nv_bfloat16, float>(x, w, bias, s_in, s_out, seq_idx, u, Bz, L, D, K, silu_on, st);
  if (xt == SSS_BF16 && ut == SSS_BF16)
    return launch_packed<__nv_bfloat16, __nv_bfloat16>(x, w, bias, s_in, s_out, seq_idx, u, Bz, L, D, K, silu_on, st);
  if (xt == SSS_F32 && ut == SSS_F32)
    return launch_packed<float, float>(x, w, bias, s_in, s_out, seq_idx, u, Bz, L, D, K, silu_on, st);
  return launch_packed<float, __nv_bfloat16>(x, w, bias, s_in, s_out, seq_idx, u, Bz, L, D, K, silu_on, st);
}

}  // namespace sss
