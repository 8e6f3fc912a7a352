// Causal depthwise conv1d with an explicit (K-1)-sample conv state, SiLU
// fused, final state written in the same pass.
//
// Follows "Chapter 7: state, chunking and incremental inference" (causal-conv1d
// tutorial), section "define the state with the extended sequence":
// u = [S_0..S_{K-2}, x_0..x_{L-1}], z_t = bias + sum_k w_k u_{t+k},
// F = u[L : L+K-1].
//
// GB300 mapping (HBM-bound: read x once, write u once):
//  * a thread owns VEC adjacent channels (16 bytes of x: 8 bf16 or 4 fp32)
//    and TILE consecutive tokens; a warp covers 32*VEC adjacent channels of
//    one token, so every load and store instruction is a coalesced 128-bit
//    access of a contiguous 512-byte run;
//  * the whole TILE of x is loaded into registers before any arithmetic, so
//    each thread keeps TILE independent 16-byte loads in flight;
//  * the K-1 samples before the tile come from x (L2 hits: they are the
//    previous tile's tail) or, for tile 0, from the conv state;
//  * the thread of tile 0 is the only one that reads S for its channels and
//    the only one that writes F, so state_out may alias state_in.
#include "common.cuh"

namespace sss {

constexpr int kConvMaxK = 8;

template <typename T, int VEC>
struct __align__((sizeof(T) * VEC) >= 16 ? 16 : (sizeof(T) * VEC)) Pack {
  T e[VEC];
};

template <typename TX, typename TU, int VEC, int TILE, int KT>
__global__ void __launch_bounds__(256, 3)
conv_state_fwd_kernel(const TX* __restrict__ x, const float* __restrict__ w,
                      const float* __restrict__ bias, const TX* s_in, TX* s_out,
                      TU* __restrict__ u, int64_t L, int64_t D, int K_rt,
                      int apply_silu, int64_t n_dvec, int64_t n_tiles, int64_t n_items) {
  constexpr int MK = KT > 0 ? KT : kConvMaxK;  // register window capacity
  const int K = KT > 0 ? KT : K_rt;
  using PX = Pack<TX, VEC>;
  const int64_t item = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (item >= n_items) return;
  const int64_t dvec = item % n_dvec;
  const int64_t rest = item / n_dvec;
  const int64_t tile = rest % n_tiles;
  const int64_t b = rest / n_tiles;
  const int64_t d0 = dvec * VEC;
  const int64_t t0 = tile * TILE;
  const int64_t nt = (L - t0) < TILE ? (L - t0) : TILE;

  // the tile's inputs: all loads are issued before any arithmetic
  PX xr[TILE];
#pragma unroll
  for (int i = 0; i < TILE; ++i)
    if (i < nt) xr[i] = *reinterpret_cast<const PX*>(x + (b * L + t0 + i) * D + d0);

  // window: the K-1 extended-sequence samples before token t0, oldest first.
  // Tile 0 reads them from the conv state S (t0 - (K-1) + j < 0 there);
  // later tiles read the previous tile's tail of x (TILE >= K-1).
  float win[MK - 1 > 0 ? MK - 1 : 1][VEC];
#pragma unroll
  for (int j = 0; j < MK - 1; ++j) {
#pragma unroll
    for (int v = 0; v < VEC; ++v) win[j][v] = 0.0f;  // unused entries (j >= K-1) stay 0
    if (j < K - 1) {
      if (tile == 0) {
#pragma unroll
        for (int v = 0; v < VEC; ++v)
          win[j][v] = s_in ? to_f32(s_in[(b * D + d0 + v) * (K - 1) + j]) : 0.0f;
      } else {
        const PX p = *reinterpret_cast<const PX*>(x + (b * L + t0 - (K - 1) + j) * D + d0);
#pragma unroll
        for (int v = 0; v < VEC; ++v) win[j][v] = to_f32(p.e[v]);
      }
    }
  }

  // weights: wk[k] multiplies window sample k, wx the current input
  float wk[MK - 1 > 0 ? MK - 1 : 1][VEC];
  float wx[VEC], bs[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) {
    bs[v] = bias ? bias[d0 + v] : 0.0f;
    wx[v] = w[(d0 + v) * K + (K - 1)];
#pragma unroll
    for (int k = 0; k < MK - 1; ++k) wk[k][v] = (k < K - 1) ? w[(d0 + v) * K + k] : 0.0f;
  }

#pragma unroll
  for (int i = 0; i < TILE; ++i) {
    if (i < nt) {
      float xv[VEC], z[VEC];
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        xv[v] = to_f32(xr[i].e[v]);
        float acc = bs[v];
#pragma unroll
        for (int k = 0; k < MK - 1; ++k) acc = fmaf(wk[k][v], win[k][v], acc);
        acc = fmaf(wx[v], xv[v], acc);
        z[v] = apply_silu ? silu(acc) : acc;
      }
      st_vec<TU, VEC>(u + (b * L + t0 + i) * D + d0, z);
      // slide the window by one sample (entries k >= K-1 stay unused: wk = 0)
#pragma unroll
      for (int k = 0; k < MK - 2; ++k)
#pragma unroll
        for (int v = 0; v < VEC; ++v) win[k][v] = (k < K - 2) ? win[k + 1][v] : win[k][v];
#pragma unroll
      for (int k = 0; k < MK - 1; ++k)
        if (k == K - 2) {
#pragma unroll
          for (int v = 0; v < VEC; ++v) win[k][v] = xv[v];
        }
    }
  }

  // final state F_j = ext[L + j].  Only tile 0 reads S for these channels and
  // it writes F last, in increasing j: when L + j < K-1 it reads S[L + j],
  // an entry it has not written yet (L + j >= j), so state_out may alias
  // state_in.
  if (tile == 0 && s_out) {
    for (int j = 0; j < K - 1; ++j) {
      const int64_t e = L + j;
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        TX fv;
        if (e < K - 1)
          fv = s_in ? s_in[(b * D + d0 + v) * (K - 1) + e] : from_f32<TX>(0.0f);
        else
          fv = x[(b * L + (e - (K - 1))) * D + d0 + v];
        s_out[(b * D + d0 + v) * (K - 1) + j] = fv;
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
  const int64_t n_items = Bz * n_tiles * n_dvec;
  if (n_items == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (n_items + threads - 1) / threads;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  auto args = [&](auto kern) {
    kern<<<unsigned(blocks), threads, 0, st>>>(
        static_cast<const TX*>(x), w, bias, static_cast<const TX*>(s_in),
        static_cast<TX*>(s_out), static_cast<TU*>(u), L, D, K, silu_on, n_dvec,
        n_tiles, n_items);
  };
  if (K == 4)
    args(conv_state_fwd_kernel<TX, TU, VEC, TILE, 4>);
  else if (K == 3)
    args(conv_state_fwd_kernel<TX, TU, VEC, TILE, 3>);
  else if (K == 2)
    args(conv_state_fwd_kernel<TX, TU, VEC, TILE, 2>);
  else
    args(conv_state_fwd_kernel<TX, TU, VEC, TILE, 0>);
  return cudaGetLastError();
}

template <typename TX, typename TU>
static cudaError_t conv_dispatch_u(const void* x, const float* w, const float* bias,
                                   const void* s_in, void* s_out, void* u, int64_t Bz,
                                   int64_t L, int64_t D, int K, int silu_on,
                                   cudaStream_t st) {
  constexpr int VEC = 16 / int(sizeof(TX));
  const bool aligned = (D % VEC == 0) && (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
                       (reinterpret_cast<uintptr_t>(u) % 16 == 0);
  if (aligned)
    return launch_conv<TX, TU, VEC, 8>(x, w, bias, s_in, s_out, u, Bz, L, D, K, silu_on, st);
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

}  // namespace sss
