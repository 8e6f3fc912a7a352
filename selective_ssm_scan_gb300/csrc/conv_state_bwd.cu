// Gradient of the causal depthwise conv with an explicit (K-1)-sample state.
//
// Follows "Chapter 7: state, chunking and incremental inference" (causal-conv1d
// tutorial), section "unified derivation of the backward pass with state":
// with u = [S, x], z_t = bias + sum_k w_k u_{t+k}, out_t = SiLU(z_t) and
// F = u[L : L+K-1], the upstream gradients dy = dL/dout and q = dL/dF give
//   delta_t = dy_t SiLU'(z_t),
//   dL/du_j = sum_{t,k: t+k=j} delta_t w_k + [L <= j < L+K-1] q_{j-L},
//   dS = du[0 : K-1],  dx = du[K-1 : K-1+L],
//   dw_k = sum_t delta_t u_{t+k},  dbias = sum_t delta_t   (and over the batch).
//
// GB300 mapping (HBM-bound: read x and dy once, write dx once):
//  * a CTA is 8 warps; lane l takes the channel vector d0 = (blockIdx.x * 32
//    + l) * VEC (one 128-byte line of bf16 x per warp and token), warp w the
//    tile of TT tokens t0 = (blockIdx.y * 8 + w) * TT;
//  * a thread walks its tile forward in time, j = t0 .. t0 + TT + MK - 2,
//    with two register windows: the last MK inputs x_{j-MK+1..j} and the
//    last MK values of delta.  At step j it forms z_j and delta_j, adds
//    delta_j u_{j+k} to its dw_k, and finishes du for the token MK - 1
//    behind (dx, or dS for the steps before token 0 in tile 0).  The MK - 1
//    tokens after the tile are read again by the next tile (L2 hits);
//  * loads are clamped into the sequence and masked, so they are issued
//    without branches, one batch of 6 tokens ahead of their use (two CTAs
//    of <= 128 registers a thread share an SM);
//  * dw and dbias: each thread sums its tile, the CTA sums its 8 warps in
//    shared memory and writes one row of partials to the workspace; a second
//    kernel adds the rows in a fixed order, so the result is deterministic.
#include "common.cuh"
#include "scan_tc_util.cuh"
#include "tc_ptx.cuh"

namespace sss {

namespace {
constexpr int kBwdWarps = 8;
constexpr int kBwdTile = 64;        // tokens per warp
constexpr int kBwdMaxK = 8;
constexpr int kBwdCtaTokens = kBwdWarps * kBwdTile;
constexpr int kBwdBatch = 6;        // tokens loaded ahead of their use

template <typename T, int VEC>
struct __align__(sizeof(T) * VEC) BwdPack {
  T e[VEC];
};

__device__ __forceinline__ float dsilu(float z) {
  // d/dz [z s(z)] = s (1 + z (1 - s)), s = 1 / (1 + exp(-z))
  const float s = __fdividef(1.0f, 1.0f + __expf(fminf(-z, 80.0f)));
  return s * fmaf(z, 1.0f - s, 1.0f);
}
}  // namespace

// MK: window capacity (the conv width when it is a compile-time constant,
// else kBwdMaxK with the real K <= MK at run time).
template <typename TX, typename TD, typename TO, int VEC, int MK, bool SILU>
__global__ void __launch_bounds__(kBwdWarps * 32, 2)
conv_state_bwd_kernel(const TX* __restrict__ x, const float* __restrict__ w,
                      const float* __restrict__ bias, const TX* __restrict__ s_in,
                      const TD* __restrict__ dy, const TD* __restrict__ q, TO* __restrict__ dx,
                      TO* __restrict__ dS, float* __restrict__ part, int L, int D, int K,
                      int n_dvec, int n_groups) {
  constexpr int NIT = kBwdTile + MK - 1;            // steps of the walk
  constexpr int NB = (NIT + kBwdBatch - 1) / kBwdBatch;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int dvec = blockIdx.x * 32 + lane;
  const int tg = blockIdx.y;
  const int64_t b = blockIdx.z;
  const int t0 = (tg * kBwdWarps + warp) * kBwdTile;
  const bool live = dvec < n_dvec && t0 < L;
  const int d0 = dvec * VEC;
  const int KM1 = K - 1;

  float dwp[MK][VEC], dbp[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) {
    dbp[v] = 0.0f;
#pragma unroll
    for (int k = 0; k < MK; ++k) dwp[k][v] = 0.0f;
  }

  if (live) {
    // wz[i]: weight of window slot i (slot MK-1 = newest) in z_j;
    // wd[i]: weight of delta slot i in du_{j-MK+1+KM1}; bs: bias
    float wz[MK][VEC], wd[MK][VEC], bs[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
      bs[v] = bias ? bias[d0 + v] : 0.0f;
#pragma unroll
      for (int i = 0; i < MK; ++i) {
        const int kz = i - (MK - K);   // tap of slot i in z
        const int kd = KM1 - i;        // tap of slot i in du
        wz[i][v] = kz >= 0 ? w[(d0 + v) * K + kz] : 0.0f;
        wd[i][v] = (kd >= 0 && kd < K) ? w[(d0 + v) * K + kd] : 0.0f;
      }
    }
    // x window before step 0: slot i >= 1 holds x_{t0-MK+i} (the conv state
    // before token 0, zero before that); each step shifts the window down
    // one slot and puts x_j in slot MK-1
    float xw[MK][VEC], dl[MK][VEC];
#pragma unroll
    for (int i = 0; i < MK; ++i) {
      const int tx = t0 - MK + i;
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        float val = 0.0f;
        if (i >= 1) {
          if (tx >= 0)
            val = to_f32(x[(b * L + tx) * D + d0 + v]);
          else if (tx >= -KM1 && s_in)
            val = to_f32(s_in[(b * D + d0 + v) * KM1 + KM1 + tx]);
        }
        xw[i][v] = val;
        dl[i][v] = 0.0f;  // delta before token t0: unused except (zero) before token 0
      }
    }
    const TX* xb = x + b * L * D + d0;
    const TD* gb = dy + b * L * D + d0;
    using PX = BwdPack<TX, VEC>;
    using PG = BwdPack<TD, VEC>;
    // batch nb + 1 is loaded (still packed) while batch nb is computed
    PX xn[kBwdBatch];
    PG gn[kBwdBatch];
    auto load_batch = [&](int nb) {
#pragma unroll
      for (int i = 0; i < kBwdBatch; ++i) {
        const int j = t0 + nb * kBwdBatch + i;
        const int64_t jc = j < L ? j : L - 1;  // clamped into the sequence, masked below
        xn[i] = *reinterpret_cast<const PX*>(xb + jc * D);
        gn[i] = *reinterpret_cast<const PG*>(gb + jc * D);
      }
    };
    load_batch(0);
#pragma unroll 1
    for (int nb = 0; nb < NB; ++nb) {
      PX xc[kBwdBatch];
      PG gc[kBwdBatch];
#pragma unroll
      for (int i = 0; i < kBwdBatch; ++i) {
        xc[i] = xn[i];
        gc[i] = gn[i];
      }
      if (nb + 1 < NB) load_batch(nb + 1);
#pragma unroll
      for (int i = 0; i < kBwdBatch; ++i) {
        const int s = nb * kBwdBatch + i;  // step index, j = t0 + s
        if (s < NIT) {
          const int j = t0 + s;
          const float m = j < L ? 1.0f : 0.0f;
#pragma unroll
          for (int v = 0; v < VEC; ++v) {
#pragma unroll
            for (int k = 0; k < MK - 1; ++k) xw[k][v] = xw[k + 1][v];
            xw[MK - 1][v] = to_f32(xc[i].e[v]) * m;
#pragma unroll
            for (int k = 0; k < MK - 1; ++k) dl[k][v] = dl[k + 1][v];
            float z = bs[v];
#pragma unroll
            for (int k = 0; k < MK; ++k) z = fmaf(wz[k][v], xw[k][v], z);
            const float g = to_f32(gc[i].e[v]) * m;
            const float dv = SILU ? g * dsilu(z) : g;
            dl[MK - 1][v] = dv;
            if (s < kBwdTile) {  // delta_j belongs to this tile
              dbp[v] += dv;
#pragma unroll
              for (int k = 0; k < MK; ++k) dwp[k][v] = fmaf(dv, xw[k][v], dwp[k][v]);
            }
          }
          // du for u index ju = j - (MK-1) + KM1, i.e. x token t = j - (MK-1)
          const int t = j - (MK - 1);
          const int ju = t + KM1;
          if (t >= t0 || (t0 == 0 && ju >= 0)) {
            float o[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
              float acc = 0.0f;
#pragma unroll
              for (int k = 0; k < MK; ++k) acc = fmaf(wd[k][v], dl[k][v], acc);
              o[v] = acc;
            }
            if (q && ju >= L && ju < L + KM1) {  // direct path from F = u[L : L+K-1]
#pragma unroll
              for (int v = 0; v < VEC; ++v)
                o[v] += to_f32(q[(b * D + d0 + v) * KM1 + (ju - L)]);
            }
            if (t >= t0) {
              if (t < L) st_vec<TO, VEC>(dx + (b * L + t) * D + d0, o);
            } else {
#pragma unroll
              for (int v = 0; v < VEC; ++v)
                dS[(b * D + d0 + v) * KM1 + ju] = from_f32<TO>(o[v]);
            }
          }
        }
      }
    }
  }

  // the CTA's 8 tiles summed in shared memory, in warp order
  __shared__ float red[kBwdWarps][MK + 1][32 * VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) {
#pragma unroll
    for (int k = 0; k < MK; ++k) red[warp][k][lane * VEC + v] = dwp[k][v];
    red[warp][MK][lane * VEC + v] = dbp[v];
  }
  __syncthreads();
  // row (b, tg) of the partials: [D][K+1] floats; dwp[k] holds the tap of
  // window slot k, i.e. tap k - (MK - K)
  float* row = part + (b * n_groups + tg) * int64_t(D) * (K + 1);
  for (int e = threadIdx.x; e < 32 * VEC * (K + 1); e += blockDim.x) {
    const int c = e / (K + 1), k = e % (K + 1);  // channel c of this CTA's 32*VEC
    const int d = blockIdx.x * 32 * VEC + c;
    if (d < n_dvec * VEC) {
      const int kk = k < K ? k + (MK - K) : MK;
      float acc = 0.0f;
      for (int ww = 0; ww < kBwdWarps; ++ww) acc += red[ww][kk][c];
      row[int64_t(d) * (K + 1) + k] = acc;
    }
  }
}

// ---- K = 4 fast path -----------------------------------------------------------
// The same walk for the common width K = 4 with a channel pair per lane (D a
// multiple of 64, 16-byte aligned rows) in packed f32x2 arithmetic.  The rows
// reach a warp through shared memory: each warp keeps a ring of kK4Stages
// groups of 4 tokens (its 64 channels of x and dy per token), filled by
// cp.async.bulk row copies that one lane issues kK4Stages groups ahead, so
// ~16 tokens per warp are in flight without holding registers.  A step is
// then only its arithmetic: the window turns over every 4 steps (the unrolled
// group), so no register moves; the first group (the state gradient in tile
// 0), the look-ahead group (three steps past the tile that only finish dx)
// and the sequence's last tile (masks, the direct path from F) are the only
// special cases.
namespace {
constexpr float kLog2eB = 1.4426950408889634f;
constexpr int kK4Warps = 4;                       // warps per CTA
constexpr int kK4Tile = 64;                       // tokens per warp
constexpr int kK4CtaTokens = kK4Warps * kK4Tile;  // tokens per row of partial sums
constexpr int kK4Stages = 4;                      // groups of 4 tokens in flight per warp

__device__ __forceinline__ float ex2a(float v) {  // 2^v, approximate
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float rcpa(float v) {  // 1 / v, approximate
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
// SiLU'(z) of a channel pair: s (1 + z (1 - s)) with s = 1 / (1 + 2^(-z log2 e));
// a very negative z gives 2^(..) = inf and s = 0, the limit.
__device__ __forceinline__ uint64_t dsilu2(uint64_t z) {
  float ta, tb;
  upk2(mul2(z, pk2(-kLog2eB, -kLog2eB)), ta, tb);
  float da, db;
  upk2(add2(pk2(ex2a(ta), ex2a(tb)), pk2(1.0f, 1.0f)), da, db);
  const uint64_t sg = pk2(rcpa(da), rcpa(db));
  const uint64_t oms = fma2(sg, pk2(-1.0f, -1.0f), pk2(1.0f, 1.0f));
  return mul2(sg, fma2(z, oms, pk2(1.0f, 1.0f)));
}

// a channel pair as a packed fp32 pair, and back
template <typename T> struct Pair;
template <> struct Pair<float> {
  using Raw = uint64_t;
  static __device__ __forceinline__ Raw load(const float* p) {
    return __ldg(reinterpret_cast<const unsigned long long*>(p));
  }
  static __device__ __forceinline__ uint64_t f2(Raw r) { return r; }
  static __device__ __forceinline__ void store(float* p, uint64_t v) {
    *reinterpret_cast<uint64_t*>(p) = v;
  }
};
template <> struct Pair<__nv_bfloat16> {
  using Raw = uint32_t;
  static __device__ __forceinline__ Raw load(const __nv_bfloat16* p) {
    return __ldg(reinterpret_cast<const unsigned int*>(p));
  }
  static __device__ __forceinline__ uint64_t f2(Raw r) {
    return pk2(__uint_as_float(r << 16), __uint_as_float(r & 0xFFFF0000u));
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, uint64_t v) {
    float a, b;
    upk2(v, a, b);
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    *reinterpret_cast<__nv_bfloat162*>(p) = h;
  }
};

template <typename TX, typename TD>
__host__ __device__ constexpr int k4_ring_bytes() {  // per warp: stages x 4 tokens x (x row + dy row)
  return kK4Stages * 4 * 64 * int(sizeof(TX) + sizeof(TD));
}
}  // namespace

template <typename TX, typename TD, typename TO, bool SILU>
__global__ void __launch_bounds__(kK4Warps * 32, 7)
conv_bwd_k4_kernel(const TX* __restrict__ x, const float* __restrict__ w,
                   const float* __restrict__ bias, const TX* __restrict__ s_in,
                   const TD* __restrict__ dy, const TD* __restrict__ q, TO* __restrict__ dx,
                   TO* __restrict__ dS, float* __restrict__ part, int L, int D, int n_groups,
                   int* status) {
  using namespace tc;
  using tcs::kWaitNs;
  using PX = Pair<TX>;
  using PD = Pair<TD>;
  using PO = Pair<TO>;
  constexpr int K = 4, TT = kK4Tile, NG = TT / 4;   // groups NG: the look-ahead group
  constexpr uint32_t RX = 64 * sizeof(TX), RD = 64 * sizeof(TD);  // row bytes of a warp
  constexpr uint32_t GB = 4 * (RX + RD);                          // bytes of a group
  extern __shared__ __align__(128) uint8_t k4_smem[];
  __shared__ __align__(8) uint64_t bars[kK4Warps][kK4Stages];
  __shared__ float red[kK4Warps][K + 1][64];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = blockIdx.x * 64;      // the CTA's 64 channels
  const int d0 = c0 + 2 * lane;        // this lane's channel pair
  const int tg = blockIdx.y;
  const int64_t b = blockIdx.z;
  const int t0 = (tg * kK4Warps + warp) * TT;
  uint8_t* ring = k4_smem + warp * k4_ring_bytes<TX, TD>();
  const uint32_t ring_s = smem_u32(ring);
  uint64_t dw0 = 0, dw1 = 0, dw2 = 0, dw3 = 0, dbs = 0;  // packed zeros

  if (t0 < L) {
    if (lane == 0) {
#pragma unroll
      for (int st = 0; st < kK4Stages; ++st) mbar_init(smem_u32(&bars[warp][st]), 1);
      fence_mbar_init();
    }
    __syncwarp();
    // group gi (tokens t0 + 4 gi .. + 3) into ring stage gi % kK4Stages; rows
    // at or past L are not copied (their values are masked at use)
    auto issue = [&](int gi) {
      const int st = gi % kK4Stages;
      const uint32_t bar = smem_u32(&bars[warp][st]);
      const int j0 = t0 + 4 * gi;
      const int nrow = min(4, L - j0);
      if (nrow <= 0) {
        mbar_arrive(bar);
        return;
      }
      mbar_arrive_expect_tx(bar, uint32_t(nrow) * (RX + RD));
      const uint32_t gs = ring_s + uint32_t(st) * GB;
      for (int i = 0; i < nrow; ++i) {
        bulk_load(gs + uint32_t(i) * RX, x + (b * L + j0 + i) * D + c0, RX, bar);
        bulk_load(gs + 4 * RX + uint32_t(i) * RD, dy + (b * L + j0 + i) * D + c0, RD, bar);
      }
    };
    if (lane == 0) {
#pragma unroll
      for (int gi = 0; gi < kK4Stages; ++gi)
        if (gi <= NG) issue(gi);
    }
    const uint64_t wk0 = pk2(w[d0 * K + 0], w[(d0 + 1) * K + 0]);
    const uint64_t wk1 = pk2(w[d0 * K + 1], w[(d0 + 1) * K + 1]);
    const uint64_t wk2 = pk2(w[d0 * K + 2], w[(d0 + 1) * K + 2]);
    const uint64_t wk3 = pk2(w[d0 * K + 3], w[(d0 + 1) * K + 3]);
    const uint64_t bs = bias ? pk2(bias[d0], bias[d0 + 1]) : 0ull;
    // x of tokens t0-3 .. t0-1 (the conv state before token 0, zeros without one)
    auto x_at = [&](int t) -> uint64_t {
      if (t >= 0) return PX::f2(PX::load(x + (b * L + t) * D + d0));
      if (!s_in) return 0ull;
      return pk2(to_f32(s_in[(b * D + d0) * (K - 1) + (K - 1) + t]),
                 to_f32(s_in[(b * D + d0 + 1) * (K - 1) + (K - 1) + t]));
    };
    uint64_t xm3 = x_at(t0 - 3), xm2 = x_at(t0 - 2), xm1 = x_at(t0 - 1);
    uint64_t dm3 = 0ull, dm2 = 0ull, dm1 = 0ull;  // delta of the three steps before

    // step j: z_j, delta_j, the tile's dw / dbias terms, and du of token j - 3
    auto step = [&](uint64_t xj, uint64_t gj, bool acc) -> uint64_t {
      const uint64_t z = fma2(wk3, xj, fma2(wk2, xm1, fma2(wk1, xm2, fma2(wk0, xm3, bs))));
      const uint64_t dl = SILU ? mul2(gj, dsilu2(z)) : gj;
      if (acc) {
        dbs = add2(dbs, dl);
        dw0 = fma2(dl, xm3, dw0);
        dw1 = fma2(dl, xm2, dw1);
        dw2 = fma2(dl, xm1, dw2);
        dw3 = fma2(dl, xj, dw3);
      }
      const uint64_t o = fma2(wk0, dl, fma2(wk1, dm1, fma2(wk2, dm2, mul2(wk3, dm3))));
      xm3 = xm2;
      xm2 = xm1;
      xm1 = xj;
      dm3 = dm2;
      dm2 = dm1;
      dm1 = dl;
      return o;
    };
    auto store_dx = [&](int t, uint64_t o) { PO::store(dx + (b * L + t) * D + d0, o); };
    auto store_ds = [&](int j, uint64_t o) {  // u index j < K - 1: the state's gradient
      float a, c;
      upk2(o, a, c);
      dS[(b * D + d0) * (K - 1) + j] = from_f32<TO>(a);
      dS[(b * D + d0 + 1) * (K - 1) + j] = from_f32<TO>(c);
    };
    const bool last_tile = t0 + TT + 3 >= L;  // masks and the direct path from F
    // the group's rows from the ring (waits for them), then the refill of
    // the stage with group g + kK4Stages (the fence orders the warp's
    // generic reads before the async copy's writes)
    auto take_group = [&](int g, typename PX::Raw (&xr)[4], typename PD::Raw (&gr)[4]) -> bool {
      const int st = g % kK4Stages;
      if (!mbar_wait(smem_u32(&bars[warp][st]), uint32_t((g / kK4Stages) & 1), kWaitNs)) {
        raise_status(status, SSS_ERR_TIMEOUT);
        return false;
      }
      const uint8_t* gs = ring + st * GB;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xr[i] = *reinterpret_cast<const typename PX::Raw*>(gs + i * RX + lane * sizeof(typename PX::Raw));
        gr[i] = *reinterpret_cast<const typename PD::Raw*>(gs + 4 * RX + i * RD +
                                                           lane * sizeof(typename PD::Raw));
      }
      __syncwarp();
      if (lane == 0 && g + kK4Stages <= NG) {
        fence_proxy_async_smem();
        issue(g + kK4Stages);
      }
      return true;
    };
    if (!last_tile) {
      // rows of dx are written through a pointer that steps one row a token
      TO* dxr = dx + (b * L + t0) * D + d0;  // token t0
      typename PX::Raw xr[4];
      typename PD::Raw gr[4];
      if (take_group(0, xr, gr)) {
#pragma unroll
        for (int i = 0; i < 3; ++i) {
          const uint64_t o = step(PX::f2(xr[i]), PD::f2(gr[i]), true);
          if (t0 == 0) store_ds(i, o);
        }
        PO::store(dxr, step(PX::f2(xr[3]), PD::f2(gr[3]), true));
        dxr += D;
#pragma unroll 1
        for (int g = 1; g < NG; ++g) {
          if (!take_group(g, xr, gr)) break;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            PO::store(dxr, step(PX::f2(xr[i]), PD::f2(gr[i]), true));
            dxr += D;
          }
        }
        if (take_group(NG, xr, gr)) {
#pragma unroll
          for (int i = 0; i < 3; ++i) {
            PO::store(dxr, step(PX::f2(xr[i]), PD::f2(gr[i]), false));
            dxr += D;
          }
        }
      }
    } else {
#pragma unroll 1
      for (int g = 0; g <= NG; ++g) {
        typename PX::Raw xr[4];
        typename PD::Raw gr[4];
        if (!take_group(g, xr, gr)) break;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int sidx = 4 * g + i;
          if (sidx >= TT + 3) break;
          const int j = t0 + sidx;
          const bool in = j < L;
          const uint64_t xj = in ? PX::f2(xr[i]) : 0ull;
          const uint64_t gj = in ? PD::f2(gr[i]) : 0ull;
          uint64_t o = step(xj, gj, sidx < TT);
          const int t = j - 3;
          if (t < t0) {
            if (t0 == 0) store_ds(j, o);
          } else if (t < L) {
            if (q && t >= L - (K - 1)) {
              const int f = t - (L - (K - 1));
              o = add2(o, pk2(to_f32(q[(b * D + d0) * (K - 1) + f]),
                              to_f32(q[(b * D + d0 + 1) * (K - 1) + f])));
            }
            store_dx(t, o);
          }
        }
      }
    }
  }

  // the CTA's tiles summed in shared memory, in warp order: one row of
  // partial sums per CTA (the same [D][K+1] layout as the general kernel)
  {
    float a, c;
    upk2(dw0, a, c); red[warp][0][2 * lane] = a; red[warp][0][2 * lane + 1] = c;
    upk2(dw1, a, c); red[warp][1][2 * lane] = a; red[warp][1][2 * lane + 1] = c;
    upk2(dw2, a, c); red[warp][2][2 * lane] = a; red[warp][2][2 * lane + 1] = c;
    upk2(dw3, a, c); red[warp][3][2 * lane] = a; red[warp][3][2 * lane + 1] = c;
    upk2(dbs, a, c); red[warp][4][2 * lane] = a; red[warp][4][2 * lane + 1] = c;
  }
  __syncthreads();
  float* row = part + (b * n_groups + tg) * int64_t(D) * (K + 1);
  for (int e = threadIdx.x; e < 64 * (K + 1); e += blockDim.x) {
    const int c = e / (K + 1), k = e % (K + 1);
    float acc = 0.0f;
#pragma unroll
    for (int ww = 0; ww < kK4Warps; ++ww) acc += red[ww][k][c];
    row[int64_t(c0 + c) * (K + 1) + k] = acc;
  }
}

// dw[d][k] = sum over rows of part[row][d][k] (k < K); dbias[d] = part[..][d][K].
// A CTA takes 32 consecutive entries; warp w adds rows w, w+8, ... in order,
// then the 8 warp sums are added in warp order (a fixed order for given sizes).
__global__ void __launch_bounds__(256)
conv_bwd_reduce_kernel(const float* __restrict__ part, float* __restrict__ dw,
                       float* __restrict__ dbias, int64_t rows, int D, int K) {
  // launched as a programmatic dependent of the walk: its blocks may start
  // while the walk's last CTAs run, and wait here until the walk's partial
  // rows are complete and visible (a no-op in an ordinary launch)
  dep_wait();
  __shared__ float acc_s[8][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n = int64_t(D) * (K + 1);
  const int64_t e = int64_t(blockIdx.x) * 32 + lane;
  float acc = 0.0f;
  if (e < n) {
    int64_t r = warp;
    for (; r + 24 < rows; r += 32) {
      const float a0 = part[r * n + e], a1 = part[(r + 8) * n + e];
      const float a2 = part[(r + 16) * n + e], a3 = part[(r + 24) * n + e];
      acc += a0;
      acc += a1;
      acc += a2;
      acc += a3;
    }
    for (; r < rows; r += 8) acc += part[r * n + e];
  }
  acc_s[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && e < n) {
    float s = 0.0f;
#pragma unroll
    for (int ww = 0; ww < 8; ++ww) s += acc_s[ww][lane];
    const int d = int(e / (K + 1)), k = int(e % (K + 1));
    if (k < K)
      dw[int64_t(d) * K + k] = s;
    else if (dbias)
      dbias[d] = s;
  }
}

// L = 0: F = S, so dS = q, and there is no weight or bias gradient
template <typename TD, typename TO>
__global__ void conv_bwd_empty_kernel(const TD* __restrict__ q, TO* __restrict__ dS,
                                      float* __restrict__ dw, float* __restrict__ dbias,
                                      int64_t n_state, int D, int K) {
  const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e < n_state) dS[e] = from_f32<TO>(q ? to_f32(q[e]) : 0.0f);
  if (e < int64_t(D) * K) dw[e] = 0.0f;
  if (dbias && e < D) dbias[e] = 0.0f;
}

size_t conv_state_bwd_workspace(int64_t Bz, int64_t L, int64_t D, int K) {
  if (Bz <= 0 || L <= 0 || D <= 0 || K < 1) return 0;
  // one row of partial sums per CTA row of tokens (the K = 4 walk's rows are
  // shorter; its size covers the general kernel's too)
  const int64_t rows_tokens = K == 4 ? kK4CtaTokens : kBwdCtaTokens;
  const int64_t groups = (L + rows_tokens - 1) / rows_tokens;
  return size_t(Bz * groups * D * (K + 1)) * sizeof(float);
}

bool conv_state_bwd_supports(int K) { return K >= 1 && K <= kBwdMaxK; }

template <typename TX, typename TD, typename TO, int VEC>
static cudaError_t launch_bwd(const void* x, const float* w, const float* bias, const void* s_in,
                              const void* dy, const void* q, void* dx, void* dS, float* dw,
                              float* dbias, int64_t Bz, int64_t L, int64_t D, int K, int silu_on,
                              void* ws, cudaStream_t st) {
  const int64_t n_dvec = D / VEC;
  const int64_t groups = (L + kBwdCtaTokens - 1) / kBwdCtaTokens;
  if (groups > 65535 || Bz > 65535) return cudaErrorInvalidValue;
  const dim3 grid(unsigned((n_dvec + 31) / 32), unsigned(groups), unsigned(Bz));
  float* part = static_cast<float*>(ws);
  auto args = [&](auto kern) -> cudaError_t {
    kern<<<grid, kBwdWarps * 32, 0, st>>>(
        static_cast<const TX*>(x), w, bias, static_cast<const TX*>(s_in),
        static_cast<const TD*>(dy), static_cast<const TD*>(q), static_cast<TO*>(dx),
        static_cast<TO*>(dS), part, int(L), int(D), K, int(n_dvec), int(groups));
    return cudaGetLastError();
  };
  cudaError_t e;
  if (K == 4)
    e = silu_on ? args(conv_state_bwd_kernel<TX, TD, TO, VEC, 4, true>)
                : args(conv_state_bwd_kernel<TX, TD, TO, VEC, 4, false>);
  else
    e = silu_on ? args(conv_state_bwd_kernel<TX, TD, TO, VEC, kBwdMaxK, true>)
                : args(conv_state_bwd_kernel<TX, TD, TO, VEC, kBwdMaxK, false>);
  if (e != cudaSuccess) return e;
  const int64_t n = D * (K + 1);
  conv_bwd_reduce_kernel<<<unsigned((n + 31) / 32), 256, 0, st>>>(part, dw, dbias, Bz * groups,
                                                                  int(D), K);
  return cudaGetLastError();
}

template <typename TX, typename TD, typename TO>
static cudaError_t launch_k4(const void* x, const float* w, const float* bias, const void* s_in,
                             const void* dy, const void* q, void* dx, void* dS, float* dw,
                             float* dbias, int64_t Bz, int64_t L, int64_t D, int silu_on,
                             void* ws, cudaStream_t st) {
  const int64_t groups = (L + kK4CtaTokens - 1) / kK4CtaTokens;
  if (groups > 65535 || Bz > 65535) return cudaErrorInvalidValue;
  const dim3 grid(unsigned(D / 64), unsigned(groups), unsigned(Bz));
  const int smem = kK4Warps * k4_ring_bytes<TX, TD>();
  float* part = static_cast<float*>(ws);
  auto args = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kK4Warps * 32, smem, st>>>(
        static_cast<const TX*>(x), w, bias, static_cast<const TX*>(s_in),
        static_cast<const TD*>(dy), static_cast<const TD*>(q), static_cast<TO*>(dx),
        static_cast<TO*>(dS), part, int(L), int(D), int(groups), status_word());
    return cudaGetLastError();
  };
  cudaError_t e = silu_on ? args(conv_bwd_k4_kernel<TX, TD, TO, true>)
                          : args(conv_bwd_k4_kernel<TX, TD, TO, false>);
  if (e != cudaSuccess) return e;
  // the fixed-order sum of the partial rows, launched so that its start
  // overlaps the walk's tail (it waits for the walk's memory itself)
  const int64_t n = D * 5;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned((n + 31) / 32));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, conv_bwd_reduce_kernel, static_cast<const float*>(part), dw,
                            dbias, int64_t(Bz * groups), int(D), 4);
}

template <typename TX, typename TD, typename TO>
static cudaError_t bwd_vec(const void* x, const float* w, const float* bias, const void* s_in,
                           const void* dy, const void* q, void* dx, void* dS, float* dw,
                           float* dbias, int64_t Bz, int64_t L, int64_t D, int K, int silu_on,
                           void* ws, cudaStream_t st) {
  if (L == 0) {
    const int64_t n_state = Bz * D * (K - 1);
    const int64_t n = n_state > D * K ? n_state : D * K;
    if (n == 0) return cudaSuccess;
    conv_bwd_empty_kernel<TD, TO><<<unsigned((n + 255) / 256), 256, 0, st>>>(
        static_cast<const TD*>(q), static_cast<TO*>(dS), dw, dbias, n_state, int(D), K);
    return cudaGetLastError();
  }
  // channel pairs are loaded and stored as one vector each, which needs
  // every tensor aligned to two elements
  auto al2 = [](const void* p, size_t es) {
    return (reinterpret_cast<uintptr_t>(p) % (2 * es)) == 0;
  };
  // the K = 4 walk copies whole 64-channel rows with cp.async.bulk: 16-byte
  // aligned x and dy
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) % 16) == 0; };
  if (K == 4 && D % 64 == 0 && L >= K - 1 && al16(x) && al16(dy) && al2(dx, sizeof(TO)))
    return launch_k4<TX, TD, TO>(x, w, bias, s_in, dy, q, dx, dS, dw, dbias, Bz, L, D, silu_on,
                                 ws, st);
  if (D % 2 == 0 && al2(x, sizeof(TX)) && al2(dy, sizeof(TD)) && al2(dx, sizeof(TO)))
    return launch_bwd<TX, TD, TO, 2>(x, w, bias, s_in, dy, q, dx, dS, dw, dbias, Bz, L, D, K,
                                     silu_on, ws, st);
  return launch_bwd<TX, TD, TO, 1>(x, w, bias, s_in, dy, q, dx, dS, dw, dbias, Bz, L, D, K,
                                   silu_on, ws, st);
}

cudaError_t conv_state_bwd_launch(const void* x, sss_dtype xt, const float* w, const float* bias,
                                  const void* s_in, const void* dy, sss_dtype dyt, const void* q,
                                  void* dx, sss_dtype dxt, void* dS, float* dw, float* dbias,
                                  int64_t Bz, int64_t L, int64_t D, int K, int silu_on,
                                  void* ws, cudaStream_t st) {
#define SSS_BWD(TX, TD, TO)                                                                   \
  return bwd_vec<TX, TD, TO>(x, w, bias, s_in, dy, q, dx, dS, dw, dbias, Bz, L, D, K, silu_on, \
                             ws, st)
  using bf = __nv_bfloat16;
  if (xt == SSS_BF16) {
    if (dyt == SSS_F32) {
      if (dxt == SSS_BF16) SSS_BWD(bf, float, bf);
      SSS_BWD(bf, float, float);
    }
    if (dxt == SSS_BF16) SSS_BWD(bf, bf, bf);
    SSS_BWD(bf, bf, float);
  }
  if (dyt == SSS_F32) {
    if (dxt == SSS_BF16) SSS_BWD(float, float, bf);
    SSS_BWD(float, float, float);
  }
  if (dxt == SSS_BF16) SSS_BWD(float, bf, bf);
  SSS_BWD(float, bf, float);
#undef SSS_BWD
}

}  // namespace sss
