// Tensor-core (tcgen05) chunked selective scan, one scalar decay per head,
// from an initial state.
//
// The recurrence is Eq. (1) of "Understanding and Improving Length
// Generalization in Recurrent Models" with A_t = exp(dt_t A_h).  Its unrolled
// form with a non-zero initial state, Eq. (4) (section 4.1), applied to one
// chunk of Q tokens that starts from the state h_prev left by the previous
// chunk, splits the work into dense contractions.  With the inclusive
// log-decay prefix Lam_t = sum_{r<=t} dt_r A_h inside the chunk (the
// exp(cumsum) of log-transition coefficients the pages call for):
//
//   y_t   = sum_{s<=t} exp(Lam_t - Lam_s) (C_t . B_s) x_s      (intra-chunk)
//         + exp(Lam_t) C_t h_prev                              (initial state term)
//   h_new = exp(Lam_end) h_prev + sum_s exp(Lam_end - Lam_s) x_s B_s^T
//
// Per chunk and head that is four products on the tensor cores (bf16 in,
// fp32 accumulate in tensor memory), M = Q = 128 rows each:
//   G   = C B^T                     [t][s]  (K = N)
//   Yd  = (G o M) X                 [t][p]  (K = Q, A operand from TMEM)
//   Yo  = C h_prev^T                [t][p]  (K = N)
//   S^T = B^T X~                    [n][p]  (K = Q), X~_s = exp(Lam_end - Lam_s) x_s
// The fp32 operands the pages' tolerance cannot afford to round once to bf16
// (x, G o M, h_prev, X~; B and C are bf16 inputs and stay exact) are split
// into hi + lo bf16 parts; each product takes the hi*hi, hi*lo and lo*hi terms
// it needs (the state path keeps ~2^-16 relative precision).  The state h
// itself stays in fp32 registers, one TMEM lane (= one state row n) per
// thread, across all chunks of the sequence: it never goes to HBM between
// chunks.
//
// One CTA (128 threads = the 128 TMEM lanes) owns one (batch, head) and walks
// its chunks in order; B and C chunks arrive by TMA (128-byte swizzle, OOB rows
// zero-filled so a ragged tail needs no special case), x is read by the
// threads and written into the swizzled K-major operand tiles, thread 0
// issues the MMAs.  Every wait on an mbarrier is bounded (2 s): on expiry the
// kernel raises SSS_ERR_TIMEOUT, frees its tensor memory and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace sss {
using namespace tc;

namespace {
constexpr int kQ = 128;  // chunk length = MMA M
constexpr int kP = 64;   // head dimension
constexpr int kN = 128;  // state size
constexpr int kThreads = 128;
constexpr uint32_t kTmemCols = 512;
// tensor memory columns (fp32 accumulators unless noted)
constexpr uint32_t kColG = 0;     // C B^T          [t][s]  128
constexpr uint32_t kColYd = 128;  // (G o M) x      [t][p]   64
constexpr uint32_t kColYo = 192;  // C h^T          [t][p]   64
constexpr uint32_t kColS = 256;   // B^T x~         [n][p]   64
constexpr uint32_t kColGh = 320;  // hi(G o M), bf16 pairs   64
constexpr uint32_t kColGl = 384;  // lo(G o M), bf16 pairs   64
// shared memory (bytes from a 1024-byte aligned base)
constexpr uint32_t kOffC = 0;         // C chunk  [t][n] K-major, two 64-wide n blocks
constexpr uint32_t kOffB = 32768;     // B chunk  [s][n]
constexpr uint32_t kOffUh = 65536;    // hi(x)    [p][s] K-major, two 64-wide s blocks
constexpr uint32_t kOffUl = 81920;    // lo(x)
constexpr uint32_t kOffXh = 98304;    // hi(x~)
constexpr uint32_t kOffXl = 114688;   // lo(x~)
constexpr uint32_t kOffHh = 131072;   // hi(h)    [n][p] MN-major (rows = K = n)
constexpr uint32_t kOffHl = 147456;   // lo(h)
constexpr uint32_t kOffMisc = 163840;
constexpr uint32_t kSmemBytes = kOffMisc + 2048 + 1024;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kIdG = idesc_bf16(128, 128, 0, 0);
constexpr uint32_t kIdS = idesc_bf16(128, 64, 1, 0);
constexpr uint32_t kIdYo = idesc_bf16(128, 64, 0, 1);
constexpr uint32_t kIdYd = idesc_bf16(128, 64, 0, 0);

__device__ __forceinline__ uint16_t bf16_bits(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}
__device__ __forceinline__ float bf16_val(uint16_t b) {
  return __bfloat162float(__ushort_as_bfloat16(b));
}
// hi = bf16(v), lo = bf16(v - hi): v == hi + lo to ~2^-16 relative
__device__ __forceinline__ void split(float v, uint16_t& hi, uint16_t& lo) {
  hi = bf16_bits(v);
  lo = bf16_bits(v - bf16_val(hi));
}
__device__ __forceinline__ uint32_t pack2(uint16_t lo_elem, uint16_t hi_elem) {
  return uint32_t(lo_elem) | (uint32_t(hi_elem) << 16);
}

// K-major descriptor of a [rows][128-element K] tile stored as two 64-wide K
// blocks `blk` bytes apart; K step kk covers K elements [16 kk, 16 kk + 16).
__device__ __forceinline__ uint64_t kdesc(uint32_t base, int kk, uint32_t blk) {
  return sdesc_sw128(base + uint32_t(kk >> 2) * blk + uint32_t(kk & 3) * 32u, 16, 1024);
}

// h (fp32, this thread's state row n) -> hi/lo bf16 rows of the MN-major
// B operand of C h^T.
__device__ __forceinline__ void write_h_rows(uint8_t* sm, int n, const float* hreg) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint16_t h0, l0, h1, l1;
      split(hreg[8 * c + 2 * k], h0, l0);
      split(hreg[8 * c + 2 * k + 1], h1, l1);
      hw[k] = pack2(h0, h1);
      lw[k] = pack2(l0, l1);
    }
    *reinterpret_cast<uint4*>(sm + kOffHh + sw128(n, c)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(sm + kOffHl + sw128(n, c)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
}

template <typename TX>
__device__ __forceinline__ void load_row64(const TX* row, float* u);
template <>
__device__ __forceinline__ void load_row64<float>(const float* row, float* u) {
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(row) + q);
    u[4 * q] = v.x; u[4 * q + 1] = v.y; u[4 * q + 2] = v.z; u[4 * q + 3] = v.w;
  }
}
template <>
__device__ __forceinline__ void load_row64<__nv_bfloat16>(const __nv_bfloat16* row, float* u) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(row) + q);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      u[8 * q + 2 * k] = bf16_val(uint16_t(w[k] & 0xFFFFu));
      u[8 * q + 2 * k + 1] = bf16_val(uint16_t(w[k] >> 16));
    }
  }
}

template <typename TY>
__device__ __forceinline__ void store_row64(TY* row, const float* v);
template <>
__device__ __forceinline__ void store_row64<float>(float* row, const float* v) {
#pragma unroll
  for (int q = 0; q < 16; ++q)
    reinterpret_cast<float4*>(row)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}
template <>
__device__ __forceinline__ void store_row64<__nv_bfloat16>(__nv_bfloat16* row, const float* v) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = pack2(bf16_bits(v[8 * q + 2 * k]), bf16_bits(v[8 * q + 2 * k + 1]));
    reinterpret_cast<uint4*>(row)[q] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

template <typename TX, typename TY>
__global__ void __launch_bounds__(kThreads, 1)
ssm_scan_tc_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmC,
                   const TX* __restrict__ x, const __nv_bfloat16* __restrict__ dt,
                   const float* __restrict__ A, const float* h0, float* hT,
                   TY* __restrict__ y, int L, int H, int G, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  float* lam = reinterpret_cast<float*>(sm + kOffMisc);  // [128] Lam_t
  float* gfac = lam + 128;                                 // [128] exp(R - Lam_s)
  float* red = gfac + 128;                                 // [16]  block reductions
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffMisc + 1152);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffMisc + 1152 + 16);
  const uint32_t bar_tma = smem_u32(&bars[0]);
  const uint32_t bar_mma = smem_u32(&bars[1]);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x / H, h = blockIdx.x % H, g = h / (H / G);
  const float Ah = A[h];
  const int64_t D = int64_t(H) * kP;

  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmC);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;
  const uint32_t tl = tm + (uint32_t(warp * 32) << 16);  // this warp's TMEM lanes

  // the state row n = tid, fp32, for the whole sequence
  float hreg[kP];
  const int64_t hoff = (int64_t(b) * H + h) * kP * kN;
#pragma unroll
  for (int p = 0; p < kP; ++p) hreg[p] = h0 ? h0[hoff + int64_t(p) * kN + tid] : 0.0f;
  write_h_rows(sm, tid, hreg);

  uint32_t tma_phase = 0, mma_phase = 0;
  bool failed = false;
  const int nC = (L + kQ - 1) / kQ;
  for (int c = 0; c < nC; ++c) {
    const int t0 = c * kQ;
    const int valid = min(kQ, L - t0);
    if (tid == 0) {
      mbar_arrive_expect_tx(bar_tma, 4u * 16384u);
      tma_load_3d(sb + kOffC, &tmC, g * kN, t0, b, bar_tma);
      tma_load_3d(sb + kOffC + 16384, &tmC, g * kN + 64, t0, b, bar_tma);
      tma_load_3d(sb + kOffB, &tmB, g * kN, t0, b, bar_tma);
      tma_load_3d(sb + kOffB + 16384, &tmB, g * kN + 64, t0, b, bar_tma);
    }

    // ---- log-decay prefix Lam_t over the chunk (padding tokens add 0) ----------
    const float ell =
        tid < valid ? __bfloat162float(dt[(int64_t(b) * L + t0 + tid) * H + h]) * Ah : 0.0f;
    float v = ell;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float nb = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += nb;
    }
    if (lane == 31) red[warp] = v;
    __syncthreads();
    float lam_t = v;
    for (int w = 0; w < warp; ++w) lam_t += red[w];
    lam[tid] = lam_t;
    float mn = lam_t, mx = lam_t;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (lane == 0) {
      red[4 + warp] = mn;
      red[8 + warp] = mx;
    }
    __syncthreads();
    const float lam_min = fminf(fminf(red[4], red[5]), fminf(red[6], red[7]));
    const float lam_max = fmaxf(fmaxf(red[8], red[9]), fmaxf(red[10], red[11]));
    const float lam_end = lam[kQ - 1];
    // exp(Lam_t - Lam_s) = f_t * g_s with a mid-range reference R keeps both
    // factors inside fp32 while the chunk's decay range is below 160
    const float R = 0.5f * (lam_min + lam_max);
    const bool factored = (lam_max - lam_min) <= 160.0f;
    gfac[tid] = expf(R - lam_t);
    const float f_t = expf(lam_t - R);
    const float dec_t = expf(lam_t);             // h_prev reaches token t as exp(Lam_t)
    const float xdec = expf(lam_end - lam_t);    // token s reaches the chunk end
    const float dec_end = expf(lam_end);

    // ---- x row of token s = tid -> hi/lo of x and of x~ in [p][s] tiles ------
    {
      float u[kP];
      if (tid < valid) {
        load_row64<TX>(x + (int64_t(b) * L + t0 + tid) * D + int64_t(h) * kP, u);
      } else {
#pragma unroll
        for (int p = 0; p < kP; ++p) u[p] = 0.0f;
      }
      const uint32_t sblk = uint32_t(tid >> 6) * 8192u;
      const uint32_t ins = uint32_t(tid & 63);
      const uint32_t cc = ins >> 3, bo = (ins & 7u) * 2u;
#pragma unroll
      for (int p = 0; p < kP; ++p) {
        const uint32_t off = sblk + sw128(uint32_t(p), cc) + bo;
        uint16_t uh, ul, xh, xl;
        split(u[p], uh, ul);
        split(u[p] * xdec, xh, xl);
        *reinterpret_cast<uint16_t*>(sm + kOffUh + off) = uh;
        *reinterpret_cast<uint16_t*>(sm + kOffUl + off) = ul;
        *reinterpret_cast<uint16_t*>(sm + kOffXh + off) = xh;
        *reinterpret_cast<uint16_t*>(sm + kOffXl + off) = xl;
      }
    }
    fence_proxy_async_smem();
    __syncthreads();

    // ---- products that need only the inputs: G, S, Yo ---------------------------
    bool ok = mbar_wait(bar_tma, tma_phase, kWaitNs);
    tma_phase ^= 1u;
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tm + kColG, kdesc(sb + kOffC, kk, 16384), kdesc(sb + kOffB, kk, 16384), kIdG, kk);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // B^T as an MN-major A operand: rows s, n blocks 16 KB apart
        mma_ss(tm + kColS, sdesc_sw128(sb + kOffB + kk * 2048, 16384, 1024),
               kdesc(sb + kOffXh, kk, 8192), kIdS, kk);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tm + kColS, sdesc_sw128(sb + kOffB + kk * 2048, 16384, 1024),
               kdesc(sb + kOffXl, kk, 8192), kIdS, 1);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // h^T as an MN-major B operand: rows n
        mma_ss(tm + kColYo, kdesc(sb + kOffC, kk, 16384),
               sdesc_sw128(sb + kOffHh + kk * 2048, 8192, 1024), kIdYo, kk);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tm + kColYo, kdesc(sb + kOffC, kk, 16384),
               sdesc_sw128(sb + kOffHl + kk * 2048, 8192, 1024), kIdYo, 1);
      mma_commit(bar_mma);
    }
    ok = mbar_wait(bar_mma, mma_phase, kWaitNs);
    mma_phase ^= 1u;
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    tc_fence_after();

    // ---- decay mask on G (row t = tid) -> hi/lo bf16 pairs in TMEM ------------
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // s in [32 j, 32 j + 32)
      uint32_t ph[16], pl[16];
      if (j <= warp) {
        uint32_t graw[32];
        tmem_ld_x32(tl + kColG + 32u * j, graw);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          uint16_t hh[2], ll[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int s = 32 * j + 2 * i + e;
            float m = 0.0f;
            if (s <= tid) {
              const float wgt = factored ? f_t * gfac[s] : expf(lam_t - lam[s]);
              m = __uint_as_float(graw[2 * i + e]) * wgt;
            }
            split(m, hh[e], ll[e]);
          }
          ph[i] = pack2(hh[0], hh[1]);
          pl[i] = pack2(ll[0], ll[1]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) ph[i] = pl[i] = 0u;
      }
      tmem_st_x16(tl + kColGh + 16u * j, ph);
      tmem_st_x16(tl + kColGl + 16u * j, pl);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncthreads();

    // ---- Yd = (G o M) x: hi*hi + hi*lo + lo*hi --------------------------------
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ts(tm + kColYd, tm + kColGh + 8u * kk, kdesc(sb + kOffUh, kk, 8192), kIdYd, kk);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ts(tm + kColYd, tm + kColGh + 8u * kk, kdesc(sb + kOffUl, kk, 8192), kIdYd, 1);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ts(tm + kColYd, tm + kColGl + 8u * kk, kdesc(sb + kOffUh, kk, 8192), kIdYd, 1);
      mma_commit(bar_mma);
    }
    ok = mbar_wait(bar_mma, mma_phase, kWaitNs);
    mma_phase ^= 1u;
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    tc_fence_after();

    // ---- epilogue: y row t = tid, state row n = tid ----------------------------
    {
      float yv[kP];
      uint32_t r0[32], r1[32];
      tmem_ld_x32(tl + kColYd, r0);
      tmem_ld_x32(tl + kColYd + 32, r1);
#pragma unroll
      for (int p = 0; p < 32; ++p) {
        yv[p] = __uint_as_float(r0[p]);
        yv[p + 32] = __uint_as_float(r1[p]);
      }
      tmem_ld_x32(tl + kColYo, r0);
      tmem_ld_x32(tl + kColYo + 32, r1);
#pragma unroll
      for (int p = 0; p < 32; ++p) {
        yv[p] = fmaf(dec_t, __uint_as_float(r0[p]), yv[p]);
        yv[p + 32] = fmaf(dec_t, __uint_as_float(r1[p]), yv[p + 32]);
      }
      if (tid < valid) store_row64<TY>(y + (int64_t(b) * L + t0 + tid) * D + int64_t(h) * kP, yv);
      tmem_ld_x32(tl + kColS, r0);
      tmem_ld_x32(tl + kColS + 32, r1);
#pragma unroll
      for (int p = 0; p < 32; ++p) {
        hreg[p] = fmaf(dec_end, hreg[p], __uint_as_float(r0[p]));
        hreg[p + 32] = fmaf(dec_end, hreg[p + 32], __uint_as_float(r1[p]));
      }
      write_h_rows(sm, tid, hreg);
      fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
  }

  if (failed) {
    // let whatever is still in flight land before the memory is released
    if (tid == 0) {
      raise_status(status, SSS_ERR_TIMEOUT);
      mbar_wait(bar_mma, mma_phase ^ 1u, kWaitNs / 2);
      mbar_wait(bar_tma, tma_phase ^ 1u, kWaitNs / 2);
    }
  } else if (hT) {
#pragma unroll
    for (int p = 0; p < kP; ++p) hT[hoff + int64_t(p) * kN + tid] = hreg[p];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tm, kTmemCols);
}

// ---------------------------------------------------------------------------
// operand-layout self-test: the four descriptor forms of the scan on one tile
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128, 1)
tc_selftest_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __nv_bfloat16* __restrict__ Am, const __nv_bfloat16* __restrict__ Bm,
                   float* __restrict__ out, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  constexpr uint32_t oA = 0, oB = 32768, oAt = 65536, oBt = 98304, oMisc = 114688;
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
  // A row m = tid into TMEM as bf16 pairs (columns 320..383)
  for (int j = 0; j < 4; ++j) {
    uint32_t w[16];
    for (int i = 0; i < 16; ++i) w[i] = pack2(A16[tid * 128 + 32 * j + 2 * i], A16[tid * 128 + 32 * j + 2 * i + 1]);
    tmem_st_x16(tl + 320u + 16u * j, w);
  }
  tmem_st_wait();
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  bool ok = mbar_wait(bar_tma, 0, kWaitNs);
  if (!__syncthreads_or(!ok)) {
    if (tid == 0) {
      tc_fence_after();
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tm + 0, kdesc(sb + oA, kk, 16384), kdesc(sb + oB, kk, 16384), kIdG, kk);
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tm + 128, sdesc_sw128(sb + oAt + kk * 2048, 16384, 1024), kdesc(sb + oB, kk, 16384),
               kIdS, kk);
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tm + 192, kdesc(sb + oA, kk, 16384), sdesc_sw128(sb + oBt + kk * 2048, 8192, 1024),
               kIdYo, kk);
      for (int kk = 0; kk < 8; ++kk)
        mma_ts(tm + 256, tm + 320u + 8u * kk, kdesc(sb + oB, kk, 16384), kIdYd, kk);
      mma_commit(bar_mma);
    }
    ok = mbar_wait(bar_mma, 0, kWaitNs);
    if (!__syncthreads_or(!ok)) {
      tc_fence_after();
      uint32_t r[32];
      for (int j = 0; j < 4; ++j) {
        tmem_ld_x32(tl + 32u * j, r);
        for (int i = 0; i < 32; ++i) out[0 * 16384 + tid * 128 + 32 * j + i] = __uint_as_float(r[i]);
      }
      for (int t = 1; t < 4; ++t)
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

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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
bool make_bc_map(CUtensorMap* m, const void* ptr, int64_t Bz, int64_t L, int G, int N) {
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

template <typename TX, typename TY>
cudaError_t launch_tc(const void* x, const void* dt, const float* A, const void* B, const void* C,
                      const float* h0, float* hT, void* y, int64_t Bz, int64_t L, int H, int G,
                      int* status, cudaStream_t st) {
  CUtensorMap mB, mC;
  if (!make_bc_map(&mB, B, Bz, L, G, kN) || !make_bc_map(&mC, C, Bz, L, G, kN))
    return cudaErrorInvalidValue;
  auto kern = ssm_scan_tc_kernel<TX, TY>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
  if (e != cudaSuccess) return e;
  const int64_t grid = Bz * H;
  kern<<<unsigned(grid), kThreads, kSmemBytes, st>>>(
      mB, mC, static_cast<const TX*>(x), static_cast<const __nv_bfloat16*>(dt), A, h0, hT,
      static_cast<TY*>(y), int(L), H, G, status);
  return cudaGetLastError();
}
}  // namespace

bool ssm_scan_tc_supports(sss_dtype xt, sss_dtype at, sss_dtype yt, int64_t L, int H, int P,
                          int N, int G) {
  (void)xt; (void)yt;
  return at == SSS_BF16 && P == kP && N == kN && L >= 1 && L < (int64_t(1) << 31) && H >= 1 &&
         G >= 1 && H % G == 0 && encode_fn() != nullptr;
}

cudaError_t ssm_scan_tc_launch(const void* x, sss_dtype xt, const void* dt, const float* A,
                               const void* B, const void* C, const float* h0, float* hT,
                               void* y, sss_dtype yt, int64_t Bz, int64_t L, int H, int P,
                               int N, int G, int* status, cudaStream_t st) {
  (void)P; (void)N;
  if (Bz * H > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (xt == SSS_F32 && yt == SSS_BF16)
    return launch_tc<float, __nv_bfloat16>(x, dt, A, B, C, h0, hT, y, Bz, L, H, G, status, st);
  if (xt == SSS_F32)
    return launch_tc<float, float>(x, dt, A, B, C, h0, hT, y, Bz, L, H, G, status, st);
  if (yt == SSS_BF16)
    return launch_tc<__nv_bfloat16, __nv_bfloat16>(x, dt, A, B, C, h0, hT, y, Bz, L, H, G, status, st);
  return launch_tc<__nv_bfloat16, float>(x, dt, A, B, C, h0, hT, y, Bz, L, H, G, status, st);
}

cudaError_t tc_selftest_launch(const void* A, const void* B, float* out, int* status,
                               cudaStream_t st) {
  CUtensorMap mA, mB;
  if (!make_tile_map(&mA, A) || !make_tile_map(&mB, B)) return cudaErrorInvalidValue;
  const uint32_t smem = 114688 + 64 + 1024;
  cudaError_t e = cudaFuncSetAttribute(tc_selftest_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  tc_selftest_kernel<<<1, 128, smem, st>>>(mA, mB, static_cast<const __nv_bfloat16*>(A),
                                           static_cast<const __nv_bfloat16*>(B), out, status);
  return cudaGetLastError();
}

}  // namespace sss
