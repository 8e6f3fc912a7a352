// Tensor-core (tcgen05) chunked selective scan, one scalar decay per head,
// from an initial state; optionally fused with the causal conv + SiLU that
// produces its input.
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
// fp32 accumulate in tensor memory), M = 128 rows each.  With a reference
// R = the middle of the chunk's Lam range, g_s = exp(R - Lam_s) and
// f_t = exp(Lam_t - R), the decay weight is exp(Lam_t - Lam_s) = f_t g_s, so
// with x'_s = g_s x_s:
//   G   = C B^T                     [t][s]  (K = N)
//   Yd' = (G o causal) X'           [t][p]  (K = Q, A operand from TMEM)
//   Yo  = C h_prev^T                [t][p]  (K = N)
//   S'  = B^T X'                    [n][p]  (K = Q)
//   y_t = f_t Yd'_t + exp(Lam_t) Yo_t,   h_new = exp(Lam_end) h_prev + exp(Lam_end - R) S'.
// The factors stay inside exp(+-50) while the chunk's range is <= 100; a
// chunk with a wider range uses the plain weights exp(Lam_t - Lam_s) in the
// mask and a second operand tile X~_s = exp(Lam_end - Lam_s) x_s for S.
// The fp32 operands that a single bf16 rounding would push past the
// tolerance (x', G o causal, h_prev; B and C are bf16 inputs and stay exact)
// are split into hi + lo bf16 parts and each product takes the hi*hi, hi*lo
// and lo*hi terms.  The state stays in fp32 registers (one TMEM lane = one
// state row n per consumer thread) for the whole sequence.
//
// Warp roles in one CTA = one (batch, head), 416 threads:
//   warps 0-7  producers: per chunk, Lam and the chunk's scalars (published in
//              shared memory for the other roles), the input rows (or the
//              conv of the raw input, fused), the hi/lo operand tiles of x'
//              (token-major rows = MN-major operands, 16-byte stores),
//              double-buffered so chunk c+1 is prepared during chunk c;
//   warps 8-11 consumers: the causal mask G -> G o causal (into TMEM), the
//              state carry and its hi/lo tiles, the y epilogue;
//   warp 12    issuer: TMA of the B and C chunks and every tcgen05.mma, one
//              thread; TMA for chunk c+1 starts as soon as chunk c's products
//              that read B and C are done, G(c+1) overlaps chunk c's epilogue.
// Stages hand over through mbarriers.  Every wait is bounded (2 s): on expiry
// the waiter raises SSS_ERR_TIMEOUT and sets an abort flag that makes every
// other role stop at its next wait; the issuer drains its MMAs, the CTA frees
// its tensor memory and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "scan_tc_util.cuh"
#include "tc_ptx.cuh"

namespace sss {
using namespace tc;
using namespace tcs;

namespace {
constexpr int kQ = 128;  // chunk length = MMA M
constexpr int kP = 64;   // head dimension
constexpr int kN = 128;  // state size
constexpr int kMaxK = 4; // conv width handled by the fused producer
constexpr int kProdWarps = 8;                 // warps 0-7
constexpr int kConsWarp0 = kProdWarps;        // warps 8-11 (TMEM lane quarters 0-3)
constexpr int kIssuerWarp = kConsWarp0 + 4;   // warp 12
constexpr int kThreads = (kIssuerWarp + 1) * 32;
constexpr uint32_t kTmemCols = 512;
// tensor memory columns (fp32 accumulators unless noted)
constexpr uint32_t kColG = 0;     // C B^T                          [t][s] 128
constexpr uint32_t kColGh = 128;  // hi(G o mask), bf16 pairs              64
constexpr uint32_t kColGl = 192;  // lo(G o mask), bf16 pairs              64
constexpr uint32_t kColYd = 256;  // hi(G o mask)(x'hi | x'lo) + lo x'hi [t][128]
constexpr uint32_t kColYo = 384;  // C (h_hi + h_lo)^T                [t][p]  64
constexpr uint32_t kColS = 448;   // B^T (x'hi + x'lo)                [n][p]  64
// shared memory (bytes from a 1024-byte aligned base)
constexpr uint32_t kOffC = 0;         // C chunk [t][n], K-major, two 64-wide n blocks
constexpr uint32_t kOffB = 32768;     // B chunk [s][n]
constexpr uint32_t kOffU = 65536;     // x hi/lo, 2 stages x (hi 16 KB, lo 16 KB), rows s
constexpr uint32_t kOffX = 131072;    // x~ hi (16 KB), lo (16 KB), rows s
constexpr uint32_t kOffH = 163840;    // h hi (16 KB), lo (16 KB), rows n
constexpr uint32_t kOffMisc = 196608;
constexpr uint32_t kMiscLam = 0;       // [2][128] Lam_t of the chunk (published by producers)
constexpr uint32_t kMiscGf = 1024;     // [2][128] exp(R - Lam_s), or 1 on the plain path
constexpr uint32_t kMiscXd = 2048;     // [2][128] exp(Lam_end - Lam_s) (plain path)
constexpr uint32_t kMiscRedP = 3072;   // [2][24] producer scan scratch
constexpr uint32_t kMiscScal = 3264;   // [2][4] chunk scalars: factored flag, R, Lam_end
constexpr uint32_t kMiscW = 3456;      // [64][4] conv weights of the head
constexpr uint32_t kMiscBias = 4480;   // [64]
constexpr uint32_t kMiscBars = 4736;   // 17 mbarriers
constexpr uint32_t kMiscTmem = 4888;
constexpr uint32_t kMiscAbort = 4892;
// fused path: the raw-input rows of the next chunk, staged by TMA with the
// K-1 halo rows in front (128 + 3 rows of 128 bytes, 128-byte swizzle)
constexpr uint32_t kOffXs = 202752;
constexpr uint32_t kXsRows = 128 + 3;
constexpr uint32_t kXsBytes = kXsRows * 128;
constexpr uint32_t kSmemBytes = kOffXs + kXsBytes + 1024;
// barriers
enum {
  BAR_FULL_CB = 0, BAR_TILES = 1 /*2*/, BAR_U_FREE = 3 /*2*/, BAR_X_FREE = 5, BAR_G_FULL = 6,
  BAR_GM_FULL = 7, BAR_S_FULL = 8, BAR_S_FREE = 9, BAR_YO_DONE = 10, BAR_H_FULL = 11,
  BAR_Y_FULL = 12, BAR_ACC_FREE = 13, BAR_CB_FREE = 14, BAR_DRAIN = 15, BAR_XS_FULL = 16,
  NUM_BARS = 17
};
constexpr uint32_t kIdG = idesc_bf16(128, 128, 0, 0);     // C (K-major) x B (K-major)
constexpr uint32_t kIdS = idesc_bf16(128, 64, 1, 1);      // B^T (MN-major) x x' (MN-major)
constexpr uint32_t kIdYo = idesc_bf16(128, 64, 0, 1);     // C (K-major) x h (MN-major)
constexpr uint32_t kIdYd = idesc_bf16(128, 128, 0, 1);    // hi(G o mask) (TMEM) x x'hi|lo (MN-major)
constexpr uint32_t kIdYdLo = idesc_bf16(128, 64, 0, 1);   // lo(G o mask) (TMEM) x x'hi

// Named barrier among the threads of one role (ids 1, 2; 0 is __syncthreads).

// Inclusive prefix of `v` over the NW warps of a role; also the total and the
// minimum / maximum of the prefix over the role.  `red` holds 3 NW floats.
template <int NW>
__device__ __forceinline__ float role_prefix(float v, int lane, int wq, float* red, int bar_id,
                                             float* total, float* pmin, float* pmax) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float nb = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += nb;
  }
  float mn = v, mx = v;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (lane == 31) red[wq] = v;
  if (lane == 0) {
    red[NW + wq] = mn;
    red[2 * NW + wq] = mx;
  }
  role_sync(bar_id, NW * 32);
  float off = 0.0f, run = 0.0f, gmn = 3.0e38f, gmx = -3.0e38f;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    gmn = fminf(gmn, run + red[NW + w]);
    gmx = fmaxf(gmx, run + red[2 * NW + w]);
    if (w < wq) off += red[w];
    run += red[w];
  }
  *total = run;
  *pmin = gmn;
  *pmax = gmx;
  return v + off;
}

}  // namespace

// x: the scan input u [Bz, L, H, 64] (TX = float or bf16), or with FUSED the
// raw input [Bz, L, H*64] (bf16) that the producers convolve (K <= 4, SiLU).
template <typename TX, typename TY, bool FUSED>
__global__ void __launch_bounds__(kThreads, 1)
ssm_scan_tc_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmC,
                   const __grid_constant__ CUtensorMap tmX, const TX* __restrict__ x,
                   const __nv_bfloat16* __restrict__ dt, const float* __restrict__ A,
                   const float* h0, float* hT, TY* __restrict__ y, const float* __restrict__ conv_w,
                   const float* __restrict__ conv_b, const TX* conv_s_in, TX* conv_s_out,
                   int K, int L, int H, int G, int* status,
                     const int32_t* __restrict__ seq_idx) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived from the shared array itself so that the
  // compiler keeps every access in the shared address space
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(sm);
  uint8_t* misc = sm + kOffMisc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + kMiscTmem);
  Ctl ctl{smem_u32(misc + kMiscBars), reinterpret_cast<volatile int*>(misc + kMiscAbort), status};

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x / H, h = blockIdx.x % H, g = h / (H / G);
  const float Ah = A[h];
  const int64_t D = int64_t(H) * kP;
  const int nC = (L + kQ - 1) / kQ;

  if (warp == kIssuerWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    int counts[NUM_BARS];
    for (int i = 0; i < NUM_BARS; ++i) counts[i] = 1;
    counts[BAR_TILES] = counts[BAR_TILES + 1] = kProdWarps * 32;
    counts[BAR_GM_FULL] = counts[BAR_S_FREE] = 128;
    counts[BAR_H_FULL] = counts[BAR_ACC_FREE] = 128;
    for (int i = 0; i < NUM_BARS; ++i) mbar_init(ctl.bar(i), counts[i]);
    *ctl.abort = 0;
    fence_mbar_init();
  }
  if (FUSED && tid < kP) {
    const int64_t d = int64_t(h) * kP + tid;
    float* sw = reinterpret_cast<float*>(misc + kMiscW);
    // taps right-aligned in a window of kMaxK (leading zero weights for K < kMaxK)
#pragma unroll
    for (int k = 0; k < kMaxK; ++k)
      sw[tid * kMaxK + k] = k >= kMaxK - K ? conv_w[d * K + k - (kMaxK - K)] : 0.0f;
    reinterpret_cast<float*>(misc + kMiscBias)[tid] = conv_b ? conv_b[d] : 0.0f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;

  if (warp < kProdWarps) {
    // ============================ producers ============================
    // The prefix runs with one token per thread (s = tid < 128); the inputs
    // and operand rows with thread (q, g4) = channels [8q, 8q+8) x tokens
    // [4 g4, 4 g4 + 4): every input element is read (and, fused, convolved in
    // a register window) once.
    constexpr int NT = 4;                        // tokens per thread
    constexpr int PT = kProdWarps * 32;
    const int s = tid, q = tid & 7, g4 = tid >> 3;
    float* red = reinterpret_cast<float*>(misc + kMiscRedP);
    const float* swq = reinterpret_cast<const float*>(misc + kMiscW) + 8 * q * kMaxK;
    const float* sbq = reinterpret_cast<const float*>(misc + kMiscBias) + 8 * q;
    auto stage_x = [&](int c) {  // TMA of chunk c's raw rows [t0 - 3, t0 + 128)
      mbar_arrive_expect_tx(ctl.bar(BAR_XS_FULL), kXsBytes);
      tma_load_3d(sb + kOffXs, &tmX, h * kP, c * kQ - (kMaxK - 1), b, ctl.bar(BAR_XS_FULL));
    };
    if (FUSED && s == 0) {
      prefetch_tmap(&tmX);
      stage_x(0);
    }
    int xs_issued = FUSED ? 1 : 0, xs_landed = 0;
    // on abort every loop below keeps running its named barriers with the
    // work skipped, so no thread is ever left waiting at one
    bool ok = true;
    for (int c = 0; c < nC; ++c) {
      const int t0 = c * kQ;
      const int valid = min(kQ, L - t0);
      // a token that starts a new packed sample gets kSampleStartLog: the
      // chunk's range passes kFactorRange, so it takes the plain weights
      // exp(Lam_t - Lam_s), which are 0 across the start, as is the carry
      const float ell = ok && s < valid && warp < 4
                            ? (sample_start(seq_idx, b, L, t0 + s)
                                   ? kSampleStartLog
                                   : __bfloat162float(dt[(int64_t(b) * L + t0 + s) * H + h]) * Ah)
                            : 0.0f;
      float u[NT][8];  // [token j][channel e]
      const int tb = t0 + NT * g4;  // first token of the group
      const int nv = ok ? min(NT, max(0, valid - NT * g4)) : 0;  // live tokens
      if constexpr (!FUSED) {
        // unconditional loads of clamped rows, dead tokens zeroed afterwards
        const int64_t rowbase = int64_t(b) * L * D + int64_t(h) * kP + 8 * q;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const int pc = min(tb + j, L - 1);
          const TX* row = x + rowbase + int64_t(pc) * D;
          float v[8];
          if constexpr (sizeof(TX) == 4) {
            const float4 v0 = __ldg(reinterpret_cast<const float4*>(row));
            const float4 v1 = __ldg(reinterpret_cast<const float4*>(row) + 1);
            v[0] = v0.x; v[1] = v0.y; v[2] = v0.z; v[3] = v0.w;
            v[4] = v1.x; v[5] = v1.y; v[6] = v1.z; v[7] = v1.w;
          } else {
            const uint4 r4 = __ldg(reinterpret_cast<const uint4*>(row));
            const uint32_t w4[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              v[2 * i] = __uint_as_float(w4[i] << 16);
              v[2 * i + 1] = __uint_as_float(w4[i] & 0xFFFF0000u);
            }
          }
          const float live_j = j < nv ? 1.0f : 0.0f;
#pragma unroll
          for (int e = 0; e < 8; ++e) u[j][e] = v[e] * live_j;
        }
      } else {
        // rows tb - (kMaxK-1) + i, i < NT + kMaxK - 1, from the staged tile
        // (rows outside [0, L) arrive zero-filled; rows past the last live
        // token are zeroed; positions < 0 are then taken from the conv state)
        constexpr int NR = NT + kMaxK - 1;
        if (ok) ok = ctl.wait(BAR_XS_FULL, uint32_t(c & 1));
        if (ok) xs_landed = c + 1;
        uint4 xr[NR];
#pragma unroll
        for (int i = 0; i < NR; ++i) {
          const int row = NT * g4 + i;  // staged row = position t0 - 3 + row
          const int pos = tb - (kMaxK - 1) + i;
          const uint4 v = *reinterpret_cast<const uint4*>(sm + kOffXs + sw128(row, q));
          xr[i] = (ok && nv > 0 && pos < tb + nv) ? v : make_uint4(0u, 0u, 0u, 0u);
        }
        if (tb < kMaxK - 1 && nv > 0 && conv_s_in) {
#pragma unroll
          for (int i = 0; i < kMaxK - 1; ++i) {
            const int pos = tb - (kMaxK - 1) + i;
            if (pos < 0 && pos >= -(K - 1)) {
              uint32_t w4[4];
#pragma unroll
              for (int i2 = 0; i2 < 4; ++i2) {
                const int64_t d0 = int64_t(b) * D + int64_t(h) * kP + 8 * q + 2 * i2;
                const uint16_t lo = *reinterpret_cast<const uint16_t*>(&conv_s_in[d0 * (K - 1) + (K - 1) + pos]);
                const uint16_t hi = *reinterpret_cast<const uint16_t*>(&conv_s_in[(d0 + 1) * (K - 1) + (K - 1) + pos]);
                w4[i2] = pack2(lo, hi);
              }
              xr[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
          }
        }
        // channel pair by channel pair (weights of two channels = two float4
        // broadcast reads of the staged table), all tokens per pair; token j
        // uses rows j + k with the right-aligned taps
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          const float4 wa = *reinterpret_cast<const float4*>(swq + (2 * e2) * kMaxK);
          const float4 wb = *reinterpret_cast<const float4*>(swq + (2 * e2 + 1) * kMaxK);
          const float2 bb = *reinterpret_cast<const float2*>(sbq + 2 * e2);
          const float wa_[4] = {wa.x, wa.y, wa.z, wa.w}, wb_[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            float za = bb.x, zb = bb.y;
#pragma unroll
            for (int k = 0; k < kMaxK; ++k) {
              const uint4 rv = xr[j + k];
              const uint32_t wv = e2 == 0 ? rv.x : e2 == 1 ? rv.y : e2 == 2 ? rv.z : rv.w;
              za = fmaf(wa_[k], __uint_as_float(wv << 16), za);
              zb = fmaf(wb_[k], __uint_as_float(wv & 0xFFFF0000u), zb);
            }
            u[j][2 * e2] = za;
            u[j][2 * e2 + 1] = zb;
          }
        }
        // SiLU on every value (dead tokens hold finite conv outputs of zero
        // rows), then zeroed by a multiply: no branch around the expensive part
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const float live_j = j < nv ? 1.0f : 0.0f;
#pragma unroll
          for (int e = 0; e < 8; ++e) u[j][e] = silu(u[j][e]) * live_j;
        }
      }
      // ---- Lam over the chunk (warps 0-3, one token per thread) -------------
      float lam_s = 0.0f, lam_end = 0.0f, lmin = 0.0f, lmax = 0.0f;
      if (warp < 4)
        lam_s = role_prefix<4>(ell, lane, warp, red + 12 * (c & 1), 3, &lam_end, &lmin, &lmax);
      const int st = c & 1;
      // the stage's shared arrays and tiles are free once Yd(c-2) is done
      if (ok && c >= 2) ok = ctl.wait(BAR_U_FREE + st, uint32_t(((c >> 1) + 1) & 1));
      float* lamP = reinterpret_cast<float*>(misc + kMiscLam) + 128 * st;
      float* gP = reinterpret_cast<float*>(misc + kMiscGf) + 128 * st;
      float* xdP = reinterpret_cast<float*>(misc + kMiscXd) + 128 * st;
      float* scal = reinterpret_cast<float*>(misc + kMiscScal) + 4 * st;
      if (warp < 4) {  // publish Lam and the scalars that every role uses
        const bool fac = (lmax - lmin) <= kFactorRange;
        const float R = 0.5f * (lmin + lmax);
        lamP[s] = lam_s;
        gP[s] = fac ? expf(R - lam_s) : 1.0f;
        xdP[s] = expf(lam_end - lam_s);
        if (s == 0) {
          scal[0] = fac ? 1.0f : 0.0f;
          scal[1] = R;
          scal[2] = lam_end;
        }
      }
      role_sync(1, PT);
      // every producer has read the staged tile: stage the next chunk's rows
      // while this chunk's operand tiles go out
      if (FUSED && s == 0 && ok && c + 1 < nC) {
        stage_x(c + 1);
        xs_issued = c + 2;
      }
      const bool fac = scal[0] != 0.0f;
      uint8_t* uh = sm + kOffU + st * 32768;
      if (ok) {  // x' = g_s x (plain path: g_s = 1)
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const float f = gP[NT * g4 + j];
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) split2(u[j][2 * k] * f, u[j][2 * k + 1] * f, hw[k], lw[k]);
          *reinterpret_cast<uint4*>(uh + sw128(NT * g4 + j, q)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(uh + 16384 + sw128(NT * g4 + j, q)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
      if (!fac) {  // plain path: X~_s = exp(Lam_end - Lam_s) x_s for the state product
        if (ok && c >= 1) ok = ctl.wait(BAR_X_FREE, uint32_t((c - 1) & 1));
        if (ok) {
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            const float f = xdP[NT * g4 + j];
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) split2(u[j][2 * k] * f, u[j][2 * k + 1] * f, hw[k], lw[k]);
            *reinterpret_cast<uint4*>(sm + kOffX + sw128(NT * g4 + j, q)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(sm + kOffX + 16384 + sw128(NT * g4 + j, q)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
      }
      if (ok) {
        fence_proxy_async_smem();
        mbar_arrive(ctl.bar(BAR_TILES + st));
      }
    }
    if (FUSED && s == 0 && xs_issued > xs_landed)  // a staged tile still in flight
      mbar_wait(ctl.bar(BAR_XS_FULL), uint32_t(xs_landed & 1), kWaitNs / 2);
    if constexpr (FUSED) {
      // final conv state F_j = ext[L + j]; every read of S happened in chunk 0
      role_sync(1, PT);
      if (conv_s_out && s < kP && !*ctl.abort) {
        const int64_t d = int64_t(h) * kP + s;
        TX f[kMaxK - 1];
        for (int j = 0; j < K - 1; ++j) {
          const int e = L + j;  // extended-sequence index
          f[j] = e < K - 1 ? (conv_s_in ? conv_s_in[(int64_t(b) * D + d) * (K - 1) + e]
                                        : from_f32<TX>(0.0f))
                           : x[(int64_t(b) * L + (e - (K - 1))) * D + d];
        }
        for (int j = 0; j < K - 1; ++j) conv_s_out[(int64_t(b) * D + d) * (K - 1) + j] = f[j];
      }
    }
  } else if (warp < kIssuerWarp) {
    // ===== consumers: TMEM lane r = row t (mask, y) = state row n (S, h) =====
    const int wq = warp - kConsWarp0;  // == warp % 4, the TMEM lane quarter
    const int r = 32 * wq + lane;
    const uint32_t tl = tm + (uint32_t(wq * 32) << 16);
    float hreg[kP];
    const int64_t hoff = (int64_t(b) * H + h) * kP * kN;
#pragma unroll
    for (int p = 0; p < kP; ++p) hreg[p] = h0 ? h0[hoff + int64_t(p) * kN + r] : 0.0f;
    write_split_row(sm + kOffH, sm + kOffH + 16384, r, hreg);
    fence_proxy_async_smem();
    mbar_arrive(ctl.bar(BAR_H_FULL));
    {  // blocks of G o M above the diagonal of this warp's rows stay zero
      uint32_t z[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) z[i] = 0u;
      for (int j = wq + 1; j < 4; ++j) {
        tmem_st_x16(tl + kColGh + 16u * j, z);
        tmem_st_x16(tl + kColGl + 16u * j, z);
      }
      tmem_st_wait();
    }
    bool ok = true;
    for (int c = 0; c < nC; ++c) {
      const int t0 = c * kQ;
      const int valid = min(kQ, L - t0);
      const int st = c & 1;
      // the chunk's Lam and scalars, published by the producers with the tiles
      if (ok) ok = ctl.wait(BAR_TILES + st, uint32_t((c >> 1) & 1));
      const float* lam = reinterpret_cast<const float*>(misc + kMiscLam) + 128 * st;
      const float* scal = reinterpret_cast<const float*>(misc + kMiscScal) + 4 * st;
      const bool fac = scal[0] != 0.0f;
      const float R = scal[1], lam_end = scal[2];
      const float lam_t = lam[r];
      const float f_t = fac ? expf(lam_t - R) : 1.0f;       // row scale of Yd'
      const float dec_t = expf(lam_t);                        // h_prev reaches row t
      const float dec_end = expf(lam_end);                    // h_prev reaches the chunk end
      const float s_scale = fac ? expf(lam_end - R) : 1.0f;  // scale of S'
      // ---- mask: row t = r, columns s <= t, 16 columns at a time ------------
      // (ok is made warp-uniform before every warp-collective TMEM access)
      if (ok) ok = ctl.wait(BAR_G_FULL, uint32_t(c & 1));
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc_fence_after();
        for (int j = 0; j <= wq; ++j) {
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int s0 = 32 * j + 16 * hf;
            uint32_t graw[16], ph[8], pl[8];
            tmem_ld_x16(tl + kColG + uint32_t(s0), graw);
            float m[16];
            if (fac) {  // the decay lives in x' and the row scale f_t
#pragma unroll
              for (int i = 0; i < 16; ++i) m[i] = __uint_as_float(graw[i]);
            } else {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float4 l4 = *reinterpret_cast<const float4*>(lam + s0 + 4 * i);
                m[4 * i] = __uint_as_float(graw[4 * i]) * __expf(lam_t - l4.x);
                m[4 * i + 1] = __uint_as_float(graw[4 * i + 1]) * __expf(lam_t - l4.y);
                m[4 * i + 2] = __uint_as_float(graw[4 * i + 2]) * __expf(lam_t - l4.z);
                m[4 * i + 3] = __uint_as_float(graw[4 * i + 3]) * __expf(lam_t - l4.w);
              }
            }
            if (j == wq) {  // diagonal block: s = s0 + i <= t = 32 wq + lane
#pragma unroll
              for (int i = 0; i < 16; ++i) m[i] = 16 * hf + i <= lane ? m[i] : 0.0f;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) split2(m[2 * i], m[2 * i + 1], ph[i], pl[i]);
            tmem_st_x8(tl + kColGh + uint32_t(s0 / 2), ph);
            tmem_st_x8(tl + kColGl + uint32_t(s0 / 2), pl);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(ctl.bar(BAR_GM_FULL));
      }
      // ---- state carry: row n = r ------------------------------------------
      if (ok) ok = ctl.wait(BAR_S_FULL, uint32_t(c & 1));
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          uint32_t r0[16];
          tmem_ld_x16(tl + kColS + 16u * qq, r0);
#pragma unroll
          for (int p = 0; p < 16; ++p)
            hreg[16 * qq + p] = fmaf(dec_end, hreg[16 * qq + p], s_scale * __uint_as_float(r0[p]));
        }
        tc_fence_before();
        mbar_arrive(ctl.bar(BAR_S_FREE));
      }
      if (ok) ok = ctl.wait(BAR_YO_DONE, uint32_t(c & 1));  // Yo(c) has read h_{c-1}
      if (ok) {
        write_split_row(sm + kOffH, sm + kOffH + 16384, r, hreg);
        fence_proxy_async_smem();
        mbar_arrive(ctl.bar(BAR_H_FULL));
      }
      // ---- y rows ------------------------------------------------------------
      if (ok) ok = ctl.wait(BAR_Y_FULL, uint32_t(c & 1));
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc_fence_after();
        TY* yrow = y + (int64_t(b) * L + t0 + r) * D + int64_t(h) * kP;
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          float yv[16];
          {
            uint32_t a0[16], a1[16];
            tmem_ld_x16(tl + kColYd + 16u * qq, a0);
            tmem_ld_x16(tl + kColYd + 64u + 16u * qq, a1);
#pragma unroll
            for (int p = 0; p < 16; ++p) yv[p] = f_t * (__uint_as_float(a0[p]) + __uint_as_float(a1[p]));
          }
          {
            uint32_t a0[16];
            tmem_ld_x16(tl + kColYo + 16u * qq, a0);
            if (qq == 3) {
              tc_fence_before();
              mbar_arrive(ctl.bar(BAR_ACC_FREE));
            }
#pragma unroll
            for (int p = 0; p < 16; ++p) yv[p] = fmaf(dec_t, __uint_as_float(a0[p]), yv[p]);
          }
          if (r < valid) store_row16<TY>(yrow + 16 * qq, yv);
        }
      }
    }
    if (ok && hT) {
#pragma unroll
      for (int p = 0; p < kP; ++p) hT[hoff + int64_t(p) * kN + r] = hreg[p];
    }
  } else {
   if (lane == 0) {
    // ========================= issuer (one thread) =========================
    auto tma_chunk = [&](int c) {
      mbar_arrive_expect_tx(ctl.bar(BAR_FULL_CB), 4u * 16384u);
      const int t0 = c * kQ;
      tma_load_3d(sb + kOffC, &tmC, g * kN, t0, b, ctl.bar(BAR_FULL_CB));
      tma_load_3d(sb + kOffC + 16384, &tmC, g * kN + 64, t0, b, ctl.bar(BAR_FULL_CB));
      tma_load_3d(sb + kOffB, &tmB, g * kN, t0, b, ctl.bar(BAR_FULL_CB));
      tma_load_3d(sb + kOffB + 16384, &tmB, g * kN + 64, t0, b, ctl.bar(BAR_FULL_CB));
    };
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmC);
    tma_chunk(0);
    int tma_issued = 1, tma_landed = 0;
    for (int c = 0; c < nC; ++c) {
      const int st = c & 1;
      if (!ctl.wait(BAR_FULL_CB, uint32_t(c & 1))) break;
      tma_landed = c + 1;
      if (!ctl.wait(BAR_TILES + st, uint32_t((c >> 1) & 1))) break;
      const bool fac = reinterpret_cast<const float*>(misc + kMiscScal)[4 * st] != 0.0f;
      const uint32_t uh = sb + kOffU + st * 32768;          // x' hi | lo
      const uint32_t xs = fac ? uh : sb + kOffX;             // operand of the state product
      // base descriptors; each K step adds a compile-time constant
      const uint64_t dC = sdesc_sw128(sb + kOffC, 16, 1024), dBk = sdesc_sw128(sb + kOffB, 16, 1024);
      const uint64_t dBm = sdesc_sw128(sb + kOffB, 16384, 1024);
      const uint64_t dXs = sdesc_sw128(xs, 16384, 1024), dXs2 = sdesc_sw128(xs + 16384, 16384, 1024);
      const uint64_t dH = sdesc_sw128(sb + kOffH, 16384, 1024), dH2 = sdesc_sw128(sb + kOffH + 16384, 16384, 1024);
      const uint64_t dU = sdesc_sw128(uh, 16384, 1024);
      tc_fence_after();
      // G = C B^T (mask(c-1) has read G(c-1): Yd(c-1) was issued after it)
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tm + kColG, dC + kstep(kk, 16384), dBk + kstep(kk, 16384), kIdG, kk);
      mma_commit(ctl.bar(BAR_G_FULL));
      // S' = B^T (x'hi + x'lo) into the single S buffer once state(c-1) read it;
      // B^T is the MN-major view of the B chunk
      if (c >= 1 && !ctl.wait(BAR_S_FREE, uint32_t((c - 1) & 1))) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tm + kColS, dBm + mnstep(kk), dXs + mnstep(kk), kIdS, kk);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tm + kColS, dBm + mnstep(kk), dXs2 + mnstep(kk), kIdS, 1);
      mma_commit(ctl.bar(BAR_X_FREE));
      mma_commit(ctl.bar(BAR_S_FULL));
      // Yo = C (h_hi + h_lo)^T once h_{c-1} is in place and the epilogue of
      // chunk c-1 has read Yo and Yd
      if (!ctl.wait(BAR_H_FULL, uint32_t(c & 1))) break;
      if (c >= 1 && !ctl.wait(BAR_ACC_FREE, uint32_t((c - 1) & 1))) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tm + kColYo, dC + kstep(kk, 16384), dH + mnstep(kk), kIdYo, kk);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tm + kColYo, dC + kstep(kk, 16384), dH2 + mnstep(kk), kIdYo, 1);
      mma_commit(ctl.bar(BAR_YO_DONE));
      mma_commit(ctl.bar(BAR_CB_FREE));
      // the next chunk's B and C as soon as this chunk's readers are done
      if (c + 1 < nC) {
        if (!ctl.wait(BAR_CB_FREE, uint32_t(c & 1))) break;
        tma_chunk(c + 1);
        tma_issued = c + 2;
      }
      // Yd' = hi(G o mask)(x'hi | x'lo) + lo(G o mask) x'hi
      if (!ctl.wait(BAR_GM_FULL, uint32_t(c & 1))) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) mma_ts(tm + kColYd, tm + kColGh + 8u * kk, dU + mnstep(kk), kIdYd, kk);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) mma_ts(tm + kColYd, tm + kColGl + 8u * kk, dU + mnstep(kk), kIdYdLo, 1);
      mma_commit(ctl.bar(BAR_Y_FULL));
      mma_commit(ctl.bar(BAR_U_FREE + st));
    }
    // every MMA of this CTA (and a TMA still in flight) lands before the
    // tensor memory and shared memory are released
    mma_commit(ctl.bar(BAR_DRAIN));
    mbar_wait(ctl.bar(BAR_DRAIN), 0, kWaitNs);
    if (tma_issued > tma_landed)
      mbar_wait(ctl.bar(BAR_FULL_CB), uint32_t(tma_landed & 1), kWaitNs / 2);
   }
   __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kIssuerWarp) tmem_dealloc(tm, kTmemCols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {
template <typename TX, typename TY, bool FUSED>
cudaError_t launch_tc(const void* x, const void* dt, const float* A, const void* B, const void* C,
                      const float* h0, float* hT, void* y, const float* w, const float* bias,
                      const void* s_in, void* s_out, int K, int64_t Bz, int64_t L, int H, int G,
                      int* status, const int32_t* seq_idx, cudaStream_t st) {
  CUtensorMap mB, mC, mX;
  if (!make_bc_map(&mB, B, Bz, L, G, kN) || !make_bc_map(&mC, C, Bz, L, G, kN))
    return cudaErrorInvalidValue;
  if (FUSED) {
    if (!make_x_map(&mX, x, Bz, L, int64_t(H) * kP, kXsRows)) return cudaErrorInvalidValue;
  } else {
    mX = mB;  // unused
  }
  auto kern = ssm_scan_tc_kernel<TX, TY, FUSED>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
  if (e != cudaSuccess) return e;
  kern<<<unsigned(Bz * H), kThreads, kSmemBytes, st>>>(
      mB, mC, mX, static_cast<const TX*>(x), static_cast<const __nv_bfloat16*>(dt), A, h0, hT,
      static_cast<TY*>(y), w, bias, static_cast<const TX*>(s_in), static_cast<TX*>(s_out), K,
      int(L), H, G, status, seq_idx);
  return cudaGetLastError();
}
}  // namespace

bool ssm_scan_tc_supports(sss_dtype xt, sss_dtype at, sss_dtype yt, int64_t L, int H, int P,
                          int N, int G) {
  (void)xt; (void)yt;
  return at == SSS_BF16 && P == kP && N == kN && L >= 1 && L < (int64_t(1) << 31) && H >= 1 &&
         G >= 1 && H % G == 0 && encode_fn() != nullptr;
}

bool mixer_fwd_tc_supports(sss_dtype xt, sss_dtype at, int K, int64_t L, int H, int P, int N,
                           int G) {
  return xt == SSS_BF16 && K >= 1 && K <= kMaxK && ssm_scan_tc_supports(xt, at, at, L, H, P, N, G);
}

cudaError_t ssm_scan_tc_launch(const void* x, sss_dtype xt, const void* dt, const float* A,
                               const void* B, const void* C, const float* h0, float* hT,
                               void* y, sss_dtype yt, int64_t Bz, int64_t L, int H, int P,
                               int N, int G, int* status, const int32_t* seq_idx, cudaStream_t st) {
  (void)P; (void)N;
  if (Bz * H > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
#define SSS_TC(TXT, TYT)                                                                    \
  return launch_tc<TXT, TYT, false>(x, dt, A, B, C, h0, hT, y, nullptr, nullptr, nullptr,  \
                                    nullptr, 1, Bz, L, H, G, status, seq_idx, st);
  if (xt == SSS_F32 && yt == SSS_BF16) SSS_TC(float, __nv_bfloat16)
  if (xt == SSS_F32) SSS_TC(float, float)
  if (yt == SSS_BF16) SSS_TC(__nv_bfloat16, __nv_bfloat16)
  SSS_TC(__nv_bfloat16, float)
#undef SSS_TC
}

cudaError_t mixer_fwd_tc_launch(const void* x, const float* w, const float* bias,
                                const void* s_in, void* s_out, const void* dt, const float* A,
                                const void* B, const void* C, const float* h0, float* hT,
                                void* y, sss_dtype yt, int64_t Bz, int64_t L, int H, int G, int K,
                                int* status, const int32_t* seq_idx, cudaStream_t st) {
  if (Bz * H > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (yt == SSS_BF16)
    return launch_tc<__nv_bfloat16, __nv_bfloat16, true>(x, dt, A, B, C, h0, hT, y, w, bias, s_in,
                                                         s_out, K, Bz, L, H, G, status, seq_idx, st);
  return launch_tc<__nv_bfloat16, float, true>(x, dt, A, B, C, h0, hT, y, w, bias, s_in, s_out, K,
                                               Bz, L, H, G, status, seq_idx, st);
}

}  // namespace sss
