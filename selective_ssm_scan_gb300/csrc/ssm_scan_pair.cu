// Tensor-core (tcgen05) chunked selective scan over a PAIR of heads per CTA,
// optionally fused with the causal conv + SiLU that produces its input.
//
// The arithmetic is the one of the single-head kernel (ssm_scan_tc.cu): Eq. (1)
// of "Understanding and Improving Length Generalization in Recurrent Models"
// with A_t = exp(dt_t A_h), unrolled over a chunk of tokens from the state
// left by the previous chunk (Eq. (4), section 4.1).  With the inclusive
// log-decay prefix Lam_t inside the chunk, a reference R = the middle of the
// chunk's Lam range, g_s = exp(R - Lam_s), f_t = exp(Lam_t - R) and x'_s = g_s x_s:
//
//   G  = C B^T                                        (once per chunk: the
//                                                      heads share B and C)
//   Y  = (G o causal) X' + C (e^R h_prev)^T           (one accumulator)
//   S' = B^T X'
//   y_t = f_t Y_t,      h_new = exp(Lam_end) h_prev + exp(Lam_end - R) S'.
//
// Pieces instead of fixed chunks: a piece is at most 128 tokens and ends
// before the token at which either head's Lam range would pass kFactorRange,
// so the factored weights always stay inside exp(+-50).  Ordinary inputs give
// 128-token pieces; a head with a huge decay gives shorter ones (a single
// token always qualifies: its range is 0).
//
// GB300 mapping, one CTA per (batch, head pair), 416 threads (13 warps: the
// register file then allows 128 registers a thread):
//   warps 0-3  producers: per piece, the decay prefix of both heads (one token
//              per thread) and the piece length; then per head the conv + SiLU
//              of the raw rows (TMA-staged) or the input rows and the
//              x' = g x hi/lo tiles (16-byte stores, 128-byte swizzle), two
//              items of 8 channels x 4 tokens per thread;
//   warps 4-11 consumers: warp 4 + 4 hs + q owns head hs and TMEM lanes
//              32q..32q+31: its share of the causal mask of G (32-column blocks
//              2hs, 2hs+1), then the state carry of head hs (one state row n
//              per thread, fp32 registers) and the y rows of head hs;
//   warp 12    issuer: TMA of B and C (double-buffered, one piece ahead) and
//              every tcgen05.mma, one thread.
// Tensor memory (512 columns): G [t][s] 128, hi/lo(G o causal) 64 + 64,
// Y of each head 64, S' of each head 64.  Shared memory: B/C stages 2 x 64 KB,
// one x' tile pair and one h' tile pair shared by the two heads (each head's
// tiles are written once the other head's products have read them), the
// staged raw rows, and the piece descriptors.  Per piece the MMAs run
//   G, Yo_a, S'_a, Yd_a, Yo_b, S'_b, Yd_b
// so each tile hand-over hides behind products of the other head.  Every
// wait is bounded (2 s); a timeout raises SSS_ERR_TIMEOUT and unwinds.
#include "common.cuh"
#include "scan_tc_util.cuh"
#include "tc_ptx.cuh"

namespace sss {
using namespace tc;
using namespace tcs;

namespace {
namespace pr {
constexpr int kP = 64;    // head dimension
constexpr int kN = 128;   // state size
constexpr int kMaxK = 4;  // conv width handled by the fused producer
constexpr int kProdWarps = 4;
constexpr int kConsWarp0 = 4;
constexpr int kIssuerWarp = 12;
constexpr int kThreads = (kIssuerWarp + 1) * 32;  // 416
constexpr int kPT = kProdWarps * 32;              // 128 producer threads
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColG = 0, kColGh = 128, kColGl = 192;
constexpr uint32_t kColY = 256;  // + 64 hs
constexpr uint32_t kColS = 384;  // + 64 hs
// shared memory (bytes from a 1024-byte aligned base)
constexpr uint32_t kOffBC = 0;        // stage k: C at 65536 k (two 64-wide n blocks), B at +32768
constexpr uint32_t kOffX = 131072;    // x' hi; lo at +16384 (rows s)
constexpr uint32_t kOffH = 163840;    // h' hi; lo at +16384 (rows n)
constexpr uint32_t kOffXs = 196608;   // staged raw rows [t0 - 3, t0 + 128) of one head
constexpr uint32_t kXsRows = 128 + kMaxK - 1;
constexpr uint32_t kXsBytes = kXsRows * 128;
constexpr uint32_t kOffMisc = kOffXs + kXsBytes;  // 213376
// misc (offsets from kOffMisc)
constexpr uint32_t kMiInfo = 0;       // 4 piece descriptors
constexpr uint32_t kMiRed = 4224;     // producer scan scratch [2][4][4] + piece lengths
// conv weights and bias, per (head hs, channel pair e2, channel group q) 12
// floats: the taps of channels 8q + 2e2 and 8q + 2e2 + 1 interleaved (tap k of
// the pair = floats 2k, 2k+1), the two biases, 2 pad.  The 48-byte stride puts
// the 8 groups a warp reads on distinct banks.
constexpr uint32_t kMiW = 4480;       // [2][4][8][12] floats
constexpr uint32_t kMiBars = 7552;    // mbarriers
constexpr uint32_t kMiTmem = 7808;
constexpr uint32_t kMiAbort = 7812;
constexpr uint32_t kMiscBytes = 7816;
constexpr uint32_t kSmemBytes = kOffMisc + kMiscBytes + 1024;
constexpr int kSlots = 4;

struct PieceInfo {
  int start, n, last, pad;
  float R[2], lend[2];
  float lam[2][128];
};
static_assert(sizeof(PieceInfo) * kSlots <= kMiRed, "piece ring");

enum {
  BAR_BC_FULL = 0 /*2*/, BAR_BC_FREE = 2 /*2*/, BAR_XS_FULL = 4, BAR_INFO_FULL = 5 /*4*/,
  BAR_INFO_FREE = 9 /*4*/, BAR_X_FULL = 13, BAR_X_FREE = 14, BAR_G_FULL = 15, BAR_GM_FULL = 16,
  BAR_GM_FREE = 17, BAR_H_FULL = 18 /*2*/, BAR_H_FREE = 20 /*2*/, BAR_S_FULL = 22 /*2*/,
  BAR_S_FREE = 24 /*2*/, BAR_Y_FULL = 26 /*2*/, BAR_Y_FREE = 28 /*2*/, BAR_DRAIN = 30,
  NUM_BARS = 31
};
// Barrier discipline: each barrier's completions are awaited in order by one
// role that sees every one of them, so the phase parity it waits on is never
// two phases stale.  (The h' tile pair is handed between the heads through
// two barriers, BAR_H_FREE + hs = "Yo of head hs has read the tiles", for
// that reason: arrivals on different barriers are not ordered.)
static_assert(NUM_BARS * 8 <= kMiTmem - kMiBars, "barrier area");

constexpr uint32_t kIdG = idesc_bf16(128, 128, 0, 0);   // C (K-major) x B (K-major)
constexpr uint32_t kIdS = idesc_bf16(128, 64, 1, 1);    // B^T (MN-major) x x' (MN-major)
constexpr uint32_t kIdYo = idesc_bf16(128, 64, 0, 1);   // C (K-major) x h' (MN-major)
constexpr uint32_t kIdYd = idesc_bf16(128, 64, 0, 1);   // (G o causal) (TMEM) x x' (MN-major)

// Inclusive prefix over 128 tokens held one per thread by 4 warps, for the
// two heads at once (one named barrier): per head the prefix sum and the
// prefix min / max of the prefix sum.  `red` holds 24 floats.
__device__ __forceinline__ void piece_scan2(const float (&v0)[2], int lane, int w4, float* red,
                                            int bar_id, float (&lam)[2], float (&pmin)[2],
                                            float (&pmax)[2]) {
  float v[2] = {v0[0], v0[1]}, mn[2], mx[2];
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float nb = __shfl_up_sync(0xffffffffu, v[h2], o);
      if (lane >= o) v[h2] += nb;
    }
    mn[h2] = v[h2];
    mx[h2] = v[h2];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float a = __shfl_up_sync(0xffffffffu, mn[h2], o);
      const float c = __shfl_up_sync(0xffffffffu, mx[h2], o);
      if (lane >= o) {
        mn[h2] = fminf(mn[h2], a);
        mx[h2] = fmaxf(mx[h2], c);
      }
    }
    if (lane == 31) {
      red[12 * h2 + 3 * w4] = v[h2];
      red[12 * h2 + 3 * w4 + 1] = mn[h2];
      red[12 * h2 + 3 * w4 + 2] = mx[h2];
    }
  }
  role_sync(bar_id, 128);
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    float off = 0.0f, gmn = 3.0e38f, gmx = -3.0e38f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      if (w < w4) {
        gmn = fminf(gmn, off + red[12 * h2 + 3 * w + 1]);
        gmx = fmaxf(gmx, off + red[12 * h2 + 3 * w + 2]);
        off += red[12 * h2 + 3 * w];
      }
    }
    lam[h2] = off + v[h2];
    pmin[h2] = fminf(gmn, off + mn[h2]);
    pmax[h2] = fmaxf(gmx, off + mx[h2]);
  }
}

// ---- packed fp32 pairs (two channels at once: f32x2 FMA / MUL / ADD) --------
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
__device__ __forceinline__ float ex2f(float v) {  // 2^v, approximate (a few ulp)
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float rcpf(float v) {  // 1 / v, approximate (1 ulp)
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
constexpr float kLog2e = 1.4426950408889634f;
// a bf16 pair word (channel a low, channel b high) as a packed fp32 pair
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w) {
  return pk2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
// SiLU of a pair, times g: z / (1 + e^-z) * g, with e^-z = 2^(-z log2 e)
__device__ __forceinline__ uint64_t silu_scaled2(uint64_t z, float g) {
  float ta, tb;
  upk2(mul2(z, pk2(-kLog2e, -kLog2e)), ta, tb);
  float da, db;
  upk2(add2(pk2(ex2f(ta), ex2f(tb)), pk2(1.0f, 1.0f)), da, db);
  return mul2(z, pk2(rcpf(da) * g, rcpf(db) * g));
}
// a packed pair -> bf16 hi pair and lo pair (v == hi + lo to ~2^-16)
__device__ __forceinline__ void split_pair(uint64_t v, uint32_t& hi, uint32_t& lo) {
  float a, b;
  upk2(v, a, b);
  const __nv_bfloat162 h2 = __floats2bfloat162_rn(a, b);
  hi = *reinterpret_cast<const uint32_t*>(&h2);
  float ra, rb;
  upk2(add2(v, pk2(-__uint_as_float(hi << 16), -__uint_as_float(hi & 0xFFFF0000u))), ra, rb);
  const __nv_bfloat162 l2 = __floats2bfloat162_rn(ra, rb);
  lo = *reinterpret_cast<const uint32_t*>(&l2);
}
}  // namespace pr
}  // namespace

// x: the scan input u [Bz, L, H, 64] (TX = float or bf16), or with FUSED the
// raw input [Bz, L, H*64] (bf16) that the producers convolve (K <= 4, SiLU).
// Requires (H / G) even: both heads of a pair read the same B and C group.
template <typename TX, typename TY, bool FUSED>
__global__ void __launch_bounds__(pr::kThreads, 1)
ssm_scan_pair_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmC,
                     const __grid_constant__ CUtensorMap tmX, const TX* __restrict__ x,
                     const __nv_bfloat16* __restrict__ dt, const float* __restrict__ A,
                     const float* h0, float* hT, TY* __restrict__ y,
                     const float* __restrict__ conv_w, const float* __restrict__ conv_b,
                     const TX* conv_s_in, TX* conv_s_out, int K, int L, int H, int G,
                     int* status) {
  using namespace pr;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(sm);
  uint8_t* misc = sm + kOffMisc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + kMiTmem);
  Ctl ctl{smem_u32(misc + kMiBars), reinterpret_cast<volatile int*>(misc + kMiAbort), status};
  PieceInfo* info = reinterpret_cast<PieceInfo*>(misc + kMiInfo);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int npair = H / 2;
  const int b = blockIdx.x / npair, pair = blockIdx.x % npair;
  const int g = (2 * pair) / (H / G);
  const int64_t D = int64_t(H) * kP;

  if (warp == kIssuerWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    int counts[NUM_BARS];
    for (int i = 0; i < NUM_BARS; ++i) counts[i] = 1;
    for (int i = 0; i < kSlots; ++i) {
      counts[BAR_INFO_FULL + i] = kPT;
      counts[BAR_INFO_FREE + i] = 256 + 1;  // consumers + issuer
    }
    counts[BAR_X_FULL] = kPT;
    counts[BAR_GM_FULL] = 256;
    for (int i = 0; i < 2; ++i) {
      counts[BAR_H_FULL + i] = 128;
      counts[BAR_S_FREE + i] = 128;
      counts[BAR_Y_FREE + i] = 128;
    }
    for (int i = 0; i < NUM_BARS; ++i) mbar_init(ctl.bar(i), counts[i]);
    *ctl.abort = 0;
    fence_mbar_init();
  }
  if (FUSED && tid < 2 * kP) {
    // channel tid of the pair = head hs, channel 8q + 2e2 + odd of that head
    const int64_t d = int64_t(2 * pair) * kP + tid;
    const int hs = tid >> 6, cq = (tid & 63) >> 3, e = tid & 7, e2 = e >> 1, odd = e & 1;
    float* sw = reinterpret_cast<float*>(misc + kMiW) + ((hs * 4 + e2) * 8 + cq) * 12;
    // taps right-aligned in a window of kMaxK (leading zero weights for K < kMaxK)
#pragma unroll
    for (int k = 0; k < kMaxK; ++k)
      sw[2 * k + odd] = k >= kMaxK - K ? conv_w[d * K + k - (kMaxK - K)] : 0.0f;
    sw[8 + odd] = conv_b ? conv_b[d] : 0.0f;
    sw[10 + odd] = 0.0f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;

  if (warp < kProdWarps) {
    // ============================ producers ============================
    // decay phase: thread = token tk of the piece, both heads; operand phase:
    // item i = tid + 128 rd (rd = 0, 1) = channels [8q, 8q+8) x tokens
    // [4 g4, 4 g4 + 4) of one head, q = i & 7, g4 = i >> 3
    constexpr int NT = 4;
    constexpr int NR = NT + kMaxK - 1;  // staged rows an item reads
    const int tk = tid;
    const int q = tid & 7;
    float* red = reinterpret_cast<float*>(misc + kMiRed);
    int* nred = reinterpret_cast<int*>(misc + kMiRed + 24 * 4);
    const float Aa = A[2 * pair], Ab = A[2 * pair + 1];
    auto stage_x = [&](int start, int hs) {  // TMA of raw rows [start - 3, start + 128)
      mbar_arrive_expect_tx(ctl.bar(BAR_XS_FULL), kXsBytes);
      tma_load_3d(sb + kOffXs, &tmX, (2 * pair + hs) * kP, start - (kMaxK - 1), b,
                  ctl.bar(BAR_XS_FULL));
    };
    if (FUSED && tid == 0) {
      prefetch_tmap(&tmX);
      stage_x(0, 0);
    }
    int xs_issued = FUSED ? 1 : 0, xs_landed = 0;
    // dt of the next piece's token, loaded one piece ahead
    auto load_dt = [&](int start, int hh) -> float {
      const int t = start + tk;
      return t < L ? __bfloat162float(dt[(int64_t(b) * L + t) * H + 2 * pair + hh]) : 0.0f;
    };
    float dt_next[2] = {load_dt(0, 0), load_dt(0, 1)};
    bool ok = true;
    int p = 0;
    for (int c = 0;; ++c) {
      const int slot = c & (kSlots - 1);
      PieceInfo* inf = info + slot;
      // ---- decay prefix of both heads, piece length ----------------------
      const float ell[2] = {ok ? dt_next[0] * Aa : 0.0f, ok ? dt_next[1] * Ab : 0.0f};
      float lam[2], pmin[2], pmax[2];
      piece_scan2(ell, lane, warp, red, 1, lam, pmin, pmax);
      const bool live_tok = p + tk < L;
      const unsigned bal0 = __ballot_sync(0xffffffffu, live_tok && (pmax[0] - pmin[0]) <= kFactorRange);
      const unsigned bal1 = __ballot_sync(0xffffffffu, live_tok && (pmax[1] - pmin[1]) <= kFactorRange);
      if (lane == 0) {
        nred[warp] = __popc(bal0);
        nred[4 + warp] = __popc(bal1);
      }
      role_sync(1, kPT);
      int n = min(nred[0] + nred[1] + nred[2] + nred[3], nred[4] + nred[5] + nred[6] + nred[7]);
      n = max(n, 1);  // token 0 always qualifies while p < L
      const bool last = p + n >= L;
      if (!last) {
        dt_next[0] = load_dt(p + n, 0);
        dt_next[1] = load_dt(p + n, 1);
      }
      // ---- publish the piece descriptor ----------------------------------
      if (ok && c >= kSlots) ok = ctl.wait(BAR_INFO_FREE + slot, uint32_t(((c / kSlots) - 1) & 1));
      inf->lam[0][tk] = lam[0];
      inf->lam[1][tk] = lam[1];
      if (tk == n - 1) {
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          inf->R[h2] = 0.5f * (pmin[h2] + pmax[h2]);
          inf->lend[h2] = lam[h2];
        }
      }
      if (tid == 0) {
        inf->start = p;
        inf->n = n;
        inf->last = last ? 1 : 0;
      }
      role_sync(1, kPT);
      mbar_arrive(ctl.bar(BAR_INFO_FULL + slot));
      // ---- per head: inputs, x' = g x hi/lo tiles ------------------------
#pragma unroll 1
      for (int hs = 0; hs < 2; ++hs) {
        const int head = 2 * pair + hs;
        const float R = inf->R[hs];
        uint32_t hw[NT][4], lw[NT][4];
        const int xu = 2 * c + hs;  // use of the x' tile pair
        if (FUSED) {
          const int su = 2 * c + hs;  // staging use
          if (ok) ok = ctl.wait(BAR_XS_FULL, uint32_t(su & 1));
          if (ok) xs_landed = su + 1;
        }
#pragma unroll 1
        for (int rd = 0; rd < 2; ++rd) {
          const int g4 = (tid >> 3) + 16 * rd;
          const int tb = 4 * g4;                            // first token (in the piece)
          const int nv = ok ? min(NT, max(0, n - tb)) : 0;  // live tokens
          // x' = g_s x with g_s = exp(R - Lam_s), 0 for dead tokens
          float gv[NT];
#pragma unroll
          for (int j = 0; j < NT; ++j)
            gv[j] = j < nv ? ex2f((R - inf->lam[hs][tb + j]) * kLog2e) : 0.0f;
          if constexpr (!FUSED) {
            const int64_t rowbase = int64_t(b) * L * D + int64_t(head) * kP + 8 * q;
#pragma unroll
            for (int j = 0; j < NT; ++j) {
              const int pc = min(p + tb + j, L - 1);
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
#pragma unroll
              for (int k = 0; k < 4; ++k)
                split_pair(mul2(pk2(v[2 * k], v[2 * k + 1]), pk2(gv[j], gv[j])), hw[j][k], lw[j][k]);
            }
          } else {
            // staged rows tb + i = positions p + tb - 3 + i
            uint4 xr[NR];
#pragma unroll
            for (int i = 0; i < NR; ++i)
              xr[i] = *reinterpret_cast<const uint4*>(sm + kOffXs + sw128(tb + i, q));
            if (p == 0 && tb < kMaxK - 1 && nv > 0) {
              // positions < 0: the conv state S (zeros without one)
#pragma unroll
              for (int i = 0; i < kMaxK - 1; ++i) {
                const int pos = tb - (kMaxK - 1) + i;
                if (pos < 0) {
                  uint32_t w4[4] = {0u, 0u, 0u, 0u};
                  if (conv_s_in && pos >= -(K - 1)) {
#pragma unroll
                    for (int i2 = 0; i2 < 4; ++i2) {
                      const int64_t d0 = int64_t(b) * D + int64_t(head) * kP + 8 * q + 2 * i2;
                      const uint16_t lo = *reinterpret_cast<const uint16_t*>(&conv_s_in[d0 * (K - 1) + (K - 1) + pos]);
                      const uint16_t hi = *reinterpret_cast<const uint16_t*>(&conv_s_in[(d0 + 1) * (K - 1) + (K - 1) + pos]);
                      w4[i2] = pack2(lo, hi);
                    }
                  }
                  xr[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
              }
            }
            if (rd == 1) {
              // every producer has its rows in registers (the empty asm reads
              // them, so each load has returned before the barrier): stage the
              // next head's (or piece's) rows, the TMA write ordered after the
              // generic-proxy reads by the proxy fence
#pragma unroll
              for (int i = 0; i < NR; ++i)
                asm volatile("" ::"r"(xr[i].x), "r"(xr[i].y), "r"(xr[i].z), "r"(xr[i].w) : "memory");
              role_sync(1, kPT);
              if (tid == 0 && ok) {
                fence_proxy_async_smem();
                if (hs == 0) {
                  stage_x(p, 1);
                  xs_issued = 2 * c + 2;
                } else if (!last) {
                  stage_x(p + n, 0);
                  xs_issued = 2 * c + 3;
                }
              }
            }
            // channel pair by channel pair: conv, SiLU, g, split, two channels
            // per packed fp32 operation
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const float* sw = reinterpret_cast<const float*>(misc + kMiW) + ((hs * 4 + e2) * 8 + q) * 12;
              const float4 w01 = *reinterpret_cast<const float4*>(sw);
              const float4 w23 = *reinterpret_cast<const float4*>(sw + 4);
              const float2 bb = *reinterpret_cast<const float2*>(sw + 8);
              const uint64_t wk[4] = {pk2(w01.x, w01.y), pk2(w01.z, w01.w), pk2(w23.x, w23.y),
                                      pk2(w23.z, w23.w)};
              uint64_t xv[NR];
#pragma unroll
              for (int i = 0; i < NR; ++i) {
                const uint32_t wv = e2 == 0 ? xr[i].x : e2 == 1 ? xr[i].y : e2 == 2 ? xr[i].z : xr[i].w;
                xv[i] = bf2_to_f2(wv);
              }
#pragma unroll
              for (int j = 0; j < NT; ++j) {
                uint64_t z = pk2(bb.x, bb.y);
#pragma unroll
                for (int k = 0; k < kMaxK; ++k) z = fma2(wk[k], xv[j + k], z);
                split_pair(silu_scaled2(z, gv[j]), hw[j][e2], lw[j][e2]);
              }
            }
          }
          // the tile pair is free once the previous use's products are done
          if (rd == 0 && ok && xu >= 1) ok = ctl.wait(BAR_X_FREE, uint32_t((xu - 1) & 1));
          if (ok) {
#pragma unroll
            for (int j = 0; j < NT; ++j) {
              *reinterpret_cast<uint4*>(sm + kOffX + sw128(tb + j, q)) =
                  make_uint4(hw[j][0], hw[j][1], hw[j][2], hw[j][3]);
              *reinterpret_cast<uint4*>(sm + kOffX + 16384 + sw128(tb + j, q)) =
                  make_uint4(lw[j][0], lw[j][1], lw[j][2], lw[j][3]);
            }
          }
        }
        if (ok) {
          fence_proxy_async_smem();
          mbar_arrive(ctl.bar(BAR_X_FULL));
        }
      }
      if (last) break;
      p += n;
    }
    if (FUSED && tid == 0) {  // staged tiles still in flight
      for (int su = xs_landed; su < xs_issued; ++su)
        mbar_wait(ctl.bar(BAR_XS_FULL), uint32_t(su & 1), kWaitNs / 2);
    }
    if constexpr (FUSED) {
      // final conv state F_j = ext[L + j] of both heads' channels; every read
      // of S happened in piece 0
      role_sync(1, kPT);
      if (conv_s_out && !*ctl.abort) {
        const int64_t d = int64_t(2 * pair) * kP + tid;
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
    // ===== consumers: head hs, TMEM lanes of quarter q (row t = state row n = r) =====
    const int cw = warp - kConsWarp0;
    const int q = warp & 3;  // == warp % 4: the TMEM lane quarter this warp may access
    const int hs = cw >> 2;
    const int r = 32 * q + lane;
    const int head = 2 * pair + hs;
    const uint32_t tl = tm + (uint32_t(q * 32) << 16);
    const uint32_t colY = kColY + 64u * hs, colS = kColS + 64u * hs;
    float hreg[kP];
    const int64_t hoff = (int64_t(b) * H + head) * kP * kN;
#pragma unroll
    for (int pp = 0; pp < kP; ++pp) hreg[pp] = h0 ? h0[hoff + int64_t(pp) * kN + r] : 0.0f;
    {  // blocks of G o causal above the diagonal of this quarter stay zero
      uint32_t z[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) z[i] = 0u;
      for (int j = 2 * hs; j < 2 * hs + 2; ++j) {
        if (j > q) {
          tmem_st_x16(tl + kColGh + 16u * j, z);
          tmem_st_x16(tl + kColGl + 16u * j, z);
        }
      }
      tmem_st_wait();
    }
    uint8_t* htile = sm + kOffH;
    // every wait is followed by a warp vote, so the warp leaves the loop
    // together (its TMEM accesses are warp-collective)
    auto wait_all = [&](int bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, ctl.wait(bar, parity));
    };
    bool ok = true;
    if (hs == 0) {  // h' for Yo_a of piece 0: e^{R_0} h0
      ok = wait_all(BAR_INFO_FULL, 0u);
      if (ok) {
        write_split_row(htile, htile + 16384, r, hreg, expf(info[0].R[0]));
        fence_proxy_async_smem();
        mbar_arrive(ctl.bar(BAR_H_FULL));
      }
    }
    for (int c = 0; ok; ++c) {
      const int slot = c & (kSlots - 1);
      const PieceInfo* inf = info + slot;
      if (!(ok = wait_all(BAR_INFO_FULL + slot, uint32_t((c / kSlots) & 1)))) break;
      const int n = inf->n, start = inf->start;
      const bool last = inf->last != 0;
      const float R = inf->R[hs], lend = inf->lend[hs], lam_t = inf->lam[hs][r];
      // ---- mask share: rows of quarter q, 32-column blocks 2hs, 2hs+1 ----
      if (c >= 1 && !(ok = wait_all(BAR_GM_FREE, uint32_t((c - 1) & 1)))) break;
      if (!(ok = wait_all(BAR_G_FULL, uint32_t(c & 1)))) break;
      tc_fence_after();
      for (int j = 2 * hs; j <= min(q, 2 * hs + 1); ++j) {
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          const int s0 = 32 * j + 16 * hf;
          uint32_t graw[16], ph[8], pl[8];
          tmem_ld_x16(tl + kColG + uint32_t(s0), graw);
          float m[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) m[i] = __uint_as_float(graw[i]);
          if (j == q) {  // diagonal block: s = s0 + i <= t = 32 q + lane
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
      // ---- head b: h' = e^{R_c} h_{c-1} for Yo_b(c), once Yo_a(c) has read the tiles
      if (hs == 1) {
        if (!(ok = wait_all(BAR_H_FREE + 0, uint32_t(c & 1)))) break;  // Yo_a(c) is done
        write_split_row(htile, htile + 16384, r, hreg, expf(R));
        fence_proxy_async_smem();
        mbar_arrive(ctl.bar(BAR_H_FULL + 1));
      }
      // ---- state carry: row n = r ---------------------------------------
      if (!(ok = wait_all(BAR_S_FULL + hs, uint32_t(c & 1)))) break;
      tc_fence_after();
      {
        const float dec_end = expf(lend), s_scale = expf(lend - R);
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          uint32_t r0[16];
          tmem_ld_x16(tl + colS + 16u * qq, r0);
#pragma unroll
          for (int pp = 0; pp < 16; ++pp)
            hreg[16 * qq + pp] = fmaf(dec_end, hreg[16 * qq + pp], s_scale * __uint_as_float(r0[pp]));
        }
      }
      tc_fence_before();
      mbar_arrive(ctl.bar(BAR_S_FREE + hs));
      // ---- y rows: y_t = f_t Y_t ---------------------------------------------
      if (!(ok = wait_all(BAR_Y_FULL + hs, uint32_t(c & 1)))) break;
      tc_fence_after();
      {
        const float f_t = expf(lam_t - R);
        TY* yrow = y + (int64_t(b) * L + start + r) * D + int64_t(head) * kP;
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          uint32_t a0[16];
          tmem_ld_x16(tl + colY + 16u * qq, a0);
          if (qq == 3) {  // Y is read: the next piece's products may start
            tc_fence_before();
            mbar_arrive(ctl.bar(BAR_Y_FREE + hs));
          }
          float yv[16];
#pragma unroll
          for (int pp = 0; pp < 16; ++pp) yv[pp] = f_t * __uint_as_float(a0[pp]);
          if (r < n) store_row16<TY>(yrow + 16 * qq, yv);
        }
      }
      mbar_arrive(ctl.bar(BAR_INFO_FREE + slot));
      if (last) break;
      // ---- head a: h' = e^{R_{c+1}} h_c for Yo_a(c+1), once Yo_b(c) is done
      if (hs == 0) {
        const int slot1 = (c + 1) & (kSlots - 1);
        if (!(ok = wait_all(BAR_INFO_FULL + slot1, uint32_t(((c + 1) / kSlots) & 1)))) break;
        if (!(ok = wait_all(BAR_H_FREE + 1, uint32_t(c & 1)))) break;  // Yo_b(c) is done
        write_split_row(htile, htile + 16384, r, hreg, expf(info[slot1].R[0]));
        fence_proxy_async_smem();
        mbar_arrive(ctl.bar(BAR_H_FULL));
      }
    }
    if (ok && !*ctl.abort && hT) {
#pragma unroll
      for (int pp = 0; pp < kP; ++pp) hT[hoff + int64_t(pp) * kN + r] = hreg[pp];
    }
  } else {
    if (lane == 0) {
      // ========================= issuer (one thread) =========================
      auto tma_bc = [&](int start, int st) {
        const uint32_t base = sb + kOffBC + uint32_t(st) * 65536u;
        const uint32_t bar = ctl.bar(BAR_BC_FULL + st);
        mbar_arrive_expect_tx(bar, 65536u);
        tma_load_3d(base, &tmC, g * kN, start, b, bar);
        tma_load_3d(base + 16384, &tmC, g * kN + 64, start, b, bar);
        tma_load_3d(base + 32768, &tmB, g * kN, start, b, bar);
        tma_load_3d(base + 49152, &tmB, g * kN + 64, start, b, bar);
      };
      prefetch_tmap(&tmB);
      prefetch_tmap(&tmC);
      tma_bc(0, 0);
      int tma_issued = 1, tma_landed = 0;
      for (int c = 0;; ++c) {
        const int st = c & 1, slot = c & (kSlots - 1);
        if (!ctl.wait(BAR_INFO_FULL + slot, uint32_t((c / kSlots) & 1))) break;
        const int start = info[slot].start, n = info[slot].n;
        const bool last = info[slot].last != 0;
        mbar_arrive(ctl.bar(BAR_INFO_FREE + slot));
        if (!last) {  // the next piece's B and C into the other stage
          if (c >= 1 && !ctl.wait(BAR_BC_FREE + (st ^ 1), uint32_t(((c - 1) >> 1) & 1))) break;
          tma_bc(start + n, st ^ 1);
          tma_issued = c + 2;
        }
        if (!ctl.wait(BAR_BC_FULL + st, uint32_t((c >> 1) & 1))) break;
        tma_landed = c + 1;
        const uint32_t cb = sb + kOffBC + uint32_t(st) * 65536u, bb = cb + 32768u;
        tc_fence_after();
        // G = C B^T (mask(c-1) has read G(c-1): Yd_a(c-1) waited for it)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tm + kColG, kdesc(cb, kk, 16384), kdesc(bb, kk, 16384), kIdG, kk);
        mma_commit(ctl.bar(BAR_G_FULL));
        bool good = true;
#pragma unroll 1
        for (int hs = 0; hs < 2 && good; ++hs) {
          const uint32_t dY = tm + kColY + 64u * hs, dS = tm + kColS + 64u * hs;
          // Yo = C (e^R h)^T starts the Y accumulator, once the h' tiles are
          // written and the previous y rows are read
          good = ctl.wait(BAR_H_FULL + hs, uint32_t(c & 1));
          if (good && c >= 1) good = ctl.wait(BAR_Y_FREE + hs, uint32_t((c - 1) & 1));
          if (!good) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(dY, kdesc(cb, kk, 16384), mndesc(sb + kOffH, kk), kIdYo, kk);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(dY, kdesc(cb, kk, 16384), mndesc(sb + kOffH + 16384, kk), kIdYo, 1);
          mma_commit(ctl.bar(BAR_H_FREE + hs));
          // S' = B^T (x'hi + x'lo) once the x' tiles are in and the previous
          // carry has read S'
          good = ctl.wait(BAR_X_FULL, uint32_t(hs));  // completion 2c + hs
          if (good && c >= 1) good = ctl.wait(BAR_S_FREE + hs, uint32_t((c - 1) & 1));
          if (!good) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(dS, sdesc_sw128(bb + kk * 2048, 16384, 1024), mndesc(sb + kOffX, kk), kIdS, kk);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(dS, sdesc_sw128(bb + kk * 2048, 16384, 1024), mndesc(sb + kOffX + 16384, kk),
                   kIdS, 1);
          mma_commit(ctl.bar(BAR_S_FULL + hs));
          if (hs == 1) mma_commit(ctl.bar(BAR_BC_FREE + st));
          // Yd = hi(G o c) x'hi + hi(G o c) x'lo + lo(G o c) x'hi onto Y
          if (hs == 0) good = ctl.wait(BAR_GM_FULL, uint32_t(c & 1));
          if (!good) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(dY, tm + kColGh + 8u * kk, mndesc(sb + kOffX, kk), kIdYd, 1);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(dY, tm + kColGh + 8u * kk, mndesc(sb + kOffX + 16384, kk), kIdYd, 1);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(dY, tm + kColGl + 8u * kk, mndesc(sb + kOffX, kk), kIdYd, 1);
          mma_commit(ctl.bar(BAR_Y_FULL + hs));
          mma_commit(ctl.bar(BAR_X_FREE));
          if (hs == 1) mma_commit(ctl.bar(BAR_GM_FREE));
        }
        if (!good || last) break;
      }
      // every MMA of this CTA (and TMA still in flight) lands before the
      // tensor memory and shared memory are released
      mma_commit(ctl.bar(BAR_DRAIN));
      mbar_wait(ctl.bar(BAR_DRAIN), 0, kWaitNs);
      for (int i = tma_landed; i < tma_issued; ++i)
        mbar_wait(ctl.bar(BAR_BC_FULL + (i & 1)), uint32_t((i >> 1) & 1), kWaitNs / 2);
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
cudaError_t launch_pair(const void* x, const void* dt, const float* A, const void* B,
                        const void* C, const float* h0, float* hT, void* y, const float* w,
                        const float* bias, const void* s_in, void* s_out, int K, int64_t Bz,
                        int64_t L, int H, int G, int* status, cudaStream_t st) {
  using namespace pr;
  CUtensorMap mB, mC, mX;
  if (!make_bc_map(&mB, B, Bz, L, G, kN) || !make_bc_map(&mC, C, Bz, L, G, kN))
    return cudaErrorInvalidValue;
  if (FUSED) {
    if (!make_x_map(&mX, x, Bz, L, int64_t(H) * kP, kXsRows)) return cudaErrorInvalidValue;
  } else {
    mX = mB;  // unused
  }
  auto kern = ssm_scan_pair_kernel<TX, TY, FUSED>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
  if (e != cudaSuccess) return e;
  kern<<<unsigned(Bz * (H / 2)), kThreads, kSmemBytes, st>>>(
      mB, mC, mX, static_cast<const TX*>(x), static_cast<const __nv_bfloat16*>(dt), A, h0, hT,
      static_cast<TY*>(y), w, bias, static_cast<const TX*>(s_in), static_cast<TX*>(s_out), K,
      int(L), H, G, status);
  return cudaGetLastError();
}
}  // namespace

// The pair kernel takes bf16 dt/B/C, P = 64, N = 128 and pairs of heads that
// share a B/C group.
bool ssm_scan_pair_supports(sss_dtype at, int64_t L, int H, int P, int N, int G) {
  return at == SSS_BF16 && P == pr::kP && N == pr::kN && L >= 1 && L < (int64_t(1) << 31) &&
         H >= 2 && G >= 1 && H % G == 0 && (H / G) % 2 == 0 && encode_fn() != nullptr;
}

cudaError_t ssm_scan_pair_launch(const void* x, sss_dtype xt, const void* dt, const float* A,
                                 const void* B, const void* C, const float* h0, float* hT,
                                 void* y, sss_dtype yt, int64_t Bz, int64_t L, int H, int G,
                                 int* status, cudaStream_t st) {
  if (Bz * (H / 2) > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
#define SSS_PAIR(TXT, TYT)                                                                    \
  return launch_pair<TXT, TYT, false>(x, dt, A, B, C, h0, hT, y, nullptr, nullptr, nullptr,  \
                                      nullptr, 1, Bz, L, H, G, status, st);
  if (xt == SSS_F32 && yt == SSS_BF16) SSS_PAIR(float, __nv_bfloat16)
  if (xt == SSS_F32) SSS_PAIR(float, float)
  if (yt == SSS_BF16) SSS_PAIR(__nv_bfloat16, __nv_bfloat16)
  SSS_PAIR(__nv_bfloat16, float)
#undef SSS_PAIR
}

cudaError_t mixer_fwd_pair_launch(const void* x, const float* w, const float* bias,
                                  const void* s_in, void* s_out, const void* dt, const float* A,
                                  const void* B, const void* C, const float* h0, float* hT,
                                  void* y, sss_dtype yt, int64_t Bz, int64_t L, int H, int G,
                                  int K, int* status, cudaStream_t st) {
  if (Bz * (H / 2) > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (yt == SSS_BF16)
    return launch_pair<__nv_bfloat16, __nv_bfloat16, true>(x, dt, A, B, C, h0, hT, y, w, bias,
                                                           s_in, s_out, K, Bz, L, H, G, status, st);
  return launch_pair<__nv_bfloat16, float, true>(x, dt, A, B, C, h0, hT, y, w, bias, s_in, s_out,
                                                 K, Bz, L, H, G, status, st);
}

}  // namespace sss
