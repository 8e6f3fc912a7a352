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
//   h_new = exp(Lam_end - R) (e^R h_prev + B^T X'),   y_t = f_t Y_t.
//
// The state columns of tensor memory hold sigma = e^R h_prev before the
// chunk's state product and accumulate B^T X' on top of it, so the state
// product needs no columns of its own; between chunks sigma is rescaled to
// the next chunk's reference: sigma <- e^{R'} (e^{Lam_end - R} sigma), two
// factors each inside exp(+-50).
//
// Pieces instead of fixed chunks: a piece is at most 128 tokens and ends
// before the token at which either head's Lam range would pass kFactorRange,
// so the factored weights always stay inside exp(+-50).  Ordinary inputs give
// 128-token pieces; a head with a huge decay gives shorter ones (a single
// token always qualifies: its range is 0).
//
// GB300 mapping, one CTA per (batch, head pair), 640 threads in five
// warpgroups whose register budgets are set with setmaxnreg:
//   warps 0-7   producers (112 registers): per piece and head the conv + SiLU
//               of the raw rows (TMA-staged) or the input rows and the
//               x' = g x hi/lo values, 8 channels x 4 tokens per thread
//               (packed f32x2 arithmetic), stored for both heads at once;
//   warps 8-11  state (96): warp 8 + q owns TMEM lanes 32q.. (state rows n):
//               the rescale of sigma between pieces, the h' tiles (the hi/lo
//               split of the rescaled sigma) and hT;
//   warps 12-15 output (80): TMEM lanes 32q.. as token rows t: the y rows;
//   the state warps also mask and split G (rows t of their lane quarter);
//   warp 16     issuer: every tcgen05.mma and commit, one thread;
//   warp 17     decay: per piece, the log-decay prefix of both heads (4 tokens
//               per lane), the piece length and the chunk scalars, published
//               in a ring of 4 piece descriptors up to 4 pieces ahead;
//   warp 18     loader: the TMA of each piece's B and C, one thread.
// The two heads' x' tiles (and h' tiles) sit side by side as the two 64-wide
// halves of one N = 128 operand, so every product covers both heads in one
// M = 128, N = 128 MMA:
//   G = C B^T,  S_ab += B^T [x'_a | x'_b],  Y_ab = C [h'_a | h'_b]^T + (G o c) [x'_a | x'_b].
// Tensor memory (512 columns): G [t][s] 128 (the masked hi/lo split of G is
// written over G, block by block), two Y buffers (pieces alternate) and the
// state sigma of both heads, 128 each: the state never leaves the SM between
// pieces.  Shared memory: the piece's C and B (32 KB each), the x' tiles (hi
// and lo, 64 KB), the h' tiles (64 KB), the staged raw rows and the piece
// descriptors.  Per piece the MMAs run in the order
//   Yo(c), G(c), S(c), Yd(c)
// so that every hand-over has an MMA group of slack: the state warps rescale
// sigma while Yd(c-1) runs, the masks of G(c) are written while S(c) runs,
// C(c+1) loads while S(c) and Yd(c) run and B(c+1) while Yd(c) and Yo(c+1)
// run, the x' tiles of piece c+1 are stored while Yo(c+1) and G(c+1) run,
// and the y rows of piece c are read while piece c+1 runs.  Every wait is
// bounded (2 s); a timeout raises SSS_ERR_TIMEOUT and unwinds.
#include <type_traits>

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
constexpr int kProdWarps = 8;
constexpr int kOutWarp0 = 12;
constexpr int kIssuerWarp = 16;
constexpr int kDecayWarp = 17;
constexpr int kLoaderWarp = 18;
constexpr int kWarps = 20;
constexpr int kThreads = kWarps * 32;              // 640
constexpr int kPT = kProdWarps * 32;               // 256 producer threads
constexpr int kCT = 128;                           // state threads; output threads
// Registers a thread per warpgroup after setmaxnreg.  The launch gives every
// thread 96 (65536 / 640, in steps of 8); the budgets below add up to the
// same 61440: producers 2 x 128 x 112, state 128 x 96, output 128 x 80,
// issuer / decay / loader 128 x 80 (each the least that compiles without
// spills: a spilled register reloads through an L1 that the shared-memory
// carve-out leaves small, often from L2).  The host checks the launch count before
// every launch: a split whose sum exceeded the launch's registers would make
// setmaxnreg.inc wait forever.
constexpr uint32_t kLaunchRegs = 96;
constexpr uint32_t kRegProd = 112, kRegState = 96, kRegOut = 80, kRegCtl = 80;
static_assert(kPT * kRegProd + kCT * kRegState + kCT * kRegOut + 128 * kRegCtl ==
                  uint32_t(kThreads) * kLaunchRegs,
              "register budgets");
constexpr uint32_t kTmemCols = 512;
// tensor memory columns: G [t][s] fp32, overwritten block by block by the
// masked split (32-column block j: hi pairs at 32j, lo pairs at 32j + 16);
// Y buffer u [t][p] at 128 + 128 u; the state sigma [n][p]; head b at + 64
constexpr uint32_t kColG = 0;
constexpr uint32_t kColY = 128;
constexpr uint32_t kColH = 384;
// shared memory (bytes from a 1024-byte aligned base)
constexpr uint32_t kOffC = 0;         // C of the piece [t][n] (two 64-wide n blocks)
constexpr uint32_t kOffB = 32768;     // B of the piece [s][n]
constexpr uint32_t kOffX = 65536;     // x' hi of head hs at + 16384 hs, lo at + 32768 + 16384 hs (rows s)
constexpr uint32_t kOffH = 131072;    // h' hi of head hs at + 16384 hs, lo at + 32768 + 16384 hs (rows n)
constexpr uint32_t kOffXs = 196608;   // staged raw rows [t0 - 3, t0 + 128) of one head
constexpr uint32_t kXsRows = 128 + kMaxK - 1;
constexpr uint32_t kXsBytes = kXsRows * 128;
constexpr uint32_t kOffMisc = kOffXs + kXsBytes;  // 213376
// misc (offsets from kOffMisc)
constexpr uint32_t kMiInfo = 0;       // 4 piece descriptors
constexpr uint32_t kMiRed = 4224;     // (unused)
// conv weights and bias times -log2(e), per (head hs, channel pair e2, channel
// group q) 12 floats: the taps of channels 8q + 2e2 and 8q + 2e2 + 1 interleaved
// (tap k of the pair = floats 2k, 2k+1), the two biases, 2 pad.  The 48-byte stride puts
// the 8 groups a warp reads on distinct banks.
constexpr uint32_t kMiW = 4480;       // [2][4][8][12] floats
constexpr uint32_t kMiBars = 7552;    // mbarriers
constexpr uint32_t kMiTmem = 7840;
constexpr uint32_t kMiAbort = 7844;
constexpr uint32_t kMiscBytes = 7848;
// per output warp, 32 rows x 64 bytes of bf16 y: the warp writes its rows
// here and reads them back as whole 64-byte row segments, so one global store
// instruction covers 8 rows instead of 32 partial lines
constexpr uint32_t kOffYs = (kOffMisc + kMiscBytes + 127u) & ~127u;
constexpr uint32_t kYsWarpBytes = 32 * 64;
constexpr uint32_t kSmemBytes = kOffYs + 4 * kYsWarpBytes + 1024;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
constexpr int kSlots = 4;

struct PieceInfo {
  int start, n, last, pad;
  float R[2], lend[2];
  float lam[2][128];
};
static_assert(sizeof(PieceInfo) * kSlots <= kMiRed, "piece ring");

enum {
  BAR_C_FULL = 0, BAR_B_FULL = 1, BAR_XS_FULL = 2, BAR_INFO_FULL = 3 /*4*/,
  BAR_INFO_FREE = 7 /*4*/, BAR_X_FULL = 11, BAR_G_DONE = 12, BAR_S_DONE = 13,
  BAR_Y_FULL = 14 /*2*/, BAR_GM_FULL = 16, BAR_H_FULL = 17, BAR_Y_FREE = 18 /*2*/,
  BAR_DRAIN = 20, NUM_BARS = 21
};
// Barrier discipline: each barrier's completions are awaited in order by
// threads that see every one of them, and no waiter can fall two phases
// behind (the phase it waits for gates the work that would complete the
// next one), so the parity it waits on is never stale.  A commit (about as
// costly to issue as an MMA) makes its barrier track every MMA issued before
// it, so one commit per product group serves every role that needs it:
//   G_DONE(c)  after G(c):  the masks may read G; C may be reloaded (Yo(c)
//              has read it too);
//   S_DONE(c)  after S(c):  sigma may be rescaled (Yo(c) has read the h'
//              tiles); B may be reloaded (G(c) has read it too); with STATE
//              the x' tiles are free;
//   Y_FULL(c)  after Yd(c), one barrier per Y buffer: the y rows may be read;
//              the x' tiles are free; G(c+1) may overwrite the masked split.
static_assert(NUM_BARS * 8 <= kMiTmem - kMiBars, "barrier area");

constexpr uint32_t kIdG = idesc_bf16(128, 128, 0, 0);   // C (K-major) x B (K-major)
constexpr uint32_t kIdS = idesc_bf16(128, 128, 1, 1);   // B^T (MN-major) x [x'_a | x'_b] (MN-major)
constexpr uint32_t kIdYo = idesc_bf16(128, 128, 0, 1);  // C (K-major) x [h'_a | h'_b] (MN-major)
constexpr uint32_t kIdYd = idesc_bf16(128, 128, 0, 1);  // (G o causal) (TMEM) x [x'_a | x'_b]

// registers per thread of this warpgroup (every warp of the warpgroup runs it)
template <uint32_t R>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}
template <uint32_t R>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
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
constexpr float kLn2 = 0.6931471805599453f;
// SiLU of a pair, times g, from z' = -z log2(e) (the conv's weights and bias
// carry the factor -log2(e), so the conv yields z' directly):
//   SiLU(z) g = z g / (1 + e^-z) = (z' gn) / (1 + 2^z'),  gn = -ln(2) g.
// One reciprocal per channel: a large z' gives 2^z' = inf and a zero, which
// is SiLU's limit there (no cap on the exponent is needed).
__device__ __forceinline__ uint64_t silu_scaled2(uint64_t zp, float gn) {
  float ta, tb;
  upk2(zp, ta, tb);
  float da, db;
  upk2(add2(pk2(ex2f(ta), ex2f(tb)), pk2(1.0f, 1.0f)), da, db);
  return mul2(mul2(zp, pk2(gn, gn)), pk2(rcpf(da), rcpf(db)));
}
// a packed pair -> one bf16 pair word (round to nearest even, element 0 low)
__device__ __forceinline__ uint32_t bf2_pack(uint64_t v) {
  float a, b;
  upk2(v, a, b);
  const __nv_bfloat162 h2 = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h2);
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
// STATE: only the final state is wanted (the first pass of the span split):
// no G, mask, Yo, Yd, h' tiles or y rows; per piece the producers' x' tiles,
// the S' MMAs and the carry.
namespace {
namespace pr {
// Causal mask and hi/lo split of the rows of G in this warp's TMEM lane
// quarter q (rows t = 32 q + lane), 32-column blocks j of parity `par`: blocks
// above the diagonal become zeros, the diagonal block keeps s <= t.  The
// block's 32 fp32 columns are read first; its hi pairs go over the first 16,
// its lo pairs over the last 16.
__device__ __forceinline__ void mask_split_g(uint32_t tl, int q, int lane, int par) {
#pragma unroll 1
  for (int j = par; j < 4; j += 2) {
    uint32_t ph[16], pl[16];
    if (j <= q) {
      uint32_t g2[2][16];
      tmem_ld_x16_nowait(tl + kColG + uint32_t(32 * j), g2[0]);
      tmem_ld_x16_nowait(tl + kColG + uint32_t(32 * j + 16), g2[1]);
      tmem_ld_wait();
      reg_fence16(g2[0]);
      reg_fence16(g2[1]);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float m[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) m[i] = __uint_as_float(g2[hf][i]);
        if (j == q) {  // diagonal block: s = 32 j + 16 hf + i <= t = 32 q + lane
#pragma unroll
          for (int i = 0; i < 16; ++i) m[i] = 16 * hf + i <= lane ? m[i] : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) split2(m[2 * i], m[2 * i + 1], ph[8 * hf + i], pl[8 * hf + i]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) ph[i] = pl[i] = 0u;
    }
    tmem_st_x16(tl + kColG + uint32_t(32 * j), ph);
    tmem_st_x16(tl + kColG + uint32_t(32 * j + 16), pl);
  }
  tmem_st_wait();
}
}  // namespace pr
}  // namespace

// x: the scan input u [Bz, L, H, 64] (TX = float or bf16), or with FUSED the
// raw input [Bz, L, H*64] (bf16) that the producers convolve (K <= 4, SiLU).
// Requires (H / G) even: both heads of a pair read the same B and C group.
// STATE: only the final state is wanted (the first pass of the span split):
// no G, mask, Yo, Yd, h' tiles or y rows; per piece the producers' x' tiles,
// the S MMAs and the rescale of sigma.
template <typename TX, typename TY, bool FUSED, bool PACKED, bool STATE>
__global__ void __launch_bounds__(pr::kThreads, 1)
ssm_scan_pair_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmC,
                     const __grid_constant__ CUtensorMap tmX, const TX* __restrict__ x,
                     const __nv_bfloat16* __restrict__ dt, const float* __restrict__ A,
                     const float* h0, float* hT, TY* __restrict__ y,
                     const float* __restrict__ conv_w, const float* __restrict__ conv_b,
                     const TX* conv_s_in, TX* conv_s_out, int K, int L, int H, int G,
                     int* status, const int32_t* __restrict__ seq_idx) {
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
  // launched as a dependent of the previous kernel of the span split: its
  // outputs (conv and SSM states) are complete and visible from here on
  dep_wait();

  if (warp == kIssuerWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    int counts[NUM_BARS];
    for (int i = 0; i < NUM_BARS; ++i) counts[i] = 1;
    for (int i = 0; i < kSlots; ++i) {
      counts[BAR_INFO_FULL + i] = 32;                       // the decay warp
      counts[BAR_INFO_FREE + i] = kPT + 2 * kCT + 2;        // + issuer, loader
    }
    counts[BAR_H_FULL] = kCT;
    counts[BAR_GM_FULL] = kCT;
    counts[BAR_Y_FREE] = counts[BAR_Y_FREE + 1] = kCT;
    counts[BAR_X_FULL] = kPT;
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
      sw[2 * k + odd] = k >= kMaxK - K ? -kLog2e * conv_w[d * K + k - (kMaxK - K)] : 0.0f;
    sw[8 + odd] = conv_b ? -kLog2e * conv_b[d] : 0.0f;
    sw[10 + odd] = 0.0f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;

  if (warp < kProdWarps) {
    regs_inc<kRegProd>();
    // ============================ producers ============================
    // thread (q, g4) = channels [8q, 8q+8) x tokens [4 g4, 4 g4 + 4) of one head
    constexpr int NT = 4;
    constexpr int NR = NT + kMaxK - 1;  // staged rows a thread reads
    const int q = tid & 7, g4 = tid >> 3, tb = 4 * g4;
    auto stage_x = [&](int start, int hs) {  // TMA of raw rows [start - 3, start + 128)
      mbar_arrive_expect_tx(ctl.bar(BAR_XS_FULL), kXsBytes);
      tma_load_3d(sb + kOffXs, &tmX, (2 * pair + hs) * kP, start - (kMaxK - 1), b,
                  ctl.bar(BAR_XS_FULL));
    };
    if (FUSED && tid == 0) {
      prefetch_tmap(&tmX);
      stage_x(0, 0);
      // head b's rows of piece 0 are staged once head a's are consumed: have
      // them in L2 by then (the 3 halo rows before token 0 come from S)
      tma_prefetch_3d(&tmX, (2 * pair + 1) * kP, 0, b);
    }
    int xs_issued = FUSED ? 1 : 0, xs_landed = 0;
    bool ok = true;
    for (int c = 0;; ++c) {
      const int slot = c & (kSlots - 1);
      const PieceInfo* inf = info + slot;
      // ---- the piece descriptor (start, length, decay prefix) -------------
      if (ok) ok = ctl.wait(BAR_INFO_FULL + slot, uint32_t((c / kSlots) & 1));
      const int p = inf->start, n = ok ? inf->n : 1;
      const bool last = !ok || inf->last != 0;
      // ---- per head: inputs, x' = g x hi/lo values ------------------------
      uint32_t hw2[2][NT][4], lw2[2][NT][4];  // both heads' values, stored together
#pragma unroll
      for (int hs = 0; hs < 2; ++hs) {
        const int head = 2 * pair + hs;
        const int nv = ok ? min(NT, max(0, n - tb)) : 0;  // live tokens of this thread
        const float R = inf->R[hs];
        // x' = g_s x with g_s = exp(R - Lam_s), 0 for dead tokens (fused:
        // times -ln 2, the factor SiLU takes from z')
        float gv[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j)
          gv[j] = j < nv ? (FUSED ? -kLn2 : 1.0f) * ex2f((R - inf->lam[hs][tb + j]) * kLog2e) : 0.0f;
        uint32_t(&hw)[NT][4] = hw2[hs];
        uint32_t(&lw)[NT][4] = lw2[hs];
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
          const int su = 2 * c + hs;  // staging use
          if (ok) ok = ctl.wait(BAR_XS_FULL, uint32_t(su & 1));
          if (ok) xs_landed = su + 1;
          // staged rows tb + i = positions p + tb - 3 + i
          uint4 xr[NR];
#pragma unroll
          for (int i = 0; i < NR; ++i)
            xr[i] = *reinterpret_cast<const uint4*>(sm + kOffXs + sw128(tb + i, q));
          {
            // a fold of every loaded word: once it is computed each staged
            // load has returned, so the buffer can go to the next head's (or
            // piece's) rows before any arithmetic; the proxy fence orders the
            // TMA write after these generic-proxy reads
            // (one word of each 16-byte load suffices: a vector load
            // completes as a whole)
            uint32_t fold = 0u;
#pragma unroll
            for (int i = 0; i < NR; ++i) fold ^= xr[i].x;
            asm volatile("" ::"r"(fold));
          }
          role_sync(3, kPT);
          if (tid == 0 && ok) {
            fence_proxy_async_smem();
            if (hs == 0) {
              stage_x(p, 1);
              xs_issued = su + 2;
            } else if (!last) {
              stage_x(p + n, 0);
              xs_issued = su + 2;
            }
          }
          if (PACKED && tb == 0 && inf->pad != 7) {
            // packed rows: halo positions of another sample read as zero
#pragma unroll
            for (int i = 0; i < kMaxK - 1; ++i)
              if (!((inf->pad >> i) & 1)) xr[i] = make_uint4(0u, 0u, 0u, 0u);
          }
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
      }
      mbar_arrive(ctl.bar(BAR_INFO_FREE + slot));  // done with the descriptor
      // the x' tiles are free once the previous piece's S and Yd are done
      if (ok && c >= 1)
        ok = STATE ? ctl.wait(BAR_S_DONE, uint32_t((c - 1) & 1))
                   : ctl.wait(BAR_Y_FULL + ((c - 1) & 1), uint32_t(((c - 1) >> 1) & 1));
      if (ok) {
#pragma unroll
        for (int hs = 0; hs < 2; ++hs) {
          uint8_t* xt = sm + kOffX + 16384u * hs;
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            *reinterpret_cast<uint4*>(xt + sw128(tb + j, q)) =
                make_uint4(hw2[hs][j][0], hw2[hs][j][1], hw2[hs][j][2], hw2[hs][j][3]);
            *reinterpret_cast<uint4*>(xt + 32768 + sw128(tb + j, q)) =
                make_uint4(lw2[hs][j][0], lw2[hs][j][1], lw2[hs][j][2], lw2[hs][j][3]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(ctl.bar(BAR_X_FULL));
      }
      // every producer leaves the loop at the same piece (they share named
      // barriers), failed waits included
      if (role_sync_or(3, kPT, !ok)) ok = false;
      if (last || !ok) break;
    }
    if (FUSED && tid == 0) {  // staged tiles still in flight
      for (int su = xs_landed; su < xs_issued; ++su)
        if (!mbar_wait(ctl.bar(BAR_XS_FULL), uint32_t(su & 1), kWaitNs / 2))
          raise_status(status, SSS_ERR_TIMEOUT);
    }
    if constexpr (FUSED) {
      // final conv state F_j = ext[L + j] of both heads' channels; every read
      // of S happened in piece 0
      role_sync(3, kPT);
      if (conv_s_out && tid < 2 * kP && !*ctl.abort) {
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
  } else if (warp < kOutWarp0) {
    regs_dec<kRegState>();
    // ===== state: TMEM lanes of quarter q (state row n = r), both heads =====
    const int q = warp & 3;  // == warp % 4: the TMEM lane quarter this warp may access
    const int r = 32 * q + lane;
    const uint32_t tl = tm + (uint32_t(q * 32) << 16);
    const int64_t hoff0 = (int64_t(b) * H + 2 * pair) * kP * kN;  // head a; head b + kP * kN
    // every wait is followed by a warp vote, so the warp leaves the loop
    // together (its TMEM accesses are warp-collective)
    auto wait_all = [&](int bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, ctl.wait(bar, parity));
    };
    // sigma <- t (s sigma) for both heads, 32 columns at a time; unless
    // STATE, the hi/lo split of the new values into row n = r of the h' tiles
    // (the operand of the next Yo)
    auto rescale = [&](float s0, float s1, float t0, float t1) {
#pragma unroll 1
      for (int hs = 0; hs < 2; ++hs) {
        uint8_t* ht = sm + kOffH + 16384u * hs;
        const uint64_t sp = hs ? pk2(s1, s1) : pk2(s0, s0), tp = hs ? pk2(t1, t1) : pk2(t0, t0);
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          const uint32_t col = kColH + 64u * hs + 32u * hf;
          uint32_t w0[16], w1[16];
          tmem_ld_x16_nowait(tl + col, w0);
          tmem_ld_x16_nowait(tl + col + 16, w1);
          tmem_ld_wait();
          reg_fence16(w0);
          reg_fence16(w1);
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            float a, c;
            upk2(mul2(tp, mul2(sp, pk2(__uint_as_float(w0[i]), __uint_as_float(w0[i + 1])))), a, c);
            w0[i] = __float_as_uint(a);
            w0[i + 1] = __float_as_uint(c);
            upk2(mul2(tp, mul2(sp, pk2(__uint_as_float(w1[i]), __uint_as_float(w1[i + 1])))), a, c);
            w1[i] = __float_as_uint(a);
            w1[i + 1] = __float_as_uint(c);
          }
          tmem_st_x16(tl + col, w0);
          tmem_st_x16(tl + col + 16, w1);
          if constexpr (!STATE) {
            // columns p = 32 hf .. 32 hf + 31: 16-byte chunks 4 hf .. 4 hf + 3
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              const uint32_t(&w)[16] = cc < 2 ? w0 : w1;
              const int o = 8 * (cc & 1);
              uint32_t hw[4], lw[4];
#pragma unroll
              for (int k = 0; k < 4; ++k)
                split2(__uint_as_float(w[o + 2 * k]), __uint_as_float(w[o + 2 * k + 1]), hw[k], lw[k]);
              *reinterpret_cast<uint4*>(ht + sw128(r, 4 * hf + cc)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
              *reinterpret_cast<uint4*>(ht + 32768 + sw128(r, 4 * hf + cc)) =
                  make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
          }
        }
      }
      tmem_st_wait();
      if constexpr (!STATE) fence_proxy_async_smem();
      tc_fence_before();
    };
    // sigma = h0 (zeros without h0) needs no descriptor: it goes to tensor
    // memory while the decay warp forms piece 0; then sigma = e^{R_0} h0 and
    // the h' tiles of piece 0
#pragma unroll 1
    for (int hs = 0; hs < 2; ++hs) {
#pragma unroll 1
      for (int q2 = 0; q2 < 2; ++q2) {
        uint32_t w[2][16];
#pragma unroll
        for (int pp = 0; pp < 32; ++pp) {
          const int pc = 32 * q2 + pp;
          w[pp >> 4][pp & 15] =
              __float_as_uint(h0 ? h0[hoff0 + int64_t(hs) * kP * kN + int64_t(pc) * kN + r] : 0.0f);
        }
        tmem_st_x16(tl + kColH + 64u * hs + 32u * q2, w[0]);
        tmem_st_x16(tl + kColH + 64u * hs + 32u * q2 + 16u, w[1]);
      }
    }
    tmem_st_wait();
    bool ok = wait_all(BAR_INFO_FULL, 0u);
    if (ok) {
      rescale(1.0f, 1.0f, expf(info[0].R[0]), expf(info[0].R[1]));
      mbar_arrive(ctl.bar(BAR_H_FULL));
    }
    for (int c = 0; ok; ++c) {
      const int slot = c & (kSlots - 1);
      const PieceInfo* inf = info + slot;  // (its INFO_FULL phase was awaited)
      const bool last = inf->last != 0;
      if constexpr (!STATE) {
        // masks of G(c): the rows of this quarter
        if (!(ok = wait_all(BAR_G_DONE, uint32_t(c & 1)))) break;
        tc_fence_after();
        mask_split_g(tl, q, lane, 0);
        mask_split_g(tl, q, lane, 1);
        tc_fence_before();
        mbar_arrive(ctl.bar(BAR_GM_FULL));
      }
      // sigma after S(c): h_c = e^{Lam_end - R} sigma
      if (!(ok = wait_all(BAR_S_DONE, uint32_t(c & 1)))) break;
      tc_fence_after();
      const float s[2] = {expf(inf->lend[0] - inf->R[0]), expf(inf->lend[1] - inf->R[1])};
      if (last) {
        if (hT && !*ctl.abort) {
#pragma unroll 1
          for (int hs = 0; hs < 2; ++hs) {
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              uint32_t a0[16];
              tmem_ld_x16(tl + kColH + 64u * hs + 16u * qq, a0);
#pragma unroll
              for (int pp = 0; pp < 16; ++pp)
                hT[hoff0 + int64_t(hs) * kP * kN + int64_t(16 * qq + pp) * kN + r] =
                    s[hs] * __uint_as_float(a0[pp]);
            }
          }
        }
        mbar_arrive(ctl.bar(BAR_INFO_FREE + slot));
        break;
      }
      // sigma for piece c+1: e^{R_{c+1}} h_c
      const int slot1 = (c + 1) & (kSlots - 1);
      if (!(ok = wait_all(BAR_INFO_FULL + slot1, uint32_t(((c + 1) / kSlots) & 1)))) break;
      rescale(s[0], s[1], expf(info[slot1].R[0]), expf(info[slot1].R[1]));
      mbar_arrive(ctl.bar(BAR_H_FULL));
      mbar_arrive(ctl.bar(BAR_INFO_FREE + slot));
    }
  } else if (warp < kIssuerWarp) {
    regs_dec<kRegOut>();
    // ===== output: TMEM lanes of quarter q (token row t = r), both heads =====
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const uint32_t tl = tm + (uint32_t(q * 32) << 16);
    auto wait_all = [&](int bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, ctl.wait(bar, parity));
    };
    for (int c = 0;; ++c) {
      const int slot = c & (kSlots - 1);
      if (!wait_all(BAR_INFO_FULL + slot, uint32_t((c / kSlots) & 1))) break;
      const PieceInfo* inf = info + slot;
      const int n = inf->n, start = inf->start;
      const bool last = inf->last != 0;
      if constexpr (!STATE) {
        // ---- y rows of both heads: y_t = f_t Y_t ----------------------------
        const int yb = c & 1;
        if (!wait_all(BAR_Y_FULL + yb, uint32_t((c >> 1) & 1))) break;
        tc_fence_after();
        const uint32_t tY = tl + kColY + 128u * uint32_t(yb);
        // 32 columns [32 hf, 32 hf + 32) of head hs, scaled by f_t, to y
        auto emit_half = [&](int hs, int hf, float f_t, const uint32_t (&u0)[16],
                             const uint32_t (&u1)[16]) {
          // fused, bf16 y: through the warp's buffer (64-byte row segments);
          // otherwise direct row stores
          if constexpr (FUSED && std::is_same<TY, __nv_bfloat16>::value) {
            // f_t Y as bf16 pairs: one packed multiply and one paired
            // conversion per two columns
            uint32_t w[16];
            const uint64_t ff = pk2(f_t, f_t);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              w[i] = bf2_pack(mul2(pk2(__uint_as_float(u0[2 * i]), __uint_as_float(u0[2 * i + 1])), ff));
              w[8 + i] = bf2_pack(mul2(pk2(__uint_as_float(u1[2 * i]), __uint_as_float(u1[2 * i + 1])), ff));
            }
            // row `lane` of the warp's buffer, 16-byte chunks XOR-swizzled by
            // (row / 2) % 4: both the row writes and the segment reads below
            // touch 8 distinct bank groups per 8 lanes
            uint8_t* yb8 = sm + kOffYs + uint32_t(q) * kYsWarpBytes;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
              *reinterpret_cast<uint4*>(yb8 + lane * 64 + ((cc ^ ((lane >> 1) & 3)) << 4)) =
                  make_uint4(w[4 * cc], w[4 * cc + 1], w[4 * cc + 2], w[4 * cc + 3]);
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int row = 8 * j + (lane >> 2), ch = lane & 3;
              const uint4 v = *reinterpret_cast<const uint4*>(yb8 + row * 64 + ((ch ^ ((row >> 1) & 3)) << 4));
              if (32 * q + row < n)
                *reinterpret_cast<uint4*>(y + (int64_t(b) * L + start + 32 * q + row) * D +
                                          int64_t(2 * pair + hs) * kP + 32 * hf + 8 * ch) = v;
            }
            __syncwarp();
          } else {
            TY* yrow = y + (int64_t(b) * L + start + r) * D + int64_t(2 * pair + hs) * kP + 32 * hf;
            float yv[16];
#pragma unroll
            for (int pp = 0; pp < 16; ++pp) yv[pp] = f_t * __uint_as_float(u0[pp]);
            if (r < n) store_row16<TY>(yrow, yv);
#pragma unroll
            for (int pp = 0; pp < 16; ++pp) yv[pp] = f_t * __uint_as_float(u1[pp]);
            if (r < n) store_row16<TY>(yrow + 16, yv);
          }
        };
#pragma unroll 1
        for (int hs = 0; hs < 2; ++hs) {
          const float f_t = expf(inf->lam[hs][r] - inf->R[hs]);
#pragma unroll 1
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t a0[16], a1[16];
            tmem_ld_x16_nowait(tY + 64u * hs + 32u * hf, a0);
            tmem_ld_x16_nowait(tY + 64u * hs + 32u * hf + 16u, a1);
            tmem_ld_wait();
            reg_fence16(a0);
            reg_fence16(a1);
            if (hs == 1 && hf == 1) {  // Y is read: Yo(c+2) may overwrite it
              tc_fence_before();
              mbar_arrive(ctl.bar(BAR_Y_FREE + yb));
            }
            emit_half(hs, hf, f_t, a0, a1);
          }
        }
      }
      mbar_arrive(ctl.bar(BAR_INFO_FREE + slot));
      if (last) break;
    }
  } else {
    regs_dec<kRegCtl>();
    if (warp == kIssuerWarp) {
      if (lane == 0) {
        // ========================= issuer (one thread) =========================
        const uint32_t cb = sb + kOffC, bb = sb + kOffB, xb = sb + kOffX, hb = sb + kOffH;
        // base descriptors; every K step below adds a constant to them
        const uint64_t dC = sdesc_sw128(cb, 16, 1024), dBk = sdesc_sw128(bb, 16, 1024);
        const uint64_t dBm = sdesc_sw128(bb, 16384, 1024);
        const uint64_t dXh = sdesc_sw128(xb, 16384, 1024), dXl = sdesc_sw128(xb + 32768, 16384, 1024);
        const uint64_t dHh = sdesc_sw128(hb, 16384, 1024), dHl = sdesc_sw128(hb + 32768, 16384, 1024);
        const uint32_t tG = tm + kColG, tS = tm + kColH;
        // Issuing an MMA blocks once the tensor pipe is about three MMAs
        // ahead, so every wait sits where its barrier has (almost surely)
        // completed already: between the MMAs of a group, with work queued.
        bool last = false;
        // the next piece's descriptor: consumed between the MMAs of this one
        auto take_info = [&](int cc) -> bool {
          const int sl = cc & (kSlots - 1);
          if (!ctl.wait(BAR_INFO_FULL + sl, uint32_t((cc / kSlots) & 1))) return false;
          last = info[sl].last != 0;
          mbar_arrive(ctl.bar(BAR_INFO_FREE + sl));
          return true;
        };
        bool ok = take_info(0);
        if constexpr (!STATE) {
          ok = ok && ctl.wait(BAR_H_FULL, 0u) && ctl.wait(BAR_C_FULL, 0u);
        }
        for (int c = 0; ok; ++c) {
          const bool last_c = last;
          if constexpr (!STATE) {
            const uint32_t dY = tm + kColY + 128u * uint32_t(c & 1);
            // Yo(c) = C [e^R h_a | e^R h_b]^T (hi + lo) starts Y(c); its
            // operands (C, the h' tiles, a free Y buffer) were awaited before
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) mma_ss(dY, dC + kstep(kk, 16384), dHh + mnstep(kk), kIdYo, kk);
            if (!(ok = ctl.wait(BAR_B_FULL, uint32_t(c & 1)))) break;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) mma_ss(dY, dC + kstep(kk, 16384), dHl + mnstep(kk), kIdYo, 1);
            // G(c) = C B^T, once Yd(c-1) has read the masked split that G
            // overwrites (it ran before Yo(c), so this rarely waits)
            if (c >= 1 && !(ok = ctl.wait(BAR_Y_FULL + ((c - 1) & 1), uint32_t(((c - 1) >> 1) & 1)))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tG, dC + kstep(kk, 16384), dBk + kstep(kk, 16384), kIdG, kk);
            mma_commit(ctl.bar(BAR_G_DONE));
            // S(c): sigma += B^T [x'_a | x'_b] (hi + lo), once the x' tiles are in
            if (!(ok = ctl.wait(BAR_X_FULL, uint32_t(c & 1)))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) mma_ss(tS, dBm + mnstep(kk), dXh + mnstep(kk), kIdS, 1);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) mma_ss(tS, dBm + mnstep(kk), dXl + mnstep(kk), kIdS, 1);
            mma_commit(ctl.bar(BAR_S_DONE));
            // Y(c) += hi(G o c) x'hi + hi(G o c) x'lo + lo(G o c) x'hi; K step
            // kk (tokens 16 kk ..) reads 32-column block kk / 2, half kk % 2
            if (!(ok = ctl.wait(BAR_GM_FULL, uint32_t(c & 1)))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(dY, tG + 32u * (kk >> 1) + 8u * (kk & 1), dXh + mnstep(kk), kIdYd, 1);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts(dY, tG + 32u * (kk >> 1) + 8u * (kk & 1), dXl + mnstep(kk), kIdYd, 1);
            // the next piece's descriptor, C and Y buffer, with Yd(c) queued
            if (!last_c) {
              ok = take_info(c + 1) && ctl.wait(BAR_C_FULL, uint32_t((c + 1) & 1)) &&
                   (c + 1 < 2 || ctl.wait(BAR_Y_FREE + ((c + 1) & 1), uint32_t((((c + 1) >> 1) - 1) & 1)));
            }
#pragma unroll
            for (int kk = 4; kk < 8; ++kk)
              mma_ts(dY, tG + 32u * (kk >> 1) + 8u * (kk & 1), dXl + mnstep(kk), kIdYd, 1);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(dY, tG + 32u * (kk >> 1) + 16u + 8u * (kk & 1), dXh + mnstep(kk), kIdYd, 1);
            mma_commit(ctl.bar(BAR_Y_FULL + (c & 1)));
            if (last_c || !ok) break;
            // the h' tiles and sigma of piece c+1 (rescaled after S(c))
            if (!(ok = ctl.wait(BAR_H_FULL, uint32_t((c + 1) & 1)))) break;
          } else {
            if (!(ok = ctl.wait(BAR_H_FULL, uint32_t(c & 1)) && ctl.wait(BAR_B_FULL, uint32_t(c & 1)) &&
                       ctl.wait(BAR_X_FULL, uint32_t(c & 1))))
              break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) mma_ss(tS, dBm + mnstep(kk), dXh + mnstep(kk), kIdS, 1);
            if (!last_c) ok = take_info(c + 1);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) mma_ss(tS, dBm + mnstep(kk), dXl + mnstep(kk), kIdS, 1);
            mma_commit(ctl.bar(BAR_S_DONE));
            if (last_c || !ok) break;
          }
        }
        // every MMA lands before the tensor memory and shared memory are released
        mma_commit(ctl.bar(BAR_DRAIN));
        if (!mbar_wait(ctl.bar(BAR_DRAIN), 0, kWaitNs)) raise_status(status, SSS_ERR_TIMEOUT);
      }
      __syncwarp();
    } else if (warp == kLoaderWarp) {
      if (lane == 0) {
        // ========================= loader (one thread) =========================
        // B(c) and C(c) land in their single buffers once the MMAs of piece
        // c-1 that read them are done (C after G(c-1), B after S(c-1))
        const uint32_t cb = sb + kOffC, bb = sb + kOffB;
        prefetch_tmap(&tmB);
        if constexpr (!STATE) prefetch_tmap(&tmC);
        int c_issued = 0, b_issued = 0;
        auto load_c = [&](int start) {
          const uint32_t bar = ctl.bar(BAR_C_FULL);
          mbar_arrive_expect_tx(bar, 32768u);
          tma_load_3d(cb, &tmC, g * kN, start, b, bar);
          tma_load_3d(cb + 16384, &tmC, g * kN + 64, start, b, bar);
        };
        auto load_b = [&](int start) {
          const uint32_t bar = ctl.bar(BAR_B_FULL);
          mbar_arrive_expect_tx(bar, 32768u);
          tma_load_3d(bb, &tmB, g * kN, start, b, bar);
          tma_load_3d(bb + 16384, &tmB, g * kN + 64, start, b, bar);
        };
        // piece 0 starts at token 0: its C and B go out before its descriptor
        if constexpr (!STATE) load_c(0);
        load_b(0);
        for (int c = 0;; ++c) {
          const int slot = c & (kSlots - 1);
          if (!ctl.wait(BAR_INFO_FULL + slot, uint32_t((c / kSlots) & 1))) break;
          const int start = info[slot].start;
          const bool last = info[slot].last != 0;
          mbar_arrive(ctl.bar(BAR_INFO_FREE + slot));
          if constexpr (!STATE) {
            if (c >= 1) {
              if (!ctl.wait(BAR_G_DONE, uint32_t((c - 1) & 1))) break;
              load_c(start);
            }
            c_issued = c + 1;
          }
          if (c >= 1) {
            if (!ctl.wait(BAR_S_DONE, uint32_t((c - 1) & 1))) break;
            load_b(start);
          }
          b_issued = c + 1;
          if (last) break;
        }
        // a load of each buffer is in flight at most: wait for the last one
        if (c_issued > 0 && !mbar_wait(ctl.bar(BAR_C_FULL), uint32_t((c_issued - 1) & 1), kWaitNs / 2))
          raise_status(status, SSS_ERR_TIMEOUT);
        if (b_issued > 0 && !mbar_wait(ctl.bar(BAR_B_FULL), uint32_t((b_issued - 1) & 1), kWaitNs / 2))
          raise_status(status, SSS_ERR_TIMEOUT);
      }
      __syncwarp();
    } else if (warp == kDecayWarp) {
      // ============================ decay warp ============================
      // lane l holds tokens 4l .. 4l+3 of the piece for both heads: the
      // inclusive log-decay prefix Lam, its running min / max, the piece length
      // (tokens while both heads' Lam range stays <= kFactorRange), and per head
      // R = the middle of the range and Lam_end, published in the descriptor ring
      const float Ah[2] = {A[2 * pair], A[2 * pair + 1]};
      // the log-decay l_t = dt_t A_h of the piece's tokens; a token that starts
      // a new packed sample gets kSampleStartLog, which ends the piece before
      // it (its range would pass kFactorRange) and zeroes the state it inherits
      auto load_dt = [&](int start, float (&v)[2][4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int t = start + 4 * lane + i;
          const bool reset = PACKED && t < L && sample_start(seq_idx, b, L, t);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
            v[hh][i] = t < L ? (reset ? kSampleStartLog
                                      : __bfloat162float(dt[(int64_t(b) * L + t) * H + 2 * pair + hh]) *
                                            Ah[hh])
                             : 0.0f;
        }
      };
      float dtv[2][4];
      load_dt(0, dtv);
      bool ok = true;
      int p = 0;
      for (int c = 0;; ++c) {
        const int slot = c & (kSlots - 1);
        PieceInfo* inf = info + slot;
        float lam[2][4], pmn[2][4], pmx[2][4];
        int ngood[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float run = 0.0f;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            run += dtv[hh][i];
            lam[hh][i] = run;
          }
          float incl = run;  // inclusive scan of the lanes' sums
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float nb = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += nb;
          }
          const float excl = incl - run;
          float lmn = 3.0e38f, lmx = -3.0e38f;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            lam[hh][i] += excl;
            lmn = fminf(lmn, lam[hh][i]);
            lmx = fmaxf(lmx, lam[hh][i]);
            pmn[hh][i] = lmn;
            pmx[hh][i] = lmx;
          }
          // min / max over the earlier lanes' tokens: exclusive warp scan
          float smn = lmn, smx = lmx;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float a2 = __shfl_up_sync(0xffffffffu, smn, o);
            const float c2 = __shfl_up_sync(0xffffffffu, smx, o);
            if (lane >= o) {
              smn = fminf(smn, a2);
              smx = fmaxf(smx, c2);
            }
          }
          float emn = __shfl_up_sync(0xffffffffu, smn, 1), emx = __shfl_up_sync(0xffffffffu, smx, 1);
          if (lane == 0) {
            emn = 3.0e38f;
            emx = -3.0e38f;
          }
          int cnt = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            pmn[hh][i] = fminf(pmn[hh][i], emn);
            pmx[hh][i] = fmaxf(pmx[hh][i], emx);
            const bool good = p + 4 * lane + i < L && (pmx[hh][i] - pmn[hh][i]) <= kFactorRange;
            cnt += __popc(__ballot_sync(0xffffffffu, good));
          }
          ngood[hh] = cnt;
        }
        const int n = max(1, min(ngood[0], ngood[1]));  // token 0 always qualifies while p < L
        const bool last = p + n >= L;
        float dtn[2][4];
        if (!last) load_dt(p + n, dtn);  // the next piece's dt, in flight during the publish
        if (ok && c >= kSlots) ok = ctl.wait(BAR_INFO_FREE + slot, uint32_t(((c / kSlots) - 1) & 1));
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          *reinterpret_cast<float4*>(&inf->lam[hh][4 * lane]) =
              make_float4(lam[hh][0], lam[hh][1], lam[hh][2], lam[hh][3]);
        // token n-1: lane (n-1) / 4, slot (n-1) % 4
        const int src = (n - 1) >> 2, idx = (n - 1) & 3;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float mn = pmn[hh][0], mx = pmx[hh][0], le = lam[hh][0];
#pragma unroll
          for (int i = 1; i < 4; ++i)
            if (idx == i) {
              mn = pmn[hh][i];
              mx = pmx[hh][i];
              le = lam[hh][i];
            }
          const float R = __shfl_sync(0xffffffffu, 0.5f * (mn + mx), src);
          const float lend = __shfl_sync(0xffffffffu, le, src);
          if (lane == 0) {
            inf->R[hh] = R;
            inf->lend[hh] = lend;
          }
        }
        if (lane == 0) {
          inf->start = p;
          inf->n = n;
          inf->last = last ? 1 : 0;
          // halo mask: bit j set when the conv of this piece may read position
          // p - (K-1) + j (the same packed sample as token p; positions before
          // the row carry token 0's id).  A piece never contains a sample start
          // after its first token, so only the halo can belong to another sample.
          int halo = 7;
          if (PACKED && seq_idx) {
            halo = 0;
            const int32_t me = seq_idx[int64_t(b) * L + p];
            for (int j = 0; j < kMaxK - 1; ++j) {
              const int pos = p - (kMaxK - 1) + j;
              const int32_t id = seq_idx[int64_t(b) * L + (pos < 0 ? 0 : pos)];
              if (id == me) halo |= 1 << j;
            }
          }
          inf->pad = halo;
        }
        __syncwarp();
        mbar_arrive(ctl.bar(BAR_INFO_FULL + slot));
        if (last) break;
        p += n;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int i = 0; i < 4; ++i) dtv[hh][i] = dtn[hh][i];
      }
    }
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
// The per-warpgroup register budgets assume the launch gives every thread
// kLaunchRegs registers; a build that gives another count is refused rather
// than launched (its setmaxnreg split would not add up).
template <typename F>
cudaError_t prepare_pair(F* kern) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != int(pr::kLaunchRegs)) return cudaErrorInvalidConfiguration;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(pr::kSmemBytes));
}

template <typename TX, typename TY, bool FUSED>
cudaError_t launch_pair(const void* x, const void* dt, const float* A, const void* B,
                        const void* C, const float* h0, float* hT, void* y, const float* w,
                        const float* bias, const void* s_in, void* s_out, int K, int64_t Bz,
                        int64_t L, int H, int G, int* status, const int32_t* seq_idx, cudaStream_t st,
                        bool dependent = false) {
  using namespace pr;
  CUtensorMap mB, mC, mX;
  if (!make_bc_map(&mB, B, Bz, L, G, kN) || !make_bc_map(&mC, C, Bz, L, G, kN))
    return cudaErrorInvalidValue;
  if (FUSED) {
    if (!make_x_map(&mX, x, Bz, L, int64_t(H) * kP, kXsRows)) return cudaErrorInvalidValue;
  } else {
    mX = mB;  // unused
  }
  // packed rows get their own instantiation: the ordinary one carries none of
  // their checks
  auto kern = seq_idx ? ssm_scan_pair_kernel<TX, TY, FUSED, true, false>
                      : ssm_scan_pair_kernel<TX, TY, FUSED, false, false>;
  cudaError_t e = prepare_pair(kern);
  if (e != cudaSuccess) return e;
  return launch_dep(kern, dim3(unsigned(Bz * (H / 2))), dim3(kThreads), kSmemBytes, st, dependent,
                    mB, mC, mX, static_cast<const TX*>(x), static_cast<const __nv_bfloat16*>(dt),
                    A, h0, hT, static_cast<TY*>(y), w, bias, static_cast<const TX*>(s_in),
                    static_cast<TX*>(s_out), K, int(L), H, G, status, seq_idx);
}
}  // namespace

// The pair kernel takes bf16 dt/B/C, P = 64, N = 128 and pairs of heads that
// share a B/C group.
bool ssm_scan_pair_supports(sss_dtype at, int64_t L, int H, int P, int N, int G) {
  return at == SSS_BF16 && P == pr::kP && N == pr::kN && L >= 1 && L < (int64_t(1) << 31) &&
         H >= 2 && G >= 1 && H % G == 0 && (H / G) % 2 == 0 && encode_fn() != nullptr;
}

// The state-only kernel (first pass of the span split): zero initial state,
// hT written, no y.  C is not read, so its tensor map is not encoded.
template <typename TX, bool FUSED>
cudaError_t launch_pair_state(const void* x, const void* dt, const float* A, const void* B,
                              float* hT, const float* w, const float* bias, const void* s_in,
                              int K, int64_t Bz, int64_t L, int H, int G, int* status,
                              cudaStream_t st, bool dependent) {
  using namespace pr;
  if (Bz * (H / 2) > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  CUtensorMap mB, mX;
  if (!make_bc_map(&mB, B, Bz, L, G, kN)) return cudaErrorInvalidValue;
  if (FUSED) {
    if (!make_x_map(&mX, x, Bz, L, int64_t(H) * kP, kXsRows)) return cudaErrorInvalidValue;
  } else {
    mX = mB;  // unused
  }
  auto kern = ssm_scan_pair_kernel<TX, __nv_bfloat16, FUSED, false, true>;
  cudaError_t e = prepare_pair(kern);
  if (e != cudaSuccess) return e;
  return launch_dep(kern, dim3(unsigned(Bz * (H / 2))), dim3(kThreads), kSmemBytes, st, dependent,
                    mB, mB, mX, static_cast<const TX*>(x), static_cast<const __nv_bfloat16*>(dt),
                    A, nullptr, hT, nullptr, w, bias, static_cast<const TX*>(s_in), nullptr, K,
                    int(L), H, G, status, nullptr);
}

cudaError_t ssm_scan_pair_state_launch(const void* x, sss_dtype xt, const void* dt,
                                       const float* A, const void* B, float* hT, int64_t Bz,
                                       int64_t L, int H, int G, int* status, cudaStream_t st) {
  if (xt == SSS_F32)
    return launch_pair_state<float, false>(x, dt, A, B, hT, nullptr, nullptr, nullptr, 1, Bz, L,
                                           H, G, status, st, true);
  return launch_pair_state<__nv_bfloat16, false>(x, dt, A, B, hT, nullptr, nullptr, nullptr, 1,
                                                 Bz, L, H, G, status, st, true);
}

cudaError_t mixer_fwd_pair_state_launch(const void* x, const float* w, const float* bias,
                                        const void* s_in, const void* dt, const float* A,
                                        const void* B, float* hT, int64_t Bz, int64_t L, int H,
                                        int G, int K, int* status, cudaStream_t st) {
  return launch_pair_state<__nv_bfloat16, true>(x, dt, A, B, hT, w, bias, s_in, K, Bz, L, H, G,
                                                status, st, true);
}

cudaError_t ssm_scan_pair_launch(const void* x, sss_dtype xt, const void* dt, const float* A,
                                 const void* B, const void* C, const float* h0, float* hT,
                                 void* y, sss_dtype yt, int64_t Bz, int64_t L, int H, int G,
                                 int* status, const int32_t* seq_idx, cudaStream_t st,
                                 bool dependent) {
  if (Bz * (H / 2) > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
#define SSS_PAIR(TXT, TYT)                                                                    \
  return launch_pair<TXT, TYT, false>(x, dt, A, B, C, h0, hT, y, nullptr, nullptr, nullptr,  \
                                      nullptr, 1, Bz, L, H, G, status, seq_idx, st, dependent);
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
                                  int K, int* status, const int32_t* seq_idx, cudaStream_t st,
                                  bool dependent) {
  if (Bz * (H / 2) > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (yt == SSS_BF16)
    return launch_pair<__nv_bfloat16, __nv_bfloat16, true>(x, dt, A, B, C, h0, hT, y, w, bias,
                                                           s_in, s_out, K, Bz, L, H, G, status,
                                                           seq_idx, st, dependent);
  return launch_pair<__nv_bfloat16, float, true>(x, dt, A, B, C, h0, hT, y, w, bias, s_in, s_out,
                                                 K, Bz, L, H, G, status, seq_idx, st, dependent);
}

}  // namespace sss
