// Decode attention over the low-bit dual-path MLA cache (QuantMLA page, abstract and appendix
// Figure 8; RAQ-MLA page, Figures 3-4 and appendix Table 5).
//
// Grid (B, H/16, n_q + n_split). CTA (b, hb, z) handles 16 heads of sequence b:
//   z <  n_q : a share of the protected tokens (t < S or t >= T-W) from the BF16 sink/recent
//              buffers (n_q > 1 only when there is little packed work);
//   z >= n_q : share z - n_q of the packed tokens [S, T-W), in tiles of 32 tokens streamed from
//              the page pool into a ring of shared-memory stages by bulk copies.
// Each CTA writes an unnormalized partial (O, max, sum); a second kernel merges the partials
// with a log-sum-exp reduction (one global softmax over all tokens).
//
// Packed tiles. Warp w owns latent group w (channels 128w..128w+127) and k_R chunk w
// (channels 16w..16w+15). Codes are never dequantized into a tile:
//   scores:  q . c_hat = scale_t * sum_i q_i code_ti + min_t * sum_i q_i  (per token group),
//   readout: sum_t p_t c_hat_t = sum_t (p_t scale_t) code_t + sum_t p_t min_t,
// both on tensor cores. The codes reach the products as FP16 subnormals: the bit pattern n
// (or 16n, 4^i n) of a 16-bit half is the exact value n * 2^-24 (times that power of two), so
// a single AND of a code word yields a ready operand. Matrix loads (ldmatrix) read 8x8 blocks
// of 16-bit elements straight from the staged token-major rows: plain for the score operand
// (token columns), transposed for the readout operand (token rows). The query is converted to
// FP16 with a per-head power-of-two prescale (exact for BF16 inputs) and permuted to match the
// channel order the masks produce. k_R uses its per-page channel scale folded into the query
// (split into two BF16 terms so the product stays accurate to ~2^-16).
//
// Within a CTA the four warps exchange partial scores through shared memory; the exchanges
// are skewed over mbarriers so that the scores of tile i+1 are computed while the softmax of
// tile i is still being published.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "kernels.cuh"
#include "ptx.cuh"

namespace mlaq {
namespace {

constexpr int kThreads = 128;
constexpr int kCtasPerSm = 3;  // resident CTAs per SM the register and shared budgets are sized for
constexpr int kPT = 32;        // tokens per packed tile
constexpr int kTile = 16;      // tokens per protected (BF16) tile
constexpr int kRowStride = 24;              // floats per head row in the BF16-path exchange
constexpr int kXStride = 40;                // floats per head row in the packed-path exchange
constexpr int kOutStride = 516;             // floats per head row when staging the partial output
constexpr int kBf16RowBytes = kRow * 2 + 16;  // padded BF16 row in shared memory (1168 B)
constexpr long long kWaitBudget = 4ll << 30;  // ~2 s at 2 GHz before a wait gives up
constexpr int kMaxSplitPages = 512;          // page ids of a split cached in shared memory
constexpr float kRescaleSlack = 8.f;          // softmax weights stay <= 2^8 between rescales
constexpr float kStrictScale = 255.f;         // a token scale >= this forces weights <= 1 (FP16 safety)

__host__ __device__ constexpr int cmax(int a, int b) { return a > b ? a : b; }

// Shared-memory stage of one packed tile: latent rows, k_R code blocks, latent metadata, k_R
// metadata (the page layout's regions A-D restricted to the tile's 32 tokens).
template <int BITS>
struct Geom {
  static constexpr int kRowBytes = 64 * BITS;
  static constexpr int kLat = kPT * kRowBytes;
  static constexpr int kRopeOff = kLat;             // 2 blocks of 16 tokens x 4 chunks x 128 B
  static constexpr int kMetaOff = kLat + 1024;      // 32 tokens x 4 groups x (scale, min)
  static constexpr int kRMetaOff = kMetaOff + 512;  // 64 channels x (scale, min)
  static constexpr int kStage = kRMetaOff + 256;
  static constexpr int kStages = 4;  // a power of two: stage index and phase are shifts
  static constexpr int kRegion =
      cmax(cmax(kStages * kStage, 2 * kTile * kBf16RowBytes), 16 * kOutStride * 4);
};

constexpr int kXsFloats = 2 * 4 * 16 * kXStride;  // partial scores [2 buf][4 warps][16 heads][32 tok]
constexpr int kXpFloats = 2 * 16 * kXStride;      // weights [2 buf][16 heads][32 tok]
constexpr int kNumBars = 12;                       // >= stages + 4 exchange barriers + query barrier
// Packed CTAs fetch the 16 query rows of their head block with bulk copies into the (still idle)
// partial-score buffer: latent rows padded to kQRowBytes (each 8-lane phase of the prologue's
// 16-byte reads covers 32 distinct banks), then the 16 k_R rows; completion on barrier kQueryBar.
constexpr int kQRowBytes = kLatent * 2 + 64;
constexpr int kQRopeOff = 16 * kQRowBytes;
constexpr int kQBytes = 16 * kLatent * 2 + 16 * kRope * 2;  // bytes the copies deliver
constexpr int kQueryBar = 8;
static_assert(kQRopeOff + 16 * kRope * 2 <= kXsFloats * 4, "query rows fit the partial-score buffer");

template <int BITS>
__host__ __device__ constexpr int smem_bytes() {
  return Geom<BITS>::kRegion + (kXsFloats + kXpFloats + 2 * 16 + 4 * 16) * 4 + kNumBars * 8 +
         (2 * 4 + 2 * 4 + 4) * 4 + kMaxSplitPages * 4 + kThreads * 8 * 4;
}
// kCtasPerSm CTAs (each with 1 KB reserved by the hardware) fit in an SM's 228 KB
static_assert(kCtasPerSm * (smem_bytes<4>() + 1024) <= 228 * 1024 &&
                  kCtasPerSm * (smem_bytes<2>() + 1024) <= 228 * 1024, "shared memory per SM");
static_assert(Geom<4>::kStages + 4 <= kQueryBar && Geom<2>::kStages + 4 <= kQueryBar && kQueryBar < kNumBars, "barriers");
template <int BITS>
constexpr int xflags_offset() {
  return Geom<BITS>::kRegion + (kXsFloats + kXpFloats + 2 * 16 + 4 * 16) * 4 + kNumBars * 8;
}
static_assert(xflags_offset<4>() % 16 == 0 && xflags_offset<2>() % 16 == 0, "vector loads of the exchange flags");
template <int BITS>
constexpr int qr_offset() {
  return xflags_offset<BITS>() + (2 * 4 + 2 * 4 + 4) * 4 + kMaxSplitPages * 4;
}
static_assert(qr_offset<4>() % 16 == 0 && qr_offset<2>() % 16 == 0, "vector access of the k_R query slice");
static_assert(qr_offset<4>() + kThreads * 8 * 4 == smem_bytes<4>() && qr_offset<2>() + kThreads * 8 * 4 == smem_bytes<2>(),
              "shared-memory carve");
static_assert(2 * 4 * 16 * kRowStride <= kXsFloats && 2 * 16 * kRowStride <= kXpFloats, "BF16 exchange");

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ float half_lo(uint32_t w) { return __low2float(*reinterpret_cast<const __half2*>(&w)); }
__device__ __forceinline__ float half_hi(uint32_t w) { return __high2float(*reinterpret_cast<const __half2*>(&w)); }
// 2^k as a float, k in [-126, 127]
// 2^x, relative error below 2^-22 (hardware approximation; subnormal results flush to zero)
__device__ __forceinline__ float exp2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct Shared {
  uint8_t* stages;  // packed stages, or BF16 row stages, or the output staging tile
  float* sbuf;      // packed: [2][4 warps][16 heads][kXStride]; BF16 path: [2][4][16][kRowStride]
  float* pbuf;      // packed: [2][16 heads][kXStride]; BF16 path: [2][16][kRowStride]
  float* alpha;     // [2][16]
  float* qmax;      // [4 warps][16 heads]: per-warp query maxima (prologue)
  uint64_t* bars;   // packed: stages full [kStages], scores ready [2], weights ready [2] (every thread arrives)
  int* xflags;      // [2][4] per warp and tile (16-byte aligned): bit 0 strict (a token scale >= kStrictScale), bit 1 timeout
  int* moved;       // [2][4] per warp and tile: a reference max moved (rescale the outputs)
  int* strict;      // [2] BF16 path: per exchange buffer (+2 padding)
  int* pids;        // [kMaxSplitPages] physical page ids of the split's pages (packed path)
  float* qr;        // [kThreads][8] k_R query slice of each thread (read when the page changes)
};

template <int BITS>
__device__ __forceinline__ Shared carve(uint8_t* smem) {
  Shared s;
  s.stages = smem;
  s.sbuf = reinterpret_cast<float*>(smem + Geom<BITS>::kRegion);
  s.pbuf = s.sbuf + kXsFloats;
  s.alpha = s.pbuf + kXpFloats;
  s.qmax = s.alpha + 2 * 16;
  s.bars = reinterpret_cast<uint64_t*>(s.qmax + 4 * 16);
  s.xflags = reinterpret_cast<int*>(s.bars + kNumBars);
  s.moved = s.xflags + 2 * 4;
  s.strict = s.moved + 2 * 4;
  s.pids = s.strict + 4;  // strict padded to 16 bytes: pids and qr stay 16-byte aligned
  s.qr = reinterpret_cast<float*>(s.pids + kMaxSplitPages);
  return s;
}

// Per-thread state shared by both token paths.
struct State {
  float o[16][4];  // readout accumulators: 16 blocks of 8 channels, C fragment
  float mterm[2];  // sum_t p_t * min_t for rows g, g+8 (packed path only)
  float m_run;     // reference max of head 4*warp + lane/8 (log2 units), shared by its 8 lanes
  float l_part;    // this lane's share of the running sum (reduced over the 8 lanes at the end)
};

// First half of the exchange: publish this warp's partial scores (first CTA barrier). Returns
// true if any thread saw a timeout. sh.strict[buf] (a CTA-wide flag for this sub-tile, read in
// the second half) forces an exact running max so that every weight stays <= 1.
//
// Lazy rescaling: the reference max of a head moves only when a tile exceeds it by more than
// kRescaleSlack (log2 units), so the weights stay <= 2^kRescaleSlack, the accumulators are
// rescaled rarely and the common path needs no cross-lane reduction. The result does not
// depend on the reference (it cancels in O / l and is accounted for in the LSE).
__device__ __forceinline__ bool exchange_partials(const Shared& sh, int buf, const float (&part)[2][4],
                                                  bool timed_out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  float* my = sh.sbuf + (buf * 4 + warp) * 16 * kRowStride;
#pragma unroll
  for (int nb = 0; nb < 2; ++nb) {
    *reinterpret_cast<float2*>(my + g * kRowStride + 8 * nb + 2 * q) = make_float2(part[nb][0], part[nb][1]);
    *reinterpret_cast<float2*>(my + (g + 8) * kRowStride + 8 * nb + 2 * q) = make_float2(part[nb][2], part[nb][3]);
  }
  return __syncthreads_or(timed_out) != 0;
}

// Second half: the online softmax of 4 heads per warp over the summed partials, P published
// for all warps (second CTA barrier), accumulators rescaled if some reference max moved.
__device__ __forceinline__ void softmax_publish(const Shared& sh, int buf, int t0, int lo, int hi, float scale_log2,
                                                State& st) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2;
  const bool strict = sh.strict[buf] != 0;

  const int hh = 4 * warp + (lane >> 3), tt = 2 * (lane & 7);
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float2 v = *reinterpret_cast<const float2*>(sh.sbuf + ((buf * 4 + w) * 16 + hh) * kRowStride + tt);
    s0 += v.x;
    s1 += v.y;
  }
  const bool v0 = (t0 + tt >= lo) && (t0 + tt < hi);
  const bool v1 = (t0 + tt + 1 >= lo) && (t0 + tt + 1 < hi);
  s0 = v0 ? s0 * scale_log2 : -INFINITY;
  s1 = v1 ? s1 * scale_log2 : -INFINITY;
  const float lmax = fmaxf(s0, s1);
  const float slack = strict ? 0.f : kRescaleSlack;
  const bool need = lmax > st.m_run + slack || (st.m_run == -INFINITY && lmax > -INFINITY);
  float alpha = 1.f;
  const bool moved = __any_sync(0xffffffffu, need);
  if (moved) {  // rare: some head of this warp needs a new reference max
    float tmax = lmax;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
    if (tmax > st.m_run + slack || (st.m_run == -INFINITY && tmax > -INFINITY)) {
      alpha = exp2f(st.m_run - tmax);  // 0 when the old reference was -inf
      st.l_part *= alpha;
      st.m_run = tmax;
    }
  }
  float p0 = 0.f, p1 = 0.f;
  if (st.m_run != -INFINITY) {
    p0 = v0 ? exp2f(s0 - st.m_run) : 0.f;
    p1 = v1 ? exp2f(s1 - st.m_run) : 0.f;
  }
  st.l_part += p0 + p1;
  *reinterpret_cast<float2*>(sh.pbuf + (buf * 16 + hh) * kRowStride + tt) = make_float2(p0, p1);
  if ((lane & 7) == 0) sh.alpha[buf * 16 + hh] = alpha;
  const bool any_rescale = __syncthreads_or(moved);
  if (threadIdx.x == 0) sh.strict[buf] = 0;  // consumed; the next use of this buffer sets it afresh

  if (any_rescale) {
    const float a0 = sh.alpha[buf * 16 + g], a1 = sh.alpha[buf * 16 + g + 8];
#pragma unroll
    for (int cb = 0; cb < 16; ++cb) {
      st.o[cb][0] *= a0;
      st.o[cb][1] *= a0;
      st.o[cb][2] *= a1;
      st.o[cb][3] *= a1;
    }
    st.mterm[0] *= a0;
    st.mterm[1] *= a1;
  }
}

// P fragment (rows g, g+8; tokens 2q,2q+1 and 2q+8,2q+9) from the published P.
__device__ __forceinline__ void load_p(const Shared& sh, int buf, float2 (&pf)[4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const float* pb = sh.pbuf + buf * 16 * kRowStride;
  pf[0] = *reinterpret_cast<const float2*>(pb + g * kRowStride + 2 * q);
  pf[1] = *reinterpret_cast<const float2*>(pb + (g + 8) * kRowStride + 2 * q);
  pf[2] = *reinterpret_cast<const float2*>(pb + g * kRowStride + 8 + 2 * q);
  pf[3] = *reinterpret_cast<const float2*>(pb + (g + 8) * kRowStride + 8 + 2 * q);
}

// ------------------------------------------------------------------ protected (BF16) tokens
// kPaged: every token of the sequence from a paged BF16 cache (the unquantized comparator);
// else the sink and recent tokens from the BF16 retention buffers.
template <bool kPaged>
__device__ void bf16_split(const DecodeParams& p, const Shared& sh, int b, int T, int T_old, int part,
                           const uint32_t (&qa)[8][4], const uint32_t (&qra)[4], State& st, int32_t& flags) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Several new tokens per sequence: the CTA's rows belong to position i of the q_len tokens and
  // see the prefix [0, T_vis), T_vis = T - (q_len - 1 - i); which copy a token is read from
  // follows the cache length T (the recent window is [T - W, T)).
  const int T_vis = (kPaged || p.q_len <= 1) ? T : T - (p.q_len - 1 - static_cast<int>(blockIdx.y) * 16 / p.h_pos);
  const int s_end = kPaged ? 0 : max(0, min(p.S, T_vis));
  const int r_beg = kPaged ? 0 : max(T - p.W, s_end);
  const int has_sink = s_end > 0 ? 1 : 0;
  const int n_all = has_sink + max(0, T_vis - r_beg + kTile - 1) / kTile;
  // this CTA's share of the sequence's protected tiles: [t_lo, t_lo + n_tiles)
  // (64-bit products only for the paged comparator, whose tables reach millions of tokens)
  const int t_lo = kPaged ? static_cast<int>((static_cast<long long>(n_all) * part) / p.n_q) : (n_all * part) / p.n_q;
  const int n_tiles =
      (kPaged ? static_cast<int>((static_cast<long long>(n_all) * (part + 1)) / p.n_q) : (n_all * (part + 1)) / p.n_q) -
      t_lo;
  if (n_tiles <= 0) return;
  constexpr int kStageBytes = kTile * kBf16RowBytes;
  if constexpr (kPaged) {  // validate the share's page ids before any copy reads through them
    bool bad = false;
    const int pg_lo = (t_lo * kTile) >> p.p_shift, pg_hi = (min(T, (t_lo + n_tiles) * kTile) - 1) >> p.p_shift;
    for (int pg = pg_lo + static_cast<int>(threadIdx.x); pg <= pg_hi; pg += kThreads) {
      const int32_t pid = __ldg(p.page_table + static_cast<size_t>(b) * p.max_pages + pg);
      bad |= pid < 0 || pid >= p.n_pages;
    }
    if (__syncthreads_or(bad)) {
      flags |= kErrBadPage;
      return;
    }
  }

  auto tile_range = [&](int li, int& start, int& count) {  // li: index in this CTA's share
    const int i = t_lo + li;
    if (has_sink && i == 0) {
      start = 0;
      count = s_end;
    } else {
      start = r_beg + (i - has_sink) * kTile;
      count = min(kTile, T_vis - start);
    }
  };
  auto row_ptr = [&](int t) -> const uint16_t* {
    if constexpr (kPaged) {
      const int32_t pid = __ldg(p.page_table + static_cast<size_t>(b) * p.max_pages + (t >> p.p_shift));
      return p.kv_bf16 + (static_cast<size_t>(pid) * p.P + (t & (p.P - 1))) * kRow;
    } else {
      return t < p.S ? p.sink + (static_cast<size_t>(b) * p.S + t) * kRow
                     : p.ring + (static_cast<size_t>(b) * p.W + (t % p.W)) * kRow;
    }
  };
  // Warp 0 stages tile i: lane 0 announces the stage's bytes, then lanes 0-15 each copy one row
  // (its address lookup and copy run in parallel rather than one after another).
  auto issue = [&](int i) {
    int start, count;
    tile_range(i, start, count);
    uint8_t* dst = sh.stages + (i & 1) * kStageBytes;
    uint64_t* bar = sh.bars + (i & 1);
    if (lane == 0) mbar_arrive_expect_tx(bar, kTile * kRow * 2);
    __syncwarp();
    // lanes 0-15: row `lane` from the cache; lanes 16-31: row `lane - 16` when it is pending (its
    // latent and k_R parts from the write's inputs)
    const int j = lane & (kTile - 1);
    const int t = start + (j < count ? j : 0);  // rows past the count repeat a valid row (masked later)
    const bool pend = !kPaged && t >= T_old;
    if (lane < kTile) {
      if (!pend) bulk_g2s(dst + j * kBf16RowBytes, row_ptr(t), kRow * 2, bar);
    } else if (pend) {
      const size_t r = static_cast<size_t>(__ldg(p.cu_new + b)) + static_cast<size_t>(t - T_old);
      bulk_g2s(dst + j * kBf16RowBytes, p.c_new + r * kLatent, kLatent * 2, bar);
      bulk_g2s(dst + j * kBf16RowBytes + kLatent * 2, p.kr_new + r * kRope, kRope * 2, bar);
    }
  };
  if (warp == 0) {
    issue(0);
    if (n_tiles > 1) issue(1);
  }
  for (int i = 0; i < n_tiles; ++i) {
    int start, count;
    tile_range(i, start, count);
    const bool ok = mbar_wait_bounded(sh.bars + (i & 1), (i >> 1) & 1, kWaitBudget);
    const uint8_t* sp = sh.stages + (i & 1) * kStageBytes;
    const int mi = lane >> 3, ri = lane & 7;

    float acc[2][4], racc[2][4];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[nb][e] = racc[nb][e] = 0.f;
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) {
      uint32_t r[4];
      ldsm_x4(r, sp + (8 * (mi >> 1) + ri) * kBf16RowBytes + (128 * warp + 16 * kc + 8 * (mi & 1)) * 2);
      mma_bf16_16816(acc[0], qa[kc], r[0], r[1]);
      mma_bf16_16816(acc[1], qa[kc], r[2], r[3]);
    }
    {
      uint32_t r[4];
      ldsm_x4(r, sp + (8 * (mi >> 1) + ri) * kBf16RowBytes + (kLatent + 16 * warp + 8 * (mi & 1)) * 2);
      mma_bf16_16816(racc[0], qra, r[0], r[1]);
      mma_bf16_16816(racc[1], qra, r[2], r[3]);
    }
    float part[2][4];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) part[nb][e] = acc[nb][e] + racc[nb][e];

    const int buf = i & 1;
    // positions are relative to the tile start: valid rows are [0, count)
    if (exchange_partials(sh, buf, part, !ok)) {
      flags |= kErrTimeout;
      if (threadIdx.x == 0)
        for (int j = i; j < min(i + 2, n_tiles); ++j)
          (void)mbar_wait_bounded(sh.bars + (j & 1), (j >> 1) & 1, kWaitBudget >> 4);
      break;
    }
    softmax_publish(sh, buf, 0, 0, count, p.scale_log2, st);
    float2 pf[4];
    load_p(sh, buf, pf);
    uint32_t ah[4], al[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float xh0 = __bfloat162float(__float2bfloat16_rn(pf[e].x));
      const float xh1 = __bfloat162float(__float2bfloat16_rn(pf[e].y));
      ah[e] = pack_bf16x2(xh0, xh1);
      al[e] = pack_bf16x2(pf[e].x - xh0, pf[e].y - xh1);
    }
    // fragment order: a0 (g, 2q..), a1 (g+8, 2q..), a2 (g, 2q+8..), a3 (g+8, 2q+8..)
    const uint32_t A_hi[4] = {ah[0], ah[1], ah[2], ah[3]};
    const uint32_t A_lo[4] = {al[0], al[1], al[2], al[3]};
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) {
      uint32_t r[4];
      ldsm_x4_t(r, sp + (8 * (mi & 1) + ri) * kBf16RowBytes + (128 * warp + 16 * kc + 8 * (mi >> 1)) * 2);
      mma_bf16_16816(st.o[2 * kc], A_hi, r[0], r[1]);
      mma_bf16_16816(st.o[2 * kc], A_lo, r[0], r[1]);
      mma_bf16_16816(st.o[2 * kc + 1], A_hi, r[2], r[3]);
      mma_bf16_16816(st.o[2 * kc + 1], A_lo, r[2], r[3]);
    }
    __syncthreads();  // every warp is done with this stage before it is refilled
    if (warp == 0 && i + 2 < n_tiles) {
      fence_proxy_async_smem();
      issue(i + 2);
    }
  }
}

// ------------------------------------------------------------------ packed tokens
// A matrix load of one 16-byte chunk per token gives lane (g, q) the 16-bit elements 2q, 2q+1
// of token g (score side) or elements g of tokens 2q, 2q+1 (transposed, readout side). An
// INT4 element holds 4 channels (nibble s), an INT2 element 8 channels (field i). Masking one
// nibble/field position of both halves of a register gives an FP16 operand pair whose values
// are code * 2^-24 * 2^lw; lw = 4s-style weights are folded into the query (scores) and into
// the output scale (readout).

// Channel (within the warp's 128-channel group) of query slot sigma of k-chunk kc, where the
// slots of lane q are the fragment's k indices 2q, 2q+1, 2q+8, 2q+9.
template <int BITS>
__device__ __forceinline__ int slot_channel(int kc, int sigma, int q) {
  if constexpr (BITS == 4) {
    // k-chunk 2m + s: mask position s of the words of chunk m (channels 32m + 8q + 0..7);
    // the pair (low, high half) of position s is (8q + s, 8q + 4 + s), the shifted word gives
    // (8q + 2 + s, 8q + 6 + s)
    const int off = sigma == 0 ? 0 : sigma == 1 ? 4 : sigma == 2 ? 2 : 6;
    return 32 * (kc >> 1) + 8 * q + (kc & 1) + off;
  } else {
    // k-chunk 4m + j: fields 2j, 2j+1 of the words of chunk m (channels 64m + 16q + 0..15);
    // field i of the (low, high) half is channel (16q + i, 16q + 8 + i)
    const int i = 2 * (kc & 3) + (sigma >> 1);
    return 64 * (kc >> 2) + 16 * q + 8 * (sigma & 1) + i;
  }
}
// log2 of the weight the mask leaves on slot sigma of k-chunk kc (equal for both halves of
// a register).
template <int BITS>
__device__ __forceinline__ int slot_log2w(int kc, int sigma) {
  if constexpr (BITS == 4) {
    return 4 * (kc & 1);
  } else {
    const int i = 2 * (kc & 3) + (sigma >> 1);
    return 2 * (i <= 4 ? i : i - 5);  // fields 5..7 are masked after a 10-bit shift
  }
}
// Readout block cb, column n: output channel within the group and log2 weight.
template <int BITS>
__device__ __forceinline__ int out_channel(int cb, int n) {
  if constexpr (BITS == 4) return 32 * (cb >> 2) + 4 * n + (cb & 3);
  else return 64 * (cb >> 3) + 8 * n + (cb & 7);
}
template <int BITS>
__host__ __device__ constexpr int out_log2w(int cb) {
  return BITS == 4 ? 4 * (cb & 1) : 2 * ((cb & 7) <= 4 ? (cb & 7) : (cb & 7) - 5);
}

// The same rows for a query that is not 16-byte aligned, element by element by every thread (kept
// out of line: the rare path does not weigh on the kernel's register allocation).
__device__ __noinline__ void copy_query(const DecodeParams& p, const Shared& sh, int b, int h0) {
  uint16_t* rows = reinterpret_cast<uint16_t*>(sh.sbuf);
  const uint16_t* ql = p.q_lat + (static_cast<size_t>(b) * p.H + h0) * kLatent;
  const uint16_t* qk = p.q_rope + (static_cast<size_t>(b) * p.H + h0) * kRope;
  for (int e = threadIdx.x; e < 16 * kLatent; e += kThreads)
    rows[(e / kLatent) * (kQRowBytes / 2) + e % kLatent] = __ldg(ql + e);
  for (int e = threadIdx.x; e < 16 * kRope; e += kThreads) rows[kQRopeOff / 2 + e] = __ldg(qk + e);
}

// The prologue's BF16 query words from the bulk-copied rows: lane (g, q) of warp w gets the pairs
// of channels slot_channel(kc, 2j, q), slot_channel(kc, 2j + 1, q) of rows g (qa[kc][2j]) and
// g + 8 (qa[kc][2j + 1]) from one 16-byte read per row and channel octet (INT4: the octet
// 32m + 8q .. + 7 serves k-chunks 2m and 2m + 1; INT2: two octets 64m + 16q .. + 15 serve
// k-chunks 4m .. 4m + 3), and the k_R words of rows g, g + 8 at dims 16w + 2q and 16w + 2q + 8.
template <int BITS>
__device__ __forceinline__ void load_query_smem(const uint8_t* rows, int warp, int g, int q, uint32_t (&qa)[8][4],
                                                uint32_t (&qrw)[4]) {
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const uint8_t* row = rows + (g + 8 * r) * kQRowBytes + 2 * 128 * warp;
    if constexpr (BITS == 4) {
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + 2 * (32 * m + 8 * q));
        qa[2 * m][r] = __byte_perm(v.x, v.z, 0x5410);          // channels +0, +4
        qa[2 * m][2 + r] = __byte_perm(v.y, v.w, 0x5410);      // +2, +6
        qa[2 * m + 1][r] = __byte_perm(v.x, v.z, 0x7632);      // +1, +5
        qa[2 * m + 1][2 + r] = __byte_perm(v.y, v.w, 0x7632);  // +3, +7
      }
    } else {
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const uint4 a = *reinterpret_cast<const uint4*>(row + 2 * (64 * m + 16 * q));
        const uint4 c = *reinterpret_cast<const uint4*>(row + 2 * (64 * m + 16 * q + 8));
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          qa[4 * m + t][r] = __byte_perm(aw[t], cw[t], 0x5410);      // channels 2t, 8 + 2t
          qa[4 * m + t][2 + r] = __byte_perm(aw[t], cw[t], 0x7632);  // 2t + 1, 9 + 2t
        }
      }
    }
  }
  const uint8_t* kr = rows + kQRopeOff + g * (kRope * 2) + 2 * (16 * warp + 2 * q);
  qrw[0] = *reinterpret_cast<const uint32_t*>(kr);
  qrw[1] = *reinterpret_cast<const uint32_t*>(kr + 8 * kRope * 2);
  qrw[2] = *reinterpret_cast<const uint32_t*>(kr + 16);
  qrw[3] = *reinterpret_cast<const uint32_t*>(kr + 8 * kRope * 2 + 16);
}

// Packed CTAs bulk-copy the query when both query pointers are 16-byte aligned.
__device__ __forceinline__ bool query_bulk(const DecodeParams& p) {
  return ((reinterpret_cast<uintptr_t>(p.q_lat) | reinterpret_cast<uintptr_t>(p.q_rope)) & 15u) == 0;
}

// Thread 0 of a packed CTA, first thing in the kernel: the head block's 16 latent query rows and
// 16 k_R query rows into the partial-score buffer by bulk copies (one per latent row, one for the
// k_R rows), so that their round trip overlaps the sequence-length and page-table reads. Needs
// 16-byte aligned query pointers (the rows of a block are then aligned too).
__device__ __forceinline__ void fetch_query(const DecodeParams& p, const Shared& sh, int b, int h0) {
  uint64_t* bar = sh.bars + kQueryBar;
  mbar_init(bar, 1);
  fence_mbar_init();
  fence_proxy_async_smem();
  mbar_arrive_expect_tx(bar, kQBytes);
  uint8_t* dst = reinterpret_cast<uint8_t*>(sh.sbuf);
  const uint16_t* src = p.q_lat + (static_cast<size_t>(b) * p.H + h0) * kLatent;
  for (int r = 0; r < 16; ++r) bulk_g2s(dst + r * kQRowBytes, src + r * kLatent, kLatent * 2, bar);
  bulk_g2s(dst + kQRopeOff, p.q_rope + (static_cast<size_t>(b) * p.H + h0) * kRope, 16 * kRope * 2, bar);
}

template <int BITS, bool kBalanced>
__device__ void packed_split(const DecodeParams& p, const Shared& sh, int b, int T, int split, State& st,
                             int32_t& flags) {
  const bool q_bulk = query_bulk(p);
  using G = Geom<BITS>;
  constexpr int kS = G::kStages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int h0 = blockIdx.y * 16;
  const int lo = p.S, hi = T - p.W;
  // Equal shares sized for one balanced wave over the whole batch: every packed CTA sums the
  // packed tiles of all sequences (one length per thread) and takes shares of
  // ceil(total x head blocks / slots) tiles, never fewer than an even split of the longest
  // table over the launched shares; shares beyond a sequence's end are empty.
  int share = 0;
  if constexpr (kBalanced) {
    long long sum = 0;
    const long long t_max = static_cast<long long>(p.max_pages) * p.P;
    for (int bb = threadIdx.x; bb < p.B; bb += kThreads) {
      long long Tb = __ldg(p.seq_lens + bb);
      if (Tb < 0 || Tb > t_max) Tb = 0;
      const long long l2 = p.S, h2 = Tb - p.W;
      if (h2 > l2) sum += (h2 - 1) / kPT - l2 / kPT + 1;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    long long* red = reinterpret_cast<long long*>(sh.qmax);
    if (lane == 0) red[warp] = sum;
    __syncthreads();
    sum = red[0] + red[1] + red[2] + red[3];
    __syncthreads();  // the scratch is reused below
    const long long units = sum * (p.H / 16);
    const long long by_sum = (units + p.share_slots - 1) / p.share_slots;
    const long long max_sub = (static_cast<long long>(p.max_pages) * p.P + kPT - 1) / kPT;
    const long long floor_share = (max_sub + p.n_split - 1) / p.n_split;
    share = static_cast<int>(by_sum > floor_share ? by_sum : floor_share);
  }
  int tile_begin = 0, n_my = 0;
  if (hi > lo) {
    const int first = lo / kPT, last = (hi - 1) / kPT;
    if (share > 0) {
      const long long b0 = first + static_cast<long long>(split) * share;
      const long long e0 = b0 + share < last + 1 ? b0 + share : last + 1;
      if (e0 > b0) {
        tile_begin = static_cast<int>(b0);
        n_my = static_cast<int>(e0 - b0);
      }
    } else {  // one wave: an even slice of this sequence's tiles
      const int n_total = last - first + 1;
      tile_begin = first + static_cast<int>((static_cast<long long>(n_total) * split) / p.n_split);
      const int tile_end = first + static_cast<int>((static_cast<long long>(n_total) * (split + 1)) / p.n_split);
      n_my = tile_end - tile_begin;
    }
  }
  // A table of at most kMaxSplitPages pages was copied whole into sh.pids at the kernel's start
  // (before the length was known): ids by page index. A longer one: the split's ids from here on,
  // by index relative to its first page.
  const bool whole_table = p.max_pages <= kMaxSplitPages;
  if (n_my == 0) {  // empty share (a short sequence): the merge sees sum 0 and skips it
    if (q_bulk && !mbar_wait_bounded(sh.bars + kQueryBar, 0, kWaitBudget)) flags |= kErrTimeout;  // copies landed
    if (whole_table) cp_async_wait_all();
    return;
  }
  const int pg0 = (tile_begin * kPT) >> p.p_shift;
  const int pid_base = whole_table ? 0 : pg0;  // sh.pids[pg - pid_base] holds page pg's id
  // validate the page ids this split reads; a bad id drops the split's work
  {
    bool bad = false;
    const int pg1 = n_my > 0 ? (((tile_begin + n_my) * kPT - 1) >> p.p_shift) : pg0 - 1;
    if (whole_table) {
      cp_async_wait_all();
      __syncthreads();
    }
    for (int pg = pg0 + static_cast<int>(threadIdx.x); pg <= pg1; pg += kThreads) {
      const int32_t pid = whole_table ? sh.pids[pg] : __ldg(p.page_table + static_cast<size_t>(b) * p.max_pages + pg);
      bad |= pid < 0 || pid >= p.n_pages;
      if (!whole_table && pg - pg0 < kMaxSplitPages) sh.pids[pg - pg0] = pid;  // the copies read ids from here
    }
    if (__syncthreads_or(bad)) {
      flags |= kErrBadPage;
      n_my = 0;
    }
  }

  // Tile i (local index) is one stage: four bulk copies completing on the stage's barrier.
  auto issue = [&](int i) {
    const int t0 = (tile_begin + i) * kPT;
    const int pg = t0 >> p.p_shift, tp0 = t0 & (p.P - 1);
    const int32_t pid = pg - pid_base < kMaxSplitPages ? sh.pids[pg - pid_base]
                                                       : __ldg(p.page_table + static_cast<size_t>(b) * p.max_pages + pg);
    const uint8_t* base = p.pool + static_cast<size_t>(pid) * static_cast<size_t>(p.page_bytes);
    uint8_t* dst = sh.stages + (i % kS) * G::kStage;
    uint64_t* bar = sh.bars + (i % kS);
    const size_t P = static_cast<size_t>(p.P);
    mbar_arrive_expect_tx(bar, G::kStage);
    bulk_g2s(dst, base + static_cast<size_t>(tp0) * G::kRowBytes, G::kLat, bar);
    bulk_g2s(dst + G::kRopeOff, base + P * G::kRowBytes + static_cast<size_t>(tp0 / 16) * 512, 1024, bar);
    bulk_g2s(dst + G::kMetaOff, base + P * (G::kRowBytes + 32) + static_cast<size_t>(tp0) * 16, 512, bar);
    bulk_g2s(dst + G::kRMetaOff, base + P * (G::kRowBytes + 48), 256, bar);
  };
  if (threadIdx.x == 0)
    for (int i = 0; i < kS && i < n_my; ++i) issue(i);
  int issued = n_my < kS ? n_my : kS;  // identical in every thread

  // ---- query operands: FP16 with a per-head power-of-two prescale, in the masks' channel order
  // (BF16 words first, from the rows in the partial-score buffer, which the kernel's start
  // bulk-copies there or, for a query that is not 16-byte aligned, stores element by element;
  // qrw: the k_R slice, rows g, g+8, dims 16w + {2q, 2q+1} and 16w + {2q+8, 2q+9})
  uint32_t qa[8][4], qrw[4];
  if (q_bulk) {
    if (!mbar_wait_bounded(sh.bars + kQueryBar, 0, kWaitBudget)) {
      flags |= kErrTimeout;
      (void)mbar_wait_bounded(sh.bars + kQueryBar, 0, kWaitBudget >> 4);
    }
  }
  load_query_smem<BITS>(reinterpret_cast<const uint8_t*>(sh.sbuf), warp, g, q, qa, qrw);
  float qsum[2] = {0.f, 0.f}, inv_f[2], head_scale;  // inv_f: prologue only
  {
    float mx0 = 0.f, mx1 = 0.f;
#pragma unroll
    for (int kc = 0; kc < 8; ++kc)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t v0 = qa[kc][2 * j];      // a0 / a2: row g
        const uint32_t v1 = qa[kc][2 * j + 1];  // a1 / a3: row g + 8
        qsum[0] += bf16_lo(v0) + bf16_hi(v0);
        qsum[1] += bf16_lo(v1) + bf16_hi(v1);
        mx0 = fmaxf(mx0, fmaxf(fabsf(bf16_lo(v0)), fabsf(bf16_hi(v0))));
        mx1 = fmaxf(mx1, fmaxf(fabsf(bf16_lo(v1)), fabsf(bf16_hi(v1))));
      }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      qsum[0] += __shfl_xor_sync(0xffffffffu, qsum[0], o);
      qsum[1] += __shfl_xor_sync(0xffffffffu, qsum[1], o);
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    if (q == 0) {
      sh.qmax[warp * 16 + g] = mx0;
      sh.qmax[warp * 16 + g + 8] = mx1;
    }
    __syncthreads();
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      mx0 = fmaxf(mx0, sh.qmax[w * 16 + g]);
      mx1 = fmaxf(mx1, sh.qmax[w * 16 + g + 8]);
    }
    bool range = false;
    const int E0 = prescale_exponent(mx0, range), E1 = prescale_exponent(mx1, range);
    if (range) flags |= kErrRange;
    // Partial scores are kept in units of 2^(24 - E) (the latent products' natural scale);
    // the softmax lane of head 4w + lane/8 multiplies the sum back by that head's factor.
    inv_f[0] = pow2_int(E0 - 24);
    inv_f[1] = pow2_int(E1 - 24);
    qsum[0] *= inv_f[0];
    qsum[1] *= inv_f[1];
    {
      const int hh = 4 * warp + (lane >> 3);
      float mh = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) mh = fmaxf(mh, sh.qmax[w * 16 + hh]);
      bool r2 = false;
      head_scale = p.scale_log2 * pow2_int(24 - prescale_exponent(mh, r2));
    }
#pragma unroll
    for (int kc = 0; kc < 8; ++kc)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int lw = slot_log2w<BITS>(kc, 2 * j);
        const float s0 = pow2_int(E0 - lw), s1 = pow2_int(E1 - lw);
        const uint32_t v0 = qa[kc][2 * j], v1 = qa[kc][2 * j + 1];
        qa[kc][2 * j] = pack_f16x2(bf16_lo(v0) * s0, bf16_hi(v0) * s0);
        qa[kc][2 * j + 1] = pack_f16x2(bf16_lo(v1) * s1, bf16_hi(v1) * s1);
      }
  }
  // k_R query slice: rows g, g+8, dims 16w + {2q, 2q+1, 2q+8, 2q+9}, kept in shared memory
  {
    float qr[8];
    const uint32_t u0 = qrw[0], u1 = qrw[1], u2 = qrw[2], u3 = qrw[3];
    qr[0] = bf16_lo(u0);
    qr[1] = bf16_hi(u0);
    qr[2] = bf16_lo(u2);
    qr[3] = bf16_hi(u2);
    qr[4] = bf16_lo(u1);
    qr[5] = bf16_hi(u1);
    qr[6] = bf16_lo(u3);
    qr[7] = bf16_hi(u3);
#pragma unroll
    for (int e = 0; e < 8; ++e) qr[e] *= inv_f[e >> 2];  // same units as the latent partials (exact)
    float4* dst = reinterpret_cast<float4*>(sh.qr + threadIdx.x * 8);
    dst[0] = make_float4(qr[0], qr[1], qr[2], qr[3]);
    dst[1] = make_float4(qr[4], qr[5], qr[6], qr[7]);
  }
  // per-page rope factors: query times channel scale split into two BF16 terms
  uint32_t qr_hi[4], qr_lo[4];
  float rconst[2] = {0.f, 0.f};
  int cur_pg = -1;

  // per-lane matrix-load offsets inside a stage's latent rows (chunk XOR token mod 8)
  const int r8 = lane & 7, mi = lane >> 3;
  int off_s, off_r0, off_r1;
  if constexpr (BITS == 4) {
    off_s = r8 * 256 + 16 * ((4 * warp + mi) ^ r8);                                  // + 2048 nb
    off_r0 = (8 * (mi & 1) + r8) * 256 + 16 * ((4 * warp + (mi >> 1)) ^ r8);         // chunks 0, 1
    off_r1 = (8 * (mi & 1) + r8) * 256 + 16 * ((4 * warp + 2 + (mi >> 1)) ^ r8);     // chunks 2, 3
  } else {
    off_s = (8 * (mi >> 1) + r8) * 128 + 16 * ((2 * warp + (mi & 1)) ^ r8);          // + 2048 pair
    off_r0 = (8 * (mi & 1) + r8) * 128 + 16 * ((2 * warp + (mi >> 1)) ^ r8);
    off_r1 = off_r0;
  }
  uint64_t* const xs_bar = sh.bars + kS;
  uint64_t* const xp_bar = sh.bars + kS + 2;

  // ---- scores of local tile i: partial sums over this warp's channels -> exchange buffer i&1
  auto score = [&](int i) {
    const int stg = i % kS, buf = i & 1;
    const bool ok = mbar_wait_bounded(sh.bars + stg, (i / kS) & 1, kWaitBudget);
    const uint8_t* sp = sh.stages + stg * G::kStage;
    const int pg = ((tile_begin + i) * kPT) >> p.p_shift;
    if (pg != cur_pg) {
      cur_pg = pg;
      const uint32_t* rm = reinterpret_cast<const uint32_t*>(sp + G::kRMetaOff) + 16 * warp;
      // A fragment element (row, dim): dims 2q, 2q+1 (regs 0, 1) and 2q+8, 2q+9 (regs 2, 3)
      const int dims[4] = {2 * q, 2 * q + 1, 2 * q + 8, 2 * q + 9};
      float sc[4], mn[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t w = rm[dims[e]];
        sc[e] = half_lo(w);
        mn[e] = half_hi(w);
      }
      float qr[8];
      {
        const float4 a = reinterpret_cast<const float4*>(sh.qr + threadIdx.x * 8)[0];
        const float4 c = reinterpret_cast<const float4*>(sh.qr + threadIdx.x * 8)[1];
        qr[0] = a.x; qr[1] = a.y; qr[2] = a.z; qr[3] = a.w;
        qr[4] = c.x; qr[5] = c.y; qr[6] = c.z; qr[7] = c.w;
      }
      float hi_v[8], lo_v[8], rqs[2], rbias[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        rqs[r] = 0.f;
        rbias[r] = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x = qr[4 * r + e] * sc[e];
          const float xh = __bfloat162float(__float2bfloat16_rn(x));
          const float xl = __bfloat162float(__float2bfloat16_rn(x - xh));
          hi_v[4 * r + e] = xh;
          lo_v[4 * r + e] = xl;
          rqs[r] += xh + xl;
          rbias[r] += qr[4 * r + e] * mn[e];
        }
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {
          rqs[r] += __shfl_xor_sync(0xffffffffu, rqs[r], o);
          rbias[r] += __shfl_xor_sync(0xffffffffu, rbias[r], o);
        }
        rconst[r] = rbias[r] - 128.f * rqs[r];
      }
      qr_hi[0] = pack_bf16x2(hi_v[0], hi_v[1]);
      qr_hi[1] = pack_bf16x2(hi_v[4], hi_v[5]);
      qr_hi[2] = pack_bf16x2(hi_v[2], hi_v[3]);
      qr_hi[3] = pack_bf16x2(hi_v[6], hi_v[7]);
      qr_lo[0] = pack_bf16x2(lo_v[0], lo_v[1]);
      qr_lo[1] = pack_bf16x2(lo_v[4], lo_v[5]);
      qr_lo[2] = pack_bf16x2(lo_v[2], lo_v[3]);
      qr_lo[3] = pack_bf16x2(lo_v[6], lo_v[7]);
    }

    // latent: four n-blocks of 8 tokens, eight k-chunks each (four independent chains)
    float acc[4][4];
    if constexpr (BITS == 4) {
      uint32_t R[4][4];
#pragma unroll
      for (int nb = 0; nb < 4; ++nb) ldsm_x4(R[nb], sp + nb * 2048 + off_s);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        uint32_t x8[4];
#pragma unroll
        for (int nb = 0; nb < 4; ++nb) {
          x8[nb] = R[nb][m] >> 8;
          if (m == 0) mma_f16_16816_z(acc[nb], qa[0], R[nb][m] & 0x000f000fu, x8[nb] & 0x000f000fu);
          else mma_f16_16816(acc[nb], qa[2 * m], R[nb][m] & 0x000f000fu, x8[nb] & 0x000f000fu);
        }
#pragma unroll
        for (int nb = 0; nb < 4; ++nb)
          mma_f16_16816(acc[nb], qa[2 * m + 1], R[nb][m] & 0x00f000f0u, x8[nb] & 0x00f000f0u);
      }
    } else {
      uint32_t R[4][2];
#pragma unroll
      for (int pp = 0; pp < 2; ++pp) {
        uint32_t X[4];
        ldsm_x4(X, sp + pp * 2048 + off_s);
        R[2 * pp][0] = X[0];
        R[2 * pp][1] = X[1];
        R[2 * pp + 1][0] = X[2];
        R[2 * pp + 1][1] = X[3];
      }
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int nb = 0; nb < 4; ++nb) {
          const uint32_t x = R[nb][m], xs = x >> 10;
          uint32_t u[8];
#pragma unroll
          for (int f = 0; f < 5; ++f) u[f] = x & (0x00030003u << (2 * f));
#pragma unroll
          for (int f = 5; f < 8; ++f) u[f] = xs & (0x00030003u << (2 * (f - 5)));
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (m == 0 && j == 0) mma_f16_16816_z(acc[nb], qa[0], u[0], u[1]);
            else mma_f16_16816(acc[nb], qa[4 * m + j], u[2 * j], u[2 * j + 1]);
          }
        }
    }
    // k_R chunk `warp`: two 16-token blocks, BF16 integers 128 + code (exact)
    float racc[4][4];
    uint32_t rb[4][2];
#pragma unroll
    for (int tb = 0; tb < 2; ++tb) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(sp + G::kRopeOff + (tb * 4 + warp) * 128 + lane * 4);
#pragma unroll
      for (int hb2 = 0; hb2 < 2; ++hb2) {
        rb[2 * tb + hb2][0] = and_or(w >> (8 * hb2), 0x000f000fu, 0x43004300u);
        rb[2 * tb + hb2][1] = and_or(w >> (8 * hb2 + 4), 0x000f000fu, 0x43004300u);
      }
    }
    // token metadata of group `warp` (tokens 8nb + 2q + c): the min and bias terms seed the
    // k_R accumulators, the scale multiplies the latent products
    float tsc[4][2];
    bool big = false;
#pragma unroll
    for (int nb = 0; nb < 4; ++nb)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int tok = 8 * nb + 2 * q + c;
        const uint32_t w = *reinterpret_cast<const uint32_t*>(sp + G::kMetaOff + (tok * 4 + warp) * 4);
        const float tmn = half_hi(w);
        tsc[nb][c] = half_lo(w);
        big |= tsc[nb][c] >= kStrictScale;
        racc[nb][c] = fmaf(tmn, qsum[0], rconst[0]);
        racc[nb][2 + c] = fmaf(tmn, qsum[1], rconst[1]);
      }
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) mma_bf16_16816(racc[nb], qr_hi, rb[nb][0], rb[nb][1]);
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) mma_bf16_16816(racc[nb], qr_lo, rb[nb][0], rb[nb][1]);
    float* my = sh.sbuf + (buf * 4 + warp) * 16 * kXStride;
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
      float part[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) part[e] = fmaf(tsc[nb][e & 1], acc[nb][e], racc[nb][e]);
      *reinterpret_cast<float2*>(my + g * kXStride + 8 * nb + 2 * q) = make_float2(part[0], part[1]);
      *reinterpret_cast<float2*>(my + (g + 8) * kXStride + 8 * nb + 2 * q) = make_float2(part[2], part[3]);
    }
    big = __any_sync(0xffffffffu, big);
    if (lane == 0) sh.xflags[buf * 4 + warp] = (big ? 1 : 0) | (ok ? 0 : 2);
    mbar_arrive(xs_bar + buf);
  };

  // ---- online softmax of tile i: heads 4w..4w+3, lane -> head 4w + lane/8, tokens 4*(lane%8)..+3
  auto softmax = [&](int i, bool strict) -> bool {
    const int buf = i & 1;
    const int hh = 4 * warp + (lane >> 3), tt = 4 * (lane & 7);
    const int t0 = (tile_begin + i) * kPT;
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float4 v = *reinterpret_cast<const float4*>(sh.sbuf + ((buf * 4 + w) * 16 + hh) * kXStride + tt);
      s[0] += v.x;
      s[1] += v.y;
      s[2] += v.z;
      s[3] += v.w;
    }
    float lmax = -INFINITY;
    bool valid[4];
    const bool inside = t0 >= lo && t0 + kPT <= hi;  // the common case: every token of the tile counts
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      valid[j] = inside || ((t0 + tt + j >= lo) && (t0 + tt + j < hi));
      s[j] = valid[j] ? s[j] * head_scale : -INFINITY;
      lmax = fmaxf(lmax, s[j]);
    }
    const float slack = strict ? 0.f : kRescaleSlack;
    const bool need = lmax > st.m_run + slack || (st.m_run == -INFINITY && lmax > -INFINITY);
    float alpha = 1.f;
    const bool moved = __any_sync(0xffffffffu, need);
    if (moved) {  // rare: some head of this warp needs a new reference max
      float tmax = lmax;
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
      if (tmax > st.m_run + slack || (st.m_run == -INFINITY && tmax > -INFINITY)) {
        alpha = exp2_fast(st.m_run - tmax);  // 0 when the old reference was -inf
        st.l_part *= alpha;
        st.m_run = tmax;
      }
    }
    float pv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) pv[j] = (valid[j] && st.m_run != -INFINITY) ? exp2_fast(s[j] - st.m_run) : 0.f;
    st.l_part += (pv[0] + pv[1]) + (pv[2] + pv[3]);
    *reinterpret_cast<float4*>(sh.pbuf + (buf * 16 + hh) * kXStride + tt) = make_float4(pv[0], pv[1], pv[2], pv[3]);
    if ((lane & 7) == 0) sh.alpha[buf * 16 + hh] = alpha;
    if (lane == 0) sh.moved[buf * 4 + warp] = moved ? 1 : 0;
    mbar_arrive(xp_bar + buf);
    return moved;
  };

  // ---- readout of tile i: O += (P * token scale) . codes, plus sum_t P * token min
  auto readout = [&](int i) {
    const int stg = i % kS, buf = i & 1;
    const uint8_t* sp = sh.stages + stg * G::kStage;
    const float* pb = sh.pbuf + buf * 16 * kXStride;
#pragma unroll
    for (int kc2 = 0; kc2 < 2; ++kc2) {
      // P fragment: rows g, g+8; tokens 16kc2 + 2q + {0, 1} (regs 0, 1) and + 8 (regs 2, 3)
      const int ta = 16 * kc2 + 2 * q, tb = ta + 8;
      const float2 p0 = *reinterpret_cast<const float2*>(pb + g * kXStride + ta);
      const float2 p1 = *reinterpret_cast<const float2*>(pb + (g + 8) * kXStride + ta);
      const float2 p2 = *reinterpret_cast<const float2*>(pb + g * kXStride + tb);
      const float2 p3 = *reinterpret_cast<const float2*>(pb + (g + 8) * kXStride + tb);
      const uint32_t wa0 = *reinterpret_cast<const uint32_t*>(sp + G::kMetaOff + (ta * 4 + warp) * 4);
      const uint32_t wa1 = *reinterpret_cast<const uint32_t*>(sp + G::kMetaOff + ((ta + 1) * 4 + warp) * 4);
      const uint32_t wb0 = *reinterpret_cast<const uint32_t*>(sp + G::kMetaOff + (tb * 4 + warp) * 4);
      const uint32_t wb1 = *reinterpret_cast<const uint32_t*>(sp + G::kMetaOff + ((tb + 1) * 4 + warp) * 4);
      const float sa0 = half_lo(wa0), sa1 = half_lo(wa1), sb0 = half_lo(wb0), sb1 = half_lo(wb1);
      uint32_t a[4];
      a[0] = pack_f16x2(p0.x * sa0, p0.y * sa1);
      a[1] = pack_f16x2(p1.x * sa0, p1.y * sa1);
      a[2] = pack_f16x2(p2.x * sb0, p2.y * sb1);
      a[3] = pack_f16x2(p3.x * sb0, p3.y * sb1);
      const float ma0 = half_hi(wa0), ma1 = half_hi(wa1), mb0 = half_hi(wb0), mb1 = half_hi(wb1);
      st.mterm[0] += (p0.x * ma0 + p0.y * ma1) + (p2.x * mb0 + p2.y * mb1);
      st.mterm[1] += (p1.x * ma0 + p1.y * ma1) + (p3.x * mb0 + p3.y * mb1);
      if constexpr (BITS == 4) {
#pragma unroll
        for (int mp = 0; mp < 2; ++mp) {
          uint32_t X[4];  // (tokens 0-7, chunk 2mp), (8-15, 2mp), (0-7, 2mp+1), (8-15, 2mp+1)
          ldsm_x4_t(X, sp + kc2 * 16 * 256 + (mp == 0 ? off_r0 : off_r1));
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int mm = 2 * mp + hf;
            const uint32_t x0 = X[2 * hf], x1 = X[2 * hf + 1], y0 = x0 >> 8, y1 = x1 >> 8;
            mma_f16_16816(st.o[4 * mm + 0], a, x0 & 0x000f000fu, x1 & 0x000f000fu);
            mma_f16_16816(st.o[4 * mm + 1], a, x0 & 0x00f000f0u, x1 & 0x00f000f0u);
            mma_f16_16816(st.o[4 * mm + 2], a, y0 & 0x000f000fu, y1 & 0x000f000fu);
            mma_f16_16816(st.o[4 * mm + 3], a, y0 & 0x00f000f0u, y1 & 0x00f000f0u);
          }
        }
      } else {
        uint32_t X[4];  // (tokens 0-7, chunk 0), (8-15, 0), (0-7, 1), (8-15, 1)
        ldsm_x4_t(X, sp + kc2 * 16 * 128 + off_r0);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const uint32_t x0 = X[2 * m], x1 = X[2 * m + 1], y0 = x0 >> 10, y1 = x1 >> 10;
#pragma unroll
          for (int f = 0; f < 5; ++f)
            mma_f16_16816(st.o[8 * m + f], a, x0 & (0x00030003u << (2 * f)), x1 & (0x00030003u << (2 * f)));
#pragma unroll
          for (int f = 5; f < 8; ++f)
            mma_f16_16816(st.o[8 * m + f], a, y0 & (0x00030003u << (2 * (f - 5))), y1 & (0x00030003u << (2 * (f - 5))));
        }
      }
    }
  };

  // ---- pipeline: scores of tile i+1 overlap the softmax exchange of tile i
  // (i = -1 only computes the scores of tile 0, so the score code is inlined once)
  for (int i = -1; i < n_my; ++i) {
    const int buf = i & 1;
    const uint32_t par = (i >> 1) & 1;
    if (i >= 0) {
      const bool ok = mbar_wait_bounded(xs_bar + buf, par, kWaitBudget);
      const int4 xv = *reinterpret_cast<const int4*>(sh.xflags + buf * 4);
      const int xf = (xv.x | xv.y) | (xv.z | xv.w);
      if (!ok || (xf & 2)) {
        flags |= kErrTimeout;
        if (threadIdx.x == 0)  // orderly exit: bounded waits for the copies still in flight
          for (int j = i + 1; j < issued; ++j)
            (void)mbar_wait_bounded(sh.bars + (j % kS), (j / kS) & 1, kWaitBudget >> 4);
        break;
      }
      softmax(i, (xf & 1) != 0);
    }
    if (i + 1 < n_my) score(i + 1);
    if (i < 0) continue;
    const bool ok = mbar_wait_bounded(xp_bar + buf, par, kWaitBudget);
    if (!ok) {
      flags |= kErrTimeout;
      if (threadIdx.x == 0)
        for (int j = i + 1; j < issued; ++j)
          (void)mbar_wait_bounded(sh.bars + (j % kS), (j / kS) & 1, kWaitBudget >> 4);
      break;
    }
    // every warp finished tile i-1 (its readout precedes the weights of tile i): refill its stage
    if (i >= 1 && issued < n_my) {
      if (warp == (i & 3) && lane == 0) {
        fence_proxy_async_smem();
        issue(issued);
      }
      ++issued;
    }
    const int4 mv = *reinterpret_cast<const int4*>(sh.moved + buf * 4);
    if ((mv.x | mv.y) | (mv.z | mv.w)) {
      const float a0 = sh.alpha[buf * 16 + g], a1 = sh.alpha[buf * 16 + g + 8];
#pragma unroll
      for (int cb = 0; cb < 16; ++cb) {
        st.o[cb][0] *= a0;
        st.o[cb][1] *= a0;
        st.o[cb][2] *= a1;
        st.o[cb][3] *= a1;
      }
      st.mterm[0] *= a0;
      st.mterm[1] *= a1;
    }
    readout(i);
  }

  // ---- partial output: undo the operand weights, add sum_t p_t min_t, store through a
  // shared-memory tile (the stages are free once every warp is here) for coalesced writes
  float mt0 = st.mterm[0], mt1 = st.mterm[1];
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) {
    mt0 += __shfl_xor_sync(0xffffffffu, mt0, o);
    mt1 += __shfl_xor_sync(0xffffffffu, mt1, o);
  }
  __syncthreads();
  float* tile = reinterpret_cast<float*>(sh.stages);
#pragma unroll
  for (int cb = 0; cb < 16; ++cb) {
    const float sc = pow2_int(24 - out_log2w<BITS>(cb));
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int ch = 128 * warp + out_channel<BITS>(cb, 2 * q + c);
      tile[g * kOutStride + ch] = fmaf(st.o[cb][c], sc, mt0);
      tile[(g + 8) * kOutStride + ch] = fmaf(st.o[cb][2 + c], sc, mt1);
    }
  }
  __syncthreads();
  const int NS = p.n_split + p.n_q;
  for (int idx = threadIdx.x; idx < 16 * (kLatent / 4); idx += kThreads) {
    const int row = idx / (kLatent / 4), c4 = idx % (kLatent / 4);
    const float4 v = *reinterpret_cast<const float4*>(tile + row * kOutStride + 4 * c4);
    *reinterpret_cast<float4*>(p.o_part + ((static_cast<size_t>(b) * p.H + h0 + row) * NS + split) * kLatent + 4 * c4) = v;
  }
}

// ------------------------------------------------------------------ protected-token CTA
template <bool kPaged>
__device__ void protected_split(const DecodeParams& p, const Shared& sh, int b, int T, int T_old, int part, State& st,
                                int32_t& flags) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int h0 = blockIdx.y * 16;
  // query fragments for latent group `warp` (BF16, exact, channels in order)
  uint32_t qa[8][4];
  {
    const uint32_t* r0 = reinterpret_cast<const uint32_t*>(p.q_lat + (static_cast<size_t>(b) * p.H + h0 + g) * kLatent + 128 * warp);
    const uint32_t* r1 = r0 + 8 * kLatent / 2;
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) {
      qa[kc][0] = __ldg(r0 + 8 * kc + q);
      qa[kc][1] = __ldg(r1 + 8 * kc + q);
      qa[kc][2] = __ldg(r0 + 8 * kc + 4 + q);
      qa[kc][3] = __ldg(r1 + 8 * kc + 4 + q);
    }
  }
  // k_R query slice: rows g, g+8, dims 16w + {2q, 2q+1, 2q+8, 2q+9}
  uint32_t qra[4];
  {
    const uint32_t* r0 = reinterpret_cast<const uint32_t*>(p.q_rope + (static_cast<size_t>(b) * p.H + h0 + g) * kRope + 16 * warp);
    const uint32_t* r1 = r0 + 8 * kRope / 2;
    qra[0] = __ldg(r0 + q);
    qra[1] = __ldg(r1 + q);
    qra[2] = __ldg(r0 + 4 + q);
    qra[3] = __ldg(r1 + 4 + q);
  }
  bf16_split<kPaged>(p, sh, b, T, T_old, part, qa, qra, st, flags);

  const int NS = p.n_split + p.n_q, slot = p.n_split + part;
  float* o0 = p.o_part + ((static_cast<size_t>(b) * p.H + h0 + g) * NS + slot) * kLatent + 128 * warp;
  float* o1 = p.o_part + ((static_cast<size_t>(b) * p.H + h0 + g + 8) * NS + slot) * kLatent + 128 * warp;
#pragma unroll
  for (int cb = 0; cb < 16; ++cb) {
    *reinterpret_cast<float2*>(o0 + 8 * cb + 2 * q) = make_float2(st.o[cb][0], st.o[cb][1]);
    *reinterpret_cast<float2*>(o1 + 8 * cb + 2 * q) = make_float2(st.o[cb][2], st.o[cb][3]);
  }
}

// ------------------------------------------------------------------ in-kernel merge
// When the whole grid is one resident wave, the NS CTAs of a (sequence, 16-head block) may merge
// their own partials (when the partials are many: see in_place_merge). The block's counter is one 64-bit word: arrivals in the low half (zero
// between calls), a generation in the high half. Each CTA, once its partial is stored (CTA
// barrier first), adds one arrival (release of the CTA's stores, acquire of the earlier
// arrivals'); the last arrival adds 2^32 - NS, which clears the count and advances the
// generation in one step; the others wait (bounded) until they see the count complete or the
// generation moved. No CTA can keep a waiting one's group from running: every CTA is
// resident. Returns false if the wait gave up or the count was not a valid arrival count (a
// workspace whose counters were not zero): the partials may then be incomplete.
__device__ __forceinline__ bool group_arrive(unsigned long long* ctr, int NS) {
  const unsigned long long old = atom_add_acq_rel_gpu(ctr, 1ull);
  const uint32_t t = static_cast<uint32_t>(old), g0 = static_cast<uint32_t>(old >> 32);
  if (t >= static_cast<uint32_t>(NS)) return false;
  if (t == static_cast<uint32_t>(NS - 1)) {
    red_add_release_gpu(ctr, (1ull << 32) - static_cast<unsigned long long>(NS));
    return true;
  }
  // released by the last arrival itself (count NS, reached before the reset is seen) or by the
  // reset (generation moved); the acquire of either orders every arrival's stores before ours
  const long long t0 = clock64();
  for (;;) {
    const unsigned long long v = ld_acquire_gpu(ctr);
    if (static_cast<uint32_t>(v >> 32) != g0 || static_cast<uint32_t>(v) == static_cast<uint32_t>(NS)) return true;
    if (clock64() - t0 > kWaitBudget) return false;
    __nanosleep(32);
  }
}

// The merge of one (sequence, 16-head block)'s NS partials by CTA z of its n_ctas: float4
// columns [z*2048/n_ctas, (z+1)*2048/n_ctas) of the block's output (16 heads x 128 columns). The slice of every
// partial and the partial maxima and sums of the slice's heads are first copied into shared
// memory, all requests in flight at once (16-byte asynchronous copies through L2: the partials
// were stored by other SMs during this launch), the maxima and sums as a group of their own. Once
// that group has landed (the slices still in flight), one warp per head forms the head's
// maximum M and sum L = sum_s 2^(m_s - M) l_s and turns each partial's (m_s, l_s) into its weight
// 2^(m_s - M) / L (and writes the head's log-sum-exp if the slice holds its first column); R
// lanes take one column (R a power of two, as many as fill the CTA), each summing every R-th
// weighted partial, and shuffles add the R sums. Partials of empty shares (maximum -inf) have
// weight 0 and their products are dropped by selection, never added: their rows hold whatever
// the buffer held.
// `buf` holds merge_buf_need(NS, n_ctas) bytes (checked on the host): NS partial slots merged by
// the group's n_ctas CTAs.
__host__ __device__ constexpr int merge_buf_need(int NS, int n_ctas) {
  return NS * (2048 / n_ctas + 1) * 16 + ((2048 / n_ctas) / 128 + 2) * NS * 8 + 32 + 256;
}

__device__ __forceinline__ void group_merge(const DecodeParams& p, uint8_t* buf, int b, int h0, int z, int n_ctas,
                                            int NS) {
  constexpr int kCols = 16 * (kLatent / 4);
  const int c0 = static_cast<int>(static_cast<long long>(z) * kCols / n_ctas);
  const int c1 = static_cast<int>(static_cast<long long>(z + 1) * kCols / n_ctas);
  const int n_cols = c1 - c0;
  if (n_cols <= 0) return;  // (uniform in the CTA)
  const int hA = c0 >> 7, n_h = ((c1 - 1) >> 7) - hA + 1;
  const size_t bh0 = static_cast<size_t>(b) * p.H + h0;
  // (m_s, l_s) of the slice's heads: [n_h][NS] pairs, contiguous in the partial maxima and sums;
  // copied as the enclosing 16-byte blocks (the array starts 16-byte aligned and the workspace
  // holds 16 bytes beyond it), so the rows start 0 or 8 bytes into the copy
  const size_t ml0 = (bh0 + hA) * NS * 2;  // float index of the first pair
  const float* mlg = p.ml_part + (ml0 & ~static_cast<size_t>(3));
  const int n_ml16 = static_cast<int>(((ml0 & 3) * 4 + static_cast<size_t>(n_h) * NS * 8 + 15) / 16);
  float2* mls = reinterpret_cast<float2*>(buf + (ml0 & 3) * 4);  // [n_h][NS]: (m_s, l_s), then (weight, -)
  float4* os = reinterpret_cast<float4*>(buf + n_ml16 * 16);      // [NS][n_cols]
  for (int j = threadIdx.x; j < n_ml16; j += kThreads) cp_async_cg16(buf + j * 16, mlg + 4 * j);
  cp_async_commit();  // the maxima and sums: waited for first, the weights overlap the slices' copies
  // thread -> (column, every k-th partial): k = 1 when the columns alone fill the CTA
  const int k = n_cols >= kThreads ? 1 : kThreads / n_cols;
  const int s_first = n_cols >= kThreads ? 0 : static_cast<int>(threadIdx.x) / n_cols;
  if (s_first < k)
    for (int ci = static_cast<int>(threadIdx.x) - s_first * n_cols; ci < n_cols; ci += kThreads) {
      const int c = c0 + ci;
      const float* src = p.o_part + (bh0 + (c >> 7)) * NS * kLatent + 4 * (c & 127);
      for (int s = s_first; s < NS; s += k) cp_async_cg16(os + s * n_cols + ci, src + static_cast<size_t>(s) * kLatent);
    }
  cp_async_commit();
  cp_async_wait_group<1>();
  __syncthreads();
  // per-head weights (warp w: heads w, w+4, ...)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int hh = warp; hh < n_h; hh += kThreads / 32) {
    float2* row = mls + hh * NS;
    float m = -INFINITY;
    for (int s = lane; s < NS; s += 32) m = fmaxf(m, row[s].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.f;
    if (m != -INFINITY)
      for (int s = lane; s < NS; s += 32) l += exp2f(row[s].x - m) * row[s].y;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    const bool any = m != -INFINITY && l > 0.f;
    const float inv = any ? 1.f / l : 0.f;
    __syncwarp();
    for (int s = lane; s < NS; s += 32) row[s].x = any ? exp2f(row[s].x - m) * inv : 0.f;
    if (lane == 0 && ((hA + hh) << 7) >= c0)  // the slice holds the head's first column
      p.lse[bh0 + hA + hh] = any ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
  }
  cp_async_wait_group<0>();
  __syncthreads();

  int lg = 0;  // R = 2^lg lanes per column
  while (lg < 5 && (n_cols << (lg + 1)) <= kThreads) ++lg;
  const int R = 1 << lg, per_pass = kThreads >> lg;
  const int slot = static_cast<int>(threadIdx.x) >> lg, r = static_cast<int>(threadIdx.x) & (R - 1);
  const int n_pass = (n_cols + per_pass - 1) / per_pass;
  for (int pass = 0; pass < n_pass; ++pass) {
    const int ci = pass * per_pass + slot;  // column within the slice
    const bool active = ci < n_cols;
    const int c = c0 + ci;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (active) {
      const float2* wrow = mls + ((c >> 7) - hA) * NS;
      // (every slot's row is loaded, so the loads of several slots are in flight together; an
      // empty share's sums are dropped by selection: its row may hold anything)
#pragma unroll 4
      for (int s = r; s < NS; s += R) {
        const float w = wrow[s].x;
        const float4 v = os[s * n_cols + ci];
        const float4 t = make_float4(fmaf(w, v.x, acc.x), fmaf(w, v.y, acc.y), fmaf(w, v.z, acc.z), fmaf(w, v.w, acc.w));
        if (w != 0.f) acc = t;
      }
    }
    for (int o = 1; o < R; o <<= 1) {
      acc.x += __shfl_xor_sync(0xffffffffu, acc.x, o);
      acc.y += __shfl_xor_sync(0xffffffffu, acc.y, o);
      acc.z += __shfl_xor_sync(0xffffffffu, acc.z, o);
      acc.w += __shfl_xor_sync(0xffffffffu, acc.w, o);
    }
    if (active && r == 0) *reinterpret_cast<float4*>(p.out + (bh0 + (c >> 7)) * kLatent + 4 * (c & 127)) = acc;
  }
}

// Bytes of a 16-head CTA's shared memory free for the merge once its shares are done: the stage
// region and the two exchange buffers that follow it (the barriers lie beyond).
template <int BITS>
__host__ __device__ constexpr int merge_buf_bytes() {
  return Geom<BITS>::kRegion + (kXsFloats + kXpFloats) * 4;
}

// kBalanced: equal shares sized from the whole batch (launched when more shares than one wave
// are needed); a separate instance, so the one-wave kernel carries none of its code.
template <int BITS, bool kBalanced, bool kPaged = false>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const Shared sh = carve<BITS>(smem);
  // grid (B, H/16, n_q + n_split): z < n_q serves a share of the protected tokens, z >= n_q packed
  // share z - n_q, so the hardware dispatches the protected CTAs first and then the shares split
  // by split. Partial slot: packed share s -> s, protected share q -> n_split + q.
  const bool is_bf16 = static_cast<int>(blockIdx.z) < p.n_q;
  const int split = is_bf16 ? p.n_split + static_cast<int>(blockIdx.z) : static_cast<int>(blockIdx.z) - p.n_q;
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h0 = blockIdx.y * 16;
  int32_t flags = 0;
  if (!is_bf16) {
    if (query_bulk(p)) {
      if (threadIdx.x == 0) fetch_query(p, sh, b, h0);
    } else {
      copy_query(p, sh, b, h0);  // (visible to every thread after the barrier below)
    }
  }
  const SeqLenWords len_words = decode_seq_len_load(p, b);
  // a short page table whole into sh.pids while the length is in flight (the share, and so its
  // pages, follow from the length): asynchronous 4-byte copies, waited for before the ids are read
  if (!is_bf16 && p.max_pages <= kMaxSplitPages)
    for (int pg = threadIdx.x; pg < p.max_pages; pg += kThreads)
      cp_async_ca4(sh.pids + pg, p.page_table + static_cast<size_t>(b) * p.max_pages + pg);
  int T_old;
  const int T = decode_seq_len_check(p, len_words, T_old, flags);
  if (threadIdx.x == 0) {
    if (is_bf16) {  // two row stages, one arrival each
      mbar_init(sh.bars, 1);
      mbar_init(sh.bars + 1, 1);
    } else {  // packed stages (one arrival + bytes), then the exchanges (one arrival per thread)
      for (int i = 0; i < Geom<BITS>::kStages; ++i) mbar_init(sh.bars + i, 1);
      for (int i = 0; i < 4; ++i) mbar_init(sh.bars + Geom<BITS>::kStages + i, kThreads);
    }
    fence_mbar_init();
    sh.strict[0] = sh.strict[1] = 0;
  }
  __syncthreads();

  State st;
#pragma unroll
  for (int cb = 0; cb < 16; ++cb) st.o[cb][0] = st.o[cb][1] = st.o[cb][2] = st.o[cb][3] = 0.f;
  st.mterm[0] = st.mterm[1] = 0.f;
  st.m_run = -INFINITY;
  st.l_part = 0.f;

  if (is_bf16) protected_split<kPaged>(p, sh, b, T, T_old, split - p.n_split, st, flags);
  else packed_split<BITS, kBalanced>(p, sh, b, T, split, st, flags);

  const int NS = p.n_split + p.n_q;
  float l_run = st.l_part;
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) l_run += __shfl_xor_sync(0xffffffffu, l_run, o);
  if ((lane & 7) == 0) {
    const int hh = h0 + 4 * warp + (lane >> 3);
    float* ml = p.ml_part + ((static_cast<size_t>(b) * p.H + hh) * NS + split) * 2;
    ml[0] = st.m_run;
    ml[1] = l_run;
  }
  if (!kBalanced && p.arrive != nullptr) {  // the grid is one resident wave: merge in place
    __syncthreads();  // the CTA's partial stores precede its arrival
    // (indices re-read from the launch: nothing stays live across the main loop for this)
    int ok = 0;
    if (threadIdx.x == 0) ok = group_arrive(p.arrive + (blockIdx.x * gridDim.y + blockIdx.y), gridDim.z);
    if (__syncthreads_or(ok))
      group_merge(p, sh.stages, blockIdx.x, blockIdx.y * 16, blockIdx.z, gridDim.z, p.n_split + p.n_q);
    else flags |= kErrTimeout;
  }
  flags = __reduce_or_sync(0xffffffffu, flags);
  if (lane == 0 && flags) atomicOr(p.err, flags);
}

// Merge the split partials of one (sequence, head): warp-shuffle log-sum-exp reduction of
// the split maxima and sums, then a weighted sum of the partial outputs.
__global__ void __launch_bounds__(128) combine_kernel(const DecodeParams p) {
  const int bh = blockIdx.x;
  const int NS = p.n_split + p.n_q;
  const int lane = threadIdx.x & 31;
  const float* ml = p.ml_part + static_cast<size_t>(bh) * NS * 2;
  const float* op = p.o_part + static_cast<size_t>(bh) * NS * kLatent + 4 * threadIdx.x;
  // The first batch of partial rows is requested together with the maxima (one round trip
  // instead of two); a slot whose weight is zero is dropped by selection, never multiplied, as
  // the row of an empty share holds whatever the buffer held before.
  constexpr int kBatch = 8;
  float4 v[kBatch];
#pragma unroll
  for (int u = 0; u < kBatch; ++u)
    v[u] = u < NS ? *reinterpret_cast<const float4*>(op + static_cast<size_t>(u) * kLatent) : make_float4(0.f, 0.f, 0.f, 0.f);
  float m = -INFINITY;
  for (int s = lane; s < NS; s += 32) m = fmaxf(m, ml[2 * s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float l = 0.f;
  if (m != -INFINITY)
    for (int s = lane; s < NS; s += 32) l += exp2f(ml[2 * s] - m) * ml[2 * s + 1];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (m != -INFINITY && l > 0.f) {
    for (int s0 = 0; s0 < NS; s0 += kBatch) {
      if (s0 > 0) {  // rows of empty shares (weight 0) are not loaded
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
          v[u] = s0 + u < NS && (p.share_slots == 0 || ml[2 * (s0 + u) + 1] != 0.f)
                     ? *reinterpret_cast<const float4*>(op + static_cast<size_t>(s0 + u) * kLatent)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const float w = s0 + u < NS ? exp2f(ml[2 * (s0 + u)] - m) : 0.f;
        if (w != 0.f) {
          acc.x += w * v[u].x;
          acc.y += w * v[u].y;
          acc.z += w * v[u].z;
          acc.w += w * v[u].w;
        }
      }
    }
    const float inv = 1.f / l;
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
  }
  *reinterpret_cast<float4*>(p.out + static_cast<size_t>(bh) * kLatent + 4 * threadIdx.x) = acc;
  if (threadIdx.x == 0)
    p.lse[bh] = (m == -INFINITY || !(l > 0.f)) ? -INFINITY : (m + log2f(l)) * 0.69314718055994530942f;
}

// Many partials per (sequence, head), as a long table over few sequence-head groups gives: CTA
// (bh, quarter) merges channels 128*quarter .. +127; its kWideGroups warps each take every
// kWideGroups-th batch of partials, and the warps' sums are added in shared memory.
constexpr int kWideGroups = 16;
constexpr int kWideMinSlots = 33;  // fewer partials: combine_kernel
__global__ void __launch_bounds__(32 * kWideGroups) combine_wide_kernel(const DecodeParams p) {
  __shared__ float4 red[kWideGroups - 1][32];
  const int bh = blockIdx.x, quarter = blockIdx.y;
  const int NS = p.n_split + p.n_q;
  const int grp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* ml = p.ml_part + static_cast<size_t>(bh) * NS * 2;
  const float* op = p.o_part + static_cast<size_t>(bh) * NS * kLatent + 128 * quarter + 4 * lane;
  // every warp forms the maximum and the weight sum over all partials (2 NS floats, cached)
  float m = -INFINITY;
  for (int s = lane; s < NS; s += 32) m = fmaxf(m, ml[2 * s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float l = 0.f;
  if (m != -INFINITY)
    for (int s = lane; s < NS; s += 32) l += exp2f(ml[2 * s] - m) * ml[2 * s + 1];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (m != -INFINITY && l > 0.f) {
    constexpr int kBatch = 8;
    for (int s0 = grp * kBatch; s0 < NS; s0 += kWideGroups * kBatch) {
      float w[kBatch];
      float4 v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {  // a partial of weight zero (an empty share) is not read
        w[u] = s0 + u < NS ? exp2f(ml[2 * (s0 + u)] - m) : 0.f;
        v[u] = w[u] != 0.f ? *reinterpret_cast<const float4*>(op + static_cast<size_t>(s0 + u) * kLatent)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        acc.x += w[u] * v[u].x;
        acc.y += w[u] * v[u].y;
        acc.z += w[u] * v[u].z;
        acc.w += w[u] * v[u].w;
      }
    }
  }
  if (grp > 0) red[grp - 1][lane] = acc;
  __syncthreads();
  if (grp != 0) return;
  for (int g2 = 0; g2 < kWideGroups - 1; ++g2) {
    const float4 r = red[g2][lane];
    acc.x += r.x;
    acc.y += r.y;
    acc.z += r.z;
    acc.w += r.w;
  }
  if (m != -INFINITY && l > 0.f) {
    const float inv = 1.f / l;
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
  }
  *reinterpret_cast<float4*>(p.out + static_cast<size_t>(bh) * kLatent + 128 * quarter + 4 * lane) = acc;
  if (quarter == 0 && lane == 0)
    p.lse[bh] = (m == -INFINITY || !(l > 0.f)) ? -INFINITY : (m + log2f(l)) * 0.69314718055994530942f;
}

// The merge launch for a decode call: one CTA per (sequence, head), or four wide CTAs when the
// partials are many.
cudaError_t launch_combine(const DecodeParams& p, cudaStream_t stream) {
  if (p.n_split + p.n_q >= kWideMinSlots)
    combine_wide_kernel<<<dim3(p.B * p.H, 4), 32 * kWideGroups, 0, stream>>>(p);
  else
    combine_kernel<<<p.B * p.H, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

int decode_num_splits(int B, int H, int max_pages, int P, int S, int W, int num_sms) {
  if (decode_uses_tc(H)) return decode_tc_num_splits(B, H, max_pages, P, num_sms);
  const int groups = B * (H / 16);
  const int target = kCtasPerSm * num_sms;  // one full wave of resident CTAs
  // one wave holds the packed shares and the protected CTAs of every sequence-head block
  int ns = target / (groups > 0 ? groups : 1) - decode_num_protected(B, H, max_pages, P, S, W, num_sms);
  const long long max_sub = (static_cast<long long>(max_pages) * P) / kPT;
  // Long page tables get splits of at most ~kShareTiles tiles even past one wave: a ragged batch
  // then spreads its longest sequences over many CTAs while the shares of short sequences are
  // empty and exit at once, and the hardware backfills the SMs (split-major dispatch).
  constexpr int kShareTiles = 40;
  const long long by_len = (max_sub + kShareTiles - 1) / kShareTiles;
  // (the rule only ever raises the count: a wave of shorter shares stays as it is)
  if (by_len > ns && ns < 64) ns = static_cast<int>(by_len > 64 ? 64 : by_len);
  // Minimum tiles per share: at least four (each share's partial costs the merge 2 KB per head),
  // except for up to 32 sequence-head groups, whose latency is their longest share: there short
  // tables take one-tile shares and medium ones two (their partials are then many, merged inside
  // the decode launch where they are 24 or more).
  const long long min_tiles = groups > 32 ? 4 : (max_sub <= 96 ? 1 : (max_sub <= 384 ? 2 : 4));
  int cap = static_cast<int>(max_sub / min_tiles);
  if (cap < 1) cap = 1;
  if (ns > cap) ns = cap;
  if (ns < 1) ns = 1;
  return ns;
}

int decode_num_protected(int B, int H, int max_pages, int P, int S, int W, int num_sms) {
  // Little packed work per CTA: the protected tiles would be the critical path of one CTA,
  // so they are shared by several (one 16-row tile each at most).
  const long long groups = static_cast<long long>(B) * (H / 16);
  const long long wave = static_cast<long long>(kCtasPerSm) * (num_sms > 0 ? num_sms : 1);
  const long long prot_max = (S > 0 ? 1 : 0) + (W + kTile - 1) / kTile;
  // 64-head blocks: the protected CTAs run as their own launch ahead of the packed shares, so
  // each takes one tile (a short launch instead of one long CTA per head block)
  if (decode_uses_tc(H)) return static_cast<int>(prot_max);
  const long long T = static_cast<long long>(max_pages) * P;
  const long long packed_max = T > S + W ? (T - W - 1) / kPT - S / kPT + 1 : 0;
  if (2 * groups * packed_max >= wave * prot_max) return 1;
  long long nq = wave / (4 * groups);
  return static_cast<int>(nq < 1 ? 1 : (nq > prot_max ? prot_max : nq));
}

int decode_share_slots(int B, int H, int max_pages, int P, int n_split, int n_q, int num_sms) {
  // balanced shares only when more shares are launched than one wave holds (long tables)
  const int groups = B * (H / 16);
  const int one_wave = kCtasPerSm * num_sms / (groups > 0 ? groups : 1) - 1;
  if (decode_uses_tc(H) || n_split <= (one_wave > 1 ? one_wave : 1)) return 0;
  const long long slots = static_cast<long long>(kCtasPerSm) * (num_sms > 0 ? num_sms : 1) -
                          static_cast<long long>(groups) * n_q;
  return static_cast<int>(slots > 16 ? (slots > (1 << 30) ? (1 << 30) : slots) : 16);
}

size_t decode_workspace_bytes(int B, int H, int n_slots) {
  const size_t NS = static_cast<size_t>(n_slots);
  // (+16: the merge copies the partial maxima and sums in whole 16-byte blocks)
  return kArriveBytes + static_cast<size_t>(B) * H * NS * (kLatent + 2) * sizeof(float) + 16;
}

namespace {

// Per-device launch facts of one decode kernel instance, looked up once (never inside a stream
// capture after the first call): the dynamic shared-memory opt-in is a function attribute, and
// the in-kernel merge needs the resident CTAs per SM and the SM count.
struct Residency {
  int per_sm;
  int sms;
};
template <int BITS, bool kBalanced, bool kPaged>
cudaError_t ensure_decode_setup(Residency* out) {
  static std::atomic<int> per_sm[64], sms[64];  // 0: not yet set up
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (per_sm[dev].load(std::memory_order_acquire) == 0) {
    e = cudaFuncSetAttribute(decode_kernel<BITS, kBalanced, kPaged>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes<BITS>());
    if (e != cudaSuccess) return e;
    int n = 0, m = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<BITS, kBalanced, kPaged>, kThreads,
                                                      smem_bytes<BITS>());
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&m, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    sms[dev].store(m, std::memory_order_relaxed);
    per_sm[dev].store(n > 0 ? n : -1, std::memory_order_release);
  }
  const int n = per_sm[dev].load(std::memory_order_acquire);
  out->per_sm = n > 0 ? n : 0;
  out->sms = sms[dev].load(std::memory_order_relaxed);
  return cudaSuccess;
}

// Whether a 16-head launch of `grid` (n_slots partials per sequence-head group) merges its
// partials in place: the grid must be one resident wave (so that a CTA waiting for its group
// cannot keep the others from running), the workspace must have a counter per group and the
// free shared memory must hold a CTA's slice of the partials; and the partials must be many
// (at least kMinInPlaceSlots per group). With few partials per group the merge launch is as
// fast: the in-place merge's chain of device-wide round trips (arrival, release, copies) costs
// about what the separate launch does (measured on GB300: in place wins from ~24 partials per
// group, loses ~1 us at 14).
constexpr int kMinInPlaceSlots = 24;
template <int BITS, bool kPaged>
cudaError_t in_place_merge(dim3 grid, int n_slots, bool* yes) {
  Residency res{};
  const cudaError_t e = ensure_decode_setup<BITS, false, kPaged>(&res);
  if (e != cudaSuccess) return e;
  const long long groups = static_cast<long long>(grid.x) * grid.y;
  const long long ctas = groups * grid.z;
  *yes = groups <= kMaxArriveGroups && ctas <= static_cast<long long>(res.per_sm) * res.sms &&
         n_slots >= kMinInPlaceSlots && merge_buf_need(n_slots, static_cast<int>(grid.z)) <= merge_buf_bytes<BITS>();
  return cudaSuccess;
}

// Launch of the 16-head kernel, merging the partials in place (a cooperative launch, which
// guarantees that every CTA is resident at once) or by a merge launch after it.
template <int BITS, bool kBalanced, bool kPaged>
cudaError_t launch_decode_kernel(DecodeParams p, dim3 grid, cudaStream_t stream) {
  Residency res{};
  cudaError_t e = ensure_decode_setup<BITS, kBalanced, kPaged>(&res);
  if (e != cudaSuccess) return e;
  bool fused = false;
  if (!kBalanced && p.arrive != nullptr &&
      (e = in_place_merge<BITS, kPaged>(grid, p.n_split + p.n_q, &fused)) != cudaSuccess)
    return e;
  if (!fused) p.arrive = nullptr;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes<BITS>();
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = fused ? 1 : 0;
  if ((e = cudaLaunchKernelEx(&cfg, decode_kernel<BITS, kBalanced, kPaged>, p)) != cudaSuccess) return e;
  if (fused) return cudaSuccess;
  return launch_combine(p, stream);
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
  // 64-head blocks: the packed shares run on the tensor-memory kernel, the protected shares here,
  // and a merge launch follows both
  const bool tc = decode_uses_tc(p.H);
  if (tc) {
    DecodeParams q = p;
    q.arrive = nullptr;
    const dim3 grid(p.B, p.H / 16, p.n_q);
    cudaError_t e;
    Residency res{};
    if (p.bits_c == 4) {
      if ((e = ensure_decode_setup<4, false, false>(&res)) != cudaSuccess) return e;
      decode_kernel<4, false><<<grid, kThreads, smem_bytes<4>(), stream>>>(q);
    } else {
      if ((e = ensure_decode_setup<2, false, false>(&res)) != cudaSuccess) return e;
      decode_kernel<2, false><<<grid, kThreads, smem_bytes<2>(), stream>>>(q);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_decode_tc(q, stream)) != cudaSuccess) return e;
    return launch_combine(q, stream);
  }
  const dim3 grid(p.B, p.H / 16, p.n_q + p.n_split);
  const bool bal = p.share_slots > 0;  // balanced shares: more than one wave, never merged in place
  if (p.bits_c == 4)
    return bal ? launch_decode_kernel<4, true, false>(p, grid, stream) : launch_decode_kernel<4, false, false>(p, grid, stream);
  return bal ? launch_decode_kernel<2, true, false>(p, grid, stream) : launch_decode_kernel<2, false, false>(p, grid, stream);
}

int decode_launch_count(int bits_c, int B, int H, int n_split, int n_q, int share_slots) {
  if (decode_uses_tc(H)) return 3;
  if (share_slots > 0) return 2;
  const dim3 grid(B, H / 16, n_q + n_split);
  bool fused = false;
  const cudaError_t e = bits_c == 4 ? in_place_merge<4, false>(grid, n_split + n_q, &fused)
                                    : in_place_merge<2, false>(grid, n_split + n_q, &fused);
  if (e != cudaSuccess) return -1;
  return fused ? 1 : 2;
}

// The unquantized comparator: every share a BF16 share over the paged BF16 cache.
int decode_bf16_num_parts(int B, int H, int max_pages, int P, int num_sms) {
  const int groups = B * (H / 16);
  int ns = kCtasPerSm * num_sms / (groups > 0 ? groups : 1);
  if (ns < 1) ns = 1;
  const long long max_tiles = (static_cast<long long>(max_pages) * P + kTile - 1) / kTile;
  // Few sequence-head groups already fill the GPU with one wave of shares; only where one wave
  // leaves a share well above ~128 16-token tiles (many groups, long tables) are shares made
  // smaller: a whole number of waves (at most 8), so that no partial wave trails the last.
  const long long by_len = (max_tiles + 127) / 128;
  if (by_len > 2LL * ns) {
    const long long waves = (by_len + ns - 1) / ns;
    ns = static_cast<int>((waves > 8 ? 8 : waves) * ns);
  }
  if (ns > max_tiles) ns = static_cast<int>(max_tiles);
  if (ns < 1) ns = 1;
  return ns;
}

cudaError_t launch_decode_bf16(const DecodeParams& p, cudaStream_t stream) {
  return launch_decode_kernel<4, false, true>(p, dim3(p.B, p.H / 16, p.n_q), stream);
}

// ------------------------------------------------------------------ built-in scratch
// Device-resident scratch used by mla_qcache_decode_attn_noalloc in place of a caller workspace.
// It lives for as long as the library is loaded, on every device that loads it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch for the current device. The host-side name of the array is only
// a stand-in, so the address is looked up once per device (with that device current) and cached.
// The cache slots are atomics: host threads whose first calls on a device overlap may each look
// the address up, and every one of them stores the same value.
cudaError_t noalloc_scratch(void** out) {
  static std::atomic<void*> addr[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  void* a = addr[dev].load(std::memory_order_acquire);
  if (a == nullptr) {
    e = cudaGetSymbolAddress(&a, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev].store(a, std::memory_order_release);
  }
  *out = a;
  return cudaSuccess;
}

}  // namespace mlaq

