// Decode attention over the low-bit dual-path MLA cache (QuantMLA page, abstract and appendix
// Figure 8; RAQ-MLA page, Figures 3-4 and appendix Table 5).
//
// Grid (n_split + 1, H/16, B). CTA (s, hb, b) handles 16 heads of sequence b:
//   s <  n_split : an even share of the packed tokens [S, T-W), streamed 16 tokens at a time
//                  from the page pool into a ring of shared-memory stages by bulk copies;
//   s == n_split : the protected tokens (t < S or t >= T-W) from the BF16 sink/recent buffers.
// Each CTA writes an unnormalized partial (O, max, sum); a second kernel merges the partials
// with a log-sum-exp reduction (one global softmax over all tokens).
//
// Inside a CTA, warp w owns latent group w (channels 128w..128w+127) and k_R chunk w
// (channels 16w..16w+15). Packed codes are never dequantized into a tile:
//   scores:  q . c_hat = scale_t * sum_i q_i code_ti + min_t * sum_i q_i  (per token group),
//            computed on tensor cores with the codes as exact small integers;
//   readout: sum_t p_t c_hat_t = sum_t (p_t scale_t) code_t + sum_t p_t min_t,
//            the same codes transposed in registers (movmatrix) as the B operand.
// k_R uses its per-page channel scale folded into the query (split into two BF16 terms so the
// product stays accurate to ~2^-16).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace mlaq {
namespace {

constexpr int kThreads = 128;
constexpr int kCtasPerSm = 3;  // resident CTAs per SM the register budget is sized for
constexpr int kStages = 8;
constexpr int kTile = 16;
constexpr int kRowStride = 24;              // floats per head row in the score / P exchange
constexpr int kBf16RowBytes = kRow * 2 + 16;  // padded BF16 row in shared memory (1168 B)
constexpr long long kWaitBudget = 4ll << 30;  // ~2 s at 2 GHz before a wait gives up
constexpr int kMaxSplitPages = 512;          // page ids of a split cached in shared memory
constexpr float kRescaleSlack = 8.f;          // softmax weights stay <= 2^8 between rescales
constexpr float kStrictScale = 255.f;         // a token scale >= this forces weights <= 1 (FP16 safety)

__host__ __device__ constexpr int packed_stage_bytes(int bits) { return kTile * 64 * bits + 512 + 256 + 256; }
__host__ __device__ constexpr int stage_region_bytes(int bits) {
  return (kStages * packed_stage_bytes(bits) > 2 * kTile * kBf16RowBytes) ? kStages * packed_stage_bytes(bits)
                                                                          : 2 * kTile * kBf16RowBytes;
}
constexpr int kSbufFloats = 2 * 4 * 16 * kRowStride;
constexpr int kPbufFloats = 2 * 16 * kRowStride;
__host__ __device__ constexpr int smem_bytes(int bits) {
  return stage_region_bytes(bits) + (kSbufFloats + kPbufFloats + 2 * 16) * 4 + kStages * 8 + 2 * 4 +
         kMaxSplitPages * 4;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float half_lo(uint32_t w) { return __half2float(__ushort_as_half(static_cast<uint16_t>(w & 0xffffu))); }
__device__ __forceinline__ float half_hi(uint32_t w) { return __half2float(__ushort_as_half(static_cast<uint16_t>(w >> 16))); }

struct Shared {
  uint8_t* stages;
  float* sbuf;   // [2][4 warps][16 heads][kRowStride]
  float* pbuf;   // [2][16 heads][kRowStride]
  float* alpha;  // [2][16]
  uint64_t* bars;
  int* strict;   // [2] per exchange buffer: a sub-tile needs an exact running max
  int* pids;     // [kMaxSplitPages] physical page ids of the split's pages (packed path)
};

template <int BITS>
__device__ __forceinline__ Shared carve(uint8_t* smem) {
  Shared s;
  s.stages = smem;
  s.sbuf = reinterpret_cast<float*>(smem + stage_region_bytes(BITS));
  s.pbuf = s.sbuf + kSbufFloats;
  s.alpha = s.pbuf + kPbufFloats;
  s.bars = reinterpret_cast<uint64_t*>(s.alpha + 2 * 16);
  s.strict = reinterpret_cast<int*>(s.bars + kStages);
  s.pids = s.strict + 2;
  return s;
}

// Per-thread state shared by both token paths.
struct State {
  float o[16][4];  // readout accumulators: channel block cb (8 channels), C fragment
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

// ------------------------------------------------------------------ packed tokens
template <int BITS>
__device__ void packed_split(const DecodeParams& p, const Shared& sh, int b, int T, int split,
                             const uint32_t (&qa)[8][4], const float (&qsum)[2], const float (&qr)[8],
                             State& st, int32_t& flags) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int lo = p.S, hi = T - p.W;
  int sub_begin = 0, n_my = 0;
  if (hi > lo) {
    const int first = lo / kTile, last = (hi - 1) / kTile;
    const int n_total = last - first + 1;
    sub_begin = first + static_cast<int>((static_cast<long long>(n_total) * split) / p.n_split);
    const int sub_end = first + static_cast<int>((static_cast<long long>(n_total) * (split + 1)) / p.n_split);
    n_my = sub_end - sub_begin;
  }
  // validate the page ids this split reads; a bad id drops the split's work
  {
    bool bad = false;
    const int pg0 = (sub_begin * kTile) >> p.p_shift;
    const int pg1 = n_my > 0 ? (((sub_begin + n_my) * kTile - 1) >> p.p_shift) : pg0 - 1;
    for (int pg = pg0 + static_cast<int>(threadIdx.x); pg <= pg1; pg += kThreads) {
      const int32_t pid = __ldg(p.page_table + static_cast<size_t>(b) * p.max_pages + pg);
      bad |= pid < 0 || pid >= p.n_pages;
      if (pg - pg0 < kMaxSplitPages) sh.pids[pg - pg0] = pid;  // refills read ids from here
    }
    if (__syncthreads_or(bad)) {
      flags |= kErrBadPage;
      n_my = 0;
    }
  }
  if (n_my == 0) return;

  constexpr int kStageBytes = packed_stage_bytes(BITS);
  constexpr int kLatBytes = kTile * 64 * BITS;
  const uint8_t* pool = p.pool;
  // Stage i is filled by four bulk copies, one issued by lane 0 of each warp (the stage's
  // mbarrier expects four arrivals), so no warp carries the whole producer load.
  auto issue_part = [&](int i, int part) {
    const int k = sub_begin + i;
    const int pg = (k * kTile) >> p.p_shift, tp0 = (k * kTile) & (p.P - 1);
    const int pg0 = (sub_begin * kTile) >> p.p_shift;
    const int32_t pid = pg - pg0 < kMaxSplitPages ? sh.pids[pg - pg0]
                                                 : __ldg(p.page_table + static_cast<size_t>(b) * p.max_pages + pg);
    const uint8_t* base = pool + static_cast<size_t>(pid) * static_cast<size_t>(p.page_bytes);
    uint8_t* dst = sh.stages + (i % kStages) * kStageBytes;
    uint64_t* bar = sh.bars + (i % kStages);
    if (part == 0) {
      mbar_arrive_expect_tx(bar, kLatBytes);
      bulk_g2s(dst, base + (tp0 / 8) * 4 * (128 * BITS), kLatBytes, bar);
    } else if (part == 1) {
      mbar_arrive_expect_tx(bar, 512);
      bulk_g2s(dst + kLatBytes, base + static_cast<size_t>(p.P) * 64 * BITS + (tp0 / 16) * 512, 512, bar);
    } else if (part == 2) {
      mbar_arrive_expect_tx(bar, 256);
      bulk_g2s(dst + kLatBytes + 512, base + static_cast<size_t>(p.P) * (64 * BITS + 32) + tp0 * 16, 256, bar);
    } else {
      mbar_arrive_expect_tx(bar, 256);
      bulk_g2s(dst + kLatBytes + 768, base + static_cast<size_t>(p.P) * (64 * BITS + 48), 256, bar);
    }
  };
  int issued = 0;  // identical in every thread
  if (lane == 0)
    for (int i = 0; i < kStages && i < n_my; ++i) issue_part(i, warp);
  issued = n_my < kStages ? n_my : kStages;

  // per-page rope factors: query times channel scale split into two BF16 terms
  uint32_t qr_hi[4], qr_lo[4];
  float rqs[2] = {0.f, 0.f}, rbias[2] = {0.f, 0.f};
  int cur_pg = -1;

  for (int i = 0; i < n_my; ++i) {
    const int stg = i % kStages;
    const bool ok = mbar_wait_bounded(sh.bars + stg, (i / kStages) & 1, kWaitBudget);
    const uint8_t* sp = sh.stages + stg * kStageBytes;
    const int k = sub_begin + i, t0 = k * kTile;
    const int pg = t0 >> p.p_shift;
    if (pg != cur_pg) {
      cur_pg = pg;
      const uint32_t* rm = reinterpret_cast<const uint32_t*>(sp + kLatBytes + 768) + 16 * warp;
      // A fragment element (row, dim): dims 2q, 2q+1 (regs 0, 1) and 2q+8, 2q+9 (regs 2, 3)
      const int dims[4] = {2 * q, 2 * q + 1, 2 * q + 8, 2 * q + 9};
      float sc[4], mn[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t w = rm[dims[e]];
        sc[e] = half_lo(w);
        mn[e] = half_hi(w);
      }
      float hi_v[8], lo_v[8];
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
      }
      // fragment regs: a0 (row g, dims 2q..), a1 (row g+8, dims 2q..), a2 (row g, 2q+8..), a3 (row g+8, 2q+8..)
      qr_hi[0] = pack_bf16x2(hi_v[0], hi_v[1]);
      qr_hi[1] = pack_bf16x2(hi_v[4], hi_v[5]);
      qr_hi[2] = pack_bf16x2(hi_v[2], hi_v[3]);
      qr_hi[3] = pack_bf16x2(hi_v[6], hi_v[7]);
      qr_lo[0] = pack_bf16x2(lo_v[0], lo_v[1]);
      qr_lo[1] = pack_bf16x2(lo_v[4], lo_v[5]);
      qr_lo[2] = pack_bf16x2(lo_v[2], lo_v[3]);
      qr_lo[3] = pack_bf16x2(lo_v[6], lo_v[7]);
    }

    // ---- unpack codes as BF16 integers 128 + n (exact), fragment layout of the page
    uint32_t bq[2][8][2];  // [n-block][k-chunk][reg]
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
      const uint8_t* blk = sp + (nb * 4 + warp) * (128 * BITS) + lane * (4 * BITS);
      if constexpr (BITS == 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(blk);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int s = 0; s < 4; ++s)
            bq[nb][2 * j + (s >> 1)][s & 1] = and_or(w4[j] >> (4 * s), 0x000f000fu, 0x43004300u);
      } else {
        const uint2 v = *reinterpret_cast<const uint2*>(blk);
        const uint32_t w2[2] = {v.x, v.y};
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int s = 0; s < 8; ++s)
            bq[nb][4 * j + (s >> 1)][s & 1] = and_or(w2[j] >> (2 * s), 0x00030003u, 0x43004300u);
      }
    }
    uint32_t rb[2][2];
    {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(sp + kLatBytes + warp * 128 + lane * 4);
#pragma unroll
      for (int s = 0; s < 4; ++s) rb[s >> 1][s & 1] = and_or(w >> (4 * s), 0x000f000fu, 0x43004300u);
    }

    // ---- scores on tensor cores
    // four independent accumulation chains per n-block pair keep the tensor pipe busy
    float acc[2][4], acc1[2][4], racc[2][4];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
      mma_bf16_16816_z(acc[nb], qa[0], bq[nb][0][0], bq[nb][0][1]);
      mma_bf16_16816_z(acc1[nb], qa[1], bq[nb][1][0], bq[nb][1][1]);
    }
#pragma unroll
    for (int kc = 2; kc < 8; kc += 2)
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        mma_bf16_16816(acc[nb], qa[kc], bq[nb][kc][0], bq[nb][kc][1]);
        mma_bf16_16816(acc1[nb], qa[kc + 1], bq[nb][kc + 1][0], bq[nb][kc + 1][1]);
      }
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
      mma_bf16_16816_z(racc[nb], qr_hi, rb[nb][0], rb[nb][1]);
      mma_bf16_16816(racc[nb], qr_lo, rb[nb][0], rb[nb][1]);
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[nb][e] += acc1[nb][e];
    }
    // token metadata: group `warp`, tokens 8nb + 2q + e
    float tsc[2][2], tmn[2][2];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int tok = 8 * nb + 2 * q + e;
        const uint32_t w = *reinterpret_cast<const uint32_t*>(sp + kLatBytes + 512 + (tok * 4 + warp) * 4);
        tsc[nb][e] = half_lo(w);
        tmn[nb][e] = half_hi(w);
      }
    float part[2][4];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = e >> 1, c = e & 1;
        part[nb][e] = tsc[nb][c] * (acc[nb][e] - 128.f * qsum[r]) + tmn[nb][c] * qsum[r] +
                      (racc[nb][e] - 128.f * rqs[r]) + rbias[r];
      }
    // token scales large enough that p * scale could overflow FP16 when p reaches 2^8
    const int buf = i & 1;
    if (fmaxf(fmaxf(tsc[0][0], tsc[0][1]), fmaxf(tsc[1][0], tsc[1][1])) >= kStrictScale) sh.strict[buf] = 1;

    // transpose the codes into the readout operand while the exchange is in flight:
    // 0x4300|n read as FP16 is 3.5 + n/512; subtracting 3.5 leaves n/512 exactly
#pragma unroll
    for (int kc = 0; kc < 8; ++kc)
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) bq[nb][kc][r] = hsub2_u32(movmatrix_t(bq[nb][kc][r]), 0x43004300u);

    if (exchange_partials(sh, buf, part, !ok)) {
      flags |= kErrTimeout;
      // orderly exit: bounded waits for the copies still in flight into this CTA
      if (threadIdx.x == 0)
        for (int j = i; j < issued; ++j)
          (void)mbar_wait_bounded(sh.bars + (j % kStages), (j / kStages) & 1, kWaitBudget >> 4);
      break;
    }
    // the previous stage is free once every warp passed the first exchange barrier
    if (i >= 1 && issued < n_my) {
      if (lane == 0) {
        fence_proxy_async_smem();
        issue_part(issued, warp);
      }
      ++issued;
    }
    softmax_publish(sh, buf, t0, lo, hi, p.scale_log2, st);

    // ---- readout: A = P * token scale (FP16), B = codes / 512 (FP16, exact)
    float2 pf[4];
    load_p(sh, buf, pf);
    uint32_t a[4];
    a[0] = pack_f16x2(pf[0].x * tsc[0][0], pf[0].y * tsc[0][1]);
    a[1] = pack_f16x2(pf[1].x * tsc[0][0], pf[1].y * tsc[0][1]);
    a[2] = pack_f16x2(pf[2].x * tsc[1][0], pf[2].y * tsc[1][1]);
    a[3] = pack_f16x2(pf[3].x * tsc[1][0], pf[3].y * tsc[1][1]);
    st.mterm[0] += pf[0].x * tmn[0][0] + pf[0].y * tmn[0][1] + pf[2].x * tmn[1][0] + pf[2].y * tmn[1][1];
    st.mterm[1] += pf[1].x * tmn[0][0] + pf[1].y * tmn[0][1] + pf[3].x * tmn[1][0] + pf[3].y * tmn[1][1];
#pragma unroll
    for (int kc = 0; kc < 8; ++kc)
#pragma unroll
      for (int r = 0; r < 2; ++r) mma_f16_16816(st.o[2 * kc + r], a, bq[0][kc][r], bq[1][kc][r]);
  }
}

// ------------------------------------------------------------------ protected (BF16) tokens
__device__ void bf16_split(const DecodeParams& p, const Shared& sh, int b, int T, const uint32_t (&qa)[8][4],
                           const uint32_t (&qra)[4], State& st, int32_t& flags) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s_end = min(p.S, T);
  const int r_beg = max(T - p.W, s_end);
  const int has_sink = s_end > 0 ? 1 : 0;
  const int n_tiles = has_sink + (T - r_beg + kTile - 1) / kTile;
  if (n_tiles <= 0) return;
  constexpr int kStageBytes = kTile * kBf16RowBytes;

  auto tile_range = [&](int i, int& start, int& count) {
    if (has_sink && i == 0) {
      start = 0;
      count = s_end;
    } else {
      start = r_beg + (i - has_sink) * kTile;
      count = min(kTile, T - start);
    }
  };
  auto row_ptr = [&](int t) -> const uint16_t* {
    return t < p.S ? p.sink + (static_cast<size_t>(b) * p.S + t) * kRow
                   : p.ring + (static_cast<size_t>(b) * p.W + (t % p.W)) * kRow;
  };
  auto issue = [&](int i) {
    int start, count;
    tile_range(i, start, count);
    uint8_t* dst = sh.stages + (i & 1) * kStageBytes;
    uint64_t* bar = sh.bars + (i & 1);
    mbar_arrive_expect_tx(bar, kTile * kRow * 2);
    for (int j = 0; j < kTile; ++j) {
      const int t = start + (j < count ? j : 0);  // rows past the count repeat a valid row (masked later)
      bulk_g2s(dst + j * kBf16RowBytes, row_ptr(t), kRow * 2, bar);
    }
  };
  if (threadIdx.x == 0) {
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
    if (threadIdx.x == 0 && i + 2 < n_tiles) {
      fence_proxy_async_smem();
      issue(i + 2);
    }
  }
}

template <int BITS>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const Shared sh = carve<BITS>(smem);
  const int split = blockIdx.x, hb = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int h0 = hb * 16;
  int32_t flags = 0;

  int T = __ldg(p.seq_lens + b);
  if (T < 0 || static_cast<long long>(T) > static_cast<long long>(p.max_pages) * p.P) {
    flags |= kErrSeqOverflow;
    T = 0;
  }
  if (threadIdx.x == 0) {
    // packed stages: four arrivals (one copy per warp); protected-token stages: one arrival
    for (int i = 0; i < kStages; ++i) mbar_init(sh.bars + i, split == p.n_split ? 1 : 4);
    fence_mbar_init();
    sh.strict[0] = sh.strict[1] = 0;
  }
  __syncthreads();

  // query fragments for latent group `warp` (BF16, exact) and their per-row sums
  uint32_t qa[8][4];
  float qsum[2] = {0.f, 0.f};
  {
    const uint32_t* r0 = reinterpret_cast<const uint32_t*>(p.q_lat + (static_cast<size_t>(b) * p.H + h0 + g) * kLatent + 128 * warp);
    const uint32_t* r1 = r0 + 8 * kLatent / 2;
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) {
      qa[kc][0] = __ldg(r0 + 8 * kc + q);
      qa[kc][1] = __ldg(r1 + 8 * kc + q);
      qa[kc][2] = __ldg(r0 + 8 * kc + 4 + q);
      qa[kc][3] = __ldg(r1 + 8 * kc + 4 + q);
      qsum[0] += bf16_lo(qa[kc][0]) + bf16_hi(qa[kc][0]) + bf16_lo(qa[kc][2]) + bf16_hi(qa[kc][2]);
      qsum[1] += bf16_lo(qa[kc][1]) + bf16_hi(qa[kc][1]) + bf16_lo(qa[kc][3]) + bf16_hi(qa[kc][3]);
    }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      qsum[0] += __shfl_xor_sync(0xffffffffu, qsum[0], o);
      qsum[1] += __shfl_xor_sync(0xffffffffu, qsum[1], o);
    }
  }
  // k_R query slice: rows g, g+8, dims 16w + {2q, 2q+1, 2q+8, 2q+9}
  uint32_t qra[4];
  float qr[8];
  {
    const uint32_t* r0 = reinterpret_cast<const uint32_t*>(p.q_rope + (static_cast<size_t>(b) * p.H + h0 + g) * kRope + 16 * warp);
    const uint32_t* r1 = r0 + 8 * kRope / 2;
    qra[0] = __ldg(r0 + q);
    qra[1] = __ldg(r1 + q);
    qra[2] = __ldg(r0 + 4 + q);
    qra[3] = __ldg(r1 + 4 + q);
    qr[0] = bf16_lo(qra[0]);
    qr[1] = bf16_hi(qra[0]);
    qr[2] = bf16_lo(qra[2]);
    qr[3] = bf16_hi(qra[2]);
    qr[4] = bf16_lo(qra[1]);
    qr[5] = bf16_hi(qra[1]);
    qr[6] = bf16_lo(qra[3]);
    qr[7] = bf16_hi(qra[3]);
  }

  State st;
#pragma unroll
  for (int cb = 0; cb < 16; ++cb) st.o[cb][0] = st.o[cb][1] = st.o[cb][2] = st.o[cb][3] = 0.f;
  st.mterm[0] = st.mterm[1] = 0.f;
  st.m_run = -INFINITY;
  st.l_part = 0.f;

  const bool is_bf16 = split == p.n_split;
  if (is_bf16) bf16_split(p, sh, b, T, qa, qra, st, flags);
  else packed_split<BITS>(p, sh, b, T, split, qa, qsum, qr, st, flags);

  // ---- partial results
  const int NS = p.n_split + 1;
  float mt0 = st.mterm[0], mt1 = st.mterm[1];
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) {
    mt0 += __shfl_xor_sync(0xffffffffu, mt0, o);
    mt1 += __shfl_xor_sync(0xffffffffu, mt1, o);
  }
  const float oscale = is_bf16 ? 1.f : 512.f;
  float* o0 = p.o_part + ((static_cast<size_t>(b) * p.H + h0 + g) * NS + split) * kLatent + 128 * warp;
  float* o1 = p.o_part + ((static_cast<size_t>(b) * p.H + h0 + g + 8) * NS + split) * kLatent + 128 * warp;
#pragma unroll
  for (int cb = 0; cb < 16; ++cb) {
    *reinterpret_cast<float2*>(o0 + 8 * cb + 2 * q) =
        make_float2(oscale * st.o[cb][0] + mt0, oscale * st.o[cb][1] + mt0);
    *reinterpret_cast<float2*>(o1 + 8 * cb + 2 * q) =
        make_float2(oscale * st.o[cb][2] + mt1, oscale * st.o[cb][3] + mt1);
  }
  float l_run = st.l_part;
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) l_run += __shfl_xor_sync(0xffffffffu, l_run, o);
  if ((lane & 7) == 0) {
    const int hh = h0 + 4 * warp + (lane >> 3);
    float* ml = p.ml_part + ((static_cast<size_t>(b) * p.H + hh) * NS + split) * 2;
    ml[0] = st.m_run;
    ml[1] = l_run;
  }
  flags = __reduce_or_sync(0xffffffffu, flags);
  if (lane == 0 && flags) atomicOr(p.err, flags);
}

// Merge the split partials of one (sequence, head): warp-shuffle log-sum-exp reduction of
// the split maxima and sums, then a weighted sum of the partial outputs.
__global__ void __launch_bounds__(128) combine_kernel(const DecodeParams p) {
  const int bh = blockIdx.x;
  const int NS = p.n_split + 1;
  const int lane = threadIdx.x & 31;
  const float* ml = p.ml_part + static_cast<size_t>(bh) * NS * 2;
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
    const float* op = p.o_part + static_cast<size_t>(bh) * NS * kLatent + 4 * threadIdx.x;
    for (int s = 0; s < NS; ++s) {
      const float w = exp2f(ml[2 * s] - m);
      if (w == 0.f) continue;
      const float4 v = *reinterpret_cast<const float4*>(op + static_cast<size_t>(s) * kLatent);
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
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

}  // namespace

int decode_num_splits(int B, int H, int max_pages, int P, int num_sms) {
  const int groups = B * (H / 16);
  const int target = kCtasPerSm * num_sms;  // one full wave of resident CTAs
  int ns = target / (groups > 0 ? groups : 1) - 1;
  const long long max_sub = (static_cast<long long>(max_pages) * P) / kTile;
  int cap = static_cast<int>(max_sub / 4);
  if (cap < 1) cap = 1;
  if (ns > cap) ns = cap;
  if (ns > 64) ns = 64;
  if (ns < 1) ns = 1;
  return ns;
}

size_t decode_workspace_bytes(int B, int H, int n_split) {
  const size_t NS = static_cast<size_t>(n_split) + 1;
  return static_cast<size_t>(B) * H * NS * (kLatent + 2) * sizeof(float);
}

// The dynamic shared-memory opt-in is a per-device function attribute: set it once per device
// (never inside a stream capture after the first call).
template <int BITS>
cudaError_t ensure_smem_attr() {
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!done[dev]) {
    e = cudaFuncSetAttribute(decode_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes(BITS));
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return cudaSuccess;
}

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
  const dim3 grid(p.n_split + 1, p.H / 16, p.B);
  cudaError_t e;
  if (p.bits_c == 4) {
    if ((e = ensure_smem_attr<4>()) != cudaSuccess) return e;
    decode_kernel<4><<<grid, kThreads, smem_bytes(4), stream>>>(p);
  } else {
    if ((e = ensure_smem_attr<2>()) != cudaSuccess) return e;
    decode_kernel<2><<<grid, kThreads, smem_bytes(2), stream>>>(p);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  combine_kernel<<<p.B * p.H, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ built-in scratch
// Device-resident scratch used by mla_qcache_decode_attn_noalloc in place of a caller workspace.
// It lives for as long as the library is loaded, on every device that loads it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch for the current device. The host-side name of the array is only
// a stand-in, so the address is looked up once per device (with that device current) and cached.
cudaError_t noalloc_scratch(void** out) {
  static void* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace mlaq
