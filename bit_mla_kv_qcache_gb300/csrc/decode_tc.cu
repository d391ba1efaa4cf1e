// Decode attention for head counts that are multiples of 64, on the fifth-generation tensor
// cores (QuantMLA page, abstract and appendix Figure 8; RAQ-MLA page, Figures 3-4 and
// appendix Table 5).
//
// Grid (B, H/64, n_split). CTA (b, hq, split) handles heads 64hq .. 64hq+63 of sequence b over
// share `split` of the packed tokens [S, T-W), in tiles of 128 tokens; thread (lane t, half h)
// loads token t's code chunks of channel half h of every latent group. Per tile:
//   1. scores, exact products, one latent group at a time: the group's codes enter tensor memory
//      as FP16 subnormals (a masked code field n at bit offset k of a half is exactly
//      n * 2^(k-24)), the A operand of tcgen05.mma kind::f16; the query (B, in shared memory)
//      carries the inverse field weight, so the tensor cores produce
//      R_g[t][h] = 2^(E-24) sum_{c in g} q_c code_tc (FP32 in tensor memory, two accumulators so
//      one group drains while the next is multiplied). The threads, one token per lane, apply
//      the token's group scale and minimum in FP32:
//      score = sum_g (scale_tg R_g + min_tg 2^(E-24) sum_{c in g} q_c) + k_R part. k_R is
//      dequantized (per-channel page scale and minimum) into the same tensor-memory operand as
//      a high and a low FP16 part, so its products carry ~2^-22 relative error. The score
//      products read only the query from shared memory, whose port the readout's operands need;
//   2. while the groups are scored, their dequantized values v = scale * code + min (FP16, one
//      rounding) go to a shared-memory tile, token-major;
//   3. softmax on the scores (one token per lane), running max per head raised only when a
//      score exceeds it by more than 2^8 (weights stay <= 2^8 in FP16);
//   4. readout O^T[512 ch x 64 heads] += V^T . P: the value tile read channel-major (M-major A),
//      B = the weights stored heads-contiguous. O accumulates in tensor memory over the share.
// Shared-memory operands use the no-swizzle canonical layout of 8x8 core matrices (128 B each):
// one token's 8 channels per 16-byte row. The latent channels inside each 8 (INT4) or 16 (INT2)
// channel block are in the order the unpack produces them (the same order in the tensor-memory
// codes and the value tile); the query follows that order and the epilogue writes each output
// row to its own channel.
// The protected (BF16) tokens are handled by the 16-head kernel's protected CTAs; the merge
// kernel combines every partial.
#include <cuda_fp16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace mlaq {
namespace {

constexpr int kTcThreads = 256;  // 8 warps; warps w and w+4 share tensor-memory lanes 32(w%4)..
constexpr int kTcHeads = 64;     // MMA N
constexpr int kTcTok = 128;      // tokens per tile: MMA M of the scores, K of the readout
constexpr long long kTcWaitBudget = 4ll << 30;
constexpr float kTcSlack = 8.f;  // weights stay <= 2^8 between raises of the running max

// shared memory (bytes)
constexpr int kTileOff = 0;
constexpr int kTileBytes = kTcTok * kLatent * 2;  // 128 tok x 512 ch FP16: core (cb, tb) at (16 cb + tb) * 128
constexpr int kQOff = kTileOff + kTileBytes;
constexpr int kQBytes = kTcHeads * kRow * 2;      // 64 heads x 576 ch FP16: core (cb, hb) at (8 cb + hb) * 128
constexpr int kPOff = kQOff + kQBytes;
constexpr int kPBytes = kTcTok * kTcHeads * 2;    // 128 tok x 64 heads FP16: core (tb, hb) at (8 tb + hb) * 128
constexpr int kMiscOff = kPOff + kPBytes;
constexpr int kBarOff = kMiscOff;                 // [0] scores done, [1] readout done, [2] query rows
constexpr int kTmemSlotOff = kMiscOff + 32;
constexpr int kMOff = kMiscOff + 64;              // running max per head (log2 units)
constexpr int kHsOff = kMOff + 256;               // MMA score -> log2 units, per head
constexpr int kRedOff = kHsOff + 256;             // [4 lane quarters][64 heads] floats
constexpr int kQsOff = kRedOff + 1024;            // [4 groups][64 heads] 2^(E-24) sum_{c in g} q_c
constexpr int kKrmOff = kQsOff + 1024;           // k_R (scale, min) of the tile's pages [4][64]
constexpr int kPidOff = kKrmOff + 1024;          // page ids of the share (first kPidCache)
constexpr int kPidCache = 256;
constexpr int kTcSmem = kPidOff + 4 * kPidCache;
static_assert(kTcSmem <= 227 * 1024, "one CTA per SM");
// The BF16 query rows of the head block, staged in the tile region before the first tile: latent
// rows padded to kQRowWords 32-bit words (the prologue's reads fall in distinct banks), then the
// k_R rows.
constexpr int kQRowWords = kLatent / 2 + 4;
constexpr int kQRopeStage = kTcHeads * kQRowWords * 4;
static_assert(kQRopeStage + kTcHeads * kRope * 2 <= kTileBytes && (kQRowWords * 4) % 16 == 0, "query staging");
static_assert(kTileOff % 1024 == 0 && kQOff % 1024 == 0 && kPOff % 1024 == 0, "operand alignment");

// tensor memory columns (512 allocated; FP32 accumulators, lane = row)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;       // O^T of latent group g (128 channels x 64 heads) at 64 g
constexpr uint32_t kColSA = 256;    // score buffers S^T (128 tokens x 64 heads)
constexpr uint32_t kColSB = 320;
constexpr uint32_t kColA = 384;     // A operand of the score products: one latent group's codes (128 tokens
                                    // x 128 channels, a pair per column), then k_R:
constexpr uint32_t kColKrHi = 384;  // k_R high FP16 parts: 128 tokens x 64 channels, a pair per column
constexpr uint32_t kColKrLo = 416;  // k_R low FP16 parts
constexpr uint32_t kColL = 448;     // per-token-lane partial sums of the weights, 64 heads

// instruction descriptors (kind::f16): D FP32, A/B FP16, M = 128, N = 64
constexpr uint32_t kIdescScore = (1u << 4) | (uint32_t(kTcHeads >> 3) << 17) | (uint32_t(kTcTok >> 4) << 24);
constexpr uint32_t kIdescRead = kIdescScore | (1u << 15) | (1u << 16);  // A and B M/N-major

// tile channel position -> latent channel (the unpack order of one code word)
template <int BITS>
__host__ __device__ constexpr int tile_to_orig(int c) {
  if (BITS == 4) {
    const int p = c & 7;
    return (c & ~7) | ((p & 1) ? 4 + (p >> 1) : (p >> 1));
  }
  const int p = c & 15, r = p >> 3, k = p & 7;
  return (c & ~15) | ((k & 1) ? 8 + 4 * r + (k >> 1) : 4 * r + (k >> 1));
}

// log2 of the field weight of tile channel position c in the code operand (INT4: nibble at bit 0
// or 4 of its half; INT2: field at bit 0, 2, 4 or 6)
template <int BITS>
__host__ __device__ constexpr int tile_log2w(int c) {
  return BITS == 4 ? 4 * (((c & 7) >> 1) & 1) : 2 * (((c & 7) >> 1) & 3);
}

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  // start, leading-dimension offset (K direction), stride offset (M/N direction), version 1,
  // no swizzle
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46);
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile("{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d),
               "l"(a), "l"(b), "r"(idesc), "r"(static_cast<uint32_t>(acc))
               : "memory");
}
__device__ __forceinline__ void tc_mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile("{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d),
               "r"(a), "l"(b), "r"(idesc), "r"(static_cast<uint32_t>(acc))
               : "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
// (1024 + n_lo, 1024 + n_hi) as FP16 -> scale * n + min, one rounding per half
__device__ __forceinline__ uint32_t dq2(uint32_t magic_codes, uint32_t s2, uint32_t m2) {
  const __half2 k1024 = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
  const __half2 n = __hsub2(*reinterpret_cast<const __half2*>(&magic_codes), k1024);
  const __half2 v = __hfma2(n, *reinterpret_cast<const __half2*>(&s2), *reinterpret_cast<const __half2*>(&m2));
  return *reinterpret_cast<const uint32_t*>(&v);
}

// per-head constants are re-read from shared memory where they are used (volatile: never
// hoisted out of the tile loop into registers)
__device__ __forceinline__ float lds_f32(const float* p) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(smem_addr(p)));
  return v;
}
__device__ __forceinline__ float4 lds_f32x4(const float* p) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(smem_addr(p)));
  return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

template <int BITS>
struct TcGeom {
  static constexpr int kRowBytes = 64 * BITS;                   // region A bytes per token
  static constexpr int kChunks = kRowBytes / 16;                // 16-byte chunks per token
  static constexpr int kItems = kTcTok * kChunks / kTcThreads;  // latent chunks per thread and tile
  static constexpr int kCpg = kItems / 4;                       // chunks per latent group and channel half
  // Thread (token lane t, channel half h) holds, for each latent group g, the kCpg chunks of
  // channels 128 g + 64 h .. 128 g + 64 h + 63 of token t; item it = kCpg g + c.
  __device__ static int chunk_of(int half, int it) { return (it / kCpg) * (kChunks / 4) + half * kCpg + it % kCpg; }
};
static_assert(TcGeom<4>::kCpg * 32 * 4 == 256 && TcGeom<2>::kCpg * 64 * 4 == 256, "a channel half of a group per thread");

// The packed data one thread unpacks for one tile, loaded a tile ahead.
template <int BITS>
struct TileRegs {
  uint4 lat[TcGeom<BITS>::kItems];     // latent code chunks of this lane's token (unpacked twice)
  uint4 tmeta;                         // (scale, min) of the 4 groups of this lane's token
  uint4 krw[2];                        // k_R code words of this lane's token, 32 channels
  uint32_t krm;                        // one k_R (scale, min) word of the tile's pages (staged)
};

__device__ __forceinline__ float half_bits_lo(uint32_t w) { return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu))); }
__device__ __forceinline__ float half_bits_hi(uint32_t w) { return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16))); }

template <int BITS>
__global__ void __launch_bounds__(kTcThreads, 1) decode_tc_kernel(const DecodeParams p) {
  using G = TcGeom<BITS>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);  // [0] scores, [1] readout
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kTmemSlotOff);
  float* m_run = reinterpret_cast<float*>(smem + kMOff);
  float* hsc = reinterpret_cast<float*>(smem + kHsOff);
  float* red = reinterpret_cast<float*>(smem + kRedOff);
  float* qs = reinterpret_cast<float*>(smem + kQsOff);
  int32_t* pids = reinterpret_cast<int32_t*>(smem + kPidOff);
  uint32_t* krm_s = reinterpret_cast<uint32_t*>(smem + kKrmOff);
  const uint32_t tile_a = smem_addr(smem + kTileOff), q_a = smem_addr(smem + kQOff), p_a = smem_addr(smem + kPOff);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x, h0 = blockIdx.y * kTcHeads, split = blockIdx.z;
  const int quarter = warp & 3, half = warp >> 2;  // TMEM lanes 32*quarter.., head/channel half
  const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
  const int NS = p.n_split + p.n_q;
  int32_t flags = 0;

  // The head block's query rows into the (still unused) tile region by bulk copies, first thing:
  // their round trip overlaps the length and page-table reads (16-byte aligned query pointers;
  // else they are read element by element below).
  const bool q_bulk = ((reinterpret_cast<uintptr_t>(p.q_lat) | reinterpret_cast<uintptr_t>(p.q_rope)) & 15u) == 0;
  uint32_t* const qlat_s = reinterpret_cast<uint32_t*>(smem + kTileOff);
  uint32_t* const qrope_s = reinterpret_cast<uint32_t*>(smem + kTileOff + kQRopeStage);
  if (q_bulk) {
    if (tid == 0) {
      mbar_init(bars + 2, 1);
      fence_mbar_init();
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bars + 2, kTcHeads * (kLatent + kRope) * 2);
    }
    __syncthreads();
    if (tid < kTcHeads)
      bulk_g2s(qlat_s + tid * kQRowWords, p.q_lat + (static_cast<size_t>(b) * p.H + h0 + tid) * kLatent, kLatent * 2,
               bars + 2);
    else if (tid == kTcHeads)
      bulk_g2s(qrope_s, p.q_rope + (static_cast<size_t>(b) * p.H + h0) * kRope, kTcHeads * kRope * 2, bars + 2);
  }

  int T_old;
  const int T = decode_seq_len(p, b, T_old, flags);
  const int lo = p.S, hi = T - p.W;
  int tile_begin = 0, n_my = 0;
  if (hi > lo) {
    const int first = lo / kTcTok, last = (hi - 1) / kTcTok;
    const int n_total = last - first + 1;
    tile_begin = first + static_cast<int>((static_cast<long long>(n_total) * split) / p.n_split);
    const int tile_end = first + static_cast<int>((static_cast<long long>(n_total) * (split + 1)) / p.n_split);
    n_my = tile_end - tile_begin;
  }
  // page ids of the share: validated, the first kPidCache kept in shared memory
  const int pg0 = (tile_begin * kTcTok) >> p.p_shift;
  if (n_my > 0) {
    const int end_tok = min(hi, (tile_begin + n_my) * kTcTok);
    const int pg1 = (end_tok - 1) >> p.p_shift;
    bool bad = false;
    for (int pg = pg0 + tid; pg <= pg1; pg += kTcThreads) {
      const int32_t pid = __ldg(p.page_table + static_cast<size_t>(b) * p.max_pages + pg);
      bad |= pid < 0 || pid >= p.n_pages;
      if (pg - pg0 < kPidCache) pids[pg - pg0] = pid;
    }
    if (__syncthreads_or(bad)) {
      flags |= kErrBadPage;
      n_my = 0;
    }
  }
  if (n_my == 0) {  // empty share: the merge sees sum 0 and skips the slot
    if (q_bulk && !mbar_wait_bounded(bars + 2, 0, kTcWaitBudget)) flags |= kErrTimeout;  // the copies landed
    if (tid < kTcHeads) {
      float* ml = p.ml_part + ((static_cast<size_t>(b) * p.H + h0 + tid) * NS + split) * 2;
      ml[0] = -INFINITY;
      ml[1] = 0.f;
    }
    flags = __reduce_or_sync(0xffffffffu, flags);
    if (lane == 0 && flags) atomicOr(p.err, flags);
    return;
  }

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    mbar_init(bars, 1);
    mbar_init(bars + 1, 1);
    fence_mbar_init();
  }

  // ---- per-tile packed loads (issued one tile ahead)
  const size_t P = static_cast<size_t>(p.P);
  auto page_base = [&](int pos) -> const uint8_t* {
    const int pg = pos >> p.p_shift;
    const int32_t pid = pg - pg0 < kPidCache ? pids[pg - pg0]
                                             : __ldg(p.page_table + static_cast<size_t>(b) * p.max_pages + pg);
    return p.pool + static_cast<size_t>(pid) * static_cast<size_t>(p.page_bytes);
  };
  TileRegs<BITS> R;
  // this lane's token row in region A of tile i (null past the end) and its XOR swizzle
  auto token_row = [&](int i, int& swz) -> const uint8_t* {
    const int pos = (tile_begin + i) * kTcTok + 32 * quarter + lane;
    const int slot = pos & (p.P - 1);
    swz = slot & 7;
    return pos < hi ? page_base(pos) + static_cast<size_t>(slot) * G::kRowBytes : nullptr;
  };
  // the code chunks of latent group g from a token row (zero past the end)
  auto load_group = [&](const uint8_t* row, int swz, int g) {
#pragma unroll
    for (int cc = 0; cc < G::kCpg; ++cc)
      R.lat[g * G::kCpg + cc] =
          row != nullptr ? __ldg(reinterpret_cast<const uint4*>(row + 16 * (G::chunk_of(half, g * G::kCpg + cc) ^ swz)))
                         : make_uint4(0u, 0u, 0u, 0u);
  };
  // the token and page metadata of tile i and its k_R codes
  auto load_meta = [&](int i) {
    const int t0 = (tile_begin + i) * kTcTok;
    const int pos = t0 + 32 * quarter + lane;
    R.tmeta = R.krw[0] = R.krw[1] = make_uint4(0u, 0u, 0u, 0u);
    if (pos < hi) {
      const uint8_t* base = page_base(pos);
      const int slot = pos & (p.P - 1);
      R.tmeta = __ldg(reinterpret_cast<const uint4*>(base + P * (G::kRowBytes + 32) + slot * 16));
      const uint8_t* regb = base + P * G::kRowBytes;
#pragma unroll
      for (int r = 0; r < 2; ++r)
        R.krw[r] = __ldg(reinterpret_cast<const uint4*>(regb + ((slot >> 4) * 4 + 2 * half + r) * 128 + (slot & 7) * 16));
    }
    // one word of region D per thread: page tid/64 of the tile, channel tid%64
    const int kpos = t0 + (tid >> 6) * p.P;
    R.krm = 0u;
    if ((tid >> 6) * p.P < kTcTok && kpos < hi)
      R.krm = __ldg(reinterpret_cast<const uint32_t*>(page_base(kpos) + P * (G::kRowBytes + 48)) + (tid & 63));
  };

  // the first tile, its latency overlapping the query's conversion
  {
    int swz;
    const uint8_t* row = token_row(0, swz);
#pragma unroll
    for (int g = 0; g < 4; ++g) load_group(row, swz, g);
  }
  load_meta(0);

  // ---- query: FP16, per-head power-of-two prescale 2^E, divided by the field weight of the
  // code operand at each tile position; per-group sums for the minimum terms. The BF16 rows are
  // in the tile region: bulk-copied at the start, or copied here with one batch of independent
  // loads when the query is not 16-byte aligned.
  {
    if (q_bulk) {
      if (!mbar_wait_bounded(bars + 2, 0, kTcWaitBudget)) {
        flags |= kErrTimeout;
        (void)mbar_wait_bounded(bars + 2, 0, kTcWaitBudget >> 4);
      }
    } else {
      // the query rows are 4-byte aligned (32-bit loads)
      const uint32_t* ql = reinterpret_cast<const uint32_t*>(p.q_lat + (static_cast<size_t>(b) * p.H + h0) * kLatent);
      const uint32_t* qr = reinterpret_cast<const uint32_t*>(p.q_rope + (static_cast<size_t>(b) * p.H + h0) * kRope);
#pragma unroll 12
      for (int it = 0; it < kTcHeads * (kRow / 2) / kTcThreads; ++it) {
        const int w = it * kTcThreads + tid, h = w / (kRow / 2), k = w - h * (kRow / 2);
        if (k < kLatent / 2) qlat_s[h * kQRowWords + k] = __ldg(ql + h * (kLatent / 2) + k);
        else qrope_s[h * (kRope / 2) + k - kLatent / 2] = __ldg(qr + h * (kRope / 2) + k - kLatent / 2);
      }
    }
    __syncthreads();
    const int h = tid >> 2, part = tid & 3;  // 4 threads per head
    // one pass over latent group `part` (its maximum magnitude and its sum) in 16-byte reads,
    // staggered so that the 8 threads of a quarter-warp (2 heads x 4 groups) hit distinct banks,
    // then this thread's quarter of the k_R row
    const uint32_t* row = qlat_s + h * kQRowWords + 64 * part;
    float mx = 0.f, gs = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint4 v = *reinterpret_cast<const uint4*>(row + 4 * ((k + 2 * part) & 15));
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = bf16_lo(w4[e]), hi = bf16_hi(w4[e]);
        mx = fmaxf(mx, fmaxf(fabsf(lo), fabsf(hi)));
        gs += lo + hi;
      }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint4 v = *reinterpret_cast<const uint4*>(qrope_s + h * (kRope / 2) + 8 * part + 4 * k);
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) mx = fmaxf(mx, fmaxf(fabsf(bf16_lo(w4[e])), fabsf(bf16_hi(w4[e]))));
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    bool range = false;
    const int E = prescale_exponent(mx, range);
    if (range) flags |= kErrRange;
    qs[part * kTcHeads + h] = gs * pow2_int(E - 24);
    if (part == 0) {
      hsc[h] = p.scale_log2 * pow2_int(24 - E);
      red[h] = static_cast<float>(E);
      m_run[h] = -INFINITY;
    }
    __syncthreads();
    for (int idx = tid; idx < kTcHeads * (kRow / 16); idx += kTcThreads) {
      const int hh = idx & (kTcHeads - 1), blk = idx >> 6;  // 16-channel block
      const int Eh = static_cast<int>(red[hh]);
      const bool lat = blk < kLatent / 16;
      const uint32_t* src = lat ? qlat_s + hh * kQRowWords + 8 * blk : qrope_s + hh * (kRope / 2) + 8 * (blk - kLatent / 16);
      const uint4 s0 = reinterpret_cast<const uint4*>(src)[0], s1 = reinterpret_cast<const uint4*>(src)[1];
      const uint32_t sw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
      float x[16];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        x[2 * k] = bf16_lo(sw[k]);
        x[2 * k + 1] = bf16_hi(sw[k]);
      }
      uint32_t o[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        // tile positions 2k, 2k+1 of this block hold the channels the unpack puts there
        float v0, v1;
        if (lat) {
          v0 = x[tile_to_orig<BITS>(2 * k) & 15] * pow2_int(Eh - tile_log2w<BITS>(2 * k));
          v1 = x[tile_to_orig<BITS>(2 * k + 1) & 15] * pow2_int(Eh - tile_log2w<BITS>(2 * k + 1));
        } else {
          v0 = x[2 * k] * pow2_int(Eh);
          v1 = x[2 * k + 1] * pow2_int(Eh);
        }
        const __half2 hv = __floats2half2_rn(v0, v1);
        o[k] = *reinterpret_cast<const uint32_t*>(&hv);
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int cb = 2 * blk + r;
        st_shared_v4(q_a + (cb * 8 + (hh >> 3)) * 128 + (hh & 7) * 16, o[4 * r], o[4 * r + 1], o[4 * r + 2],
                     o[4 * r + 3]);
      }
    }
  }

  uint32_t tmem = 0;
  // The latent codes of group g into tensor memory as weighted FP16 subnormals: the A operand of
  // the group's score products (lane = token, a channel pair per column, columns 4 m + r for the
  // m-th 8-channel block of this thread's channel half).
  auto codes_to_tmem = [&](int g) {
    uint32_t c[2][16];
#pragma unroll
    for (int cc = 0; cc < G::kCpg; ++cc) {
      const uint4 v = R.lat[g * G::kCpg + cc];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t w8 = w[k] >> 8;
        if (BITS == 4) {
          const int m = 4 * cc + k;
          uint32_t* d = &c[m >> 2][4 * (m & 3)];
          d[0] = w[k] & 0x000F000Fu;
          d[1] = w[k] & 0x00F000F0u;
          d[2] = w8 & 0x000F000Fu;
          d[3] = w8 & 0x00F000F0u;
        } else {
          const int m = 2 * k;
          uint32_t* d = &c[m >> 2][4 * (m & 3)];
          d[0] = w[k] & 0x00030003u;
          d[1] = w[k] & 0x000C000Cu;
          d[2] = w[k] & 0x00300030u;
          d[3] = w[k] & 0x00C000C0u;
          d[4] = w8 & 0x00030003u;
          d[5] = w8 & 0x000C000Cu;
          d[6] = w8 & 0x00300030u;
          d[7] = w8 & 0x00C000C0u;
        }
      }
    }
    tmem_st16(tmem + lane_base + kColA + 32 * half, c[0]);
    tmem_st16(tmem + lane_base + kColA + 32 * half + 16, c[1]);
  };
  // k_R of tile i into tensor memory (the same columns, once the latent score products are done)
  // as high and low FP16 parts
  auto unpack_kr = [&](int i) {
    const int tt = 32 * quarter + lane;
    const int pos = (tile_begin + i) * kTcTok + tt;
    const int nn = ((pos & (p.P - 1)) >> 3) & 1;
    const uint32_t* mdp = krm_s + (tt >> p.p_shift) * 64 + 32 * half;  // staged before a barrier
    uint32_t md[32];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint4 v = *reinterpret_cast<const uint4*>(mdp + 4 * k);
      md[4 * k] = v.x;
      md[4 * k + 1] = v.y;
      md[4 * k + 2] = v.z;
      md[4 * k + 3] = v.w;
    }
    uint32_t khi[16], klo[16];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const uint32_t wq[4] = {R.krw[r].x, R.krw[r].y, R.krw[r].z, R.krw[r].w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t x = (wq[q] >> (4 * (2 * nn + h))) & 0x000F000Fu;
          const int lc = 16 * r + 8 * h + 2 * q;  // local channel pair (lc, lc+1)
          const float v0 = fmaf(half_bits_lo(md[lc]), static_cast<float>(x & 0xffu), half_bits_hi(md[lc]));
          const float v1 = fmaf(half_bits_lo(md[lc + 1]), static_cast<float>(x >> 16), half_bits_hi(md[lc + 1]));
          const __half2 vh = __floats2half2_rn(v0, v1);
          const __half2 vl = __floats2half2_rn(v0 - __low2float(vh), v1 - __high2float(vh));
          khi[lc >> 1] = *reinterpret_cast<const uint32_t*>(&vh);
          klo[lc >> 1] = *reinterpret_cast<const uint32_t*>(&vl);
        }
    }
    tmem_st16(tmem + lane_base + kColKrHi + 16 * half, khi);
    tmem_st16(tmem + lane_base + kColKrLo + 16 * half, klo);
  };
  // dequantized values v = scale * code + min of group g into the shared-memory tile (the
  // readout's operand): this lane's token, this thread's channel half; a warp's 32 tokens fill
  // 512 contiguous bytes of each 8-channel block
  auto values_to_smem = [&](int g) {
    constexpr uint32_t kMagic = 0x64006400u;
    const uint32_t lm = g == 0 ? R.tmeta.x : g == 1 ? R.tmeta.y : g == 2 ? R.tmeta.z : R.tmeta.w;
    const uint32_t s2 = prmt(lm, 0u, 0x1010u), m2 = prmt(lm, 0u, 0x3232u);
    const uint32_t row = tile_a + 16 * (32 * quarter + lane);
#pragma unroll
    for (int cc = 0; cc < G::kCpg; ++cc) {
      const uint4 v = R.lat[g * G::kCpg + cc];
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (BITS == 4) {
          const int cb = 16 * g + 8 * half + 4 * cc + k;
          st_shared_v4(row + cb * 2048, dq2((w[k] & 0x000F000Fu) | kMagic, s2, m2),
                       dq2(((w[k] >> 4) & 0x000F000Fu) | kMagic, s2, m2), dq2(((w[k] >> 8) & 0x000F000Fu) | kMagic, s2, m2),
                       dq2(((w[k] >> 12) & 0x000F000Fu) | kMagic, s2, m2));
        } else {
          const int cb = 16 * g + 8 * half + 2 * k;
          st_shared_v4(row + cb * 2048, dq2((w[k] & 0x00030003u) | kMagic, s2, m2),
                       dq2(((w[k] >> 2) & 0x00030003u) | kMagic, s2, m2), dq2(((w[k] >> 4) & 0x00030003u) | kMagic, s2, m2),
                       dq2(((w[k] >> 6) & 0x00030003u) | kMagic, s2, m2));
          st_shared_v4(row + (cb + 1) * 2048, dq2(((w[k] >> 8) & 0x00030003u) | kMagic, s2, m2),
                       dq2(((w[k] >> 10) & 0x00030003u) | kMagic, s2, m2),
                       dq2(((w[k] >> 12) & 0x00030003u) | kMagic, s2, m2),
                       dq2(((w[k] >> 14) & 0x00030003u) | kMagic, s2, m2));
        }
      }
    }
  };
  // score products of latent group g (A: its codes in tensor memory; B: the query) into S_A (even
  // g) or S_B (odd g)
  auto issue_group = [&](int g) {
#pragma unroll
    for (int k = 0; k < 8; ++k)
      tc_mma_ts(tmem + ((g & 1) ? kColSB : kColSA), tmem + kColA + 8 * k, sdesc(q_a + (8 * g + k) * 2048, 1024, 128),
                kIdescScore, k > 0);
  };
  // k_R products, high and low parts, into S_A
  auto issue_kr = [&]() {
#pragma unroll
    for (int kc = 0; kc < kRope / 16; ++kc) {
      const uint64_t bq = sdesc(q_a + (kLatent / 8 + 2 * kc) * 1024, 1024, 128);
      tc_mma_ts(tmem + kColSA, tmem + kColKrHi + 8 * kc, bq, kIdescScore, kc > 0);
      tc_mma_ts(tmem + kColSA, tmem + kColKrLo + 8 * kc, bq, kIdescScore, true);
    }
  };

  krm_s[tid] = R.krm;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  tmem = *tmem_slot;

  const int hb0 = 32 * half;
  bool aborted = false;
  // commits and completed waits; a wait that timed out is not counted, so that thread 0 waits for
  // that work again (bounded) before the tensor memory is released
  int s_commits = 0, s_waits = 0, o_commits = 0, o_waits = 0;
  auto wait_s = [&]() -> bool {
    const bool ok = mbar_wait_bounded(bars, s_waits & 1, kTcWaitBudget);
    if (ok) ++s_waits;
    const bool all = !__syncthreads_or(!ok);
    tc_fence_after();
    return all;
  };
  auto sync_issue = [&]() {  // make this thread's shared and tensor-memory writes visible to the MMAs
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
  };

  int i = 0;
  for (; i < n_my; ++i) {
    const int t0 = (tile_begin + i) * kTcTok;
    if (i > 0) krm_s[tid] = R.krm;  // the previous tile's k_R unpack read it before its softmax barriers
    // group 0's codes into tensor memory; its score products queue behind the previous readout
    codes_to_tmem(0);
    tmem_wait_st();
    sync_issue();
    if (tid == 0) {
      tc_fence_after();
      issue_group(0);
      tc_commit(bars);
    }
    ++s_commits;
    // the previous readout still reads the value tile and the weights: each thread waits for it
    // before its first value store (its timeout vote rides on group 0's issue barrier)
    bool read_ok = true;
    if (o_commits > o_waits) {
      read_ok = mbar_wait_bounded(bars + 1, o_waits & 1, kTcWaitBudget);
      if (read_ok) ++o_waits;
      tc_fence_after();
    }
    // per group: once its products are done, the next group's codes (after group 3: k_R) take
    // the tensor-memory operand and are issued; then the group is drained in FP32 with this
    // token's group scale and minimum, and its values go to the shared-memory tile
    float acc[32];
    int nswz = 0;
    const uint8_t* nrow = i + 1 < n_my ? token_row(i + 1, nswz) : nullptr;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      // each thread's own wait: group g's products are done, so its code columns and the other
      // accumulator are free; the timeout vote rides on the issue barrier (the group products
      // read shared memory only for the query, written before the first tile's barrier)
      const bool ok = mbar_wait_bounded(bars, s_waits & 1, kTcWaitBudget);
      if (ok) ++s_waits;
      tc_fence_after();
      if (g < 3) codes_to_tmem(g + 1);
      else unpack_kr(i);
      tmem_wait_st();
      tc_fence_before();
      if (__syncthreads_or(!ok || !read_ok)) {
        aborted = true;
        break;
      }
      if (tid == 0) {
        tc_fence_after();
        if (g < 3) issue_group(g + 1);
        else issue_kr();
        tc_commit(bars);
      }
      ++s_commits;
      {
        const uint32_t lm = g == 0 ? R.tmeta.x : g == 1 ? R.tmeta.y : g == 2 ? R.tmeta.z : R.tmeta.w;
        const float sg = half_bits_lo(lm), mg = half_bits_hi(lm);
        float sv[32];
        tmem_ld32(tmem + lane_base + ((g & 1) ? kColSB : kColSA) + hb0, sv);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const float4 qv = lds_f32x4(qs + g * kTcHeads + hb0 + 4 * jj);
          const float qq[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float t = fmaf(sg, sv[4 * jj + e], mg * qq[e]);
            acc[4 * jj + e] = g == 0 ? t : acc[4 * jj + e] + t;
          }
        }
      }
      values_to_smem(g);
      if (i + 1 < n_my) load_group(nrow, nswz, g);  // group g's registers are free: the next tile's chunks
    }
    if (aborted) break;
    if (i + 1 < n_my) load_meta(i + 1);  // the metadata registers are free too
    if (!wait_s()) {
      aborted = true;
      break;
    }
    {
      float sa[32];
      tmem_ld32(tmem + lane_base + kColSA + hb0, sa);
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j] = fmaf(sa[j], 5.9604644775390625e-8f, acc[j]);  // 2^-24
    }

    // ---- softmax: token 32*quarter + lane, heads hb0 .. hb0+31
    const int pos = t0 + 32 * quarter + lane;
    const bool valid = pos >= lo && pos < hi;
    bool over = false;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      acc[j] = valid ? acc[j] * lds_f32(hsc + hb0 + j) : -INFINITY;
      over |= acc[j] > m_run[hb0 + j] + kTcSlack;
    }
    if (__syncthreads_or(over)) {
      // raise the running max to this tile's maximum: reduce over the 128 token lanes
      float mine = -INFINITY;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float v = acc[j];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (lane == j) mine = v;
      }
      red[quarter * 64 + hb0 + lane] = mine;
      __syncthreads();
      float alpha[32], mnew_mine = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float mo = m_run[hb0 + j];
        const float mn =
            fmaxf(mo, fmaxf(fmaxf(red[hb0 + j], red[64 + hb0 + j]), fmaxf(red[128 + hb0 + j], red[192 + hb0 + j])));
        alpha[j] = mo == -INFINITY ? 0.f : ex2(mo - mn);
        if (lane == j) mnew_mine = mn;
      }
      if (o_commits > 0) {  // rescale the accumulated output columns and weight sums of these heads
#pragma unroll 1
        for (int g = 0; g < 5; ++g) {
          float o[32];
          const uint32_t addr = tmem + lane_base + (g < 4 ? kColO + 64 * g : kColL) + hb0;
          tmem_ld32(addr, o);
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] *= alpha[j];
          tmem_st32(addr, o);
        }
        tmem_wait_st();
      }
      __syncthreads();  // every thread has read m_run
      if (quarter == 0) m_run[hb0 + lane] = mnew_mine;
      __syncthreads();
    }
    // weights: FP16, heads contiguous per token (the readout's B operand)
    {
      const int t = 32 * quarter + lane;
      uint32_t pw[16];
      float lsum[32];
      if (o_commits > 0) tmem_ld32(tmem + lane_base + kColL + hb0, lsum);
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const float p0 = valid ? ex2(acc[j] - m_run[hb0 + j]) : 0.f;
        const float p1 = valid ? ex2(acc[j + 1] - m_run[hb0 + j + 1]) : 0.f;
        const __half2 hp = __floats2half2_rn(p0, p1);
        lsum[j] = (o_commits > 0 ? lsum[j] : 0.f) + __low2float(hp);
        lsum[j + 1] = (o_commits > 0 ? lsum[j + 1] : 0.f) + __high2float(hp);
        pw[j >> 1] = *reinterpret_cast<const uint32_t*>(&hp);
      }
      tmem_st32(tmem + lane_base + kColL + hb0, lsum);
      tmem_wait_st();
#pragma unroll
      for (int blk = 0; blk < 4; ++blk)
        st_shared_v4(p_a + ((t >> 3) * 8 + (hb0 >> 3) + blk) * 128 + (t & 7) * 16, pw[4 * blk], pw[4 * blk + 1],
                     pw[4 * blk + 2], pw[4 * blk + 3]);
    }
    sync_issue();
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int g = 0; g < 4; ++g)
#pragma unroll
        for (int kt = 0; kt < kTcTok / 16; ++kt)
          tc_mma_ss(tmem + kColO + 64 * g, sdesc(tile_a + (256 * g + 2 * kt) * 128, 128, 2048),
                    sdesc(p_a + kt * 2048, 1024, 128), kIdescRead, o_commits > 0 || kt > 0);
      tc_commit(bars + 1);
    }
    ++o_commits;
  }

  if (aborted) {
    flags |= kErrTimeout;
    // bounded waits for the tensor-core work still in flight before the memory is released
    if (tid == 0) {
      if (s_commits > s_waits) (void)mbar_wait_bounded(bars, s_waits & 1, kTcWaitBudget >> 4);
      if (o_commits > o_waits) (void)mbar_wait_bounded(bars + 1, o_waits & 1, kTcWaitBudget >> 4);
    }
  } else {
    const bool ok = mbar_wait_bounded(bars + 1, o_waits & 1, kTcWaitBudget);
    if (ok) ++o_waits;
    if (__syncthreads_or(!ok)) {
      flags |= kErrTimeout;
      aborted = true;
      if (tid == 0 && o_commits > o_waits) (void)mbar_wait_bounded(bars + 1, o_waits & 1, kTcWaitBudget >> 4);
    }
  }
  tc_fence_after();

  if (!aborted) {
    // ---- partial output: O^T rows are tile channels; each goes to its latent channel
    const int r = 32 * quarter + lane;
#pragma unroll 1
    for (int g = 0; g < 4; ++g) {
      float o[32];
      tmem_ld32(tmem + lane_base + kColO + 64 * g + hb0, o);
      const int ch = tile_to_orig<BITS>(128 * g + r);
      float* dst = p.o_part + ((static_cast<size_t>(b) * p.H + h0 + hb0) * NS + split) * kLatent + ch;
#pragma unroll
      for (int j = 0; j < 32; ++j) dst[static_cast<size_t>(j) * NS * kLatent] = o[j];
    }
    // sums over the 128 token lanes
    float lsum[32];
    tmem_ld32(tmem + lane_base + kColL + hb0, lsum);
    float mine = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      float v = lsum[j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == j) mine = v;
    }
    __syncthreads();
    red[quarter * 64 + hb0 + lane] = mine;
    __syncthreads();
    if (tid < kTcHeads) {
      float* ml = p.ml_part + ((static_cast<size_t>(b) * p.H + h0 + tid) * NS + split) * 2;
      ml[0] = m_run[tid];
      ml[1] = (red[tid] + red[64 + tid]) + (red[128 + tid] + red[192 + tid]);
    }
  } else if (tid < kTcHeads) {
    float* ml = p.ml_part + ((static_cast<size_t>(b) * p.H + h0 + tid) * NS + split) * 2;
    ml[0] = -INFINITY;
    ml[1] = 0.f;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  flags = __reduce_or_sync(0xffffffffu, flags);
  if (lane == 0 && flags) atomicOr(p.err, flags);
}

template <int BITS>
cudaError_t ensure_tc_attr() {
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!done[dev]) {
    e = cudaFuncSetAttribute(decode_tc_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return cudaSuccess;
}

}  // namespace

int decode_tc_num_splits(int B, int H, int max_pages, int P, int num_sms) {
  // one CTA per SM: exactly one wave of shares (a second, partial wave would double the time)
  const int groups = B * (H / kTcHeads);
  int ns = num_sms / (groups > 0 ? groups : 1);
  const long long max_tiles = (static_cast<long long>(max_pages) * P + kTcTok - 1) / kTcTok;
  if (ns > max_tiles) ns = static_cast<int>(max_tiles);
  if (ns > 128) ns = 128;
  if (ns < 1) ns = 1;
  return ns;
}

cudaError_t launch_decode_tc(const DecodeParams& p, cudaStream_t stream) {
  cudaError_t e;
  const dim3 grid(p.B, p.H / kTcHeads, p.n_split);
  if (p.bits_c == 4) {
    if ((e = ensure_tc_attr<4>()) != cudaSuccess) return e;
    decode_tc_kernel<4><<<grid, kTcThreads, kTcSmem, stream>>>(p);
  } else {
    if ((e = ensure_tc_attr<2>()) != cudaSuccess) return e;
    decode_tc_kernel<2><<<grid, kTcThreads, kTcSmem, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace mlaq
