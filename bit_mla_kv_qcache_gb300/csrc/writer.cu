// Fused cache writer (QuantMLA page, appendix Figure 8; RAQ-MLA page, appendix Table 5).
//
// Per new token (one CTA each): BF16 retention in the sink buffer / recent ring, per-token
// clip of the latent at a nearest-rank quantile of |c|, per-128-channel-group quantization
// with an FP16 minimum (rounded down) and FP16 scale (rounded up), and the bit-packed store
// into the token's page slot. Per page that fills during the call (four CTAs, 16 channels each):
// per-channel quantization of k_R over the page's P tokens, earlier tokens read from the ring.
//
// Every code is decided exactly: the nearest level is found from a float estimate and then
// confirmed against the exact midpoints min + (j + 1/2) * scale, which are formed without
// rounding (in float when a directed-rounding pair agrees, else in double).
//
// With the cached-tensor transforms of the RAQ-MLA page (Figure 4: A_c on the latent, A_R on
// k_R) the writer caches x A in place of x: each token is then served by a cluster of eight
// CTAs that form 64 transformed latent channels each (their 64-column slice of A_c arrives by
// tensor-map copies) and hand them to the cluster's first CTA through distributed shared
// memory; page fills transform the k_R of the call's new tokens.
#include <cooperative_groups.h>
#include <cstring>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace mlaq {
namespace {

__device__ __forceinline__ void raise_err(int32_t* err, int bits) {
  if (bits) atomicOr(err, bits);
}

// Is x on the upper side of the midpoint between levels j and j+1 (exact ties go to the even
// level)?
__device__ __forceinline__ bool above_midpoint(float x, float m, float s, int j) {
  const float h = (static_cast<float>(j) + 0.5f) * s;  // <= 16 significant bits: exact
  const float t_lo = __fadd_rd(m, h);
  const float t_hi = __fadd_ru(m, h);
  bool gt, eq;
  if (t_lo == t_hi) {  // m + h is exactly representable in float
    gt = x > t_lo;
    eq = x == t_lo;
  } else {  // exact in double (at most 46 significant bits)
    const double T = static_cast<double>(m) + static_cast<double>(h);
    const double xd = static_cast<double>(x);
    gt = xd > T;
    eq = xd == T;
  }
  return gt || (eq && ((j + 1) & 1) == 0);
}

__device__ __forceinline__ int quant_code(float x, float m, float s, float inv_s, int L) {
  if (!(s > 0.f)) return 0;
  int k = __float2int_rn(__fsub_rn(x, m) * inv_s);
  k = min(max(k, 0), L);
  while (k > 0 && !above_midpoint(x, m, s, k - 1)) --k;
  while (k < L && above_midpoint(x, m, s, k)) ++k;
  return k;
}

struct QParams {
  float m, s, inv_s;
  uint32_t meta;  // scale bits | min bits << 16
  int flags;
};

// FP16 minimum rounded down and FP16 scale rounded up from the exact range [lo, hi]:
// RU16(RU32(RU32(hi - m) / L)) equals RU16((hi - m) / L) because each upward rounding lands at
// or below the FP16 result (L * scale is exact in float).
__device__ __forceinline__ QParams make_qparams(float lo, float hi, int L) {
  QParams q;
  q.flags = 0;
  __half mh = __float2half_rd(lo);
  float m = __half2float(mh);
  if (isinf(m)) {
    q.flags |= kErrRange;
    m = -65504.f;
  }
  float d = __fsub_ru(hi, m);
  float r = __fdiv_ru(d, static_cast<float>(L));
  __half sh = __float2half_ru(r);
  float s = __half2float(sh);
  if (isinf(s) || hi > 65504.f) {
    q.flags |= kErrRange;
    s = 65504.f;
  }
  q.m = m;
  q.s = s;
  q.inv_s = s > 0.f ? 1.f / s : 0.f;
  uint32_t mb = __half_as_ushort(__float2half_rn(m));  // m, s are FP16 values: exact
  uint32_t sb = __half_as_ushort(__float2half_rn(s));
  if ((mb & 0x7fffu) == 0) mb = 0;  // zero is stored as +0
  if ((sb & 0x7fffu) == 0) sb = 0;
  q.meta = sb | (mb << 16);
  return q;
}

__device__ __forceinline__ int find_seq(const int32_t* cu, int B, int r) {
  int lo = 0, hi = B - 1;  // largest b with cu[b] <= r
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= r) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// ------------------------------------------------------------------ cached-tensor transforms
// x'_j = sum_i x_i A[i][j] for a BF16 row x and a BF16 matrix A [dim][dim] (row-major): the
// float32 sum runs over i = 0, 1, ..., dim-1 from +0, one rounded product (exact for two BF16
// values) and one rounded addition per step (this file is built without contraction), and is
// rounded to BF16 to nearest-even.
constexpr int kXfCtas = 8;  // CTAs (one cluster) per token when rows are transformed

__device__ __forceinline__ float bf16_bits_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
__device__ __forceinline__ uint16_t f32_bf16_bits(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }

// The CTA's slice of a latent transform (columns col0 .. col0 + 63 of a [512][512]) arrives in
// shared memory as four tensor-map boxes of 128 rows x 64 columns (16 KB each, all in flight at
// once, one barrier each); thread tid < 64 runs the sum of column col0 + tid over the rows in
// order as the boxes land. A_R ([64][64], 8 KB, contiguous) is one bulk copy. Every wait is
// bounded; a wait that gives up is agreed on by the whole CTA, the copies still in flight are
// waited for (bounded), and false is returned.
constexpr int kXfCols = kLatent / kXfCtas;                    // 64 columns per CTA
constexpr int kXfBlockRows = 128;                             // rows per box
constexpr int kXfBlocks = kLatent / kXfBlockRows;             // 4
constexpr int kXfBoxBytes = kXfBlockRows * kXfCols * 2;       // 16 KB
constexpr int kXfRopeOff = kXfBlocks * kXfBoxBytes;           // A_R after the boxes
constexpr int kXfSmemBytes = kXfRopeOff + kRope * kRope * 2;  // 72 KB of dynamic shared memory
constexpr int kXfBars = kXfBlocks + 1;                        // one per box, one for A_R
constexpr long long kXfWaitBudget = 4ll << 30;                // ~2 s at 2 GHz

__device__ __forceinline__ void xf_bars_init(uint64_t* bars) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < kXfBars; ++i) mbar_init(bars + i, 1);
    fence_mbar_init();
  }
  __syncthreads();
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// Thread 0 requests A_R (one copy) into the bytes after the boxes.
__device__ __forceinline__ void xf_issue_rope(const uint16_t* a_r, uint8_t* smem, uint64_t* bar) {
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar, kRope * kRope * 2);
    bulk_g2s(smem + kXfRopeOff, a_r, kRope * kRope * 2, bar);
  }
}

// Thread 0 requests the four boxes of columns col0 .. col0 + 63 (col0 * 2 bytes is a multiple of 16).
__device__ __forceinline__ void xf_issue_latent(const CUtensorMap* map, int col0, uint8_t* smem, uint64_t* bars) {
  if (threadIdx.x == 0) {
    for (int rb = 0; rb < kXfBlocks; ++rb) {
      mbar_arrive_expect_tx(bars + rb, kXfBoxBytes);
      tma_load_2d(smem + rb * kXfBoxBytes, map, col0, rb * kXfBlockRows, bars + rb);
    }
  }
}

// OR of a predicate over the kXfCols threads (warps 0-1) that run the sums, on barrier 1 (the
// other warps of the CTA are free meanwhile).
__device__ __forceinline__ bool sum_warps_or(bool v) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred pi, po; setp.ne.u32 pi, %1, 0; barrier.cta.red.or.pred po, 1, %2, pi; selp.u32 %0, 1, 0, po; }"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "n"(kXfCols)
      : "memory");
  return r != 0;
}

// Called by threads 0 .. kXfCols-1 only (thread 0 issued the boxes).
__device__ bool latent_slice_transform(const float* s_x, const uint8_t* smem, uint64_t* bars, uint16_t& out) {
  float acc = 0.f;
  for (int rb = 0; rb < kXfBlocks; ++rb) {
    const bool ok = mbar_wait_bounded(bars + rb, 0, kXfWaitBudget);
    if (sum_warps_or(!ok)) {
      if (threadIdx.x == 0)
        for (int j = rb; j < kXfBlocks; ++j) (void)mbar_wait_bounded(bars + j, 0, kXfWaitBudget >> 4);
      return false;
    }
    const uint16_t* blk = reinterpret_cast<const uint16_t*>(smem + rb * kXfBoxBytes) + threadIdx.x;
    const float* xb = s_x + rb * kXfBlockRows;
#pragma unroll 16
    for (int i = 0; i < kXfBlockRows; ++i) acc = acc + xb[i] * bf16_bits_f32(blk[i * kXfCols]);
  }
  out = f32_bf16_bits(acc);
  return true;
}

// Channel j < 64 of k_R A_R from the staged A_R (the CTA waits for it first).
__device__ bool rope_transform(const float* s_k, const uint8_t* smem, uint64_t* bar, int j, uint16_t& out) {
  const bool ok = mbar_wait_bounded(bar, 0, kXfWaitBudget);
  if (__syncthreads_or(!ok)) {
    if (threadIdx.x == 0) (void)mbar_wait_bounded(bar, 0, kXfWaitBudget >> 4);
    return false;
  }
  if (j < kRope) {
    const uint16_t* ar = reinterpret_cast<const uint16_t*>(smem + kXfRopeOff) + j;
    float acc = 0.f;
#pragma unroll 16
    for (int i = 0; i < kRope; ++i) acc = acc + s_k[i] * bf16_bits_f32(ar[i * kRope]);
    out = f32_bf16_bits(acc);
  }
  return true;
}

// Channels j and j+1 (j even) of k_R A_R for one k_R row in global memory, A_R staged in shared
// memory (page fills of the call's new tokens).
__device__ __forceinline__ uint32_t transform_rope_pair(const uint16_t* x, const uint16_t* ar, int j) {
  uint32_t xv[kRope / 2];  // the row's 32-bit words, all loads in flight together (rows are 4-byte aligned)
#pragma unroll
  for (int v = 0; v < kRope / 2; ++v) xv[v] = __ldg(reinterpret_cast<const uint32_t*>(x) + v);
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int i = 0; i < kRope; ++i) {
    const float xi = (i & 1) ? bf16_hi(xv[i >> 1]) : bf16_lo(xv[i >> 1]);
    const uint32_t av = *reinterpret_cast<const uint32_t*>(ar + i * kRope + j);
    a0 = a0 + xi * bf16_lo(av);
    a1 = a1 + xi * bf16_hi(av);
  }
  return static_cast<uint32_t>(f32_bf16_bits(a0)) | (static_cast<uint32_t>(f32_bf16_bits(a1)) << 16);
}

// Where row r goes: its sequence, that sequence's row offsets and length, and the id of the
// page that receives it (loads only; the caller checks them). -1 where a load was not made.
struct RowRef {
  int b, r0, r1, s0;
  int32_t pid;
};
__device__ __forceinline__ RowRef resolve_row(const WriteParams& p, int r) {
  RowRef z{-1, 0, 0, -1, -1};
  if (r < p.B) {
    z.r0 = __ldg(p.cu_new + r);
    z.r1 = __ldg(p.cu_new + r + 1);
    if (z.r0 == r && z.r1 == r + 1) z.b = r;
  }
  if (z.b < 0) {
    z.b = find_seq(p.cu_new, p.B, r);
    z.r0 = __ldg(p.cu_new + z.b);
    z.r1 = __ldg(p.cu_new + z.b + 1);
  }
  if (r < z.r0 || r >= z.r1 || z.r1 - z.r0 > p.max_new) return z;
  z.s0 = __ldg(p.seq_lens + z.b);
  if (z.s0 < 0) return z;
  const int64_t pg = (static_cast<int64_t>(z.s0) + (r - z.r0)) / p.P;
  if (pg < p.max_pages) z.pid = __ldg(p.page_table + static_cast<size_t>(z.b) * p.max_pages + pg);
  return z;
}

// The cluster of token row r: CTA `rank` forms latent channels 64 rank .. 64 rank + 63 (one per
// thread of its first two warps), CTA 1 also the 64 k_R channels; after the cluster barrier the
// first CTA gathers the row in the per-token layout (thread: latent channels 4 tid .. 4 tid + 3;
// warp-0 lanes: k_R channels 2 lane, 2 lane + 1). Every CTA of the cluster passes both barriers.
__device__ void transform_token(const WriteParams& p, const CUtensorMap* a_map, int r, uint8_t* smem, uint2& cv,
                                uint32_t& kr2, RowRef& ref) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  const int rank = static_cast<int>(cl.block_rank());
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __shared__ float s_x[kRow];
  __shared__ __align__(16) uint16_t s_y[kXfCols + kRope];
  __shared__ __align__(8) uint64_t bars[kXfBars];
  __shared__ RowRef s_ref;
  xf_bars_init(bars);
  const bool rope_here = rank == 1 && p.a_r != nullptr;
  if (p.a_c) xf_issue_latent(a_map, kXfCols * rank, smem, bars);
  if (rope_here) xf_issue_rope(p.a_r, smem, bars + kXfBlocks);
  const uint16_t* c_row = p.c_new + static_cast<size_t>(r) * kLatent;
  const uint16_t* k_row = p.kr_new + static_cast<size_t>(r) * kRope;
  const uint2 raw = __ldg(reinterpret_cast<const uint2*>(c_row) + tid);
  s_x[4 * tid] = bf16_lo(raw.x);
  s_x[4 * tid + 1] = bf16_hi(raw.x);
  s_x[4 * tid + 2] = bf16_lo(raw.y);
  s_x[4 * tid + 3] = bf16_hi(raw.y);
  if (tid < kRope / 2) {
    const uint32_t k = __ldg(reinterpret_cast<const uint32_t*>(k_row) + tid);
    s_x[kLatent + 2 * tid] = bf16_lo(k);
    s_x[kLatent + 2 * tid + 1] = bf16_hi(k);
  }
  __syncthreads();
  bool ok = true;
  if (tid < kXfCols) {  // warps 0-1: this CTA's 64 latent channels
    uint16_t y = __ldg(c_row + kXfCols * rank + tid);
    if (p.a_c) ok = latent_slice_transform(s_x, smem, bars, y);
    s_y[tid] = y;
  } else if (rank == 0 && tid == kXfCols) {  // meanwhile the first CTA finds where the row goes
    s_ref = resolve_row(p, r);
  }
  if (rank == 1 && tid < kRope) s_y[kXfCols + tid] = __ldg(k_row + tid);
  if (rope_here) {
    uint16_t yr = 0;
    if (rope_transform(s_x + kLatent, smem, bars + kXfBlocks, tid, yr)) {
      if (tid < kRope) s_y[kXfCols + tid] = yr;
    } else {
      ok = false;
    }
  }
  if (!ok && tid == 0) raise_err(p.err, kErrTimeout);
  cl.sync();  // every slice written
  if (rank == 0) {
    // channel 4 tid lives in CTA 4 tid / 64
    const uint16_t* src = cl.map_shared_rank(s_y, (4 * tid) / kXfCols);
    cv = *reinterpret_cast<const uint2*>(src + ((4 * tid) & (kXfCols - 1)));
    if (warp == 0) kr2 = *reinterpret_cast<const uint32_t*>(cl.map_shared_rank(s_y, 1) + kXfCols + 2 * lane);
    ref = s_ref;
  }
  cl.sync();  // the slices stay in place until the first CTA has read them
}

// ------------------------------------------------------------------ per-token work (one CTA)
// 128 threads per new token: warp w owns latent group w (channels 128w..128w+127, four per
// lane); lanes of warp 0 also carry the token's k_R (two channels each) for the retention copy.
// kGiven: the row arrives in cv / kr2 (transformed by the token's cluster) instead of from c_new.
// kGiven: the row arrives in cv / kr2 (transformed by the token's cluster) and where it goes in
// ref, instead of from c_new and the offset, length and page-table loads.
template <bool kGiven>
__device__ void write_token(const WriteParams& p, int r, int (&s_cnt)[2][4], uint2 cv, uint32_t kr2,
                            const RowRef& ref) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // decode steps write one row per sequence (cu_new[b] = b): then row r belongs to sequence r,
  // found with two independent loads instead of a dependent binary search
  int b = -1, r0 = 0, r1 = 0;
  if constexpr (kGiven) {
    b = ref.b;
    r0 = ref.r0;
    r1 = ref.r1;
  } else {
    if (r < p.B) {
      r0 = __ldg(p.cu_new + r);
      r1 = __ldg(p.cu_new + r + 1);
      if (r0 == r && r1 == r + 1) b = r;
    }
    if (b < 0) {
      b = find_seq(p.cu_new, p.B, r);
      r0 = __ldg(p.cu_new + b);
      r1 = __ldg(p.cu_new + b + 1);
    }
  }
  if (r < r0 || r >= r1 || r1 - r0 > p.max_new) {  // inconsistent row offsets
    if (tid == 0) raise_err(p.err, kErrRows);
    return;
  }
  const int n_b = r1 - r0;
  const int s0 = kGiven ? ref.s0 : __ldg(p.seq_lens + b);
  if (s0 < 0) {
    if (tid == 0) raise_err(p.err, kErrSeqOverflow);
    return;
  }
  const int64_t t = static_cast<int64_t>(s0) + (r - r0);
  const int64_t t_final = static_cast<int64_t>(s0) + n_b;

  // ---- load: thread holds latent channels [4*tid, 4*tid+4); warp 0 lanes k_R [2*lane, 2*lane+2)
  if constexpr (!kGiven) {
    cv = __ldg(reinterpret_cast<const uint2*>(p.c_new + static_cast<size_t>(r) * kLatent) + tid);
    if (warp == 0) kr2 = __ldg(reinterpret_cast<const uint32_t*>(p.kr_new + static_cast<size_t>(r) * kRope) + lane);
  }

  // ---- BF16 retention (pre-quantization values)
  if (t < p.S) {
    uint16_t* row = p.sink + (static_cast<size_t>(b) * p.S + t) * kRow;
    reinterpret_cast<uint2*>(row)[tid] = cv;
    if (warp == 0) reinterpret_cast<uint32_t*>(row + kLatent)[lane] = kr2;
  }
  if (t >= t_final - p.W) {
    uint16_t* row = p.ring + (static_cast<size_t>(b) * p.W + (t % p.W)) * kRow;
    reinterpret_cast<uint2*>(row)[tid] = cv;
    if (warp == 0) reinterpret_cast<uint32_t*>(row + kLatent)[lane] = kr2;
  }

  // ---- page slot
  const int64_t pg = t / p.P;
  if (pg >= p.max_pages) {
    if (tid == 0) raise_err(p.err, kErrSeqOverflow);
    return;
  }
  const int32_t pid = kGiven ? ref.pid : __ldg(p.page_table + static_cast<size_t>(b) * p.max_pages + pg);
  if (pid < 0 || pid >= p.n_pages) {
    if (tid == 0) raise_err(p.err, kErrBadPage);
    return;
  }
  const int tp = static_cast<int>(t % p.P);
  uint8_t* page = p.pool + static_cast<size_t>(pid) * static_cast<size_t>(p.page_bytes);

  float x[4] = {bf16_lo(cv.x), bf16_hi(cv.x), bf16_lo(cv.y), bf16_hi(cv.y)};
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 4; ++i) bad |= !isfinite(x[i]);
  int flags = __syncthreads_or(bad) ? kErrNonFinite : 0;

  // ---- per-token clip: tau = clip_k-th smallest |x| over the 512 channels (nearest rank),
  // found by bisection on the BF16 magnitude bit patterns, counts reduced across the CTA
  if (p.clip_k > 0) {
    const uint32_t key[4] = {cv.x & 0x7fffu, (cv.x >> 16) & 0x7fffu, cv.y & 0x7fffu, (cv.y >> 16) & 0x7fffu};
    uint32_t lo = 0, hi = 0x7fffu;
    int it = 0;
    while (lo < hi) {
      const uint32_t mid = (lo + hi) >> 1;
      int cnt = (key[0] <= mid) + (key[1] <= mid) + (key[2] <= mid) + (key[3] <= mid);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
      if (lane == 0) s_cnt[it & 1][warp] = cnt;
      __syncthreads();
      const int total = s_cnt[it & 1][0] + s_cnt[it & 1][1] + s_cnt[it & 1][2] + s_cnt[it & 1][3];
      if (total >= p.clip_k) hi = mid;
      else lo = mid + 1;
      ++it;
    }
    const float tau = __uint_as_float(lo << 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = fminf(fmaxf(x[i], -tau), tau);
  }

  // ---- group statistics over the warp
  float lo = fminf(fminf(x[0], x[1]), fminf(x[2], x[3]));
  float hi = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  const int L = (1 << p.bits_c) - 1;
  const QParams qp = make_qparams(lo, hi, L);
  flags |= qp.flags;
  int code[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) code[i] = quant_code(x[i], qp.m, qp.s, qp.inv_s, L);

  // ---- pack into region A: the token's row keeps its channels in order (this lane's four
  // channels form 16 bits (INT4) or 8 bits (INT2) at row byte (128w + 4 lane) * bits_c / 8),
  // and the row's 16-byte chunks are stored XOR-permuted by tp mod 8. Neighbouring lanes
  // merge into one 32-bit store.
  uint8_t* row = page + static_cast<size_t>(tp) * (64 * p.bits_c);
  const int swz = tp & 7;
  if (p.bits_c == 4) {
    uint32_t v = static_cast<uint32_t>(code[0]) | (static_cast<uint32_t>(code[1]) << 4) |
                 (static_cast<uint32_t>(code[2]) << 8) | (static_cast<uint32_t>(code[3]) << 12);
    v |= __shfl_down_sync(0xffffffffu, v, 1) << 16;
    if ((lane & 1) == 0) {
      const int chunk = 4 * warp + (lane >> 3);  // logical chunk of row byte 64w + 2 lane
      *reinterpret_cast<uint32_t*>(row + 16 * (chunk ^ swz) + 2 * (lane & 7)) = v;
    }
  } else {
    uint32_t v = static_cast<uint32_t>(code[0]) | (static_cast<uint32_t>(code[1]) << 2) |
                 (static_cast<uint32_t>(code[2]) << 4) | (static_cast<uint32_t>(code[3]) << 6);
    v |= __shfl_down_sync(0xffffffffu, v, 1) << 8;
    v |= __shfl_down_sync(0xffffffffu, v, 2) << 16;
    if ((lane & 3) == 0) {
      const int chunk = 2 * warp + (lane >> 4);  // logical chunk of row byte 32w + lane
      *reinterpret_cast<uint32_t*>(row + 16 * (chunk ^ swz) + (lane & 15)) = v;
    }
  }
  // ---- latent metadata (region C)
  if (lane == 0) {
    uint8_t* meta = page + static_cast<size_t>(p.P) * (64 * p.bits_c + 32) + (tp * 4 + warp) * 4;
    *reinterpret_cast<uint32_t*>(meta) = qp.meta;
  }
  flags = __reduce_or_sync(0xffffffffu, flags);
  if (lane == 0 && flags) raise_err(p.err, flags);
}

// ------------------------------------------------------------------ page fill (four CTAs)
// A page that fills during the call is quantized by four CTAs, CTA rr taking k_R channels
// 16rr .. 16rr+15: exactly the channels of region B's fragment blocks (tb, rr) and of their
// region D entries, so the four write disjoint bytes.
constexpr int kFillSplit = 4;
constexpr int kFillCh = kRope / kFillSplit;  // 16
constexpr int kFillStride = kFillCh + 1;     // row stride of the staged values (floats)
constexpr int kFillSubsets = 8;              // token subsets reduced in parallel per channel

__host__ __device__ constexpr size_t fill_smem_floats(int P) {
  return static_cast<size_t>(P) * kFillStride + 2 * kFillSubsets * kFillCh + 3 * kFillCh;
}

template <bool kTransform>
__device__ void fill_page(const WriteParams& p, int b, int f, int rr, float* smem) {
  const int tid = threadIdx.x;
  const int r0 = __ldg(p.cu_new + b), r1 = __ldg(p.cu_new + b + 1);
  const int s0 = __ldg(p.seq_lens + b);
  const int n = r1 - r0;
  // the length after this call, into a second array (the token and fill CTAs read seq_lens)
  if (p.seq_next != nullptr && f == 0 && rr == 0 && tid == 0) p.seq_next[b] = s0 + n;
  if (s0 < 0 || n <= 0 || n > p.max_new || r0 < 0 || r1 > p.n_rows) return;  // reported by the token work
  const int64_t pg = static_cast<int64_t>(s0) / p.P + f;
  if ((pg + 1) * p.P > static_cast<int64_t>(s0) + n) return;  // this page does not fill now
  if (pg >= p.max_pages) return;
  const int32_t pid = __ldg(p.page_table + static_cast<size_t>(b) * p.max_pages + pg);
  const int P = p.P;
  float* vals = smem;                                        // [P][kFillStride]
  float* red = vals + static_cast<size_t>(P) * kFillStride;  // [2][kFillSubsets][kFillCh]
  float* stats = red + 2 * kFillSubsets * kFillCh;           // [kFillCh][3]

  // A_R for the new tokens' k_R (after the staged values, 16-byte aligned for P % 32 == 0)
  const uint16_t* ar_s = reinterpret_cast<const uint16_t*>(smem + fill_smem_floats(P));
  if constexpr (kTransform) {
    if (p.a_r) {
      uint4* dst = reinterpret_cast<uint4*>(smem + fill_smem_floats(P));
      for (int v = threadIdx.x; v < kRope * kRope / 8; v += blockDim.x)
        dst[v] = __ldg(reinterpret_cast<const uint4*>(p.a_r) + v);
      __syncthreads();
    }
  }
  // gather this CTA's 32 bytes of every token of the page (earlier tokens from the ring, new
  // ones from the input), all loads of a thread in flight together; the page id is checked
  // after them (the loads do not depend on it)
  constexpr int kMaxIt = 128 * 8 / 128;  // at most 128 tokens x 8 words, over 128 threads
  const int n_items = P * 8;
  uint32_t w[kMaxIt];
#pragma unroll
  for (int it = 0; it < kMaxIt; ++it) {
    const int i = threadIdx.x + 128 * it;
    w[it] = 0;
    if (i < n_items) {
      const int u = i >> 3, e = i & 7;
      const int64_t tt = pg * P + u;
      const uint32_t* src;
      if (tt < s0) {
        src = reinterpret_cast<const uint32_t*>(p.ring + (static_cast<size_t>(b) * p.W + (tt % p.W)) * kRow + kLatent);
      } else {
        const uint16_t* k_row = p.kr_new + static_cast<size_t>(r0 + (tt - s0)) * kRope;
        if constexpr (kTransform) {
          if (p.a_r) {  // a new token's k_R is cached as k_R A_R
            w[it] = transform_rope_pair(k_row, ar_s, kFillCh * rr + 2 * e);
            continue;
          }
        }
        src = reinterpret_cast<const uint32_t*>(k_row);
      }
      w[it] = __ldg(src + kFillCh / 2 * rr + e);
    }
  }
  if (pid < 0 || pid >= p.n_pages) return;
  uint8_t* page = p.pool + static_cast<size_t>(pid) * static_cast<size_t>(p.page_bytes);
#pragma unroll
  for (int it = 0; it < kMaxIt; ++it) {
    const int i = threadIdx.x + 128 * it;
    if (i < n_items) {
      const int u = i >> 3, e = i & 7;
      vals[u * kFillStride + 2 * e] = bf16_lo(w[it]);
      vals[u * kFillStride + 2 * e + 1] = bf16_hi(w[it]);
    }
  }
  __syncthreads();

  // per-channel range: eight token subsets per channel, then the eight partial ranges
  int flags = 0;
  {
    const int c = tid & (kFillCh - 1), sub = tid >> 4;  // 128 threads = 16 channels x 8 subsets
    float lo = vals[sub * kFillStride + c], hi = lo;
    bool bad = !isfinite(lo);
    for (int u = sub + kFillSubsets; u < P; u += kFillSubsets) {
      const float v = vals[u * kFillStride + c];
      bad |= !isfinite(v);
      lo = fminf(lo, v);
      hi = fmaxf(hi, v);
    }
    red[sub * kFillCh + c] = lo;
    red[(kFillSubsets + sub) * kFillCh + c] = hi;
    if (__syncthreads_or(bad)) flags |= kErrNonFinite;
  }
  if (tid < kFillCh) {
    float lo = red[tid], hi = red[kFillSubsets * kFillCh + tid];
#pragma unroll
    for (int sub = 1; sub < kFillSubsets; ++sub) {
      lo = fminf(lo, red[sub * kFillCh + tid]);
      hi = fmaxf(hi, red[(kFillSubsets + sub) * kFillCh + tid]);
    }
    const QParams qp = make_qparams(lo, hi, 15);
    flags |= qp.flags;
    stats[3 * tid] = qp.m;
    stats[3 * tid + 1] = qp.s;
    stats[3 * tid + 2] = qp.inv_s;
    const int j = kFillCh * rr + tid;
    *reinterpret_cast<uint32_t*>(page + static_cast<size_t>(P) * (64 * p.bits_c + 48) + j * 4) = qp.meta;
  }
  __syncthreads();
  // codes: the 32-bit words of region B's fragment blocks (tb, rr), one per iteration
  uint8_t* regb = page + static_cast<size_t>(P) * 64 * p.bits_c;
  for (int wi = tid; wi < P * 2; wi += blockDim.x) {
    const int tb = wi >> 5, ln = wi & 31;
    const int q = ln & 3, g8 = ln >> 2;
    uint32_t word = 0;
#pragma unroll
    for (int nn = 0; nn < 2; ++nn)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int o = 0; o < 2; ++o) {
          const int u = 16 * tb + 8 * nn + g8;
          const int c = 8 * h + 2 * q + o;
          const int code = quant_code(vals[u * kFillStride + c], stats[3 * c], stats[3 * c + 1], stats[3 * c + 2], 15);
          word |= static_cast<uint32_t>(code) << (4 * (2 * nn + h + 4 * o));
        }
    *reinterpret_cast<uint32_t*>(regb + ((tb * 4 + rr) * 128 + ln * 4)) = word;
  }
  if (flags && tid == 0) raise_err(p.err, flags);
}

// Blocks [0, token_blocks x per-token CTAs) serve the new rows, the rest the page fills.
template <bool kTransform>
__device__ __forceinline__ void write_body(const WriteParams& p, const CUtensorMap* a_map) {
  extern __shared__ __align__(128) float smem_f[];
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (__ldg(p.cu_new) != 0 || __ldg(p.cu_new + p.B) != p.n_rows) raise_err(p.err, kErrRows);
  }
  constexpr int kPerToken = kTransform ? kXfCtas : 1;
  if (static_cast<int>(blockIdx.x) < p.token_blocks * kPerToken) {
    __shared__ int s_cnt[2][4];
    if constexpr (kTransform) {
      const int r = blockIdx.x / kXfCtas;
      uint2 cv = make_uint2(0u, 0u);
      uint32_t kr2 = 0;
      RowRef ref{-1, 0, 0, -1, -1};
      transform_token(p, a_map, r, reinterpret_cast<uint8_t*>(smem_f), cv, kr2, ref);
      if (blockIdx.x % kXfCtas != 0) return;  // the cluster's first CTA writes the token
      write_token<true>(p, r, s_cnt, cv, kr2, ref);
    } else {
      write_token<false>(p, blockIdx.x, s_cnt, make_uint2(0u, 0u), 0u, RowRef{-1, 0, 0, -1, -1});
    }
    return;
  }
  const int idx = blockIdx.x - p.token_blocks * kPerToken;
  const int per_seq = p.fill_per_seq * kFillSplit;
  if (per_seq == 0) return;  // a padding CTA of a launch without page fills
  const int b = idx / per_seq, f = (idx % per_seq) / kFillSplit, rr = idx % kFillSplit;
  if (b < p.B) fill_page<kTransform>(p, b, f, rr, smem_f);
}

__global__ void __launch_bounds__(128) write_kernel(const WriteParams p) { write_body<false>(p, nullptr); }

// Rows transformed on the way in: clusters of eight CTAs along x (token clusters, then the fill
// CTAs, padded to whole clusters with CTAs past the last sequence, which exit).
__global__ void __cluster_dims__(kXfCtas, 1, 1) __launch_bounds__(128)
    write_xf_kernel(const WriteParams p, const __grid_constant__ CUtensorMap a_map) {
  write_body<true>(p, &a_map);
}

// Standalone transform: CTA (row, part) forms channels 64 part .. 64 part + 63 of one row (all
// 64 for dim 64), with the arithmetic and staging of the fused writer, so either route caches
// the same bits.
__global__ void __launch_bounds__(128) row_transform_kernel(int dim, const uint16_t* x, const uint16_t* a,
                                                            uint16_t* out, int32_t* err,
                                                            const __grid_constant__ CUtensorMap a_map) {
  extern __shared__ __align__(128) uint8_t xf_smem[];
  __shared__ float s_x[kLatent];
  __shared__ __align__(8) uint64_t bars[kXfBars];
  xf_bars_init(bars);
  const size_t r = blockIdx.x;
  if (dim == kRope) xf_issue_rope(a, xf_smem, bars + kXfBlocks);
  else xf_issue_latent(&a_map, kXfCols * blockIdx.y, xf_smem, bars);
  for (int i = threadIdx.x; i < dim; i += 128) s_x[i] = bf16_bits_f32(__ldg(x + r * dim + i));
  __syncthreads();
  uint16_t y = 0;
  bool ok = true;
  if (dim == kRope) ok = rope_transform(s_x, xf_smem, bars + kXfBlocks, threadIdx.x, y);
  else if (threadIdx.x < kXfCols) ok = latent_slice_transform(s_x, xf_smem, bars, y);
  if (!ok) {
    if (threadIdx.x == 0) raise_err(err, kErrTimeout);
    return;
  }
  const int j = (dim == kRope ? 0 : kXfCols * static_cast<int>(blockIdx.y)) + static_cast<int>(threadIdx.x);
  if (threadIdx.x < (dim == kRope ? kRope : kXfCols)) out[r * dim + j] = y;
}

// Tensor map of a BF16 [512][512] row-major matrix for boxes of 128 rows x 64 columns (the
// encoder comes from the driver through the runtime, so nothing links against libcuda).
cudaError_t encode_latent_map(const uint16_t* a, CUtensorMap* map) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cudaErrorNotSupported;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kLatent), static_cast<cuuint64_t>(kLatent)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kLatent) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kXfCols), static_cast<cuuint32_t>(kXfBlockRows)};
  const cuuint32_t elem[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t*>(a), dims, strides, box, elem,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

__global__ void __launch_bounds__(256) advance_kernel(const int32_t* cu_new, int32_t* seq_lens, int B) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) seq_lens[b] += __ldg(cu_new + b + 1) - __ldg(cu_new + b);
}

}  // namespace

cudaError_t launch_advance(const int32_t* cu_new, int32_t* seq_lens, int B, cudaStream_t stream) {
  advance_kernel<<<(B + 255) / 256, 256, 0, stream>>>(cu_new, seq_lens, B);
  return cudaGetLastError();
}

cudaError_t launch_write(const WriteParams& p, cudaStream_t stream) {
  const bool xf = p.a_c != nullptr || p.a_r != nullptr;
  int64_t blocks = static_cast<int64_t>(p.token_blocks) * (xf ? kXfCtas : 1) +
                   static_cast<int64_t>(p.B) * p.fill_per_seq * kFillSplit;
  if (blocks == 0) return cudaSuccess;
  if (xf) blocks = (blocks + kXfCtas - 1) / kXfCtas * kXfCtas;  // whole clusters
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  const size_t smem = p.fill_per_seq > 0 ? fill_smem_floats(p.P) * sizeof(float) : 0;  // <= 10 KB
  if (xf) {
    CUtensorMap a_map;
    memset(&a_map, 0, sizeof a_map);
    if (p.a_c != nullptr) {
      const cudaError_t em = encode_latent_map(p.a_c, &a_map);
      if (em != cudaSuccess) return em;
    }
    static bool attr_done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_done[dev]) {
      e = cudaFuncSetAttribute(write_xf_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kXfSmemBytes);
      if (e != cudaSuccess) return e;
      attr_done[dev] = true;
    }
    const size_t fill_xf = p.fill_per_seq > 0 ? fill_smem_floats(p.P) * sizeof(float) + kRope * kRope * 2 : 0;
    const size_t smem_xf = p.token_blocks > 0 ? static_cast<size_t>(kXfSmemBytes) : 0;
    write_xf_kernel<<<static_cast<unsigned>(blocks), 128, smem_xf > fill_xf ? smem_xf : fill_xf, stream>>>(p, a_map);
  } else {
    write_kernel<<<static_cast<unsigned>(blocks), 128, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_row_transform(int n_rows, int dim, const uint16_t* x, const uint16_t* a, uint16_t* out,
                                 int32_t* err, cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(row_transform_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kXfSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  CUtensorMap a_map;
  memset(&a_map, 0, sizeof a_map);
  if (dim == kLatent && (e = encode_latent_map(a, &a_map)) != cudaSuccess) return e;
  row_transform_kernel<<<dim3(static_cast<unsigned>(n_rows), dim == kLatent ? kXfCtas : 1), 128, kXfSmemBytes,
                         stream>>>(dim, x, a, out, err, a_map);
  return cudaGetLastError();
}

}  // namespace mlaq
