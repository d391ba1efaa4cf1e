// Fused cache writer (QuantMLA page, appendix Figure 8; RAQ-MLA page, appendix Table 5).
//
// Per new token (one warp each): BF16 retention in the sink buffer / recent ring, per-token
// clip of the latent at a nearest-rank quantile of |c|, per-128-channel-group quantization
// with an FP16 minimum (rounded down) and FP16 scale (rounded up), and the bit-packed store
// into the token's page slot. Per page that fills during the call (one CTA each): per-channel
// quantization of k_R over the page's P tokens, earlier tokens read from the ring.
//
// Every code is decided exactly: the nearest level is found from a float estimate and then
// confirmed against the exact midpoints min + (j + 1/2) * scale, which are formed without
// rounding (in float when a directed-rounding pair agrees, else in double).
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

// ------------------------------------------------------------------ per-token work (one warp)
__device__ void write_token(const WriteParams& p, int r, int lane) {
  // decode steps write one row per sequence (cu_new[b] = b): then row r belongs to sequence r,
  // found with two independent loads instead of a dependent binary search
  int b = -1, r0 = 0, r1 = 0;
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
  if (r < r0 || r >= r1) {  // inconsistent row offsets
    if (lane == 0) raise_err(p.err, kErrRows);
    return;
  }
  const int n_b = r1 - r0;
  if (n_b > p.max_new) {
    if (lane == 0) raise_err(p.err, kErrRows);
    return;
  }
  const int s0 = __ldg(p.seq_lens + b);
  if (s0 < 0) {
    if (lane == 0) raise_err(p.err, kErrSeqOverflow);
    return;
  }
  const int64_t t = static_cast<int64_t>(s0) + (r - r0);
  const int64_t t_final = static_cast<int64_t>(s0) + n_b;

  // ---- load: lane holds latent channels [16*lane, 16*lane+16) and k_R channels [2*lane, 2*lane+2)
  const uint4* crow = reinterpret_cast<const uint4*>(p.c_new + static_cast<size_t>(r) * kLatent) + 2 * lane;
  const uint4 c0 = __ldg(crow), c1 = __ldg(crow + 1);
  const uint32_t kr2 = __ldg(reinterpret_cast<const uint32_t*>(p.kr_new + static_cast<size_t>(r) * kRope) + lane);

  // ---- BF16 retention (pre-quantization values)
  if (t < p.S) {
    uint16_t* row = p.sink + (static_cast<size_t>(b) * p.S + t) * kRow;
    reinterpret_cast<uint4*>(row)[2 * lane] = c0;
    reinterpret_cast<uint4*>(row)[2 * lane + 1] = c1;
    reinterpret_cast<uint32_t*>(row + kLatent)[lane] = kr2;
  }
  if (t >= t_final - p.W) {
    uint16_t* row = p.ring + (static_cast<size_t>(b) * p.W + (t % p.W)) * kRow;
    reinterpret_cast<uint4*>(row)[2 * lane] = c0;
    reinterpret_cast<uint4*>(row)[2 * lane + 1] = c1;
    reinterpret_cast<uint32_t*>(row + kLatent)[lane] = kr2;
  }

  // ---- page slot
  const int64_t pg = t / p.P;
  if (pg >= p.max_pages) {
    if (lane == 0) raise_err(p.err, kErrSeqOverflow);
    return;
  }
  const int32_t pid = __ldg(p.page_table + static_cast<size_t>(b) * p.max_pages + pg);
  if (pid < 0 || pid >= p.n_pages) {
    if (lane == 0) raise_err(p.err, kErrBadPage);
    return;
  }
  const int tp = static_cast<int>(t % p.P);
  uint8_t* page = p.pool + static_cast<size_t>(pid) * static_cast<size_t>(p.page_bytes);

  float x[16];
  const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = bf16_lo(cw[i]);
    x[2 * i + 1] = bf16_hi(cw[i]);
  }
  int flags = 0;
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 16; ++i) bad |= !isfinite(x[i]);
  if (__any_sync(0xffffffffu, bad)) flags |= kErrNonFinite;

  // ---- per-token clip: tau = clip_k-th smallest |x| (nearest-rank order statistic)
  if (p.clip_k > 0) {
    uint32_t key[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      key[2 * i] = cw[i] & 0x7fffu;
      key[2 * i + 1] = (cw[i] >> 16) & 0x7fffu;
    }
    uint32_t lo = 0, hi = 0x7fffu;
    while (lo < hi) {
      const uint32_t mid = (lo + hi) >> 1;
      int cnt = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) cnt += key[i] <= mid;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
      if (cnt >= p.clip_k) hi = mid;
      else lo = mid + 1;
    }
    const float tau = __uint_as_float(lo << 16);
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = fminf(fmaxf(x[i], -tau), tau);
  }

  // ---- group statistics over lanes [8g, 8g+8)
  float lo = x[0], hi = x[0];
#pragma unroll
  for (int i = 1; i < 16; ++i) {
    lo = fminf(lo, x[i]);
    hi = fmaxf(hi, x[i]);
  }
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  const int L = (1 << p.bits_c) - 1;
  const QParams qp = make_qparams(lo, hi, L);
  flags |= qp.flags;

  int code[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) code[i] = quant_code(x[i], qp.m, qp.s, qp.inv_s, L);

  // ---- pack into the documented fragment layout (region A)
  const int g = lane >> 3, k = lane & 7;
  uint8_t* blk = page + static_cast<size_t>(((tp >> 3) * 4 + g) * (128 * p.bits_c));
  const int lane_base = 4 * (tp & 7);
  if (p.bits_c == 4) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t w = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int o = 0; o < 2; ++o)
          w |= static_cast<uint32_t>(code[8 * h + 2 * q + o]) << (4 * (2 * (k & 1) + h + 4 * o));
      w |= __shfl_xor_sync(0xffffffffu, w, 1);
      if ((k & 1) == 0)
        *reinterpret_cast<uint32_t*>(blk + (lane_base + q) * 16 + (k >> 1) * 4) = w;
    }
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t w = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int o = 0; o < 2; ++o)
          w |= static_cast<uint32_t>(code[8 * h + 2 * q + o]) << (2 * (2 * (k & 3) + h + 8 * o));
      w |= __shfl_xor_sync(0xffffffffu, w, 1);
      w |= __shfl_xor_sync(0xffffffffu, w, 2);
      if ((k & 3) == 0)
        *reinterpret_cast<uint32_t*>(blk + (lane_base + q) * 8 + (k >> 2) * 4) = w;
    }
  }
  // ---- latent metadata (region C)
  if (k == 0) {
    uint8_t* meta = page + static_cast<size_t>(p.P) * (64 * p.bits_c + 32) + (tp * 4 + g) * 4;
    *reinterpret_cast<uint32_t*>(meta) = qp.meta;
  }
  flags = __reduce_or_sync(0xffffffffu, flags);
  if (lane == 0) raise_err(p.err, flags);
}

// ------------------------------------------------------------------ page fill (one CTA)
__device__ void fill_page(const WriteParams& p, int b, int f, float* vals, float* stats) {
  const int tid = threadIdx.x;
  const int r0 = __ldg(p.cu_new + b), r1 = __ldg(p.cu_new + b + 1);
  const int s0 = __ldg(p.seq_lens + b);
  const int n = r1 - r0;
  if (s0 < 0 || n <= 0 || n > p.max_new || r0 < 0 || r1 > p.n_rows) return;  // reported by the token work
  const int64_t pg = static_cast<int64_t>(s0) / p.P + f;
  if ((pg + 1) * p.P > static_cast<int64_t>(s0) + n) return;  // this page does not fill now
  if (pg >= p.max_pages) return;
  const int32_t pid = __ldg(p.page_table + static_cast<size_t>(b) * p.max_pages + pg);
  if (pid < 0 || pid >= p.n_pages) return;
  uint8_t* page = p.pool + static_cast<size_t>(pid) * static_cast<size_t>(p.page_bytes);
  const int P = p.P;

  // gather the page's k_R values: earlier tokens from the ring, new ones from the input
  for (int idx = tid; idx < P * 32; idx += blockDim.x) {
    const int u = idx >> 5, jj = idx & 31;
    const int64_t tt = pg * P + u;
    const uint32_t* src;
    if (tt < s0)
      src = reinterpret_cast<const uint32_t*>(p.ring + (static_cast<size_t>(b) * p.W + (tt % p.W)) * kRow + kLatent);
    else
      src = reinterpret_cast<const uint32_t*>(p.kr_new + static_cast<size_t>(r0 + (tt - s0)) * kRope);
    const uint32_t w = src[jj];
    vals[u * 65 + 2 * jj] = bf16_lo(w);
    vals[u * 65 + 2 * jj + 1] = bf16_hi(w);
  }
  __syncthreads();
  int flags = 0;
  if (tid < kRope) {
    float lo = vals[tid], hi = vals[tid];
    bool bad = false;
    for (int u = 0; u < P; ++u) {
      const float v = vals[u * 65 + tid];
      bad |= !isfinite(v);
      lo = fminf(lo, v);
      hi = fmaxf(hi, v);
    }
    const QParams qp = make_qparams(lo, hi, 15);
    flags |= qp.flags | (bad ? kErrNonFinite : 0);
    stats[3 * tid] = qp.m;
    stats[3 * tid + 1] = qp.s;
    stats[3 * tid + 2] = qp.inv_s;
    *reinterpret_cast<uint32_t*>(page + static_cast<size_t>(P) * (64 * p.bits_c + 48) + tid * 4) = qp.meta;
  }
  __syncthreads();
  // codes, one 32-bit word of region B per iteration
  uint8_t* regb = page + static_cast<size_t>(P) * 64 * p.bits_c;
  for (int wi = tid; wi < P * 8; wi += blockDim.x) {
    const int tb = wi >> 7, rr = (wi >> 5) & 3, ln = wi & 31;
    const int q = ln & 3, g8 = ln >> 2;
    uint32_t word = 0;
#pragma unroll
    for (int nn = 0; nn < 2; ++nn)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int o = 0; o < 2; ++o) {
          const int u = 16 * tb + 8 * nn + g8;
          const int j = 16 * rr + 8 * h + 2 * q + o;
          const int c = quant_code(vals[u * 65 + j], stats[3 * j], stats[3 * j + 1], stats[3 * j + 2], 15);
          word |= static_cast<uint32_t>(c) << (4 * (2 * nn + h + 4 * o));
        }
    *reinterpret_cast<uint32_t*>(regb + ((tb * 4 + rr) * 128 + ln * 4)) = word;
  }
  if (flags) raise_err(p.err, flags);
}

__global__ void __launch_bounds__(128) write_kernel(const WriteParams p) {
  extern __shared__ float smem_f[];
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (__ldg(p.cu_new) != 0 || __ldg(p.cu_new + p.B) != p.n_rows) raise_err(p.err, kErrRows);
  }
  if (static_cast<int>(blockIdx.x) < p.token_blocks) {
    const int r = blockIdx.x * 4 + (threadIdx.x >> 5);
    if (r < p.n_rows) write_token(p, r, threadIdx.x & 31);
    return;
  }
  const int idx = blockIdx.x - p.token_blocks;
  const int b = idx / p.fill_per_seq, f = idx % p.fill_per_seq;
  if (b < p.B) fill_page(p, b, f, smem_f, smem_f + p.P * 65);
}

}  // namespace

cudaError_t launch_write(const WriteParams& p, cudaStream_t stream) {
  const int blocks = p.token_blocks + p.B * p.fill_per_seq;
  if (blocks == 0) return cudaSuccess;
  const size_t smem = p.fill_per_seq > 0 ? (static_cast<size_t>(p.P) * 65 + 3 * kRope) * sizeof(float) : 0;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(write_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  write_kernel<<<blocks, 128, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mlaq
