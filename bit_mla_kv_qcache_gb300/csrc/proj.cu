// Projections either side of the decode attention (RAQ-MLA page, Figure 4): the query is
// absorbed into the latent space (q_nope W_UK, with A_c^-1 folded into W_UK offline), k_R is
// compensated on the query side (q_rope R, one 64 x 64 matrix for every head), and the latent
// readout leaves through W_UV (A_c^-1 folded in). All three are Y[b, h, :] = X[b, h, :] W[h]:
// per head a product with few rows (the decode batch) and a weight matrix read once, so the
// bound is the weight bytes from HBM.
//
// CTA (column block, head, batch block): 32 output columns of one head for up to 64 batch
// rows; warp w takes rows 16 w .. 16 w + 15 (one m16 tile) over all 32 columns (four n8
// tiles) and the whole K. The CTA's W slice [K][32] and X rows [64][K] are staged in shared
// memory by 16-byte asynchronous copies (float32 X is rounded to BF16 on the way in), rows
// padded by 16 bytes so that the 8 x 8 matrix loads hit distinct banks; products on the tensor
// cores (mma.sync m16n8k16, BF16 in, float32 accumulation), BF16 output rounded to nearest even.
#include <cuda_bf16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace mlaq {
namespace {

constexpr int kProjCols = 32;      // output columns per CTA
constexpr int kProjRows = 64;      // batch rows per CTA (4 warps x m16)
constexpr int kProjThreads = 128;
constexpr int kWStride = kProjCols * 2 + 16;  // bytes per staged W row (80)

__host__ __device__ constexpr int x_stride(int K) { return K * 2 + 16; }
__host__ __device__ constexpr size_t proj_smem_bytes(int K) {
  return static_cast<size_t>(K) * kWStride + static_cast<size_t>(kProjRows) * x_stride(K);
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Two products may share a launch (the query absorption and the k_R compensation): column
// blocks [0, nx0) belong to p0, the rest to p1; both have the same B and H.
struct ProjPair {
  ProjParams p0, p1;
  int nx0;
};

template <bool kXF32, bool kYF32>
__global__ void __launch_bounds__(kProjThreads) proj_kernel(const ProjPair pp) {
  extern __shared__ __align__(128) uint8_t smem[];
  const bool second = static_cast<int>(blockIdx.x) >= pp.nx0;
  const ProjParams& p = second ? pp.p1 : pp.p0;
  uint8_t* ws = smem;
  uint8_t* xs = smem + static_cast<size_t>(p.K) * kWStride;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = kProjCols * (static_cast<int>(blockIdx.x) - (second ? pp.nx0 : 0));
  const int h = blockIdx.y, b0 = kProjRows * blockIdx.z;
  const int xst = x_stride(p.K);
  // rows read by the warps that have batch rows: [b0, b0 + 16 * active warps)
  const int rows = min(kProjRows, (p.B - b0 + 15) / 16 * 16);

  // ---- stage W[h][:, n0 .. n0 + 31] (four 16-byte chunks per row)
  const uint16_t* wh = p.w + static_cast<size_t>(h) * p.w_head_stride + n0;
  for (int i = tid; i < p.K * 4; i += kProjThreads) {
    const int k = i >> 2, c = i & 3;
    cp_async16(ws + k * kWStride + 16 * c, wh + static_cast<size_t>(k) * p.N + 8 * c);
  }
  // ---- stage X rows b0 .. b0 + rows - 1 of head h (rows past the batch are zero); float32
  // rows are read eight chunks per thread at a time (all loads in flight before any store)
  const int chunks = p.K / 8;  // 16-byte BF16 chunks per row
  const int items = rows * chunks;
  if constexpr (kXF32) {
    constexpr int kU = 8;
    for (int i0 = tid; i0 < items; i0 += kProjThreads * kU) {
      float4 u[kU], v[kU];
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int i = i0 + j * kProjThreads, r = i / chunks, c = i % chunks, b = b0 + r;
        u[j] = v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < items && b < p.B) {
          const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.x) +
                                                              (static_cast<size_t>(b) * p.H + h) * p.K) + 2 * c;
          u[j] = __ldg(src);
          v[j] = __ldg(src + 1);
        }
      }
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int i = i0 + j * kProjThreads;
        if (i < items)
          *reinterpret_cast<uint4*>(xs + (i / chunks) * xst + 16 * (i % chunks)) =
              make_uint4(pack_bf16(u[j].x, u[j].y), pack_bf16(u[j].z, u[j].w), pack_bf16(v[j].x, v[j].y),
                         pack_bf16(v[j].z, v[j].w));
      }
    }
  } else {
    for (int i = tid; i < items; i += kProjThreads) {
      const int r = i / chunks, c = i % chunks, b = b0 + r;
      uint8_t* dst = xs + r * xst + 16 * c;
      if (b >= p.B)
        *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
      else
        cp_async16(dst, static_cast<const uint16_t*>(p.x) + (static_cast<size_t>(b) * p.H + h) * p.K + 8 * c);
    }
  }
  cp_async_wait_all();
  __syncthreads();
  if (b0 + 16 * warp >= p.B) return;  // this warp's rows are all past the batch

  float acc[4][4];
#pragma unroll
  for (int t = 0; t < 4; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  const uint8_t* a_base = xs + (16 * warp + (lane & 15)) * xst + 16 * (lane >> 4);
  const uint8_t* b_base = ws + ((lane & 7) + 8 * ((lane >> 3) & 1)) * kWStride + 16 * (lane >> 4);
  for (int k0 = 0; k0 < p.K; k0 += 16) {
    uint32_t a[4], b01[4], b23[4];
    ldsm_x4(a, a_base + 2 * k0);
    ldsm_x4_t(b01, b_base + k0 * kWStride);       // n8 tiles 0, 1
    ldsm_x4_t(b23, b_base + k0 * kWStride + 32);  // n8 tiles 2, 3
    mma_bf16_16816(acc[0], a, b01[0], b01[1]);
    mma_bf16_16816(acc[1], a, b01[2], b01[3]);
    mma_bf16_16816(acc[2], a, b23[0], b23[1]);
    mma_bf16_16816(acc[3], a, b23[2], b23[3]);
  }

  // ---- store: thread (g, q) holds rows g, g + 8 and columns 8 t + 2 q, 8 t + 2 q + 1
  const int g = lane >> 2, q = lane & 3;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int b = b0 + 16 * warp + g + 8 * half;
    if (b >= p.B) continue;
    const size_t row = (static_cast<size_t>(b) * p.H + h) * p.N + n0 + 2 * q;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float v0 = acc[t][2 * half], v1 = acc[t][2 * half + 1];
      if constexpr (kYF32)
        *reinterpret_cast<float2*>(static_cast<float*>(p.y) + row + 8 * t) = make_float2(v0, v1);
      else
        *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.y) + row + 8 * t) = pack_bf16(v0, v1);
    }
  }
}

template <bool kXF32, bool kYF32>
cudaError_t launch_proj_t(const ProjPair& pp, int nx, cudaStream_t stream) {
  const ProjParams& p = pp.p0;
  const size_t smem = proj_smem_bytes(pp.p0.K > pp.p1.K ? pp.p0.K : pp.p1.K);
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(proj_kernel<kXF32, kYF32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(proj_smem_bytes(kProjMaxK)));
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const dim3 grid(nx, p.H, (p.B + kProjRows - 1) / kProjRows);
  proj_kernel<kXF32, kYF32><<<grid, kProjThreads, smem, stream>>>(pp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_proj(const ProjParams& p0, const ProjParams* p1, cudaStream_t stream) {
  if (p0.B == 0) return cudaSuccess;
  ProjPair pp{p0, p1 ? *p1 : p0, p0.N / kProjCols};
  const int nx = pp.nx0 + (p1 ? p1->N / kProjCols : 0);
  if (p1 && (p1->B != p0.B || p1->H != p0.H || p1->x_f32 != p0.x_f32 || p1->y_f32 != p0.y_f32))
    return cudaErrorInvalidValue;
  if (p0.x_f32)
    return p0.y_f32 ? launch_proj_t<true, true>(pp, nx, stream) : launch_proj_t<true, false>(pp, nx, stream);
  return p0.y_f32 ? launch_proj_t<false, true>(pp, nx, stream) : launch_proj_t<false, false>(pp, nx, stream);
}

}  // namespace mlaq
