// Kernel parameter blocks and launchers shared by the C ABI layer (abi.cu) and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace mlaq {

constexpr int kLatent = 512;
constexpr int kRope = 64;
constexpr int kRow = 576;
constexpr int kGroup = 128;

// Device error bits (same values as MLA_QCACHE_DEV_* in the public header).
constexpr int kErrBadPage = 1;
constexpr int kErrSeqOverflow = 2;
constexpr int kErrNonFinite = 4;
constexpr int kErrRange = 8;
constexpr int kErrRows = 16;
constexpr int kErrTimeout = 32;

struct WriteParams {
  int B, n_rows, max_new, max_pages;
  int P, S, W, bits_c, clip_k;  // clip_k: rank of the clip order statistic (0 = no clip)
  int64_t n_pages;
  int64_t page_bytes;
  const uint16_t* c_new;
  const uint16_t* kr_new;
  const int32_t* cu_new;
  const int32_t* seq_lens;
  const int32_t* page_table;
  uint8_t* pool;
  uint16_t* sink;
  uint16_t* ring;
  int32_t* err;
  int32_t* seq_next;  // optional: lengths after the call (written by page-fill CTA 0 of each sequence)
  const uint16_t* a_c;  // optional BF16 [512][512]: the latent is cached as c A_c
  const uint16_t* a_r;  // optional BF16 [64][64]: k_R is cached as k_R A_R
  int token_blocks;  // blocks [0, token_blocks) do per-token work (one token per block)
  int fill_per_seq;  // page-fill blocks per sequence after the token blocks
};

// One launch doing per-token packing/retention (token_blocks > 0) and/or page fills.
cudaError_t launch_write(const WriteParams& p, cudaStream_t stream);
// out = x A row by row (BF16 rows of dim 64 or 512), the arithmetic of the transforming writer.
cudaError_t launch_row_transform(int n_rows, int dim, const uint16_t* x, const uint16_t* a, uint16_t* out,
                                 int32_t* err, cudaStream_t stream);
// Y[b, h, :] = X[b, h, :] W[h] for X [B][H][K] (BF16, or float32 rounded to BF16) and W
// [H][K][N] BF16 (w_head_stride elements between heads, 0 = one matrix for every head);
// Y [B][H][N] BF16 or float32. K % 16 == 0, 16 <= K <= kProjMaxK, N % 32 == 0.
constexpr int kProjMaxK = 512;
struct ProjParams {
  int B, H, K, N;
  const void* x;
  bool x_f32;
  const uint16_t* w;
  size_t w_head_stride;
  void* y;
  bool y_f32;
};
// p1 (optional): a second product of the same B, H and operand types in the same launch.
cudaError_t launch_proj(const ProjParams& p0, const ProjParams* p1, cudaStream_t stream);
// A kernel whose bounded wait must give up: ORs kErrTimeout into *err.
cudaError_t launch_wait_selftest(int32_t* err, cudaStream_t stream);
// seq_lens[b] += cu_new[b+1] - cu_new[b] for b in [0, B).
cudaError_t launch_advance(const int32_t* cu_new, int32_t* seq_lens, int B, cudaStream_t stream);

struct DecodeParams {
  const uint16_t* q_lat;
  const uint16_t* q_rope;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const uint8_t* pool;
  const uint16_t* sink;
  const uint16_t* ring;
  const uint16_t* kv_bf16;  // paged BF16 cache of the unquantized comparator (else nullptr)
  // Arrival counters of the in-kernel merge, one 64-bit word per (sequence, 16-head block):
  // count (low half, zero between calls) and generation (high half), in the workspace's first
  // kArriveBytes. nullptr: the partials are merged by a separate launch.
  unsigned long long* arrive;
  float* o_part;  // [B][H][NS][512] partial (unnormalized) outputs
  float* ml_part; // [B][H][NS][2] partial (max in log2 units, sum)
  float* out;     // [B][H][512]
  float* lse;     // [B][H]
  int32_t* err;
  int64_t n_pages;
  int64_t page_bytes;
  float scale_log2;  // softmax_scale * log2(e)
  int B, H, max_pages, P, S, W, bits_c;
  int p_shift;  // log2(P): page sizes are powers of two
  int n_split;  // shares of the packed tokens (partial slots 0 .. n_split-1)
  int n_q;      // CTAs sharing the protected (BF16) tokens (partial slots n_split .. n_split+n_q-1)
  int share_slots;  // resident CTA slots of one wave left for packed shares (16-head kernel);
                    // > 0: balanced equal shares (more shares launched than one wave holds)
  int q_len;        // new tokens decoded per sequence (rows [position][head]; 0 or 1: one)
  int h_pos;        // rows per position (H / q_len), a multiple of 16
  // Rows not yet written to the cache (decode of the cache as the write of these rows will
  // leave it): sequence b's rows cu_new[b] .. cu_new[b+1]-1 are its tokens seq_lens[b] ..;
  // cu_new == nullptr: none. They are read from here instead of the sink/recent buffers.
  const uint16_t* c_new;   // [rows][512] BF16
  const uint16_t* kr_new;  // [rows][64] BF16
  const int32_t* cu_new;   // [B+1]
  int max_new;             // bound on the rows per sequence (larger counts are an error)
};

#ifdef __CUDACC__
// Sequence b's length seen by a decode: the cached length plus its pending rows. Out-of-range
// values set an error bit and count as an empty sequence; `T_old` receives the cached length
// (the first pending token). In two steps, so that a kernel can issue other work between the
// loads and the first use of their values.
struct SeqLenWords {
  int T, c0, c1;  // seq_lens[b]; cu_new[b], cu_new[b+1] (0, 0 without pending rows)
};
__device__ __forceinline__ SeqLenWords decode_seq_len_load(const DecodeParams& p, int b) {
  SeqLenWords w;
  w.T = __ldg(p.seq_lens + b);
  w.c0 = w.c1 = 0;
  if (p.cu_new != nullptr) {
    w.c0 = __ldg(p.cu_new + b);
    w.c1 = __ldg(p.cu_new + b + 1);
  }
  return w;
}
__device__ __forceinline__ int decode_seq_len_check(const DecodeParams& p, const SeqLenWords& w, int& T_old,
                                                    int32_t& flags) {
  const int T = w.T;
  int n_new = w.c1 - w.c0;
  if (p.cu_new != nullptr && (n_new < 0 || n_new > p.max_new)) {
    flags |= kErrRows;
    n_new = 0;
  }
  if (T < 0 || static_cast<long long>(T) + n_new > static_cast<long long>(p.max_pages) * p.P) {
    flags |= kErrSeqOverflow;
    T_old = 0;
    return 0;
  }
  T_old = T;
  return T + n_new;
}
__device__ __forceinline__ int decode_seq_len(const DecodeParams& p, int b, int& T_old, int32_t& flags) {
  return decode_seq_len_check(p, decode_seq_len_load(p, b), T_old, flags);
}
#endif

// Number of packed-token shares, and of CTAs for the protected tokens, of each (sequence,
// 16-head block) for a problem size (depends on the SM count).
int decode_num_splits(int B, int H, int max_pages, int P, int S, int W, int num_sms);
int decode_num_protected(int B, int H, int max_pages, int P, int S, int W, int num_sms);
// Workspace layout of a decode call: kArriveBytes of merge counters (zero between calls), then the
// partial outputs and the partial maxima and sums.
constexpr size_t kArriveBytes = 8192;
constexpr int kMaxArriveGroups = static_cast<int>(kArriveBytes / 8);
size_t decode_workspace_bytes(int B, int H, int n_slots);  // n_slots = n_split + n_q
int decode_share_slots(int B, int H, int max_pages, int P, int n_split, int n_q, int num_sms);
// Head counts that are multiples of 64 run the packed shares on tcgen05 tensor cores (64 heads
// per CTA, one CTA per SM); the others on the 16-head warp-level kernel.
inline bool decode_uses_tc(int H) { return H % 64 == 0; }
int decode_tc_num_splits(int B, int H, int max_pages, int P, int num_sms);
cudaError_t launch_decode_tc(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream);
// Kernel launches of one decode call on the current device (1: partials merged in place; 2: a
// merge launch follows; 3: 64-head blocks), or -1 on a CUDA error.
int decode_launch_count(int bits_c, int B, int H, int n_split, int n_q, int share_slots);
// Unquantized comparator: decode over a paged BF16 cache [n_pages][P][576] (every share BF16).
int decode_bf16_num_parts(int B, int H, int max_pages, int P, int num_sms);
cudaError_t launch_decode_bf16(const DecodeParams& p, cudaStream_t stream);

// Built-in decode scratch for callers that cannot allocate (mla_qcache_decode_attn_noalloc).
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
cudaError_t noalloc_scratch(void** out);

}  // namespace mlaq
