// C ABI entry points (declared in include/mla_qcache.h): host-side validation, problem
// decomposition and kernel launches on the caller's stream. No allocation, no synchronization.
#include <cmath>
#include <cstdint>

#include <cuda_runtime.h>

#include "kernels.cuh"
#include "mla_qcache.h"

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_config(const mla_qcache_config* c) {
  if (!c) return MLA_QCACHE_ERR_NULL;
  if (c->bits_c != 2 && c->bits_c != 4) return MLA_QCACHE_ERR_CONFIG;
  if (c->bits_r != 4) return MLA_QCACHE_ERR_CONFIG;
  const int P = c->page_size;
  if (P != 32 && P != 64 && P != 128) return MLA_QCACHE_ERR_CONFIG;  // a 32-token decode tile never straddles pages
  if (c->n_sink < 0 || c->n_sink > 16) return MLA_QCACHE_ERR_CONFIG;
  if (c->n_recent < P || c->n_recent > 1024) return MLA_QCACHE_ERR_CONFIG;
  if (!(c->clip_q >= 0.0f && c->clip_q <= 1.0f)) return MLA_QCACHE_ERR_CONFIG;
  return MLA_QCACHE_OK;
}

int64_t page_bytes_of(const mla_qcache_config* c) {
  return static_cast<int64_t>(c->page_size) * (64 * c->bits_c + 48) + 256;
}

int current_sm_count(int* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_QCACHE_ERR_CUDA;
  if (cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MLA_QCACHE_ERR_CUDA;
  return MLA_QCACHE_OK;
}

}  // namespace

extern "C" {

int mla_qcache_config_check(const mla_qcache_config* cfg) { return check_config(cfg); }

size_t mla_qcache_page_bytes(const mla_qcache_config* cfg) {
  if (check_config(cfg) != MLA_QCACHE_OK) return 0;
  return static_cast<size_t>(page_bytes_of(cfg));
}

size_t mla_qcache_workspace_bytes(const mla_qcache_config* cfg, int32_t B, int32_t H, int32_t max_pages) {
  if (check_config(cfg) != MLA_QCACHE_OK || B < 1 || H < 16 || H > 256 || H % 16 || max_pages < 1) return 0;
  int sms = 0;
  if (current_sm_count(&sms) != MLA_QCACHE_OK) return 0;
  const int ns = mlaq::decode_num_splits(B, H, max_pages, cfg->page_size, cfg->n_sink, cfg->n_recent, sms);
  const int nq = mlaq::decode_num_protected(B, H, max_pages, cfg->page_size, cfg->n_sink, cfg->n_recent, sms);
  return mlaq::decode_workspace_bytes(B, H, ns + nq);
}

}  // extern "C"

static int write_impl(const mla_qcache_config* cfg, int32_t B, int32_t n_rows, const uint16_t* c_new,
                     const uint16_t* kr_new, const int32_t* cu_new, const int32_t* seq_lens, int32_t max_new,
                     const int32_t* page_table, int32_t max_pages, uint8_t* pool, int64_t n_pages,
                     uint16_t* sink_buf, uint16_t* recent_buf, int32_t* err_word, int32_t* seq_next, void* stream,
                     const uint16_t* a_c = nullptr, const uint16_t* a_r = nullptr) {
  int st = check_config(cfg);
  if (st != MLA_QCACHE_OK) return st;
  if (B < 1 || B > (1 << 20) || n_rows < 0 || max_pages < 1 || n_pages < 1) return MLA_QCACHE_ERR_SHAPE;
  if (n_rows == 0) {  // nothing to write; the next lengths equal the current ones
    if (seq_next == nullptr) return MLA_QCACHE_OK;
    if (!seq_lens) return MLA_QCACHE_ERR_NULL;
    if (!aligned(seq_lens, 4) || !aligned(seq_next, 4)) return MLA_QCACHE_ERR_ALIGN;
    return cudaMemcpyAsync(seq_next, seq_lens, static_cast<size_t>(B) * sizeof(int32_t), cudaMemcpyDeviceToDevice,
                           static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MLA_QCACHE_OK
               : MLA_QCACHE_ERR_CUDA;
  }
  if (max_new < 1) return MLA_QCACHE_ERR_SHAPE;
  // one CTA per row (a cluster of eight when the rows are transformed, the grid then padded to
  // whole clusters) plus four per page that may fill, in one grid dimension
  const int64_t row_ctas = (a_c || a_r) ? static_cast<int64_t>(n_rows) * 8 + 7 : n_rows;
  if (static_cast<int64_t>(B) * (max_new / cfg->page_size + 1) * 4 + row_ctas > 0x7fffffff)
    return MLA_QCACHE_ERR_SHAPE;
  if (!c_new || !kr_new || !cu_new || !seq_lens || !page_table || !pool || !recent_buf || !err_word)
    return MLA_QCACHE_ERR_NULL;
  if (cfg->n_sink > 0 && !sink_buf) return MLA_QCACHE_ERR_NULL;
  if (!aligned(c_new, 16) || !aligned(kr_new, 4) || !aligned(pool, 16) || !aligned(recent_buf, 16) ||
      (sink_buf && !aligned(sink_buf, 16)) || !aligned(cu_new, 4) || !aligned(seq_lens, 4) ||
      !aligned(page_table, 4) || !aligned(err_word, 4) || (seq_next && !aligned(seq_next, 4)) ||
      (a_c && !aligned(a_c, 16)) || (a_r && !aligned(a_r, 16)))
    return MLA_QCACHE_ERR_ALIGN;

  mlaq::WriteParams p{};
  p.B = B;
  p.n_rows = n_rows;
  p.max_new = max_new;
  p.max_pages = max_pages;
  p.P = cfg->page_size;
  p.S = cfg->n_sink;
  p.W = cfg->n_recent;
  p.bits_c = cfg->bits_c;
  p.clip_k = 0;
  if (cfg->clip_q > 0.0f) {
    int k = static_cast<int>(std::ceil(static_cast<double>(cfg->clip_q) * 512.0));
    p.clip_k = k < 1 ? 1 : (k > 512 ? 512 : k);
  }
  p.n_pages = n_pages;
  p.page_bytes = page_bytes_of(cfg);
  p.c_new = c_new;
  p.kr_new = kr_new;
  p.cu_new = cu_new;
  p.seq_lens = seq_lens;
  p.page_table = page_table;
  p.pool = pool;
  p.sink = sink_buf;
  p.ring = recent_buf;
  p.err = err_word;
  p.seq_next = seq_next;
  p.a_c = a_c;
  p.a_r = a_r;
  const int token_blocks = n_rows;  // one CTA (or cluster) per new token
  const int fill_per_seq = max_new / p.P + 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (max_new <= p.W - p.P + 1) {
    // No new token can overwrite a ring row that a page fill of this call still reads.
    p.token_blocks = token_blocks;
    p.fill_per_seq = fill_per_seq;
    e = mlaq::launch_write(p, s);
  } else {
    // Page fills first (they read earlier tokens from the ring), then the per-token work.
    p.token_blocks = 0;
    p.fill_per_seq = fill_per_seq;
    e = mlaq::launch_write(p, s);
    if (e == cudaSuccess) {
      p.token_blocks = token_blocks;
      p.fill_per_seq = 0;
      p.seq_next = nullptr;  // written by the first launch
      e = mlaq::launch_write(p, s);
    }
  }
  return e == cudaSuccess ? MLA_QCACHE_OK : MLA_QCACHE_ERR_CUDA;
}

extern "C" {

int mla_qcache_write(const mla_qcache_config* cfg, int32_t B, int32_t n_rows, const uint16_t* c_new,
                     const uint16_t* kr_new, const int32_t* cu_new, const int32_t* seq_lens, int32_t max_new,
                     const int32_t* page_table, int32_t max_pages, uint8_t* pool, int64_t n_pages,
                     uint16_t* sink_buf, uint16_t* recent_buf, int32_t* err_word, void* stream) {
  return write_impl(cfg, B, n_rows, c_new, kr_new, cu_new, seq_lens, max_new, page_table, max_pages, pool, n_pages,
                    sink_buf, recent_buf, err_word, nullptr, stream);
}

int mla_qcache_write_advance(const mla_qcache_config* cfg, int32_t B, int32_t n_rows, const uint16_t* c_new,
                             const uint16_t* kr_new, const int32_t* cu_new, const int32_t* seq_lens,
                             int32_t* seq_lens_next, int32_t max_new, const int32_t* page_table, int32_t max_pages,
                             uint8_t* pool, int64_t n_pages, uint16_t* sink_buf, uint16_t* recent_buf,
                             int32_t* err_word, void* stream) {
  if (!seq_lens_next) return MLA_QCACHE_ERR_NULL;
  if (B >= 1 && seq_lens) {  // the two length arrays must not overlap
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(seq_lens), b0 = reinterpret_cast<uintptr_t>(seq_lens_next);
    const uintptr_t len = static_cast<uintptr_t>(B) * sizeof(int32_t);
    if (a0 < b0 + len && b0 < a0 + len) return MLA_QCACHE_ERR_SHAPE;
  }
  return write_impl(cfg, B, n_rows, c_new, kr_new, cu_new, seq_lens, max_new, page_table, max_pages, pool, n_pages,
                    sink_buf, recent_buf, err_word, seq_lens_next, stream);
}

int mla_qcache_write_transformed(const mla_qcache_config* cfg, int32_t B, int32_t n_rows, const uint16_t* c_new,
                                 const uint16_t* kr_new, const int32_t* cu_new, const int32_t* seq_lens,
                                 int32_t* seq_lens_next, int32_t max_new, const uint16_t* a_c, const uint16_t* a_r,
                                 const int32_t* page_table, int32_t max_pages, uint8_t* pool, int64_t n_pages,
                                 uint16_t* sink_buf, uint16_t* recent_buf, int32_t* err_word, void* stream) {
  if (seq_lens_next && B >= 1 && seq_lens) {  // the two length arrays must not overlap
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(seq_lens), b0 = reinterpret_cast<uintptr_t>(seq_lens_next);
    const uintptr_t len = static_cast<uintptr_t>(B) * sizeof(int32_t);
    if (a0 < b0 + len && b0 < a0 + len) return MLA_QCACHE_ERR_SHAPE;
  }
  return write_impl(cfg, B, n_rows, c_new, kr_new, cu_new, seq_lens, max_new, page_table, max_pages, pool, n_pages,
                    sink_buf, recent_buf, err_word, seq_lens_next, stream, a_c, a_r);
}

int mla_qcache_row_transform(int32_t n_rows, int32_t dim, const uint16_t* x, const uint16_t* a, uint16_t* out,
                             int32_t* err_word, void* stream) {
  if (n_rows < 0 || (dim != 64 && dim != 512)) return MLA_QCACHE_ERR_SHAPE;
  if (n_rows == 0) return MLA_QCACHE_OK;
  if (!x || !a || !out || !err_word) return MLA_QCACHE_ERR_NULL;
  if (!aligned(x, 2) || !aligned(a, 16) || !aligned(out, 2) || !aligned(err_word, 4)) return MLA_QCACHE_ERR_ALIGN;
  const uintptr_t xs = reinterpret_cast<uintptr_t>(x), os = reinterpret_cast<uintptr_t>(out);
  const uintptr_t len = static_cast<uintptr_t>(n_rows) * static_cast<uintptr_t>(dim) * 2;
  if (xs < os + len && os < xs + len) return MLA_QCACHE_ERR_SHAPE;  // in place is not supported
  const cudaError_t e =
      mlaq::launch_row_transform(n_rows, dim, x, a, out, err_word, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_QCACHE_OK : MLA_QCACHE_ERR_CUDA;
}

static int proj_checks(int32_t B, int32_t H, int32_t K, int32_t N, const void* x, const void* w, const void* y) {
  if (B < 0 || B > (1 << 22) || H < 1 || H > 256 || K < 16 || K > mlaq::kProjMaxK || K % 16 || N < 32 || N % 32)
    return MLA_QCACHE_ERR_SHAPE;
  if (B > 0 && (!x || !w || !y)) return MLA_QCACHE_ERR_NULL;
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16)) return MLA_QCACHE_ERR_ALIGN;
  return MLA_QCACHE_OK;
}

int mla_qcache_decode_plan(const mla_qcache_config* cfg, int32_t B, int32_t H, int32_t max_pages, int32_t num_sms,
                           int32_t* plan) {
  const int st = check_config(cfg);
  if (st != MLA_QCACHE_OK) return st;
  if (!plan) return MLA_QCACHE_ERR_NULL;
  if (B < 1 || H < 16 || H > 256 || H % 16 || max_pages < 1 || num_sms < 1) return MLA_QCACHE_ERR_SHAPE;
  const int ns = mlaq::decode_num_splits(B, H, max_pages, cfg->page_size, cfg->n_sink, cfg->n_recent, num_sms);
  const int nq = mlaq::decode_num_protected(B, H, max_pages, cfg->page_size, cfg->n_sink, cfg->n_recent, num_sms);
  plan[0] = ns;
  plan[1] = nq;
  plan[2] = mlaq::decode_share_slots(B, H, max_pages, cfg->page_size, ns, nq, num_sms);
  plan[3] = mlaq::decode_uses_tc(H) ? 1 : 0;
  plan[4] = mlaq::decode_bf16_num_parts(B, H, max_pages, cfg->page_size, num_sms);
  return MLA_QCACHE_OK;
}

int mla_qcache_decode_launches(const mla_qcache_config* cfg, int32_t B, int32_t H, int32_t max_pages) {
  const int st = check_config(cfg);
  if (st != MLA_QCACHE_OK) return st;
  if (B < 1 || B > 65535 || H < 16 || H > 256 || H % 16 || max_pages < 1) return MLA_QCACHE_ERR_SHAPE;
  int sms = 0;
  const int st2 = current_sm_count(&sms);
  if (st2 != MLA_QCACHE_OK) return st2;
  const int ns = mlaq::decode_num_splits(B, H, max_pages, cfg->page_size, cfg->n_sink, cfg->n_recent, sms);
  const int nq = mlaq::decode_num_protected(B, H, max_pages, cfg->page_size, cfg->n_sink, cfg->n_recent, sms);
  const int slots = mlaq::decode_share_slots(B, H, max_pages, cfg->page_size, ns, nq, sms);
  const int n = mlaq::decode_launch_count(cfg->bits_c, B, H, ns, nq, slots);
  return n > 0 ? n : MLA_QCACHE_ERR_CUDA;
}

int mla_qcache_absorb_query(int32_t B, int32_t H, int32_t d_nope, const uint16_t* q_nope, const uint16_t* w_uk,
                            const uint16_t* q_rope, const uint16_t* r_comp, uint16_t* q_lat, uint16_t* q_rope_out,
                            void* stream) {
  int st = proj_checks(B, H, d_nope, mlaq::kLatent, q_nope, w_uk, q_lat);
  if (st != MLA_QCACHE_OK) return st;
  if ((r_comp == nullptr) != (q_rope_out == nullptr)) return MLA_QCACHE_ERR_NULL;
  if (r_comp && (st = proj_checks(B, H, mlaq::kRope, mlaq::kRope, q_rope, r_comp, q_rope_out)) != MLA_QCACHE_OK)
    return st;
  if (B == 0) return MLA_QCACHE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  mlaq::ProjParams p{B, H, d_nope, mlaq::kLatent, q_nope, false, w_uk,
                     static_cast<size_t>(d_nope) * mlaq::kLatent, q_lat, false};
  const mlaq::ProjParams pr{B, H, mlaq::kRope, mlaq::kRope, q_rope, false, r_comp, 0, q_rope_out, false};
  const cudaError_t e = mlaq::launch_proj(p, r_comp ? &pr : nullptr, s);  // one launch for both
  return e == cudaSuccess ? MLA_QCACHE_OK : MLA_QCACHE_ERR_CUDA;
}

int mla_qcache_up_project(int32_t B, int32_t H, int32_t d_v, const float* o, const uint16_t* w_uv, float* out,
                          void* stream) {
  const int st = proj_checks(B, H, mlaq::kLatent, d_v, o, w_uv, out);
  if (st != MLA_QCACHE_OK) return st;
  if (B == 0) return MLA_QCACHE_OK;
  const mlaq::ProjParams p{B, H, mlaq::kLatent, d_v, o, true, w_uv, static_cast<size_t>(mlaq::kLatent) * d_v, out,
                           true};
  const cudaError_t e = mlaq::launch_proj(p, nullptr, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_QCACHE_OK : MLA_QCACHE_ERR_CUDA;
}

int mla_qcache_selftest_wait_timeout(int32_t* err_word, void* stream) {
  if (!err_word) return MLA_QCACHE_ERR_NULL;
  if (!aligned(err_word, 4)) return MLA_QCACHE_ERR_ALIGN;
  const cudaError_t e = mlaq::launch_wait_selftest(err_word, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_QCACHE_OK : MLA_QCACHE_ERR_CUDA;
}

int mla_qcache_advance(const int32_t* cu_new, int32_t* seq_lens, int32_t B, void* stream) {
  if (!cu_new || !seq_lens) return MLA_QCACHE_ERR_NULL;
  if (B < 1) return MLA_QCACHE_ERR_SHAPE;
  if (!aligned(cu_new, 4) || !aligned(seq_lens, 4)) return MLA_QCACHE_ERR_ALIGN;
  const cudaError_t e = mlaq::launch_advance(cu_new, seq_lens, B, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_QCACHE_OK : MLA_QCACHE_ERR_CUDA;
}

}  // extern "C"

// H: rows per sequence (q_len positions x H / q_len heads, position-major).
// Rows of a write that has not run yet (mla_qcache_decode_attn_pending); cu_new == nullptr: none.
struct PendingRows {
  const uint16_t* c_new = nullptr;
  const uint16_t* kr_new = nullptr;
  const int32_t* cu_new = nullptr;
  int32_t max_new = 0;
};

static int decode_impl(const mla_qcache_config* cfg, int32_t B, int32_t H, int32_t q_len, const uint16_t* q_lat,
                       const uint16_t* q_rope, const int32_t* page_table, int32_t max_pages,
                       const int32_t* seq_lens, const uint8_t* pool, int64_t n_pages, const uint16_t* sink_buf,
                       const uint16_t* recent_buf, float softmax_scale, float* out, float* lse, void* workspace,
                       size_t workspace_bytes, int32_t* err_word, void* stream, const PendingRows& pend = PendingRows()) {
  int st = check_config(cfg);
  if (st != MLA_QCACHE_OK) return st;
  if (B < 1 || B > 65535 || H < 16 || H > 256 || H % 16 || max_pages < 1 || n_pages < 1)
    return MLA_QCACHE_ERR_SHAPE;
  if (q_len < 1 || H % q_len || (H / q_len) % 16 || q_len - 1 > cfg->n_recent) return MLA_QCACHE_ERR_SHAPE;
  if (!q_lat || !q_rope || !page_table || !seq_lens || !pool || !recent_buf || !out || !lse || !workspace ||
      !err_word)
    return MLA_QCACHE_ERR_NULL;
  if (cfg->n_sink > 0 && !sink_buf) return MLA_QCACHE_ERR_NULL;
  if (!aligned(q_lat, 4) || !aligned(q_rope, 4) || !aligned(pool, 16) || !aligned(recent_buf, 16) ||
      (sink_buf && !aligned(sink_buf, 16)) || !aligned(out, 16) || !aligned(lse, 4) || !aligned(workspace, 16) ||
      !aligned(page_table, 4) || !aligned(seq_lens, 4) || !aligned(err_word, 4))
    return MLA_QCACHE_ERR_ALIGN;
  int sms = 0;
  st = current_sm_count(&sms);
  if (st != MLA_QCACHE_OK) return st;
  const int ns = mlaq::decode_num_splits(B, H, max_pages, cfg->page_size, cfg->n_sink, cfg->n_recent, sms);
  const int nq = mlaq::decode_num_protected(B, H, max_pages, cfg->page_size, cfg->n_sink, cfg->n_recent, sms);
  const size_t need = mlaq::decode_workspace_bytes(B, H, ns + nq);
  if (workspace_bytes < need) return MLA_QCACHE_ERR_WORKSPACE;

  mlaq::DecodeParams p{};
  p.q_lat = q_lat;
  p.q_rope = q_rope;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.pool = pool;
  p.sink = sink_buf;
  p.ring = recent_buf;
  p.arrive = static_cast<unsigned long long*>(workspace);
  p.o_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + mlaq::kArriveBytes);
  p.ml_part = p.o_part + static_cast<size_t>(B) * H * (ns + nq) * mlaq::kLatent;
  p.out = out;
  p.lse = lse;
  p.err = err_word;
  p.n_pages = n_pages;
  p.page_bytes = page_bytes_of(cfg);
  p.scale_log2 = static_cast<float>(static_cast<double>(softmax_scale) * 1.4426950408889634074);
  p.B = B;
  p.H = H;
  p.max_pages = max_pages;
  p.P = cfg->page_size;
  p.p_shift = 0;
  while ((1 << p.p_shift) < p.P) ++p.p_shift;
  p.S = cfg->n_sink;
  p.W = cfg->n_recent;
  p.bits_c = cfg->bits_c;
  p.n_split = ns;
  p.n_q = nq;
  p.share_slots = mlaq::decode_share_slots(B, H, max_pages, cfg->page_size, ns, nq, sms);
  p.q_len = q_len;
  p.h_pos = H / q_len;
  p.c_new = pend.c_new;
  p.kr_new = pend.kr_new;
  p.cu_new = pend.cu_new;
  p.max_new = pend.max_new;
  const cudaError_t e = mlaq::launch_decode(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_QCACHE_OK : MLA_QCACHE_ERR_CUDA;
}

extern "C" {

int mla_qcache_decode_attn(const mla_qcache_config* cfg, int32_t B, int32_t H, const uint16_t* q_lat,
                           const uint16_t* q_rope, const int32_t* page_table, int32_t max_pages,
                           const int32_t* seq_lens, const uint8_t* pool, int64_t n_pages,
                           const uint16_t* sink_buf, const uint16_t* recent_buf, float softmax_scale, float* out,
                           float* lse, void* workspace, size_t workspace_bytes, int32_t* err_word, void* stream) {
  return decode_impl(cfg, B, H, 1, q_lat, q_rope, page_table, max_pages, seq_lens, pool, n_pages, sink_buf,
                     recent_buf, softmax_scale, out, lse, workspace, workspace_bytes, err_word, stream);
}

int mla_qcache_decode_attn_pending(const mla_qcache_config* cfg, int32_t B, int32_t H, const uint16_t* q_lat,
                                   const uint16_t* q_rope, const int32_t* page_table, int32_t max_pages,
                                   const int32_t* seq_lens, const uint16_t* c_new, const uint16_t* kr_new,
                                   const int32_t* cu_new, int32_t max_new, const uint8_t* pool, int64_t n_pages,
                                   const uint16_t* sink_buf, const uint16_t* recent_buf, float softmax_scale,
                                   float* out, float* lse, void* workspace, size_t workspace_bytes, int32_t* err_word,
                                   void* stream) {
  int st = check_config(cfg);
  if (st != MLA_QCACHE_OK) return st;
  // the pending rows must lie in the recent window, and every token they push out of it must
  // already sit in a full page: max_new <= W - P + 1
  if (max_new < 0 || max_new > cfg->n_recent - cfg->page_size + 1) return MLA_QCACHE_ERR_SHAPE;
  if (!c_new || !kr_new || !cu_new) return MLA_QCACHE_ERR_NULL;
  if (!aligned(c_new, 16) || !aligned(kr_new, 16) || !aligned(cu_new, 4)) return MLA_QCACHE_ERR_ALIGN;
  PendingRows pend;
  pend.c_new = c_new;
  pend.kr_new = kr_new;
  pend.cu_new = cu_new;
  pend.max_new = max_new;
  return decode_impl(cfg, B, H, 1, q_lat, q_rope, page_table, max_pages, seq_lens, pool, n_pages, sink_buf,
                     recent_buf, softmax_scale, out, lse, workspace, workspace_bytes, err_word, stream, pend);
}

int mla_qcache_decode_attn_multi(const mla_qcache_config* cfg, int32_t B, int32_t H, int32_t q_len,
                                 const uint16_t* q_lat, const uint16_t* q_rope, const int32_t* page_table,
                                 int32_t max_pages, const int32_t* seq_lens, const uint8_t* pool, int64_t n_pages,
                                 const uint16_t* sink_buf, const uint16_t* recent_buf, float softmax_scale,
                                 float* out, float* lse, void* workspace, size_t workspace_bytes, int32_t* err_word,
                                 void* stream) {
  if (q_len < 1 || H < 1 || static_cast<int64_t>(q_len) * H > 256) return MLA_QCACHE_ERR_SHAPE;
  return decode_impl(cfg, B, q_len * H, q_len, q_lat, q_rope, page_table, max_pages, seq_lens, pool, n_pages,
                     sink_buf, recent_buf, softmax_scale, out, lse, workspace, workspace_bytes, err_word, stream);
}

size_t mla_qcache_bf16_workspace_bytes(int32_t B, int32_t H, int32_t max_pages, int32_t page_size) {
  if (B < 1 || H < 16 || H > 256 || H % 16 || max_pages < 1 ||
      (page_size != 32 && page_size != 64 && page_size != 128))
    return 0;
  int sms = 0;
  if (current_sm_count(&sms) != MLA_QCACHE_OK) return 0;
  return mlaq::decode_workspace_bytes(B, H, mlaq::decode_bf16_num_parts(B, H, max_pages, page_size, sms));
}

int mla_qcache_decode_attn_bf16(int32_t B, int32_t H, const uint16_t* q_lat, const uint16_t* q_rope,
                                const int32_t* page_table, int32_t max_pages, int32_t page_size,
                                const int32_t* seq_lens, const uint16_t* kv_pool, int64_t n_pages,
                                float softmax_scale, float* out, float* lse, void* workspace,
                                size_t workspace_bytes, int32_t* err_word, void* stream) {
  if (B < 1 || B > (1 << 20) || H < 16 || H > 256 || H % 16 || max_pages < 1 || n_pages < 1)
    return MLA_QCACHE_ERR_SHAPE;
  if (page_size != 32 && page_size != 64 && page_size != 128) return MLA_QCACHE_ERR_CONFIG;
  if (!q_lat || !q_rope || !page_table || !seq_lens || !kv_pool || !out || !lse || !workspace || !err_word)
    return MLA_QCACHE_ERR_NULL;
  if (!aligned(q_lat, 4) || !aligned(q_rope, 4) || !aligned(kv_pool, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
      !aligned(workspace, 16) || !aligned(page_table, 4) || !aligned(seq_lens, 4) || !aligned(err_word, 4))
    return MLA_QCACHE_ERR_ALIGN;
  int sms = 0;
  int st = current_sm_count(&sms);
  if (st != MLA_QCACHE_OK) return st;
  const int parts = mlaq::decode_bf16_num_parts(B, H, max_pages, page_size, sms);
  if (workspace_bytes < mlaq::decode_workspace_bytes(B, H, parts)) return MLA_QCACHE_ERR_WORKSPACE;
  mlaq::DecodeParams p{};
  p.q_lat = q_lat;
  p.q_rope = q_rope;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.kv_bf16 = kv_pool;
  p.arrive = static_cast<unsigned long long*>(workspace);
  p.o_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + mlaq::kArriveBytes);
  p.ml_part = p.o_part + static_cast<size_t>(B) * H * parts * mlaq::kLatent;
  p.out = out;
  p.lse = lse;
  p.err = err_word;
  p.n_pages = n_pages;
  p.scale_log2 = static_cast<float>(static_cast<double>(softmax_scale) * 1.4426950408889634074);
  p.B = B;
  p.H = H;
  p.max_pages = max_pages;
  p.P = page_size;
  p.p_shift = 0;
  while ((1 << p.p_shift) < p.P) ++p.p_shift;
  p.bits_c = 4;
  p.n_split = 0;  // every share is a BF16 share
  p.n_q = parts;
  const cudaError_t e = mlaq::launch_decode_bf16(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_QCACHE_OK : MLA_QCACHE_ERR_CUDA;
}

int mla_qcache_decode_attn_noalloc(const mla_qcache_config* cfg, int32_t B, int32_t H, const uint16_t* q_lat,
                                   const uint16_t* q_rope, const int32_t* page_table, int32_t max_pages,
                                   const int32_t* seq_lens, const uint8_t* pool, int64_t n_pages,
                                   const uint16_t* sink_buf, const uint16_t* recent_buf, float softmax_scale,
                                   float* out, float* lse, int32_t* err_word, void* stream) {
  int st = check_config(cfg);
  if (st != MLA_QCACHE_OK) return st;
  if (B < 1 || B > 65535 || H < 16 || H > 256 || H % 16 || max_pages < 1 || n_pages < 1)
    return MLA_QCACHE_ERR_SHAPE;
  int sms = 0;
  st = current_sm_count(&sms);
  if (st != MLA_QCACHE_OK) return st;
  const int ns = mlaq::decode_num_splits(B, H, max_pages, cfg->page_size, cfg->n_sink, cfg->n_recent, sms);
  const int nq = mlaq::decode_num_protected(B, H, max_pages, cfg->page_size, cfg->n_sink, cfg->n_recent, sms);
  if (mlaq::decode_workspace_bytes(B, H, ns + nq) > mlaq::kNoAllocScratchBytes) return MLA_QCACHE_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  if (mlaq::noalloc_scratch(&scratch) != cudaSuccess) return MLA_QCACHE_ERR_CUDA;
  return mla_qcache_decode_attn(cfg, B, H, q_lat, q_rope, page_table, max_pages, seq_lens, pool, n_pages, sink_buf,
                                recent_buf, softmax_scale, out, lse, scratch, mlaq::kNoAllocScratchBytes, err_word,
                                stream);
}

size_t mla_qcache_noalloc_scratch_bytes(void) { return mlaq::kNoAllocScratchBytes; }

const char* mla_qcache_strerror(int32_t status) {
  switch (status) {
    case MLA_QCACHE_OK: return "ok";
    case MLA_QCACHE_ERR_NULL: return "a required pointer is NULL";
    case MLA_QCACHE_ERR_CONFIG: return "unsupported cache configuration";
    case MLA_QCACHE_ERR_SHAPE: return "invalid size argument (B, H, rows, pages or max_new)";
    case MLA_QCACHE_ERR_ALIGN: return "pointer not aligned as documented";
    case MLA_QCACHE_ERR_WORKSPACE: return "workspace too small";
    case MLA_QCACHE_ERR_CUDA: return "CUDA runtime error while launching";
    case MLA_QCACHE_ERR_SCRATCH_LIMIT:
      return "problem needs more scratch than the built-in buffer of mla_qcache_decode_attn_noalloc holds";
    default: return "unknown status";
  }
}

}  // extern "C"
