/*
 * mla_qcache.h -- C ABI of the low-bit dual-path MLA KV cache for GB300 (sm_103a).
 *
 * Two operations make up the decode hot path of Multi-Head Latent Attention over a
 * quantized, paged cache:
 *
 *   mla_qcache_write        fused cache writer: per-token latent quantize + pack, BF16
 *                           retention of sink and recent tokens, and per-page k_R
 *                           quantization once a page fills.
 *   mla_qcache_decode_attn  single-token decode attention over the packed pages plus the
 *                           BF16 protected tokens, one global softmax, latent-space readout.
 *
 * Sources (the web pages this library follows):
 *   [QuantMLA]  the QuantMLA page (function-aligned dual-path quantization of MLA caches):
 *               abstract (native low-bit kernel that unpacks and dequantizes inside
 *               attention), Figure 3 caption (packed cache plus BF16 sink/recent buffers),
 *               Figure 5 caption (C4R4 with sink4/local128), appendix Figure 8 caption
 *               (fused writer, switch to the packed copy on eviction, one global softmax).
 *   [RAQ-MLA]   the RAQ-MLA page (Role-Aware Quantization for Multi-Head Latent Attention
 *               Caches): abstract and Figures 3-4 (what is cached: latent c_KV and post-RoPE k_R;
 *               absorbed read path), appendix Table 5 (quantizer configuration), appendix
 *               Table 6 (cache page of 64 or 128 tokens).
 *
 * Conventions for every entry point:
 *   - All data pointers are DEVICE pointers unless stated otherwise. The caller owns every
 *     buffer; the library allocates nothing and never synchronizes the stream.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream). Work is
 *     enqueued asynchronously on it.
 *   - BF16 values are passed as their 16-bit patterns (uint16_t), FP16 metadata likewise.
 *   - The synchronous return value is a status (MLA_QCACHE_OK or a negative MLA_QCACHE_ERR_*).
 *     On a negative status nothing was enqueued.
 *   - Problems that can only be seen on the device (bad page id, overflowing sequence,
 *     non-finite input, ...) are OR-ed into *err_word (a device int32 that the caller zeroes
 *     and reads after synchronizing) as MLA_QCACHE_DEV_* bits. The offending work is skipped;
 *     kernels never trap.
 */
#ifndef MLA_QCACHE_H
#define MLA_QCACHE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Fixed MLA dimensions ([RAQ-MLA] Table 5; DeepSeek-V2/GLM-shaped MLA). */
#define MLA_QCACHE_LATENT_DIM 512 /* rank of the compressed latent c_KV */
#define MLA_QCACHE_ROPE_DIM 64    /* dimension of the post-RoPE positional key k_R */
#define MLA_QCACHE_GROUP 128      /* latent channels per quantization group */
#define MLA_QCACHE_ROW_DIM 576    /* one BF16 buffer row: c (512) followed by k_R (64) */

/* Synchronous status codes. */
#define MLA_QCACHE_OK 0
#define MLA_QCACHE_ERR_NULL (-1)      /* a required pointer is NULL */
#define MLA_QCACHE_ERR_CONFIG (-2)    /* unsupported configuration (bits, page, sink, recent) */
#define MLA_QCACHE_ERR_SHAPE (-3)     /* bad B, H, row count, max_pages, n_pages, max_new */
#define MLA_QCACHE_ERR_ALIGN (-4)     /* a pointer is not aligned as documented */
#define MLA_QCACHE_ERR_WORKSPACE (-5) /* workspace too small */
#define MLA_QCACHE_ERR_CUDA (-6)      /* a CUDA runtime call failed (launch, attribute, ...) */
#define MLA_QCACHE_ERR_SCRATCH_LIMIT (-7) /* too large for the built-in scratch (noalloc variant) */

/* Device-side error bits, OR-ed into *err_word. */
#define MLA_QCACHE_DEV_BAD_PAGE 1      /* page-table entry outside [0, n_pages) */
#define MLA_QCACHE_DEV_SEQ_OVERFLOW 2  /* a position >= max_pages * page_size, or seq_len < 0 */
#define MLA_QCACHE_DEV_NONFINITE 4     /* NaN or Inf in a value to quantize */
#define MLA_QCACHE_DEV_RANGE 8         /* a group min/max outside the finite FP16 range */
#define MLA_QCACHE_DEV_ROWS 16         /* cu_new inconsistent with n_rows or max_new */
#define MLA_QCACHE_DEV_TIMEOUT 32      /* a bounded device wait expired (work abandoned) */

/*
 * Cache configuration.
 *   bits_c     latent code width: 4 (C4) or 2 (C2). 2^bits_c levels, L = 2^bits_c - 1.
 *   bits_r     k_R code width: must be 4 (R4).
 *   page_size  P, tokens per cache page: 32, 64 or 128, and P <= n_recent (the pages use 64
 *              and 128; decode streams 32-token tiles that never straddle a page).
 *   n_sink     S, leading tokens kept in BF16 ("sink4"): 0..16.
 *   n_recent   W, trailing tokens kept in BF16 ("local128"): P..1024.
 *   clip_q     per-token clip quantile of |c| for the latent, in (0, 1]; 0 disables the clip.
 *              [RAQ-MLA] Table 5 lists a 0.94 clip under the INT2 latent.
 *
 * Quantizer ([RAQ-MLA] Table 5; the exact roundings are this library's reading, since the
 * pages only say "FP16 scale and minimum"). For a set of values x (one latent group of 128
 * channels of one token, or one k_R channel over the P tokens of one page):
 *   lo = min x, hi = max x
 *   min   = the largest finite FP16 value <= lo                  (round down)
 *   scale = the smallest FP16 value >= 0 with min + L*scale >= hi (round up of (hi-min)/L)
 *   code(x) = the k in [0, L] minimising |x - (min + k*scale)|, exact ties to the even k
 *   dequantized value: min + code * scale
 * so |dequant - x| <= scale/2 holds exactly. Clip (latent only, when clip_q > 0): tau is the
 * k-th smallest |c_i| over the 512 channels of the token with k = ceil(clip_q * 512) (a
 * nearest-rank order statistic), and each c_i is replaced by min(max(c_i, -tau), tau) before
 * the group statistics.
 */
typedef struct {
  int32_t bits_c;
  int32_t bits_r;
  int32_t page_size;
  int32_t n_sink;
  int32_t n_recent;
  float clip_q;
} mla_qcache_config;

/*
 * Physical page layout (this library's own; the pages say only "packed cache
 * representations" and give no byte layout). One contiguous region of
 * mla_qcache_page_bytes() bytes per physical page of P tokens; t is the token's index in
 * its page (position mod P), c a latent channel (0..511), j a k_R channel (0..63).
 *
 *   Region A, latent codes, offset 0, size P*64*bits_c bytes.
 *     One row of R = 64*bits_c bytes per token, row t at t*R. Inside a row the channels are
 *     in order: byte k holds channels 2k (low nibble) and 2k+1 (high nibble) for bits_c == 4,
 *     channels 4k+i at bits [2i, 2i+2) for bits_c == 2. The row's 16-byte chunks are stored
 *     XOR-permuted: logical chunk k/16 sits at chunk (k/16) ^ (t%8), i.e. byte
 *     t*R + 16*((k/16) ^ (t%8)) + k%16.
 *     (So eight consecutive tokens' copies of one logical chunk fall on eight distinct
 *     16-byte bank groups: an 8x8 matrix load of 16-bit elements, one row per token, reads
 *     them without bank conflicts, plain or transposed. Element e of logical chunk j holds
 *     channels 32j + 4e + s at bits 4s (INT4) or 64j + 8e + i at bits 2i (INT2).)
 *   Region B, k_R codes (4 bits), offset P*64*bits_c, size 32*P bytes.
 *     Blocks of 16 tokens x 16 channels: block (t/16, j/16) starts at ((t/16)*4 + j/16)*128.
 *     A block is 32 lanes of one 32-bit word, lane = 4*(t%8) + q. With e = j%16,
 *     q = (e%8)/2, h = e/8, o = e%2, n = (t%16)/8: field s = 2*n + h, bits [4*(s+4*o), +4).
 *   Region C, latent metadata, offset P*(64*bits_c + 32), size 16*P bytes.
 *     Token t, group g at (t*4 + g)*4: FP16 scale (2 bytes) then FP16 minimum (2 bytes).
 *   Region D, k_R metadata, offset P*(64*bits_c + 48), size 256 bytes.
 *     Channel j at j*4: FP16 scale then FP16 minimum, over the P tokens of the page.
 *
 *   Effective bits ([RAQ-MLA] Table 5): latent (64*bits_c + 16)*8/512 = 2.25 (C2) or 4.25
 *   (C4) bits/element; k_R (32*P + 256)*8/(64*P) = 4 + 32/P = 4.25 (P=128) or 4.50 (P=64).
 *
 * BF16 buffers ([QuantMLA] Figure 8): sink_buf [B][n_sink][576] holds positions 0..S-1;
 * recent_buf [B][n_recent][576] is a ring, position t in slot t % W. A row is c (512) then
 * k_R (64), the pre-quantization (unclipped) values.
 *
 * Which tokens attention reads from BF16 ("protected"), for a sequence of T cached tokens:
 * t < S or t >= T - W. Every other token is read from its packed copy. Because P <= W, a
 * token that is not protected lies in a full page whose k_R is already quantized.
 */

/* Bytes of one physical page, or 0 for an invalid configuration. */
size_t mla_qcache_page_bytes(const mla_qcache_config* cfg);

/* MLA_QCACHE_OK if the configuration is supported, else MLA_QCACHE_ERR_CONFIG/NULL. */
int mla_qcache_config_check(const mla_qcache_config* cfg);

/*
 * Bytes of device workspace mla_qcache_decode_attn needs for B sequences, H heads and a
 * page table of max_pages columns (the split of the KV axis depends on these and on the
 * SM count of the current device). Returns 0 on invalid arguments.
 */
size_t mla_qcache_workspace_bytes(const mla_qcache_config* cfg, int32_t B, int32_t H,
                                  int32_t max_pages);

/*
 * Fused cache writer ([QuantMLA] Figure 8; [RAQ-MLA] Table 5).
 *
 * For each sequence b in [0, B), rows cu_new[b] .. cu_new[b+1]-1 of c_new / kr_new are the
 * new tokens at positions seq_lens[b], seq_lens[b]+1, ... (seq_lens[b] = tokens already
 * cached before this call; the caller advances it afterwards). For every new token t:
 *   - the latent is clipped (if clip_q > 0), quantized per 128-channel group and its codes
 *     and metadata are stored in page page_table[b][t/P], slot t%P (regions A and C);
 *   - if t < S, its BF16 row is stored in sink_buf[b][t];
 *   - if t is among the last W positions after this call, its BF16 row is stored in
 *     recent_buf[b][t%W] (earlier rows of this call would be overwritten anyway);
 *   - if t is the last token of its page, the page's k_R is quantized per channel over the
 *     page's P tokens (regions B and D), reading earlier tokens of the page from the ring.
 * A token leaving the recent window needs no work: its packed copy already exists.
 *
 * Arguments:
 *   c_new      [n_rows][512] BF16, kr_new [n_rows][64] BF16 (post-RoPE), row-major.
 *   cu_new     [B+1] int32, non-decreasing, cu_new[0] = 0, cu_new[B] = n_rows.
 *   seq_lens   [B] int32, tokens cached before this call.
 *   max_new    host int: upper bound on cu_new[b+1]-cu_new[b] (1 for a decode step).
 *   page_table [B][max_pages] int32 physical page ids; entries for every position written
 *              must be valid (the caller allocates pages before writing into them).
 *   pool       [n_pages][page_bytes] bytes, 16-byte aligned.
 *   sink_buf   [B][S][576] BF16 (may be NULL when S == 0); recent_buf [B][W][576] BF16.
 *   err_word   device int32 receiving MLA_QCACHE_DEV_* bits (required).
 * Errors: NULL pointer, bad config, B < 1, n_rows < 0, max_new < 1 (with n_rows > 0),
 * n_rows + 4 * B * (max_new / P + 1) above 2^31 - 1, max_pages < 1, n_pages < 1, misaligned
 * pool or buffers -> negative status, nothing run.
 */
int mla_qcache_write(const mla_qcache_config* cfg, int32_t B, int32_t n_rows,
                     const uint16_t* c_new, const uint16_t* kr_new, const int32_t* cu_new,
                     const int32_t* seq_lens, int32_t max_new, const int32_t* page_table,
                     int32_t max_pages, uint8_t* pool, int64_t n_pages, uint16_t* sink_buf,
                     uint16_t* recent_buf, int32_t* err_word, void* stream);

/*
 * Decode of the cache as a pending write will leave it, without waiting for that write
 * ([QuantMLA] Figure 8: every token gets a packed copy on arrival and is read from it once it
 * leaves the recent window). The arguments are those of mla_qcache_decode_attn plus the
 * write's rows: c_new, kr_new, cu_new and max_new as mla_qcache_write takes them, seq_lens the
 * lengths BEFORE that write. Sequence b is decoded at length T = seq_lens[b] + (cu_new[b+1] -
 * cu_new[b]); its pending tokens seq_lens[b] .. T-1 are read from c_new / kr_new (they are the
 * newest, hence BF16-protected), every other token from the cache.
 *
 * Because P <= W, the pending write changes nothing else this decode reads: the packed copies
 * it adds belong to tokens inside the recent window, a page it fills holds only such tokens,
 * and the ring slots it overwrites belong to tokens that left the window. So the write
 * (mla_qcache_write or mla_qcache_write_advance with the same rows and lengths) may run
 * concurrently on another stream, provided it finishes before the next call that reads this
 * cache. Only the plain writer qualifies: with a transformed writer the cache holds x A, not
 * the rows given here.
 *   max_new    0 <= max_new <= W - P + 1 (1 for a decode step at P = W = 128), so that every
 *              token the pending rows push out of the window already lies in a full page.
 *   c_new, kr_new 16-byte aligned; cu_new 4-byte aligned.
 * Errors: as mla_qcache_decode_attn; bad max_new -> MLA_QCACHE_ERR_SHAPE; a NULL row pointer ->
 * MLA_QCACHE_ERR_NULL; misaligned rows -> MLA_QCACHE_ERR_ALIGN. On the device, a sequence whose
 * row count is negative or above max_new sets MLA_QCACHE_DEV_ROWS and is decoded without
 * pending rows; T beyond max_pages * P sets MLA_QCACHE_DEV_SEQ_OVERFLOW (empty sequence).
 */
int mla_qcache_decode_attn_pending(const mla_qcache_config* cfg, int32_t B, int32_t H,
                                   const uint16_t* q_lat, const uint16_t* q_rope,
                                   const int32_t* page_table, int32_t max_pages,
                                   const int32_t* seq_lens, const uint16_t* c_new,
                                   const uint16_t* kr_new, const int32_t* cu_new, int32_t max_new,
                                   const uint8_t* pool, int64_t n_pages, const uint16_t* sink_buf,
                                   const uint16_t* recent_buf, float softmax_scale, float* out,
                                   float* lse, void* workspace, size_t workspace_bytes,
                                   int32_t* err_word, void* stream);

/*
 * Decode of several new tokens per sequence in one call (a speculative draft verified in one
 * step, or a short chunk): the q_len tokens are the cache's last ones, written before the
 * call, and position i (0 <= i < q_len) attends to the cache tokens t < T - (q_len - 1 - i),
 * itself included. Which copy a token is read from follows the cache length T as in
 * mla_qcache_decode_attn (BF16 for t < S or t >= T - W, else the packed copy), so every
 * position sees the same packed range and only the BF16 recent rows differ in their end; a
 * position whose prefix is empty gets out = 0, lse = -inf. (The pages decode one token per
 * step; this is the plainest extension: causal attention among the new tokens.)
 *   H          heads per position, a multiple of 16; q_len * H <= 256; q_len - 1 <= W.
 *   q_lat      [B][q_len][H][512] BF16, q_rope [B][q_len][H][64] BF16 (position-major rows);
 *   out, lse   [B][q_len][H][512] float32, [B][q_len][H] float32.
 *   workspace  mla_qcache_workspace_bytes(cfg, B, q_len * H, max_pages) bytes (first 8192
 *              bytes zero, as for mla_qcache_decode_attn).
 * Other arguments and errors as mla_qcache_decode_attn (with q_len * H rows); bad q_len ->
 * MLA_QCACHE_ERR_SHAPE. q_len = 1 is mla_qcache_decode_attn. At q_len * H a multiple of 64 the
 * packed pages are read once for all positions (64 rows per tensor-memory CTA).
 */
int mla_qcache_decode_attn_multi(const mla_qcache_config* cfg, int32_t B, int32_t H, int32_t q_len,
                                 const uint16_t* q_lat, const uint16_t* q_rope, const int32_t* page_table,
                                 int32_t max_pages, const int32_t* seq_lens, const uint8_t* pool, int64_t n_pages,
                                 const uint16_t* sink_buf, const uint16_t* recent_buf, float softmax_scale,
                                 float* out, float* lse, void* workspace, size_t workspace_bytes, int32_t* err_word,
                                 void* stream);

/*
 * Unquantized comparator: the same single-token decode attention over a paged BF16 cache
 * (every token exact; the latency the quantized cache is measured against, QuantMLA page,
 * appendix Table 9 form: delta = t_quantized / t_BF16 - 1).
 *   kv_pool    [n_pages][page_size][576] BF16 (c then k_R per token), 16-byte aligned; token
 *              t of sequence b lives in row t % page_size of page page_table[b][t / page_size].
 *   page_size  32, 64 or 128. Other arguments as mla_qcache_decode_attn (no sink/recent
 *              buffers, no quantization config); workspace of mla_qcache_bf16_workspace_bytes
 *              (first 8192 bytes zero, as for mla_qcache_decode_attn).
 * Errors: as mla_qcache_decode_attn; a bad page id sets MLA_QCACHE_DEV_BAD_PAGE and drops the
 * share that would read it.
 */
size_t mla_qcache_bf16_workspace_bytes(int32_t B, int32_t H, int32_t max_pages, int32_t page_size);
int mla_qcache_decode_attn_bf16(int32_t B, int32_t H, const uint16_t* q_lat, const uint16_t* q_rope,
                                const int32_t* page_table, int32_t max_pages, int32_t page_size,
                                const int32_t* seq_lens, const uint16_t* kv_pool, int64_t n_pages,
                                float softmax_scale, float* out, float* lse, void* workspace,
                                size_t workspace_bytes, int32_t* err_word, void* stream);

/*
 * Fused cache writer with the length update: exactly mla_qcache_write, and in the same launch
 * seq_lens_next[b] = seq_lens[b] + cu_new[b+1] - cu_new[b] for every b in [0, B) (a decode
 * step then needs no separate length kernel). seq_lens_next [B] is a device int32 array,
 * 4-byte aligned, that must not overlap seq_lens (the writer's CTAs read seq_lens while the
 * new lengths are stored); callers alternate two length arrays from step to step. With
 * n_rows == 0 the lengths are copied on `stream`.
 * Errors: those of mla_qcache_write; seq_lens_next NULL -> MLA_QCACHE_ERR_NULL; overlapping
 * seq_lens -> MLA_QCACHE_ERR_SHAPE; misaligned -> MLA_QCACHE_ERR_ALIGN.
 */
int mla_qcache_write_advance(const mla_qcache_config* cfg, int32_t B, int32_t n_rows,
                             const uint16_t* c_new, const uint16_t* kr_new, const int32_t* cu_new,
                             const int32_t* seq_lens, int32_t* seq_lens_next, int32_t max_new,
                             const int32_t* page_table, int32_t max_pages, uint8_t* pool,
                             int64_t n_pages, uint16_t* sink_buf, uint16_t* recent_buf,
                             int32_t* err_word, void* stream);

/*
 * Cache writer over transformed rows (RAQ-MLA page, Figure 4: the latent is cached in the basis
 * of an invertible A_c, applied after the RMSNorm, and k_R in that of A_R, applied after RoPE;
 * the read path folds A_c^-1 into the up-projections and compensates k_R on the query side).
 * Exactly mla_qcache_write (or mla_qcache_write_advance when seq_lens_next is not NULL) of the
 * rows c A_c and k_R A_R in place of c and k_R, in one launch ("fused", RAQ-MLA page, appendix
 * Table 9): the page bytes, the BF16 sink/recent rows and the error bits are those that writer
 * stores for the transformed rows.
 *   a_c   NULL or BF16 [512][512] row-major, 16-byte aligned: latent channel j is cached as
 *         the BF16 value of sum_i c_i a_c[i][j].
 *   a_r   NULL or BF16 [64][64] row-major, 16-byte aligned: the same for k_R.
 * Arithmetic (the page fixes none; this is the reading taken): each sum is accumulated in
 * float32 in the order i = 0, 1, ... starting from +0, one rounded product (exact for two BF16
 * values) and one rounded addition per step, and rounded to BF16 to nearest-even; every
 * transformed value, and so every code, is therefore reproducible bit for bit.
 * Each new row is served by a cluster of eight CTAs (64 transformed latent channels each; the
 * CTA's 64-column slice of a_c arrives in shared memory by tensor-map copies). A copy wait that
 * gives up sets MLA_QCACHE_DEV_TIMEOUT (the row is then not valid).
 * Errors: those of mla_qcache_write / mla_qcache_write_advance; misaligned a_c / a_r ->
 * MLA_QCACHE_ERR_ALIGN; 8 * n_rows + 4 * B * (max_new / P + 1) + 7 above 2^31 - 1 ->
 * MLA_QCACHE_ERR_SHAPE. A transformed value that overflows sets MLA_QCACHE_DEV_NONFINITE.
 */
int mla_qcache_write_transformed(const mla_qcache_config* cfg, int32_t B, int32_t n_rows,
                                 const uint16_t* c_new, const uint16_t* kr_new, const int32_t* cu_new,
                                 const int32_t* seq_lens, int32_t* seq_lens_next, int32_t max_new,
                                 const uint16_t* a_c, const uint16_t* a_r, const int32_t* page_table,
                                 int32_t max_pages, uint8_t* pool, int64_t n_pages, uint16_t* sink_buf,
                                 uint16_t* recent_buf, int32_t* err_word, void* stream);

/*
 * Standalone transform ("standalone", RAQ-MLA page, appendix Table 9: A_c as its own kernel
 * before the cache write): out[r] = x[r] A for n_rows BF16 rows of dim 64 or 512, with the
 * arithmetic of mla_qcache_write_transformed (so transforming first and then calling
 * mla_qcache_write caches the same bytes). x, out: device BF16, 2-byte aligned; a: 16-byte
 * aligned; out must not overlap x. One CTA per row and 64 output channels. err_word: device
 * int32, 4-byte aligned; a copy wait that gives up ORs MLA_QCACHE_DEV_TIMEOUT into it.
 * Errors: dim not 64 / 512 or n_rows < 0 or overlap -> MLA_QCACHE_ERR_SHAPE; NULL ->
 * MLA_QCACHE_ERR_NULL; misaligned -> MLA_QCACHE_ERR_ALIGN; n_rows == 0 runs nothing.
 */
int mla_qcache_row_transform(int32_t n_rows, int32_t dim, const uint16_t* x, const uint16_t* a, uint16_t* out,
                             int32_t* err_word, void* stream);

/*
 * The launch plan of a decode call for a problem size and an SM count (no GPU needed; what
 * mla_qcache_decode_attn and mla_qcache_workspace_bytes use with the current device's count):
 *   plan[0]  packed-token shares per (sequence, 16- or 64-head block)
 *   plan[1]  CTAs sharing the BF16 (sink and recent) tokens per (sequence, 16-head block)
 *   plan[2]  > 0: the balanced 16-head instance with this many CTA slots for packed shares
 *            (more shares than one wave holds); 0: even slices of each sequence
 *   plan[3]  1: the packed tokens run on the 64-head tensor-memory kernel (H % 64 == 0)
 *   plan[4]  shares of the unquantized comparator (mla_qcache_decode_attn_bf16) at this
 *            configuration's page size
 * plan: host int32[5]. Errors: bad config -> MLA_QCACHE_ERR_CONFIG; NULL -> MLA_QCACHE_ERR_NULL;
 * B < 1, H not a multiple of 16 in 16..256, max_pages < 1, num_sms < 1 -> MLA_QCACHE_ERR_SHAPE.
 */
int mla_qcache_decode_plan(const mla_qcache_config* cfg, int32_t B, int32_t H, int32_t max_pages, int32_t num_sms,
                           int32_t* plan);

/*
 * Kernel launches one mla_qcache_decode_attn call of this shape makes on the current device:
 * 1 (the partials merged inside the decode launch), 2 (a merge launch follows) or 3 (64-head
 * blocks: protected shares, tensor-memory shares, merge). For sizing CUDA graphs and counting
 * launches; the first call sets the kernels' shared-memory attribute, as a first decode call
 * does. Returns the count, or a negative status: bad config -> MLA_QCACHE_ERR_CONFIG/NULL; bad
 * sizes -> MLA_QCACHE_ERR_SHAPE; a failed runtime query -> MLA_QCACHE_ERR_CUDA.
 */
int mla_qcache_decode_launches(const mla_qcache_config* cfg, int32_t B, int32_t H, int32_t max_pages);

/*
 * Query absorption (RAQ-MLA page, Figure 4: the decode scores the latent directly, so the
 * query's no-position part is carried into the latent space through W_UK, with A_c^-1 folded
 * into W_UK offline; k_R's transform is compensated on the query side):
 *   q_lat[b][h][:]      = BF16( q_nope[b][h][:] . w_uk[h] )        w_uk [H][d_nope][512]
 *   q_rope_out[b][h][:] = BF16( q_rope[b][h][:] . r_comp )         r_comp [64][64], every head
 * All BF16, row-major, 16-byte aligned; products on the tensor cores with float32 accumulation,
 * each result rounded to BF16 to nearest-even (relative error within one BF16 rounding plus the
 * float32 accumulation). r_comp and q_rope_out are both NULL (no compensation: pass q_rope to
 * the decode unchanged) or both set. The outputs are the decode's q_lat / q_rope.
 *   d_nope   a multiple of 16, 16..512 (128 for DeepSeek-V2-shaped layers). B 0..2^22, H 1..256.
 * Errors: bad sizes -> MLA_QCACHE_ERR_SHAPE; NULL (with B > 0) -> MLA_QCACHE_ERR_NULL;
 * misaligned -> MLA_QCACHE_ERR_ALIGN. Nothing is checked on the device.
 */
int mla_qcache_absorb_query(int32_t B, int32_t H, int32_t d_nope, const uint16_t* q_nope, const uint16_t* w_uk,
                            const uint16_t* q_rope, const uint16_t* r_comp, uint16_t* q_lat, uint16_t* q_rope_out,
                            void* stream);

/*
 * Up-projection of the decode output (RAQ-MLA page, Figure 4: the readout stays in the latent
 * space and leaves through W_UV, with A_c^-1 folded into W_UV offline):
 *   out[b][h][:] = BF16(o[b][h][:]) . w_uv[h]      o [B][H][512] float32 (mla_qcache_decode_attn's
 *                                                  out), w_uv [H][512][d_v] BF16, out [B][H][d_v]
 *                                                  float32
 * The attention output enters the tensor cores rounded to BF16 (nearest-even), the sums are
 * float32. d_v a multiple of 32 (128 for DeepSeek-V2-shaped layers); pointers 16-byte aligned.
 * Errors: as mla_qcache_absorb_query.
 */
int mla_qcache_up_project(int32_t B, int32_t H, int32_t d_v, const float* o, const uint16_t* w_uv, float* out,
                          void* stream);

/*
 * Self-test of the device-side failure detection: launches one kernel whose only wait can never
 * complete (an mbarrier nothing arrives at), waited on with the bounded wait every kernel of
 * this library uses. After ~1 ms the wait gives up, MLA_QCACHE_DEV_TIMEOUT is OR-ed into
 * err_word (device int32, 4-byte aligned) and the kernel returns; the context stays usable.
 * Errors: NULL -> MLA_QCACHE_ERR_NULL; misaligned -> MLA_QCACHE_ERR_ALIGN.
 */
int mla_qcache_selftest_wait_timeout(int32_t* err_word, void* stream);

/*
 * Length update after a write (the pages leave the bookkeeping to the caller): for every
 * sequence b in [0, B), seq_lens[b] += cu_new[b+1] - cu_new[b], in one kernel on `stream`,
 * ordered after a preceding mla_qcache_write on the same stream. cu_new [B+1] and seq_lens [B]
 * are device int32 arrays, 4-byte aligned; seq_lens must not be read by a write still in flight
 * on another stream.
 * Errors: NULL pointer or B < 1 -> negative status, nothing run.
 */
int mla_qcache_advance(const int32_t* cu_new, int32_t* seq_lens, int32_t B, void* stream);

/*
 * Decode attention over the quantized dual-path cache ([QuantMLA] abstract and Figure 8;
 * [RAQ-MLA] Figures 3-4: absorbed query, score = q_lat . c + q_rope . k_R, latent-space
 * readout).
 *
 * For each sequence b with T = seq_lens[b] cached tokens and each head h:
 *   v_t   = BF16 row of token t if protected (t < S or t >= T-W), else its dequantized
 *           packed copy (latent codes with the token's group metadata, k_R codes with the
 *           page's channel metadata)
 *   s_t   = softmax_scale * (q_lat[b][h] . v_t[0:512] + q_rope[b][h] . v_t[512:576])
 *   out[b][h][:] = sum_t exp(s_t - m) v_t[0:512] / sum_t exp(s_t - m),  m = max_t s_t
 *   lse[b][h]    = m + ln(sum_t exp(s_t - m))   (natural log; -inf and out = 0 when T = 0)
 * All tokens share one softmax normalization.
 *
 * Arguments:
 *   H          heads: a multiple of 16, 16..256.
 *   q_lat      [B][H][512] BF16 absorbed query, q_rope [B][H][64] BF16.
 *   page_table [B][max_pages] int32, seq_lens [B] int32 (0 <= T <= max_pages * P).
 *   pool, sink_buf, recent_buf as written by mla_qcache_write.
 *   out        [B][H][512] float32, lse [B][H] float32.
 *   workspace  device scratch of at least mla_qcache_workspace_bytes(cfg, B, H, max_pages)
 *              bytes, 256-byte aligned. Its first 8192 bytes are the split merge's arrival
 *              counters: zero them once before the first call on this workspace (for example
 *              cudaMemset after allocating it); every call leaves them zero, whatever its
 *              shape, so one workspace serves calls of any size. The rest is scratch whose
 *              contents are meaningless after the call. Calls sharing one workspace must not
 *              overlap. Counters that are not zero make the call report
 *              MLA_QCACHE_DEV_TIMEOUT (the merge of a sequence whose shares see an invalid
 *              count is abandoned, at the latest after the bounded wait) and may stay invalid:
 *              after that bit, zero the first 8192 bytes again.
 * How the partials are merged: when the call's CTAs fit on the GPU at once (one wave) and each
 * (sequence, 16-head block) has many partials (24 or more), its CTAs merge their own partials at
 * the end of the decode launch (a cooperative launch: every CTA is resident); otherwise a
 * second launch merges them (mla_qcache_decode_launches tells which).
 * Errors: as for the writer, plus H not a multiple of 16 or > 256, workspace too small.
 */
int mla_qcache_decode_attn(const mla_qcache_config* cfg, int32_t B, int32_t H,
                           const uint16_t* q_lat, const uint16_t* q_rope,
                           const int32_t* page_table, int32_t max_pages,
                           const int32_t* seq_lens, const uint8_t* pool, int64_t n_pages,
                           const uint16_t* sink_buf, const uint16_t* recent_buf,
                           float softmax_scale, float* out, float* lse, void* workspace,
                           size_t workspace_bytes, int32_t* err_word, void* stream);

/*
 * Decode attention that allocates nothing, for callers that cannot call cudaMalloc: for
 * example a plugin inside a host runtime that owns all device memory through its own
 * allocator and forbids direct allocations, or a latency-critical serving loop that must
 * never trigger a device allocation (which can synchronize the device or fail under a memory
 * budget fixed at startup). There is no counterpart on the pages; it is the same computation
 * as mla_qcache_decode_attn with the same arguments minus the workspace.
 *
 * Instead of a caller workspace it uses a scratch array compiled into this library: a static
 * device buffer of mla_qcache_noalloc_scratch_bytes() bytes (16 MiB) that every GPU which
 * loads the library holds until the process exits. Problems whose split partials do not fit
 * (mla_qcache_workspace_bytes() above that size) are rejected with
 * MLA_QCACHE_ERR_SCRATCH_LIMIT and nothing is launched. The entry point calls no cudaMalloc,
 * cudaFree or allocating library routine.
 *
 * The first call on a device looks up the scratch's device address (cudaGetSymbolAddress, with
 * that device current) and caches it; make that first call before any stream capture. Host
 * threads may make their first calls concurrently (the cache is atomic). cudaDeviceReset
 * reloads the library's device code, after which the cached address is stale: a process that
 * resets a device must not call this entry point on it again. Every
 * call shares the one array. Its first 8192 bytes are the merge counters described under
 * mla_qcache_decode_attn: zero when the library is loaded, left zero by every call; the rest
 * needs no initial value (each call writes every partial result it later reads). Calls that
 * overlap on the GPU (two streams, or two host threads) race on the scratch: serialize them.
 */
int mla_qcache_decode_attn_noalloc(const mla_qcache_config* cfg, int32_t B, int32_t H,
                                   const uint16_t* q_lat, const uint16_t* q_rope,
                                   const int32_t* page_table, int32_t max_pages,
                                   const int32_t* seq_lens, const uint8_t* pool, int64_t n_pages,
                                   const uint16_t* sink_buf, const uint16_t* recent_buf,
                                   float softmax_scale, float* out, float* lse, int32_t* err_word,
                                   void* stream);

/* Size in bytes of the built-in scratch used by mla_qcache_decode_attn_noalloc. */
size_t mla_qcache_noalloc_scratch_bytes(void);

/* Static description of a status code (never NULL). */
const char* mla_qcache_strerror(int32_t status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_QCACHE_H */
