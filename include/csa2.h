/*
 * csa2.h -- C ABI of libcsa2: the decode-time hot path of CSA2 compressed
 * sparse attention over an FP4 main KV cache, as hand-written CUDA kernels
 * for GB300 (sm_103a).
 *
 * The method is described on web pages about the DeepSeek-V4.1-Flash report:
 *  [ENG]  "DeepSeek-V4.1-Flash：把 KV Cache 压缩到极限的百万上下文 MoE"
 *  [HUNT] "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression"
 *  [55ZB] "552B参数干掉1.6T：DeepSeek V4.1 Flash技术深度解析"
 * The pages state the problem (three layer modes, the FP4 format, the
 * candidate pool, Top-512) but no interface; these calls follow that
 * statement.  Section names are cited per call.
 *
 * Conventions shared by every call
 *  - Every tensor pointer is DEVICE memory owned by the caller.  The library
 *    allocates nothing; scratch comes through a caller-provided workspace
 *    sized by the matching *_workspace_bytes() call.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream).  No call synchronises.
 *  - Every call returns a csa2_status; no exception crosses the ABI.
 *    Argument errors are found on the host before any launch and leave every
 *    output untouched.  csa2_last_error() gives a thread-local detail string.
 *  - Data errors found on the device (an index outside its valid range) never
 *    fault: the offending element is skipped and a bit is OR-ed into
 *    *err_flag (a caller-owned device uint32, nullable).  Read it after the
 *    stream has synchronised.
 *  - Layouts are dense row-major C arrays unless stated.  Shapes below use
 *    B batch, T query tokens per sequence, N entry capacity per sequence,
 *    D KV channels (last 64 carry RoPE), H attention heads, K selected
 *    entries, P pool blocks.
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *csa2_stream_t; /* same type as cudaStream_t */

typedef enum {
    CSA2_OK = 0,
    CSA2_ERR_INVALID_ARG = 1,  /* bad shape, null or misaligned pointer, bad mode */
    CSA2_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. a D/dv pair)  */
    CSA2_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required     */
    CSA2_ERR_CUDA = 4,         /* a CUDA runtime error at launch                 */
    CSA2_ERR_DEVICE_FLAG = 5,  /* reserved for callers that map *err_flag        */
    CSA2_ERR_TIMEOUT = 6       /* reserved for callers that map CSA2_FLAG_TIMEOUT */
} csa2_status;

typedef enum {
    CSA2_MODE_FULL = 0,     /* layer computes its own scores and Top-K          */
    CSA2_MODE_REINDEX = 1,  /* rescore inside the pool with the layer's own q   */
    CSA2_MODE_REUSE = 2     /* reuse the source layer's indices unchanged       */
} csa2_mode;

typedef enum { CSA2_BF16 = 0, CSA2_FP8_E4M3 = 1, CSA2_FP32 = 2 } csa2_dtype;

/* Bits OR-ed into *err_flag by the kernels. */
#define CSA2_FLAG_BAD_INDEX 0x1u  /* attention idx outside [-1, kv_len)              */
#define CSA2_FLAG_BAD_POOL 0x2u   /* pool block id outside [-1, ceil(N/8))           */
#define CSA2_FLAG_BAD_SLOT 0x4u   /* quantise dst_slot outside [0, n_slots)          */
#define CSA2_FLAG_TIMEOUT 0x8u    /* a bounded on-chip wait gave up (results invalid)  */

/* Fixed indexer shape: 4 heads of dimension 64, one 64-dim key per entry. */
#define CSA2_INDEX_HEADS 4
#define CSA2_INDEX_DIM 64
#define CSA2_POOL_BLOCK 8      /* positions per pool block                           */
#define CSA2_MAX_POOL 2048     /* at most 2048 blocks x 8 = 16384 candidates          */
#define CSA2_MAX_K 2048

/*
 * csa2_quantize_kv_fp4 -- quantise post-RoPE KV rows to the FP4 main-cache
 * format.  [ENG] section "效率组件四件", item 4 "FP4 主 KV Cache": E2M1 values
 * with one E4M3 scale per 16 channels, no second-level global scale,
 * quantised after RoPE; [HUNT] CSA2 paragraph (same format).
 *
 * For row r, group g (channels 16g..16g+15):
 *   s = E4M3(amax/6) rounded to nearest even, saturating at 448;
 *   code_c = sign(x_c) << 3 | E2M1(|x_c|/s) rounded to nearest, ties to the
 *   even code, saturating at 6 (magnitude 0 when s == 0).
 * The sign bit of a code is the sign bit of its input, also for zeros.
 *
 * kv        bf16 [rows, kv_row_stride] (first D of each row used); 16-byte
 *           aligned, kv_row_stride a multiple of 8 elements.
 * rows      >= 0 (0 is a no-op).     D: multiple of 16, 16..4096.
 * dst_slot  int64 [rows] or NULL: row r is written to cache slot dst_slot[r]
 *           (else slot r).  A slot outside [0, n_slots) is skipped and sets
 *           CSA2_FLAG_BAD_SLOT.
 * n_slots   capacity of the cache planes, in slots.
 * codes     uint8 [n_slots, D/2]: channel 2i in the low nibble of byte i,
 *           2i+1 in the high nibble; 4-byte aligned.
 * scales    uint8 [n_slots, D/16]: the E4M3 scale of each group.
 * Bytes per entry: D/2 + D/16 (324 for D = 576).
 */
csa2_status csa2_quantize_kv_fp4(const void *kv, int64_t rows, int D, int64_t kv_row_stride,
                                 const int64_t *dst_slot, int64_t n_slots, uint8_t *codes,
                                 uint8_t *scales, uint32_t *err_flag, csa2_stream_t stream);

/*
 * csa2_rope_quantize_kv_fp4 -- RoPE, then csa2_quantize_kv_fp4, in one pass
 * over pre-RoPE rows.  [ENG] section "效率组件四件", item 4 (the FP4 main KV
 * is quantised after RoPE); the pages fix neither the rotation layout nor how
 * the angles are evaluated.  Rotation: interleaved pairs (2i, 2i+1) of the
 * last rope_dim channels, with the caller's fp32 table
 *     cos_sin[pos][i] = (cos, sin),  float [n_pos, rope_dim/2, 2], 8-byte aligned:
 *     a' = (a*c) - (b*s),  b' = (a*s) + (b*c)
 * in fp32, every product and sum rounded (no fused multiply-add), then rounded
 * to bf16 (nearest even) before the quantiser sees it: the stored bytes equal
 * csa2_quantize_kv_fp4 of the rows an unfused RoPE in those steps writes.
 *
 * pos       int32 [rows]: row r uses table row pos[r]; a position outside
 *           [0, n_pos) skips the row's rotated groups and sets CSA2_FLAG_BAD_INDEX.
 * rope_dim  multiple of 16, 16..D (64 for the 576-channel entries).
 * Other arguments and rules as csa2_quantize_kv_fp4.
 */
csa2_status csa2_rope_quantize_kv_fp4(const void *kv, int64_t rows, int D, int64_t kv_row_stride,
                                      const int32_t *pos, const float *cos_sin, int64_t n_pos, int rope_dim,
                                      const int64_t *dst_slot, int64_t n_slots, uint8_t *codes, uint8_t *scales,
                                      uint32_t *err_flag, csa2_stream_t stream);

/*
 * csa2_index_score -- indexer scores of query tokens against compressed
 * entries.  [ENG] section "Hierarchical Sparse Indexer——索引成本变常数": Full
 * layers score every entry (cost linear in context); later Reindex layers
 * score only inside the candidate pool (constant cost); [HUNT] CSA2
 * paragraph: Reindex reuses the KV and rescores with its own indexer Q.
 * The pages give no score formula; this library computes
 *   score = sum_{h<4} w_h * ReLU(sum_{d<64} q_hd * k_d)
 * with exact products and fp32 accumulation.
 *
 * mode    FULL: scores [B, T, N], entry j scored iff j < kv_len[b*T+t], else
 *         -inf.  REINDEX: scores [B, T, 8P] in pool-local order l = 8p + i
 *         for key j = 8*pool_blocks[b,t,p] + i of the SAME sequence b, -inf
 *         where the block id is -1 or j >= kv_len.  REUSE: returns CSA2_OK
 *         without work.
 * q_idx   [B, T, 4, 64], w fp32 [B, T, 4], k_idx [B, N, 64]; q_dt == k_dt,
 *         either CSA2_FP8_E4M3 (no scale) or CSA2_BF16; q_idx and k_idx
 *         16-byte aligned.
 * kv_len  int32 [B*T], visible entries per query token (values > N act as N).
 * pool_blocks int32 [B, T, P] for REINDEX (1 <= P <= 2048), NULL for FULL.
 *         A block id outside [-1, ceil(N/8)) scores -inf and sets
 *         CSA2_FLAG_BAD_POOL.
 */
csa2_status csa2_index_score(csa2_mode mode, int B, int T, int64_t N, const void *q_idx,
                             csa2_dtype q_dt, const float *w, const void *k_idx, csa2_dtype k_dt,
                             const int32_t *kv_len, const int32_t *pool_blocks, int P,
                             float *scores, uint32_t *err_flag, csa2_stream_t stream);

/*
 * csa2_build_pool -- the hierarchical candidate pool.  [ENG] section
 * "Hierarchical Sparse Indexer": the decoder's first Full layer builds a
 * block-level pool of at most 2048 blocks x 8 positions = 16384 candidates.
 * Block beta covers positions [8*beta, 8*beta + 8); its score is the max of
 * scores[b,t,j] over its positions j < kv_len (a partial last block counts).
 * The pool is the Top-min(P, #blocks with a finite score) blocks, written
 * to pool_blocks [B, T, P] as block ids, -1 padded, in unspecified order.
 *
 * scores fp32 [B, T, N] (16-byte aligned when N % 4 == 0); kv_len int32
 * [B*T]; 1 <= P <= 2048; G must be 8; ceil(N/8) <= 131072.
 * workspace: csa2_build_pool_workspace_bytes() bytes (currently 0; NULL ok).
 */
csa2_status csa2_build_pool(int B, int T, int64_t N, const float *scores, const int32_t *kv_len,
                            int P, int G, int32_t *pool_blocks, void *workspace, size_t ws_bytes,
                            csa2_stream_t stream);
size_t csa2_build_pool_workspace_bytes(int B, int T, int64_t N, int P);

/*
 * csa2_topk -- Top-K selection per query token.  [ENG] CSA2 section (Top-512
 * in every layer); [55ZB] DeepSelect paragraph (the sparse attention's
 * Top-K kernel).  Selects the K largest finite scores; -inf is never
 * selected; fewer than K candidates leaves -1 in the remaining slots.  Ties
 * at the K-th value are taken toward the lower candidate position.  Output
 * order is unspecified.
 *
 * mode   FULL: scores [B, T, M], candidates j < min(kv_len[b*T+t], M) (kv_len
 *        may be NULL: all M); idx holds positions j.
 *        REINDEX: scores [B, T, 8P] from csa2_index_score(REINDEX), M == 8P;
 *        a selected l = 8p + i is written as 8*pool_blocks[b,t,p] + i.
 *        REUSE: returns CSA2_OK, idx untouched (the layer consumes its source
 *        layer's idx buffer).
 * idx    int32 [B, T, K], 1 <= K <= 2048.  M <= 393216 (larger rows:
 *        CSA2_ERR_UNSUPPORTED).
 * workspace: csa2_topk_workspace_bytes() bytes (currently 0; NULL ok).
 */
csa2_status csa2_topk(csa2_mode mode, int B, int T, int64_t M, const float *scores,
                      const int32_t *kv_len, const int32_t *pool_blocks, int P, int K, int32_t *idx,
                      void *workspace, size_t ws_bytes, csa2_stream_t stream);
size_t csa2_topk_workspace_bytes(int B, int T, int64_t M, int K);

/*
 * csa2_index_topk -- fused decode indexer: the result of csa2_index_score
 * (same mode, FP8 E4M3 q_idx and k_idx only) followed by csa2_topk, and for
 * FULL with pool_out also by csa2_build_pool (G = 8), without writing the
 * scores out.  [ENG] Hierarchical Sparse Indexer and CSA2 section (score,
 * pool, Top-512 per layer); the fusion itself is not on the pages.
 *
 * Arguments as in csa2_index_score and csa2_topk: q_idx [B, T, 4, 64],
 * w fp32 [B, T, 4], k_idx [B, N, 64], kv_len int32 [B*T], REINDEX pool_blocks
 * int32 [B, T, P]; idx int32 [B, T, K], 1 <= K <= 2048; FULL pool_out int32
 * [B, T, P_out] or NULL, 1 <= P_out <= 2048.  Candidates per row (N for
 * FULL, 8P for REINDEX) <= 349184 (larger rows: CSA2_ERR_UNSUPPORTED).  Selection rules, ties, -1 padding and the
 * err_flag bits are those of the unfused calls.  bf16 indexer tensors:
 * CSA2_ERR_INVALID_ARG (use the unfused calls).  REUSE: returns CSA2_OK.
 */
csa2_status csa2_index_topk(csa2_mode mode, int B, int T, int64_t N, const void *q_idx, csa2_dtype q_dt,
                            const float *w, const void *k_idx, csa2_dtype k_dt, const int32_t *kv_len,
                            const int32_t *pool_blocks, int P, int K, int32_t *idx, int32_t *pool_out,
                            int P_out, uint32_t *err_flag, csa2_stream_t stream);

/*
 * csa2_index_topk_dense -- the same result as csa2_index_score (FULL, FP8)
 * followed by csa2_topk, for many query tokens per sequence (a prefill
 * chunk), without writing the [B, T, N] score matrix.  [ENG] Hierarchical
 * Sparse Indexer (Full layers score every entry, Top-512 per query); the
 * fusion and its passes are not on the pages.
 *
 * Two kernels on the stream:
 *  1. tensor-core scoring of every (query, key), keeping only the maximum of
 *     each aligned block of 8 positions;
 *  2. per query, tau = the K-th largest block maximum and the K blocks that
 *     reach it (ties at tau broken arbitrarily); every score outside them is
 *     <= tau <= the K-th largest score, so the Top-K of the 8K scores inside
 *     them (rescored from the FP8 keys) is a Top-K of the row.  The two
 *     kernels may round a score differently in the last bits of fp32, which
 *     can only move a selection among scores tied at the K-th value within
 *     that rounding.
 * Selection rules, ties, -1 padding: those of csa2_topk (FULL).
 *
 * q_idx FP8 E4M3 [B, T, 4, 64], w fp32 [B, T, 4], k_idx FP8 E4M3 [B, N, 64]
 * (both 16-byte aligned), kv_len int32 [B*T] (required), idx int32
 * [B, T, K], 1 <= K <= 2048, N <= 262144 (else CSA2_ERR_UNSUPPORTED).
 * workspace: csa2_index_topk_dense_workspace_bytes() bytes, 16-byte
 * aligned (the block maxima, 4 bytes per 8 positions per query); too
 * small: CSA2_ERR_WORKSPACE.  err_flag: CSA2_FLAG_TIMEOUT.
 */
csa2_status csa2_index_topk_dense(int B, int T, int64_t N, const void *q_idx, csa2_dtype q_dt, const float *w,
                                  const void *k_idx, csa2_dtype k_dt, const int32_t *kv_len, int K, int32_t *idx,
                                  uint32_t *err_flag, void *workspace, size_t ws_bytes, csa2_stream_t stream);
size_t csa2_index_topk_dense_workspace_bytes(int B, int T, int64_t N, int K);

/*
 * csa2_sparse_attn_fp4 -- attention of each query head over its selected FP4
 * entries.  The pages give no formula (the [ENG] inference bullet names
 * FlashMLA fused attention as the kernel of Reuse layers); read MLA-style:
 * for query row (b,t,h) and valid selected entries J,
 *   z_j = sm_scale * sum_{c<D} q[c] * Khat[j][c]
 *   out[c] = sum_j softmax(z)_j * Khat[j][c]   for c < dv
 *   lse = log sum_j exp(z_j)
 * Khat is the dequantised entry (E2M1 value x its group's E4M3 scale,
 * exact in f16), computed on chip from the FP4 planes; V is its first dv
 * channels.  The scores and P V run on the tensor cores with fp32
 * accumulation; P is rounded to f16.
 * An empty J gives out = 0 and lse = -inf.
 * mode  any: REUSE layers pass their source layer's idx (and KV, or their
 *       own KV) unchanged ([ENG] CSA2 section; [55ZB], [HUNT] CSA2 paragraphs).
 *
 * q       bf16 [B, T, H, D], 16-byte aligned, finite; on the D = 576 path each
 *         (token, head) row's largest |q| must be below 2^76 (the row is
 *         scaled by a power of two into f16).  Supported (D, dv, H):
 *         D = 576, dv = 512, H a multiple of 64; D = 128, dv = 64, H a
 *         multiple of 16.
 * codes   uint8 [B*N, D/2], scales uint8 [B*N, D/16]: entry j of sequence
 *         b is row b*N + j (the layout csa2_quantize_kv_fp4 writes);
 *         codes 16-byte aligned, scales 4-byte aligned.
 * idx     int32 [B, T, K], entries j in [0, kv_len) or -1 (skipped);
 *         anything else is skipped and sets CSA2_FLAG_BAD_INDEX.  K <= 2048.
 * kv_len  int32 [B*T] or NULL (= N).
 * out     fp32 [B, T, H, dv] (out_dt must be CSA2_FP32), 16-byte aligned;
 *         lse fp32 [B, T, H] or NULL.
 * err_flag  CSA2_FLAG_BAD_INDEX as above; CSA2_FLAG_TIMEOUT if a bounded
 *         on-chip wait gave up (that launch's results are invalid).
 * workspace csa2_sparse_attn_workspace_bytes() bytes: 0 for D = 576 with
 *         K <= 512 (a cluster of CTAs merges its partials on chip), else the
 *         split-KV partials; NULL allowed when 0.
 */
csa2_status csa2_sparse_attn_fp4(csa2_mode mode, int B, int T, int H, int D, int dv,
                                 const void *q, const uint8_t *codes, const uint8_t *scales,
                                 int64_t N, const int32_t *idx, int K, const int32_t *kv_len,
                                 float sm_scale, void *out, csa2_dtype out_dt, float *lse,
                                 uint32_t *err_flag, void *workspace, size_t ws_bytes,
                                 csa2_stream_t stream);
size_t csa2_sparse_attn_workspace_bytes(int B, int T, int H, int D, int dv, int K);

/*
 * csa2_sparse_attn_fp4_prefetch -- csa2_sparse_attn_fp4, plus an L2 prefetch
 * hint for the layer that attends next with the same indices.  In a CSA2
 * group the Reuse layers attend with their source layer's idx ([ENG] CSA2
 * section; [HUNT] CSA2 paragraph), so while this layer's attention computes
 * (its HBM traffic is over once its own rows have landed) the rows that idx
 * selects in the next layer's planes can already travel to L2, and the next
 * launch gathers them from there.
 *
 * Arguments, results and errors are those of csa2_sparse_attn_fp4, plus
 * next_codes / next_scales: FP4 planes of the same shape and layout as
 * codes / scales (codes 16-byte, scales 4-byte aligned), or both NULL (then
 * this is exactly csa2_sparse_attn_fp4).  They are only read as a hint: no
 * result depends on them, nothing waits for them, and they may be written
 * afterwards.  The hint is issued on the D = 576, K <= 512 path only.
 */
csa2_status csa2_sparse_attn_fp4_prefetch(csa2_mode mode, int B, int T, int H, int D, int dv,
                                          const void *q, const uint8_t *codes, const uint8_t *scales,
                                          int64_t N, const int32_t *idx, int K, const int32_t *kv_len,
                                          float sm_scale, void *out, csa2_dtype out_dt, float *lse,
                                          uint32_t *err_flag, void *workspace, size_t ws_bytes,
                                          const uint8_t *next_codes, const uint8_t *next_scales,
                                          csa2_stream_t stream);

/*
 * csa2_swa_attn_fp8 -- the sliding-window branch over an FP8 window KV,
 * merged with the sparse branch.  [ENG] "效率组件四件" item 4 (the SWA KV stays
 * FP8); [HUNT] (every layer also has a sliding window).  The pages give neither
 * the window size nor the FP8 layout; READINGS: window rows are E4M3 without a
 * scale, K = all D channels, V = the first dv (as the sparse branch), and query
 * row (b, t) attends to the first swa_len[b*T+t] rows of sequence b's window
 * (all visible: the caller keeps the last window of tokens there).  The
 * merge is the softmax over both branches' entries:
 *     M = max(lse_w, lse_s), a = e^(lse_w - M), c = e^(lse_s - M),
 *     out = (a o_w + c o_s) / (a + c),  lse = M + log(a + c).
 *
 * q          bf16 [B, T, H, D], D = 576, dv = 512, H a multiple of 64; each
 *            (token, head) row's largest |q| below 2^76, as in the sparse branch.
 *            The window's E4M3 values enter the MMAs as exact f16.
 * swa_kv     E4M3 [B, W, D], 1 <= W <= 512, 16-byte aligned.
 * swa_len    int32 [B*T], clamped to [0, W].
 * o_sparse, lse_sparse  fp32 [B, T, H, dv] and [B, T, H] from
 *            csa2_sparse_attn_fp4, or both NULL (window branch alone).
 * out        fp32 [B, T, H, dv]; may be o_sparse itself (merged in place).
 * lse        fp32 [B, T, H] merged log-sum-exp, or NULL.
 * An empty window with lse_s = -inf gives out = 0, lse = -inf.
 */
csa2_status csa2_swa_attn_fp8(int B, int T, int H, int D, int dv, const void *q, const uint8_t *swa_kv, int W,
                              const int32_t *swa_len, float sm_scale, const float *o_sparse, const float *lse_sparse,
                              float *out, float *lse, uint32_t *err_flag, csa2_stream_t stream);

/*
 * csa2_sparse_attn_fp4_noalloc -- csa2_sparse_attn_fp4 without a caller
 * workspace.  The pages have no counterpart to this call: it exists for
 * callers that may not allocate device memory at all, such as an engine that
 * plans every byte of its device memory before it starts serving, or code
 * that must not call cudaMalloc/cudaFree because those calls can synchronise
 * the device.  The split-KV scratch lives in one array built into the library
 * (csa2_sparse_attn_noalloc_max_scratch_bytes() bytes, 20 MiB; every
 * supported shape fits on a 152-SM GB300) that every GPU
 * loading the library holds until the process exits.
 *
 * Arguments, layouts, results and errors are those of csa2_sparse_attn_fp4
 * (minus workspace/ws_bytes); the call allocates nothing.  A shape whose
 * scratch (csa2_sparse_attn_workspace_bytes) exceeds the array returns
 * CSA2_ERR_WORKSPACE with an explanation.  The array's device addresses are
 * kept in a table of 64 devices: a call on a device ordinal of 64 or more
 * that needs scratch returns CSA2_ERR_UNSUPPORTED.  The first call on each device
 * looks up the array's device address with that device current; make that
 * first call before any stream capture.  All calls on a device share the
 * array and it keeps the previous call's contents (each call overwrites every
 * partial it reads, so no clearing is needed): calls that overlap on the GPU
 * (for instance on two streams of the same device) race.
 */
csa2_status csa2_sparse_attn_fp4_noalloc(csa2_mode mode, int B, int T, int H, int D, int dv,
                                         const void *q, const uint8_t *codes, const uint8_t *scales,
                                         int64_t N, const int32_t *idx, int K, const int32_t *kv_len,
                                         float sm_scale, void *out, csa2_dtype out_dt, float *lse,
                                         uint32_t *err_flag, csa2_stream_t stream);
size_t csa2_sparse_attn_noalloc_max_scratch_bytes(void);

/*
 * csa2_selftest_bounded_wait -- exercises the library's bounded wait on an
 * mbarrier (the one every tensor-core kernel uses for its TMA copies and
 * MMAs) with an arrival that never comes: one CTA polls an mbarrier nothing
 * arrives on, gives up after max_polls polls (1 <= max_polls <= 2^22), sets
 * CSA2_FLAG_TIMEOUT in *err_flag (device, required) and returns, leaving the
 * context usable.  Test infrastructure for the failure path; no fault, trap
 * or unbounded spin is involved.
 */
csa2_status csa2_selftest_bounded_wait(uint32_t max_polls, uint32_t *err_flag, csa2_stream_t stream);

/* Status helpers. */
const char *csa2_status_string(csa2_status s);
const char *csa2_last_error(void); /* thread-local detail of the last non-OK status */
int csa2_version(void);            /* major*10000 + minor*100 + patch */

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H */
