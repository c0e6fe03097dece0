/*
 * qsa.h -- C ABI of libqsa: indexer-selected (QSA-style) block-sparse attention
 * on one GB300 (sm_103a).
 *
 * For every query row the path (1) scores each complete compressed block of
 * `ratio` tokens as  s_b = sum_h w_h * max(0, q_I,h . k_I,b),  (2) keeps the
 * K = budget/ratio best blocks (ties to the lower block index) plus the
 * incomplete tail block, and (3) runs GQA softmax attention (scale 1/sqrt(D))
 * over the raw K/V rows of the kept tokens, gathered from a paged cache.
 *
 * Sources (web pages, by title and section):
 *   [VA6]  "Agentic shootout -- Atlas x Flash-Next research", report
 *          "Flash-Next support: vLLM vs Atlas", (a) item 6 "QSA sparse
 *          attention + indexer": mean-pooled compressed keys whose page table
 *          follows the main KV cache, weight-free scoring, block top-k with
 *          budget/ratio groups, expansion to budget + ratio - 1 token indices
 *          (-1 padded), one opaque index -> KV update -> sparse attend step.
 *   [PR16] same page, "PR 16 review: qwen4exp serving in Atlas (Claude's
 *          review)", (a): relu-score top-512 + tail, inert <= 2051 visible.
 *   [LC3]  same page, "Flash-Next support: llama.cpp vs Atlas", (a) item 3:
 *          blocks cut the position line; the tail block is always visible.
 *   [VP5]  same page, "Flash-Next support: vLLM vs Atlas" (d) item 10: alias
 *          the compressed cache's page mapping to the main block table at
 *          1/ratio density.
 *   [INV]  "Atlas Flash-Next defect investigations", Report A: Defect 1
 *          (decode at pos requires pos == ingested; rewind sets
 *          ingested -= dropped), Defect 4 (16-byte alignment of every base
 *          pointer and pitch; sticky CUDA errors are fatal), Defect 5
 *          (capacity is checked when tokens are appended, never mid-step).
 *
 * Conventions for every entry point
 *   - Pointers marked "device" are device memory owned by the caller; the
 *     library never allocates, frees, synchronises, or copies device data to
 *     the host. All work is enqueued on the caller's `stream`, in order.
 *   - Tensors are dense, row-major, C-contiguous, with the shapes given.
 *     bf16 values are passed as their 16-bit patterns (qsa_bf16).
 *   - Every pointer that a kernel reads or writes with vector accesses
 *     (pools, K/V/q inputs, outputs, workspace) must be 16-byte aligned.
 *   - Every call returns a qsa_status. Host-detected problems are returned
 *     before anything is enqueued. Problems only the device can see (a
 *     position that does not match the ingested counter, a page id outside the
 *     pool, a position beyond the page table) are written to the caller's
 *     device word `*status` with an atomic first-error-wins compare-and-swap;
 *     the caller reads it after synchronising. A non-zero status means the
 *     outputs of that step are undefined.
 *   - The fused step (qsa_decode) makes no host synchronisation and no
 *     allocation, so it can be captured in a CUDA graph.
 */
#ifndef QSA_H
#define QSA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t qsa_bf16; /* bit pattern of a bfloat16 value */

typedef enum qsa_status {
  QSA_OK = 0,
  QSA_ERR_INVALID_ARG = 1,  /* null or misaligned pointer, bad size or stride */
  QSA_ERR_UNSUPPORTED = 2,  /* configuration outside the supported set */
  QSA_ERR_CAPACITY = 3,     /* append beyond the pages the table provides */
  QSA_ERR_WORKSPACE = 4,    /* workspace smaller than qsa_workspace_bytes() */
  QSA_ERR_CUDA = 5,         /* a launch failed (recoverable) */
  QSA_ERR_CUDA_FATAL = 6,   /* sticky CUDA error: the context is lost */
  QSA_ERR_DESYNC = 7,       /* device: append position != ingested counter */
  QSA_ERR_PAGE = 8,         /* device: page id outside [0, num_pages) */
  QSA_ERR_REWIND = 9,       /* device: rewind by more than was ingested */
  QSA_ERR_TIMEOUT = 10,     /* device: an internal wait of a kernel expired (1 s);
                               the kernel released its resources and returned */
  QSA_ERR_REUSE = 11        /* device: a reused selection's position is not in
                               [0, row position], or its token set exceeds
                               qsa_max_attend_tokens() */
} qsa_status;

/* Shape of the method. Supported set (checked by qsa_config_check):
 *   ratio      power of two in [2, 16]          tokens per compressed block
 *   budget     multiple of ratio                token budget, K = budget/ratio
 *   K          1 <= K <= 2048
 *   n_idx_heads (H_I) in [1, 64]                indexer query heads
 *   idx_dim    (d_I) 64 or 128                  indexer key/query dim
 *   n_q_heads  (Hq), n_kv_heads (Hkv) in {1,2,4}, Hq % Hkv == 0,
 *              Hq / Hkv <= 8                    GQA
 *   head_dim   (D) 128
 *   page_size  (P) 64, multiple of ratio        tokens per cache page
 *   index_format QSA_INDEX_BF16, QSA_INDEX_MXFP8 or QSA_INDEX_MXFP4 (the
 *              MX ones with P / ratio >= 8 blocks per page)  compressed-key plane
 *   local_window in [0, 16384]                  always-kept recent tokens
 * The indexer has one key head (MQA), as the pages require.
 *
 * Index formats. QSA_INDEX_BF16: compressed keys are bf16 and the index
 * queries are scored as given. QSA_INDEX_MXFP8 ("Agentic shootout", "Flash-Next
 * support: vLLM vs Atlas", the report whose (a) item 3 is "QSA sparse
 * attention + n-gram indexer", Scores bullet: MXFP8 quantisation of the index
 * queries and of the indexer cache; "ATOM Model Support Guide", DeepSeek-V4.1,
 * Cache bullet: an fp8 index plane with E8M0 scales): every compressed key is
 * stored as OCP MXFP8 -- per 32 consecutive values one E8M0 scale
 * 2^(floor(log2 amax) - 8) (2^-127 for an all-zero block) and E4M3 elements,
 * value / scale rounded to nearest-even and clamped to +-448 -- and the fused
 * step puts each index query head through the same quantisation before
 * scoring. The key quantised is the bf16 compressed key of QSA_INDEX_BF16;
 * scores are exact sums of the quantised values' products in fp32.
 *
 * Local window ("Agentic shootout", "Flash-Next support: llama.cpp vs Atlas",
 * (d) adoption plan, phase 2, item 6: the last 128 tokens are always kept, a
 * union with the top-k set; llama.cpp's indexer_local_blocks): with
 * local_window = W > 0 every row attends to its selected blocks, its tail and
 * its last W visible tokens. The selection itself is unchanged; the token set
 * is the selected tokens before min(V - W, n_blk * ratio) followed by every
 * token from there to the row. Attention then takes up to budget + W +
 * ratio - 1 tokens (qsa_max_attend_tokens, qsa_workspace_bytes grow with W). */
#define QSA_INDEX_BF16 0
#define QSA_INDEX_MXFP8 1
#define QSA_INDEX_MXFP4 2 /* as MXFP8 with E2M1 elements (0, 0.5, 1, 1.5, 2, 3, 4, 6)
                             and scale 2^(floor(log2 amax) - 2) ("ATOM Model
                             Support Guide", DeepSeek-V4.1, Cache bullet: an fp4
                             index plane in E2M1 + E8M0 arithmetic); queries too */
typedef struct qsa_config {
  int ratio;
  int budget;
  int n_idx_heads;
  int idx_dim;
  int n_q_heads;
  int n_kv_heads;
  int head_dim;
  int page_size;
  int index_format; /* QSA_INDEX_BF16 (0) or QSA_INDEX_MXFP8 (1) */
  int local_window; /* always-kept recent tokens per row (0: none) */
} qsa_config;

/* The query rows of one step. The step appends rows_per_seq (R) tokens to
 * each of n_seq sequences; every appended token is a query row. Rows are
 * sequence-major: row i*R + j is token j of sequence i, at logical position
 * pos0[i] + j, and it sees V = pos0[i] + j + 1 tokens (its own included;
 * rows of one sequence are causal among themselves).
 *   decode:  R = 1;   speculative verify: R = draft rows + 1;
 *   chunked prefill:  n_seq = 1, R = chunk length.
 * seq_ids must be distinct within a call. */
typedef struct qsa_rows {
  int n_seq;
  int rows_per_seq;
  const int32_t *seq_ids;   /* device [n_seq]: slot in page_table / ingested */
  int32_t *pos0;            /* device [n_seq]: position of the first row */
  const int32_t *pos0_host; /* optional host copy of pos0 (NULL if absent);
                               when given, capacity is checked on the host
                               and reported as QSA_ERR_CAPACITY before any
                               launch */
  int advance;              /* non-zero: qsa_append / qsa_decode also add R to
                               pos0[i] on the device when they advance the
                               ingested counter, as the step's last action, so
                               a step captured in a CUDA graph can be replayed
                               for consecutive decode steps without the
                               positions and counters drifting apart
                               ("Agentic shootout", "PR 16 review: qwen4exp
                               serving in Atlas", (c) item 4: the ingested
                               counter froze at the capture step while the
                               sequence advanced) */
  const int32_t *mrope_pos; /* optional device [n_seq * rows_per_seq][3] int32:
                               each row's (t, h, w) position for interleaved
                               MRoPE (row i * R + j is token pos0[i] + j),
                               read only when a pre-indexer or attention
                               option has an MRoPE section; NULL: every row is
                               a text token, (p, p, p) */
} qsa_rows;

/* Paged cache of all sequences ([VA6], [VP5]). Logical token t of the
 * sequence in slot s lives in page page_table[s][t / P] at offset t % P.
 * Compressed block b of that sequence lives in the same page id of the block
 * pool, as block row rr = b % (P/ratio) of that page: the block pool shares
 * the main page table at 1/ratio density. All pools have num_pages pages.
 *
 * Inside a block-pool page (P/ratio rows of d_I bf16 values) the rows are
 * stored in tiles of G = min(P/ratio, 8) rows by 8 values: element (rr, d)
 * sits at
 *     ((rr / G) * (d_I / 8) + d / 8) * 8 * G + (rr % G) * 8 + d % 8
 * (the tensor cores' K-major core-matrix order), so one contiguous copy of a
 * page is a ready operand of the scoring contraction. The block pool is
 * written only by qsa_append and read only by qsa_index_score / qsa_decode.
 *
 * With QSA_INDEX_MXFP8 a block-pool page is qsa_idxblk_page_bytes() =
 * bpp * (d_I + d_I/32) bytes (bpp = P/ratio blocks): first the E4M3 elements,
 * element (rr, d) at byte
 *     ((rr / 8) * (d_I / 16) + d / 16) * 128 + (rr % 8) * 16 + d % 16
 * (core matrices of 8 blocks x 16 bytes), then the E8M0 scale bytes, scale
 * (rr, c) of values 32c .. 32c+31 at byte bpp * d_I + rr * (d_I / 32) + c.
 * With QSA_INDEX_MXFP4 a page is bpp * (d_I/2 + d_I/32) bytes: E2M1 pairs,
 * element (rr, d) in byte ((rr / 8) * (d_I / 32) + d / 32) * 128 + (rr % 8) * 16
 * + (d % 32) / 2 (the low nibble for even d), then the scale bytes at
 * bpp * d_I / 2 + rr * (d_I / 32) + c. */
typedef struct qsa_cache {
  const int32_t *page_table; /* device [n_slots, max_pages] */
  int n_slots;
  int max_pages;             /* pages per sequence: capacity max_pages * P */
  int num_pages;             /* pages in each pool */
  qsa_bf16 *k_pool;          /* device [num_pages, P, Hkv, D] */
  qsa_bf16 *v_pool;          /* device [num_pages, P, Hkv, D] */
  qsa_bf16 *idxraw_pool;     /* device [num_pages, P, d_I]   raw index keys */
  void *idxblk_pool;         /* device block keys (tiled, above): bf16 [num_pages, P/ratio * d_I],
                                or with QSA_INDEX_MXFP8 bytes [num_pages, qsa_idxblk_page_bytes()] */
  int32_t *ingested;         /* device [n_slots]: tokens ingested per slot */
  int32_t *blkpos_pool;      /* device [num_pages, P/ratio, 4] int32, 16-byte aligned:
                                the (t, h, w) triple of each block's first token
                                (4th value unused), written by appends through a
                                pre-indexer with an MRoPE section and read when a
                                later append completes the block; NULL when no
                                MRoPE section is used */
} qsa_cache;

/* Message for a status code (static string). */
const char *qsa_strerror(int status);

/* Test hook of the failure path ("Atlas Flash-Next defect investigations",
 * Report A, Defect 4: an error is reported, never laundered into success).
 * Sets the time limit, in nanoseconds, after which an internal wait of the
 * index-score kernel gives up: the CTA records QSA_ERR_TIMEOUT in the status
 * word, waits a bounded 2 ms for its own copies and tensor-core work to land,
 * frees its tensor memory and returns, so the context stays usable. 0 restores
 * the default (1 s); other values are clamped to [1 us, 10 s]. The value is
 * read when a launch is issued (a captured graph keeps the value it was
 * captured with). Returns the previous limit. Meant for tests; a production
 * caller has no reason to change it. */
unsigned long long qsa_set_wait_limit_ns(unsigned long long ns);

/* 0 (QSA_OK) if the configuration is in the supported set above, else
 * QSA_ERR_UNSUPPORTED (QSA_ERR_INVALID_ARG for a NULL pointer). */
int qsa_config_check(const qsa_config *cfg);

/* Bytes of one block-pool page for the configuration's index format
 * (P/ratio * d_I * 2 for bf16, P/ratio * (d_I + d_I/32) for MXFP8); 0 on an
 * invalid configuration. */
size_t qsa_idxblk_page_bytes(const qsa_config *cfg);

/* Bytes of workspace that qsa_decode and qsa_gather_attn need for up to
 * max_rows query rows and up to max_blocks_per_row complete blocks per row
 * (max_blocks_per_row >= max_pages * P / ratio covers every row). Returns 0 on
 * an invalid configuration. */
size_t qsa_workspace_bytes(const qsa_config *cfg, int max_rows, int max_blocks_per_row);

/* Append: ingest R new tokens per sequence ([VA6] KV update + raw key store +
 * group compress; [INV] Defect 1 counter discipline).
 * For each sequence i (slot s = seq_ids[i]) the kernel first checks
 * pos0[i] == ingested[s] (else QSA_ERR_DESYNC, nothing written for i) and
 * pos0[i] + R <= max_pages * P (else QSA_ERR_CAPACITY). It then writes the
 * tokens' K, V and raw index-key rows into the pools, pools every block the
 * new tokens complete (k_b = bf16_rne(sum_j raw_{b*ratio+j} / ratio), fp32
 * sum), and sets ingested[s] = pos0[i] + R.
 *   k_new, v_new  device [n_seq*R, Hkv, D] bf16
 *   idx_k_new     device [n_seq*R, d_I] bf16
 *   status        device int32, see conventions */
int qsa_append(const qsa_config *cfg, const qsa_rows *rows, const qsa_cache *cache,
               const qsa_bf16 *k_new, const qsa_bf16 *v_new, const qsa_bf16 *idx_k_new,
               int32_t *status, cudaStream_t stream);

/* Rewind ([INV] Defect 1 fix: ingested -= dropped, pooled = ingested/ratio):
 * for each i, ingested[seq_ids[i]] -= n_drop[i]. A negative n_drop or one
 * larger than the ingested count leaves the counter unchanged and records
 * QSA_ERR_REWIND. Rows past the new end become dead and are overwritten by
 * the next append; a block made incomplete is re-pooled from its new raw rows
 * when an append completes it again.
 *   seq_ids, n_drop  device [n_seq] int32 */
int qsa_rewind(const qsa_config *cfg, int n_seq, const int32_t *seq_ids, const int32_t *n_drop,
               int32_t *ingested, int32_t *status, cudaStream_t stream);

/* Index score ([PR16] relu-score, [VA6] scoring against compressed keys):
 * for every row with n_blk = V / ratio > K complete blocks, writes
 * scores[row * ld_scores + b] = sum_h w[row,h] * max(0, q_idx[row,h,:] . k_b)
 * for b < n_blk (bf16 products, fp32 accumulation). Rows with n_blk <= K are
 * skipped: every block is selected there, so no score is needed. With
 * QSA_INDEX_MXFP8 the keys are the MXFP8 plane's values and each query head is
 * MXFP8-rounded inside the kernel (as qsa_quantize_index_q; rounding twice
 * changes nothing), the score of the fused step.
 *   q_idx   device [rows, H_I, d_I] bf16
 *   w       device [rows, H_I] fp32
 *   scores  device [rows, ld_scores] fp32; ld_scores >= max_pages*P/ratio,
 *           multiple of 4
 *   status  optional device int32 (NULL: device-detected problems are not
 *           recorded); the same holds for qsa_topk_select and qsa_gather_attn */
int qsa_index_score(const qsa_config *cfg, const qsa_rows *rows, const qsa_cache *cache,
                    const qsa_bf16 *q_idx, const float *w, float *scores, int ld_scores,
                    int32_t *status, cudaStream_t stream);

/* MX round trip of index query heads (the query side of the MX planes, which
 * the scorer applies itself): each d_I vector's blocks of 32 values are
 * quantised as the keys are -- MXFP4 when cfg's index_format is
 * QSA_INDEX_MXFP4, else MXFP8 -- and written back as bf16 (every MX value is
 * exact in bf16).
 *   q_idx, q_out  device [n_rows, H_I, d_I] bf16 (q_out == q_idx allowed) */
int qsa_quantize_index_q(const qsa_config *cfg, int n_rows, const qsa_bf16 *q_idx, qsa_bf16 *q_out,
                         cudaStream_t stream);

/* Top-K select ([VA6] block top-k; ties to the lower block index): for every
 * row, if n_blk <= K all blocks are selected; otherwise the K blocks with
 * the largest score under the total order (score descending, block index
 * ascending). Writes sel[row*K + i] ascending, padded with -1 to K entries,
 * and n_sel[row] = number of selected blocks. Scores are compared as fp32
 * (+0 and -0 are equal; +inf and -inf are ordinary values; a NaN score is
 * outside the contract and ranks above +inf).
 *   scores  device [rows, ld_scores] fp32 (from qsa_index_score), 16-byte
 *           aligned, ld_scores a multiple of 4 (else QSA_ERR_INVALID_ARG)
 *   sel     device [rows, K] int32;  n_sel  device [rows] int32 */
int qsa_topk_select(const qsa_config *cfg, const qsa_rows *rows, const float *scores,
                    int ld_scores, int32_t *sel, int32_t *n_sel, int32_t *status,
                    cudaStream_t stream);

/* Gather attention ([VA6] sparse paged GQA; [LC3] tail always visible): for
 * every row, the token set T = {b*ratio + j : b in sel, j < ratio} U
 * [n_blk*ratio, V) is gathered through the page table, and each query head h
 * (KV head g = h*Hkv/Hq) gets o_h = sum_{t in T} softmax_t(q_h . K_t,g /
 * sqrt(D)) V_t,g, split across CTAs and merged, rounded to bf16.
 *   q    device [rows, Hq, D] bf16
 *   sel, n_sel as written by qsa_topk_select
 *   out  device [rows, Hq, D] bf16
 *   ws   device workspace of ws_bytes >= qsa_workspace_bytes(cfg, rows, *) */
int qsa_gather_attn(const qsa_config *cfg, const qsa_rows *rows, const qsa_cache *cache,
                    const qsa_bf16 *q, const int32_t *sel, const int32_t *n_sel, qsa_bf16 *out,
                    void *ws, size_t ws_bytes, int32_t *status, cudaStream_t stream);

/* The fused step ([VA6]: one opaque index -> KV update -> sparse attend
 * transaction): qsa_append, then qsa_index_score, qsa_topk_select and
 * qsa_gather_attn for every appended row. Makes no host synchronisation and
 * no allocation; capturable in a CUDA graph. The device status word collects
 * errors of all stages.
 *   sel_out, n_sel_out  optional device [rows, K] / [rows] int32 (NULL: kept
 *                       in the workspace)
 *   ws                  device workspace, ws_bytes >=
 *                       qsa_workspace_bytes(cfg, rows, max_pages*P/ratio)
 * With QSA_INDEX_MXFP8 the step's scorer MXFP8-rounds the index queries (as
 * qsa_quantize_index_q) before scoring; q_idx itself is not written. */
int qsa_decode(const qsa_config *cfg, const qsa_rows *rows, const qsa_cache *cache,
               const qsa_bf16 *k_new, const qsa_bf16 *v_new, const qsa_bf16 *idx_k_new,
               const qsa_bf16 *q_idx, const float *w, const qsa_bf16 *q,
               int32_t *sel_out, int32_t *n_sel_out, qsa_bf16 *out,
               void *ws, size_t ws_bytes, int32_t *status, cudaStream_t stream);

/* Pre-indexer ("Agentic shootout", "Flash-Next support: vLLM vs Atlas", (a)
 * item 6, and the same report's description of the fused pre-indexer kernel:
 * the indexer's q/k heads go through Gemma RMSNorm -- gain weight + 1, fp32
 * accumulation -- and the same NeoX RoPE as main attention; a compressed key is
 * the mean-pool, then the norm, then RoPE at the block's first position).
 *   y   = x / sqrt(mean(x^2) + eps) * (1 + gamma)
 *   RoPE at position p: for i < rotary_dim/2 the pair (y_i, y_{i+rotary_dim/2})
 *       turns by p * rope_theta^(-2i/rotary_dim); dims >= rotary_dim are kept.
 * The pages leave epsilon and the RoPE base open: both are inputs. The angle is
 * formed and reduced to [-pi, pi] in double (each pair's frequency computed once
 * per call on the host); its sine / cosine, the norm and the rotation run in
 * fp32; results are rounded to bf16. Raw index keys are stored as given. */
typedef struct qsa_pre_indexer {
  const float *gamma_q; /* device [d_I] fp32: query-norm gains */
  const float *gamma_k; /* device [d_I] fp32: compressed-key-norm gains */
  float eps;            /* >= 0 */
  float rope_theta;     /* > 0 */
  int rotary_dim;       /* 0 (no RoPE), 64, or d_I */
  int mrope_section[3]; /* interleaved MRoPE ("Agentic shootout", "Flash-Next
                           support: vLLM vs Atlas", (a) item 6 and its fused
                           pre-indexer notes): (t, h, w) section sizes in
                           rotary pairs, adding up to rotary_dim / 2; NeoX pair
                           i turns by the row's h when i % 3 == 1 and
                           i < 3 * h, by its w when i % 3 == 2 and i < 3 * w,
                           by its t otherwise; a compressed key turns at its
                           block's first token's triple (the cache's
                           blkpos_pool keeps it). All zero: plain RoPE. */
} qsa_pre_indexer;

/* qsa_append whose completed blocks go through the pre-indexer:
 * k_b = bf16(RoPE_{b*ratio}(GemmaRMSNorm(mean of the block's raw keys)))
 * (then MXFP8-quantised with QSA_INDEX_MXFP8).
 * A cache must be filled with one kind of append throughout. */
int qsa_append_pre(const qsa_config *cfg, const qsa_pre_indexer *pre, const qsa_rows *rows,
                   const qsa_cache *cache, const qsa_bf16 *k_new, const qsa_bf16 *v_new,
                   const qsa_bf16 *idx_k_new, int32_t *status, cudaStream_t stream);

/* The index queries of the rows through the pre-indexer:
 * q_out[row, h] = bf16(RoPE_{row position}(GemmaRMSNorm(q_idx[row, h]))),
 * then, with QSA_INDEX_MXFP8, the MXFP8 round trip of qsa_quantize_index_q.
 *   q_idx, q_out  device [rows, H_I, d_I] bf16, distinct buffers */
int qsa_pre_index_q(const qsa_config *cfg, const qsa_pre_indexer *pre, const qsa_rows *rows,
                    const qsa_bf16 *q_idx, qsa_bf16 *q_out, cudaStream_t stream);

/* Bytes of workspace qsa_decode_pre needs: qsa_workspace_bytes plus the
 * pre-indexed query rows. */
size_t qsa_workspace_bytes_pre(const qsa_config *cfg, int max_rows, int max_blocks_per_row);

/* The fused step through the pre-indexer: as qsa_decode, with the appended
 * blocks pooled as in qsa_append_pre and the index queries pre-indexed (into
 * the workspace; q_idx itself is not written) before scoring. */
int qsa_decode_pre(const qsa_config *cfg, const qsa_pre_indexer *pre, const qsa_rows *rows,
                   const qsa_cache *cache, const qsa_bf16 *k_new, const qsa_bf16 *v_new,
                   const qsa_bf16 *idx_k_new, const qsa_bf16 *q_idx, const float *w, const qsa_bf16 *q,
                   int32_t *sel_out, int32_t *n_sel_out, qsa_bf16 *out, void *ws, size_t ws_bytes,
                   int32_t *status, cudaStream_t stream);

/* Main-attention options of the fused step ("Agentic shootout", "Flash-Next
 * support: vLLM vs Atlas", (a) item 6, Dataflow bullet: GQA with a sigmoid
 * output gate, always on, GemmaRMSNorm q/k heads, a fused QK-norm + RoPE +
 * gate path). Each member is optional:
 *   gamma_q  device [D] fp32: every query head of the step becomes
 *            bf16(RoPE_{row position}(GemmaRMSNorm(q_h))) (gains 1 + gamma_q) in the
 *            workspace; q itself is not written
 *   gamma_k  device [D] fp32: every appended key head is stored as
 *            bf16(RoPE_{token position}(GemmaRMSNorm(k_h))); a cache must be filled
 *            with one kind of append throughout (qsa_append_ex with the same gamma_k)
 *   eps, rope_theta, rotary_dim   as in qsa_pre_indexer (rotary_dim 0, 64 or D)
 *   gate     device [rows, Hq, D] bf16: the output is o * sigmoid(gate),
 *            elementwise, before its bf16 rounding
 * The pages leave the gate's granularity, epsilon and the RoPE base open:
 * elementwise, and both inputs. */
typedef struct qsa_attn_options {
  const float *gamma_q;
  const float *gamma_k;
  float eps;
  float rope_theta;
  int rotary_dim;
  const qsa_bf16 *gate;
  int mrope_section[3]; /* as in qsa_pre_indexer: q and k heads turn at their
                           own row's (t, h, w) (qsa_rows.mrope_pos); all zero:
                           plain RoPE */
} qsa_attn_options;

/* qsa_append / qsa_append_pre with optional index pre-indexer and main
 * attention options (only gamma_k acts here). Either pointer may be NULL. */
int qsa_append_ex(const qsa_config *cfg, const qsa_pre_indexer *pre, const qsa_attn_options *attn,
                  const qsa_rows *rows, const qsa_cache *cache, const qsa_bf16 *k_new,
                  const qsa_bf16 *v_new, const qsa_bf16 *idx_k_new, int32_t *status, cudaStream_t stream);

/* Bytes of workspace qsa_decode_ex needs with any options: qsa_workspace_bytes
 * plus the prepared index and main query rows. */
size_t qsa_workspace_bytes_ex(const qsa_config *cfg, int max_rows, int max_blocks_per_row);

/* The fused step with optional index pre-indexer (as qsa_decode_pre) and main
 * attention options (above). With both NULL it is qsa_decode. */
int qsa_decode_ex(const qsa_config *cfg, const qsa_pre_indexer *pre, const qsa_attn_options *attn,
                  const qsa_rows *rows, const qsa_cache *cache, const qsa_bf16 *k_new, const qsa_bf16 *v_new,
                  const qsa_bf16 *idx_k_new, const qsa_bf16 *q_idx, const float *w, const qsa_bf16 *q,
                  int32_t *sel_out, int32_t *n_sel_out, qsa_bf16 *out, void *ws, size_t ws_bytes,
                  int32_t *status, cudaStream_t stream);

/* Tokens one row's attention can take: the split plan covers
 * ceil((budget + ratio - 1) / 112) splits of 112 tokens. A reused selection
 * (below) may be used while its token set stays within this count. Returns 0
 * on an invalid configuration. */
int qsa_max_attend_tokens(const qsa_config *cfg);

/* Gather attention with a reused selection ("Agentic shootout", "Flash-Next
 * support: vLLM vs Atlas", (a) item 6: with MTP, later draft steps reuse the
 * step-0 selection while the side caches keep updating; "Flash-Next support:
 * llama.cpp vs Atlas", (a) item 3: a shared indexer layer reuses the previous
 * full layer's top-k). sel / n_sel were selected by the row at position
 * sel_pos[row] <= the row's position (for a shared layer, the same position).
 * The row attends over the reused blocks plus every token from that
 * position's block boundary to the row:
 *     T = {b*ratio + j : b in sel, j < ratio}  U  [((sel_pos+1)/ratio)*ratio, V).
 * Nothing is scored or selected. |T| must stay <= qsa_max_attend_tokens(),
 * else QSA_ERR_REUSE is recorded (as for sel_pos outside [0, position]).
 *   sel_pos  device [rows] int32
 *   other arguments as qsa_gather_attn */
int qsa_gather_attn_reuse(const qsa_config *cfg, const qsa_rows *rows, const qsa_cache *cache,
                          const qsa_bf16 *q, const int32_t *sel, const int32_t *n_sel,
                          const int32_t *sel_pos, qsa_bf16 *out, void *ws, size_t ws_bytes,
                          int32_t *status, cudaStream_t stream);

/* The fused step with a reused selection: qsa_append (the side caches keep
 * updating: raw keys, pooled blocks, K/V, counters), then
 * qsa_gather_attn_reuse for every appended row, then the counter commit.
 * Skips index scoring and top-K selection. No host synchronisation, no
 * allocation; capturable in a CUDA graph. Arguments as qsa_decode without the
 * indexer query and weights, plus the reused selection (sel, n_sel, sel_pos;
 * device [rows, K], [rows], [rows] int32). ws_bytes >= qsa_workspace_bytes(cfg,
 * rows, max_pages*P/ratio). */
int qsa_decode_reuse(const qsa_config *cfg, const qsa_rows *rows, const qsa_cache *cache,
                     const qsa_bf16 *k_new, const qsa_bf16 *v_new, const qsa_bf16 *idx_k_new,
                     const qsa_bf16 *q, const int32_t *sel, const int32_t *n_sel,
                     const int32_t *sel_pos, qsa_bf16 *out, void *ws, size_t ws_bytes,
                     int32_t *status, cudaStream_t stream);

/* Size of the fixed scratch array behind qsa_gather_attn_static. */
#define QSA_STATIC_SCRATCH_BYTES (32u << 20)

/* Gather attention without a workspace (the pages have no counterpart; this
 * is a convenience of this library). Same computation, arguments and outputs
 * as qsa_gather_attn, minus ws / ws_bytes: the split partials live in a
 * QSA_STATIC_SCRATCH_BYTES array compiled into the library, for callers that
 * cannot allocate device memory themselves (a plugin that only receives the
 * framework's input and output tensors, or a loop where cudaMalloc is not
 * allowed). The call allocates nothing.
 *   - Every GPU that loads the library holds that array until the process
 *     exits. A call whose partials would not fit (about 316 KB per row at
 *     Hq = 32, budget 2048: up to 106 rows) returns QSA_ERR_WORKSPACE.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents; calls that overlap on the GPU race and give wrong results.
 *     Nothing in it needs to start at zero.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture. */
int qsa_gather_attn_static(const qsa_config *cfg, const qsa_rows *rows, const qsa_cache *cache,
                           const qsa_bf16 *q, const int32_t *sel, const int32_t *n_sel,
                           qsa_bf16 *out, int32_t *status, cudaStream_t stream);

/* Host-to-device copy of a step's inputs inside the stream's chain of kernels
 * (the pages have no counterpart: this is the library's way to feed a fused
 * step from host memory without breaking the programmatic launch chain that a
 * copy-engine node would break). A kernel reads `bytes` bytes at `src` in host
 * memory the device can reach -- pinned (cudaHostAlloc, cudaHostRegister), or
 * any host memory where the GPU accesses pageable memory through a coherent
 * CPU-GPU link; checked with cudaHostGetDevicePointer -- and writes them to
 * `dst` in device memory. It is launched as a programmatic dependent of the previous kernel on
 * the stream and copies before it waits for that kernel, so the copy overlaps
 * the kernel's tail; a library kernel launched after it on the stream sees the
 * copy and everything before it.
 *   dst    device, 16-byte aligned; must not be read by the kernel launched
 *          just before this call on the stream (give each step its own buffer)
 *   src    host memory the device can reach, 16-byte aligned
 *   bytes  a multiple of 16
 * Returns QSA_ERR_INVALID_ARG for a NULL or misaligned pointer, a size that is
 * not a multiple of 16, or a source the device cannot reach (nothing is
 * launched then). */
int qsa_stage_in(void *dst, const void *src, size_t bytes, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H */
