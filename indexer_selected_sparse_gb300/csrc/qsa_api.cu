// extern "C" entry points of libqsa: argument validation, workspace layout,
// and the launch sequence of each operation (declared in include/qsa.h).
//
// Host-side checks follow the lessons of "Atlas Flash-Next defect
// investigations", Report A: Defect 4 (every base pointer and pitch 16-byte
// aligned; sticky CUDA errors are fatal, never laundered into success) and
// Defect 5 (capacity is checked when tokens are appended, against the pages
// the caller's table provides, never as a mid-step abort).
#include <cmath>
#include <cstring>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

bool is_pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }
int ilog2(int v) {
  int l = 0;
  while ((1 << l) < v) ++l;
  return l;
}
size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

// Argument checks and conversions shared by every entry point (declared in
// qsa_internal.cuh, so that every translation unit validates alike).
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_cfg(const qsa_config *c) {
  if (!c) return QSA_ERR_INVALID_ARG;
  if (!is_pow2(c->ratio) || c->ratio < 2 || c->ratio > 16) return QSA_ERR_UNSUPPORTED;
  if (c->budget <= 0 || c->budget % c->ratio != 0) return QSA_ERR_UNSUPPORTED;
  const int k = c->budget / c->ratio;
  if (k < 1 || k > kMaxTopK) return QSA_ERR_UNSUPPORTED;
  if (c->n_idx_heads < 1 || c->n_idx_heads > 64) return QSA_ERR_UNSUPPORTED;
  if (c->idx_dim != 64 && c->idx_dim != 128) return QSA_ERR_UNSUPPORTED;
  if (c->head_dim != kHeadDim) return QSA_ERR_UNSUPPORTED;
  if (c->n_kv_heads != 1 && c->n_kv_heads != 2 && c->n_kv_heads != 4) return QSA_ERR_UNSUPPORTED;
  if (c->n_q_heads < c->n_kv_heads || c->n_q_heads % c->n_kv_heads != 0) return QSA_ERR_UNSUPPORTED;
  if (c->n_q_heads / c->n_kv_heads > 8) return QSA_ERR_UNSUPPORTED;
  if (c->page_size != 64 || c->page_size % c->ratio != 0) return QSA_ERR_UNSUPPORTED;
  if (c->index_format != QSA_INDEX_BF16 && c->index_format != QSA_INDEX_MXFP8 && c->index_format != QSA_INDEX_MXFP4)
    return QSA_ERR_UNSUPPORTED;
  if (c->local_window < 0 || c->local_window > kMaxLocalWindow) return QSA_ERR_UNSUPPORTED;
  // an MX plane is scored on the tensor-core path: 8 or more blocks per page
  if (c->index_format != QSA_INDEX_BF16 && c->page_size / c->ratio < 8) return QSA_ERR_UNSUPPORTED;
  return QSA_OK;
}

Shape make_shape(const qsa_config *c) {
  Shape s;
  s.ratio = c->ratio;
  s.budget = c->budget;
  s.topk = c->budget / c->ratio;
  s.h_idx = c->n_idx_heads;
  s.d_idx = c->idx_dim;
  s.hq = c->n_q_heads;
  s.hkv = c->n_kv_heads;
  s.d = c->head_dim;
  s.page = c->page_size;
  s.log2_ratio = ilog2(c->ratio);
  s.log2_page = ilog2(c->page_size);
  s.idx_fp8 = c->index_format == QSA_INDEX_MXFP8 || c->index_format == QSA_INDEX_MXFP4 ? 1 : 0;
  s.idx_fp4 = c->index_format == QSA_INDEX_MXFP4 ? 1 : 0;
  s.window = c->local_window;
  return s;
}

int check_rows(const qsa_rows *r) {
  if (!r) return QSA_ERR_INVALID_ARG;
  if (r->n_seq < 0 || r->rows_per_seq < 0) return QSA_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(r->n_seq) * r->rows_per_seq;
  if (rows > 65535) return QSA_ERR_INVALID_ARG;  // one grid row per query row
  if (rows > 0 && (!r->seq_ids || !r->pos0)) return QSA_ERR_INVALID_ARG;
  return QSA_OK;
}

int check_cache(const qsa_cache *c, bool need_kv, bool need_idx) {
  if (!c || !c->page_table || c->max_pages < 1 || c->num_pages < 1 || c->n_slots < 1)
    return QSA_ERR_INVALID_ARG;
  if (need_kv && (!c->k_pool || !c->v_pool || !aligned16(c->k_pool) || !aligned16(c->v_pool)))
    return QSA_ERR_INVALID_ARG;
  if (need_idx && (!c->idxraw_pool || !c->idxblk_pool || !aligned16(c->idxraw_pool) ||
                   !aligned16(c->idxblk_pool)))
    return QSA_ERR_INVALID_ARG;
  return QSA_OK;
}

CacheView view(const qsa_cache *c) {
  CacheView v;
  v.page_table = c->page_table;
  v.max_pages = c->max_pages;
  v.num_pages = c->num_pages;
  v.k_pool = c->k_pool;
  v.v_pool = c->v_pool;
  v.idxraw_pool = c->idxraw_pool;
  v.idxblk_pool = c->idxblk_pool;
  return v;
}

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return QSA_OK;
  switch (e) {
    case cudaErrorIllegalAddress:
    case cudaErrorLaunchFailure:
    case cudaErrorMisalignedAddress:
    case cudaErrorIllegalInstruction:
    case cudaErrorHardwareStackError:
    case cudaErrorInvalidAddressSpace:
    case cudaErrorInvalidPc:
    case cudaErrorAssert:
    case cudaErrorLaunchTimeout:
      return QSA_ERR_CUDA_FATAL;
    default:
      cudaGetLastError();  // clear a non-sticky error
      return QSA_ERR_CUDA;
  }
}

namespace {

int host_capacity_check(const qsa_rows *r, const qsa_cache *c, int page_size) {
  if (!r->pos0_host) return QSA_OK;
  const long long cap = static_cast<long long>(c->max_pages) * page_size;
  for (int i = 0; i < r->n_seq; ++i) {
    const long long p = r->pos0_host[i];
    if (p < 0 || p + r->rows_per_seq > cap) return QSA_ERR_CAPACITY;
  }
  return QSA_OK;
}

// Workspace layout of the fused step: [partials][scores][sel][n_sel], each
// region 256-byte aligned.
struct WsLayout {
  size_t partials, scores, sel, n_sel, total;
};

WsLayout ws_layout(const Shape &sh, int rows, int ld) {
  WsLayout l;
  l.partials = 0;
  size_t off = round_up(attn_partial_bytes(sh, rows), 256);
  l.scores = off;
  off += round_up(static_cast<size_t>(rows) * ld * sizeof(float), 256);
  l.sel = off;
  off += round_up(static_cast<size_t>(rows) * sh.topk * sizeof(int32_t), 256);
  l.n_sel = off;
  off += round_up(static_cast<size_t>(rows) * sizeof(int32_t), 256);
  l.total = off;
  return l;
}

int ld_for(int max_blocks) { return static_cast<int>(round_up(max_blocks > 0 ? max_blocks : 1, 4)); }

// Bytes of the pre-indexed index queries of `rows` rows (fused step with a pre-indexer).
size_t q_prep_bytes(const Shape &sh, int rows) {
  return static_cast<size_t>(rows) * sh.h_idx * sh.d_idx * sizeof(uint16_t);
}

// Pre-indexer parameters: gains present where needed, eps >= 0, theta > 0,
// rotary dims 0, 64 or d_I (whole NeoX pairs per warp lane).
// An MRoPE section: all zero (plain RoPE), or three non-negative pair counts
// adding up to rotary_dim / 2.
bool mrope_on(const int sec[3]) { return sec[0] != 0 || sec[1] != 0 || sec[2] != 0; }

int check_mrope(const int sec[3], int rotary_dim) {
  if (!mrope_on(sec)) return QSA_OK;
  if (sec[0] < 0 || sec[1] < 0 || sec[2] < 0 || rotary_dim == 0) return QSA_ERR_INVALID_ARG;
  if (static_cast<long long>(sec[0]) + sec[1] + sec[2] != rotary_dim / 2) return QSA_ERR_INVALID_ARG;
  return QSA_OK;
}

// The rows' triples (4-byte aligned when given) with an MRoPE section, and the
// cache's block-position pool when keys are pooled through one.
int check_mrope_buffers(const qsa_rows *rows, const qsa_cache *cache, bool on_q, bool on_blk) {
  if ((on_q || on_blk) && rows && rows->mrope_pos && (reinterpret_cast<uintptr_t>(rows->mrope_pos) & 3))
    return QSA_ERR_INVALID_ARG;
  if (on_blk && (!cache || !cache->blkpos_pool || !aligned16(cache->blkpos_pool))) return QSA_ERR_INVALID_ARG;
  return QSA_OK;
}

// The MRoPE buffers one call needs: the rows' triples when any of its RoPE
// uses a section, the cache's block-position pool when it pools keys through a
// pre-indexer with one.
int check_mrope_call(const qsa_pre_indexer *pre, const qsa_attn_options *att, const qsa_rows *rows,
                     const qsa_cache *cache) {
  const bool pre_on = pre && mrope_on(pre->mrope_section);
  const bool on_q = pre_on || (att && mrope_on(att->mrope_section));
  const bool on_blk = cache && pre_on && pre->gamma_k;
  return check_mrope_buffers(rows, cache, on_q, on_blk);
}

Mrope mrope_of(const int sec[3], const qsa_rows *rows) {
  Mrope m;
  m.on = mrope_on(sec);
  if (m.on) {
    m.sec_h = sec[1];
    m.sec_w = sec[2];
    m.pos = rows ? rows->mrope_pos : nullptr;
  }
  return m;
}

int check_pre(const qsa_config *c, const qsa_pre_indexer *p, bool need_q, bool need_k) {
  if (!p) return QSA_ERR_INVALID_ARG;
  if ((need_q && !p->gamma_q) || (need_k && !p->gamma_k)) return QSA_ERR_INVALID_ARG;
  if (!(p->eps >= 0.f) || !(p->rope_theta > 0.f) || p->eps > 1e30f || p->rope_theta > 1e30f)
    return QSA_ERR_INVALID_ARG;
  if (p->rotary_dim != 0 && p->rotary_dim != 64 && p->rotary_dim != c->idx_dim) return QSA_ERR_UNSUPPORTED;
  return check_mrope(p->mrope_section, p->rotary_dim);
}

// rows: the call's rows (their MRoPE triples); cache: where blocks are pooled
// (its block-position pool), nullptr for query-only calls.
PreArgs pre_args(const qsa_pre_indexer *p, const uint16_t *q_in, uint16_t *q_out, const qsa_rows *rows,
                 const qsa_cache *cache) {
  PreArgs a;
  a.gamma_q = p->gamma_q;
  a.gamma_k = p->gamma_k;
  a.eps = p->eps;
  a.rot = p->rotary_dim;
  const double pi = std::acos(-1.0);
  for (int i = 0; i < a.rot / 2; ++i)
    a.half_turns[i] = std::pow(static_cast<double>(p->rope_theta), -2.0 * i / a.rot) / pi;
  a.q_in = q_in;
  a.q_out = q_out;
  a.mr = mrope_of(p->mrope_section, rows);
  if (a.mr.on && cache) a.blkpos = cache->blkpos_pool;
  return a;
}



// The fused step; pre != nullptr: through the pre-indexer (the append kernel
// pre-indexes the step's query rows into the workspace, the score kernel reads
// them after its dependency wait).
// Main-attention options: gains present where given, eps >= 0, theta > 0,
// rotary dims 0, 64 or D.
int check_attn(const qsa_attn_options *a) {
  if (!a) return QSA_OK;
  if (!(a->eps >= 0.f) || !(a->rope_theta > 0.f) || a->eps > 1e30f || a->rope_theta > 1e30f)
    return QSA_ERR_INVALID_ARG;
  if (a->rotary_dim != 0 && a->rotary_dim != 64 && a->rotary_dim != kHeadDim) return QSA_ERR_UNSUPPORTED;
  if (a->gate && !aligned16(a->gate)) return QSA_ERR_INVALID_ARG;
  return check_mrope(a->mrope_section, a->rotary_dim);
}

AttnPrep attn_prep(const qsa_attn_options *a, const uint16_t *q_in, uint16_t *q_out, const qsa_rows *rows) {
  AttnPrep p;
  p.mr = mrope_of(a->mrope_section, rows);
  p.gamma_q = a->gamma_q;
  p.gamma_k = a->gamma_k;
  p.eps = a->eps;
  p.rot = a->rotary_dim;
  p.q_in = q_in;
  p.q_out = q_out;
  const double pi = std::acos(-1.0);
  for (int i = 0; i < p.rot / 2; ++i)
    p.half_turns[i] = std::pow(static_cast<double>(a->rope_theta), -2.0 * i / p.rot) / pi;
  return p;
}

// Bytes of the prepared main query rows of `rows` rows.
size_t q_main_bytes(const Shape &sh, int rows) {
  return static_cast<size_t>(rows) * sh.hq * kHeadDim * sizeof(uint16_t);
}

int decode_impl(const qsa_config *cfg, const qsa_pre_indexer *pre, const qsa_attn_options *att,
                const qsa_rows *rows,
                const qsa_cache *cache, const qsa_bf16 *k_new, const qsa_bf16 *v_new,
                const qsa_bf16 *idx_k_new, const qsa_bf16 *q_idx, const float *w, const qsa_bf16 *q,
                int32_t *sel_out, int32_t *n_sel_out, qsa_bf16 *out, void *ws, size_t ws_bytes,
                int32_t *status, cudaStream_t stream) {
  int rc;
  if ((rc = check_cfg(cfg)) != QSA_OK) return rc;
  if ((rc = check_rows(rows)) != QSA_OK) return rc;
  if ((rc = check_cache(cache, true, true)) != QSA_OK) return rc;
  if (!cache->ingested || !status) return QSA_ERR_INVALID_ARG;
  if ((rc = check_mrope_call(pre, att, rows, cache)) != QSA_OK) return rc;
  const int n_rows = rows->n_seq * rows->rows_per_seq;
  if (n_rows == 0) return QSA_OK;
  if (!k_new || !v_new || !idx_k_new || !q_idx || !w || !q || !out || !ws)
    return QSA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(idx_k_new) || !aligned16(q_idx) ||
      !aligned16(q) || !aligned16(out) || !aligned16(ws))
    return QSA_ERR_INVALID_ARG;
  if ((rc = host_capacity_check(rows, cache, cfg->page_size)) != QSA_OK) return rc;
  const Shape sh = make_shape(cfg);
  const int cap_tokens = cache->max_pages * cfg->page_size;
  const int ld = ld_for(cap_tokens / cfg->ratio);
  const WsLayout L = ws_layout(sh, n_rows, ld);
  // through the pre-indexer the step's index queries are prepared into the
  // workspace by the append kernel, and the score kernel reads them there (with
  // an MX plane the score kernel rounds its query tiles itself)
  const bool q_prep = pre != nullptr;
  const bool q_main = att && att->gamma_q;  // main queries normed + roped into the workspace
  const size_t idx_bytes = q_prep ? round_up(q_prep_bytes(sh, n_rows), 256) : 0;
  const size_t need = L.total + idx_bytes + (q_main ? round_up(q_main_bytes(sh, n_rows), 256) : 0);
  if (ws_bytes < need) return QSA_ERR_WORKSPACE;
  uint8_t *base = static_cast<uint8_t *>(ws);
  float *scores = reinterpret_cast<float *>(base + L.scores);
  int32_t *sel = sel_out ? sel_out : reinterpret_cast<int32_t *>(base + L.sel);
  int32_t *n_sel = n_sel_out ? n_sel_out : reinterpret_cast<int32_t *>(base + L.n_sel);
  uint16_t *q_pre = q_prep ? reinterpret_cast<uint16_t *>(base + L.total) : nullptr;
  uint16_t *q_att = q_main ? reinterpret_cast<uint16_t *>(base + L.total + idx_bytes) : nullptr;
  const CacheView cv = view(cache);
  const int R = rows->rows_per_seq;

  PreArgs pa;
  if (pre) pa = pre_args(pre, q_idx, q_pre, rows, cache);
  pa.q_in = q_prep ? q_idx : nullptr;
  pa.q_out = q_pre;
  AttnPrep ap;
  if (att) ap = attn_prep(att, q_main ? q : nullptr, q_att, rows);
  cudaError_t e = launch_append(sh, rows->n_seq, R, rows->seq_ids, rows->pos0, cache->page_table,
                                cache->max_pages, cache->num_pages, cache->k_pool, cache->v_pool,
                                cache->idxraw_pool, cache->idxblk_pool, cache->ingested, k_new,
                                v_new, idx_k_new, status, true, stream, &pa, att ? &ap : nullptr);
  if (e == cudaSuccess)
    e = launch_score(sh, rows->n_seq, R, rows->seq_ids, rows->pos0, cv, q_prep ? q_pre : q_idx, w, scores, ld,
                     status, true, stream, q_prep);
  if (e == cudaSuccess)
    e = launch_select(sh, rows->n_seq, R, rows->pos0, scores, ld, sel, n_sel, ld, cap_tokens,
                      status, true, stream);
  // the counter (and, with rows->advance, pos0) moves last, inside the merge
  // kernel: every stage before it reads the pre-step position
  CommitArgs commit;
  commit.n_seq = rows->n_seq;
  commit.R = R;
  commit.capacity = cap_tokens;
  commit.advance = rows->advance;
  commit.seq_ids = rows->seq_ids;
  commit.pos0 = rows->pos0;
  commit.ingested = cache->ingested;
  // the attention derives each row's selected count (min(n_blk, K)) instead of
  // loading n_sel: one dependent load less after its wait
  if (e == cudaSuccess)
    e = launch_attn(sh, rows->n_seq, R, rows->seq_ids, rows->pos0, cv, q_main ? q_att : q, sel, nullptr, out,
                    base + L.partials, status, true, commit, stream, nullptr, att ? att->gate : nullptr);
  return cuda_status(e);
}

// A step's inputs from pinned host memory into device memory, as a kernel in
// the stream's programmatic chain: every CTA copies its 16-byte pieces, then
// waits for the previous kernel and only then lets the next one launch, so the
// copy overlaps the previous kernel's tail and the chain's ordering (a kernel
// never overlaps one two back) is kept.
constexpr int kStageThreads = 256;

__global__ void __launch_bounds__(kStageThreads)
stage_in_kernel(uint4 *__restrict__ dst, const uint4 *__restrict__ src, size_t n16) {
  // four loads in flight per thread before their stores (host memory is a
  // long round trip away)
  const size_t stride = static_cast<size_t>(gridDim.x) * kStageThreads;
  for (size_t i0 = static_cast<size_t>(blockIdx.x) * kStageThreads + threadIdx.x; i0 < n16; i0 += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i0 + u * stride < n16) v[u] = src[i0 + u * stride];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i0 + u * stride < n16) dst[i0 + u * stride] = v[u];
  }
  pdl_wait();
  pdl_trigger();
}
}  // namespace
}  // namespace qsa

using namespace qsa;

extern "C" {

const char *qsa_strerror(int status) {
  switch (status) {
    case QSA_OK: return "ok";
    case QSA_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad size or stride)";
    case QSA_ERR_UNSUPPORTED: return "configuration outside the supported set";
    case QSA_ERR_CAPACITY: return "append beyond the pages the page table provides (max_pages * page_size tokens)";
    case QSA_ERR_WORKSPACE: return "workspace smaller than qsa_workspace_bytes()";
    case QSA_ERR_CUDA: return "CUDA launch error";
    case QSA_ERR_CUDA_FATAL: return "sticky CUDA error: the context is lost";
    case QSA_ERR_DESYNC: return "append position does not match the ingested counter";
    case QSA_ERR_PAGE: return "page id outside the pool";
    case QSA_ERR_REWIND: return "rewind by more tokens than were ingested";
    case QSA_ERR_TIMEOUT: return "an internal wait of a kernel expired";
    case QSA_ERR_REUSE: return "reused selection: position outside [0, row position] or token set beyond qsa_max_attend_tokens()";
    default: return "unknown status";
  }
}

int qsa_config_check(const qsa_config *cfg) { return check_cfg(cfg); }

size_t qsa_idxblk_page_bytes(const qsa_config *cfg) {
  if (check_cfg(cfg) != QSA_OK) return 0;
  const int bpp = cfg->page_size / cfg->ratio;
  if (cfg->index_format == QSA_INDEX_MXFP4) return static_cast<size_t>(fp4_page_bytes(bpp, cfg->idx_dim));
  return cfg->index_format == QSA_INDEX_MXFP8 ? static_cast<size_t>(fp8_page_bytes(bpp, cfg->idx_dim))
                                              : static_cast<size_t>(bpp) * cfg->idx_dim * sizeof(uint16_t);
}

int qsa_quantize_index_q(const qsa_config *cfg, int n_rows, const qsa_bf16 *q_idx, qsa_bf16 *q_out,
                         cudaStream_t stream) {
  int rc;
  if ((rc = check_cfg(cfg)) != QSA_OK) return rc;
  if (n_rows < 0) return QSA_ERR_INVALID_ARG;
  if (n_rows == 0) return QSA_OK;
  if (!q_idx || !q_out) return QSA_ERR_INVALID_ARG;
  Shape sh = make_shape(cfg);
  sh.idx_fp8 = 1;  // an MX round trip whatever the cache's format: MXFP4 for an MXFP4 plane, else MXFP8
  PreArgs pa;      // no pre-indexer: no gains, no positions
  return cuda_status(launch_pre_index_q(sh, n_rows, 1, nullptr, pa, q_idx, q_out, false, stream));
}

int qsa_max_attend_tokens(const qsa_config *cfg) {
  if (check_cfg(cfg) != QSA_OK) return 0;
  return attn_max_tokens(make_shape(cfg));
}

size_t qsa_workspace_bytes(const qsa_config *cfg, int max_rows, int max_blocks_per_row) {
  if (check_cfg(cfg) != QSA_OK || max_rows < 0 || max_blocks_per_row < 0) return 0;
  const Shape sh = make_shape(cfg);
  return ws_layout(sh, max_rows, ld_for(max_blocks_per_row)).total;
}

int qsa_append(const qsa_config *cfg, const qsa_rows *rows, const qsa_cache *cache,
               const qsa_bf16 *k_new, const qsa_bf16 *v_new, const qsa_bf16 *idx_k_new,
               int32_t *status, cudaStream_t stream) {
  int rc;
  if ((rc = check_cfg(cfg)) != QSA_OK) return rc;
  if ((rc = check_rows(rows)) != QSA_OK) return rc;
  if ((rc = check_cache(cache, true, true)) != QSA_OK) return rc;
  if (!cache->ingested || !status) return QSA_ERR_INVALID_ARG;
  const long long n_rows = static_cast<long long>(rows->n_seq) * rows->rows_per_seq;
  if (n_rows == 0) return QSA_OK;
  if (!k_new || !v_new || !idx_k_new || !aligned16(k_new) || !aligned16(v_new) || !aligned16(idx_k_new))
    return QSA_ERR_INVALID_ARG;
  if ((rc = host_capacity_check(rows, cache, cfg->page_size)) != QSA_OK) return rc;
  const Shape sh = make_shape(cfg);
  cudaError_t e = launch_append(sh, rows->n_seq, rows->rows_per_seq, rows->seq_ids, rows->pos0,
                                cache->page_table, cache->max_pages, cache->num_pages,
                                cache->k_pool, cache->v_pool, cache->idxraw_pool, cache->idxblk_pool,
                                cache->ingested, k_new, v_new, idx_k_new, status, false, stream);
  if (e == cudaSuccess)
    e = launch_commit(rows->n_seq, rows->rows_per_seq, cache->max_pages * cfg->page_size,
                      rows->seq_ids, rows->pos0, cache->ingested, rows->advance, false, stream);
  return cuda_status(e);
}

int qsa_rewind(const qsa_config *cfg, int n_seq, const int32_t *seq_ids, const int32_t *n_drop,
               int32_t *ingested, int32_t *status, cudaStream_t stream) {
  int rc;
  if ((rc = check_cfg(cfg)) != QSA_OK) return rc;
  if (n_seq < 0) return QSA_ERR_INVALID_ARG;
  if (n_seq == 0) return QSA_OK;
  if (!seq_ids || !n_drop || !ingested || !status) return QSA_ERR_INVALID_ARG;
  return cuda_status(launch_rewind(n_seq, seq_ids, n_drop, ingested, status, stream));
}

int qsa_index_score(const qsa_config *cfg, const qsa_rows *rows, const qsa_cache *cache,
                    const qsa_bf16 *q_idx, const float *w, float *scores, int ld_scores,
                    int32_t *status, cudaStream_t stream) {
  int rc;
  if ((rc = check_cfg(cfg)) != QSA_OK) return rc;
  if ((rc = check_rows(rows)) != QSA_OK) return rc;
  if ((rc = check_cache(cache, false, true)) != QSA_OK) return rc;
  if (static_cast<long long>(rows->n_seq) * rows->rows_per_seq == 0) return QSA_OK;
  if (!q_idx || !w || !scores || !aligned16(q_idx) || !aligned16(scores)) return QSA_ERR_INVALID_ARG;
  const long long max_blk = static_cast<long long>(cache->max_pages) * cfg->page_size / cfg->ratio;
  if (ld_scores < max_blk || ld_scores % 4 != 0) return QSA_ERR_INVALID_ARG;
  const Shape sh = make_shape(cfg);
  return cuda_status(launch_score(sh, rows->n_seq, rows->rows_per_seq, rows->seq_ids, rows->pos0,
                                  view(cache), q_idx, w, scores, ld_scores, status, false, stream));
}

int qsa_topk_select(const qsa_config *cfg, const qsa_rows *rows, const float *scores,
                    int ld_scores, int32_t *sel, int32_t *n_sel, int32_t *status,
                    cudaStream_t stream) {
  int rc;
  if ((rc = check_cfg(cfg)) != QSA_OK) return rc;
  if ((rc = check_rows(rows)) != QSA_OK) return rc;
  if (static_cast<long long>(rows->n_seq) * rows->rows_per_seq == 0) return QSA_OK;
  // rows are read with 16-byte loads
  if (!scores || !sel || !n_sel || !aligned16(scores) || ld_scores < 4 || ld_scores % 4 != 0)
    return QSA_ERR_INVALID_ARG;
  const Shape sh = make_shape(cfg);
  // rows whose visible count exceeds ld_scores * ratio are rejected in-kernel
  const long long cap = static_cast<long long>(ld_scores) * cfg->ratio + cfg->ratio - 1;
  return cuda_status(launch_select(sh, rows->n_seq, rows->rows_per_seq, rows->pos0, scores,
                                   ld_scores, sel, n_sel, ld_scores,
                                   cap > 0x7fffffff ? 0x7fffffff : static_cast<int>(cap), status,
                                   false, stream));
}

int qsa_gather_attn(const qsa_config *cfg, const qsa_rows *rows, const qsa_cache *cache,
                    const qsa_bf16 *q, const int32_t *sel, const int32_t *n_sel, qsa_bf16 *out,
                    void *ws, size_t ws_bytes, int32_t *status, cudaStream_t stream) {
  int rc;
  if ((rc = check_cfg(cfg)) != QSA_OK) return rc;
  if ((rc = check_rows(rows)) != QSA_OK) return rc;
  if ((rc = check_cache(cache, true, false)) != QSA_OK) return rc;
  const int n_rows = rows->n_seq * rows->rows_per_seq;
  if (n_rows == 0) return QSA_OK;
  if (!q || !sel || !n_sel || !out || !ws || !aligned16(q) || !aligned16(out) || !aligned16(ws))
    return QSA_ERR_INVALID_ARG;
  const Shape sh = make_shape(cfg);
  if (ws_bytes < attn_partial_bytes(sh, n_rows)) return QSA_ERR_WORKSPACE;
  return cuda_status(launch_attn(sh, rows->n_seq, rows->rows_per_seq, rows->seq_ids, rows->pos0,
                                 view(cache), q, sel, n_sel, out, ws, status, false, CommitArgs{},
                                 stream));
}

int qsa_decode(const qsa_config *cfg, const qsa_rows *rows, const qsa_cache *cache,
               const qsa_bf16 *k_new, const qsa_bf16 *v_new, const qsa_bf16 *idx_k_new,
               const qsa_bf16 *q_idx, const float *w, const qsa_bf16 *q, int32_t *sel_out,
               int32_t *n_sel_out, qsa_bf16 *out, void *ws, size_t ws_bytes, int32_t *status,
               cudaStream_t stream) {
  return decode_impl(cfg, nullptr, nullptr, rows, cache, k_new, v_new, idx_k_new, q_idx, w, q, sel_out, n_sel_out,
                     out, ws, ws_bytes, status, stream);
}

size_t qsa_workspace_bytes_pre(const qsa_config *cfg, int max_rows, int max_blocks_per_row) {
  if (check_cfg(cfg) != QSA_OK || max_rows < 0 || max_blocks_per_row < 0) return 0;
  const Shape sh = make_shape(cfg);
  const WsLayout L = ws_layout(sh, max_rows, ld_for(max_blocks_per_row));
  return L.total + round_up(q_prep_bytes(sh, max_rows), 256);
}

int qsa_append_pre(const qsa_config *cfg, const qsa_pre_indexer *pre, const qsa_rows *rows,
                   const qsa_cache *cache, const qsa_bf16 *k_new, const qsa_bf16 *v_new,
                   const qsa_bf16 *idx_k_new, int32_t *status, cudaStream_t stream) {
  int rc;
  if ((rc = check_cfg(cfg)) != QSA_OK) return rc;
  if ((rc = check_pre(cfg, pre, false, true)) != QSA_OK) return rc;
  if ((rc = check_rows(rows)) != QSA_OK) return rc;
  if ((rc = check_cache(cache, true, true)) != QSA_OK) return rc;
  if (!cache->ingested || !status) return QSA_ERR_INVALID_ARG;
  const long long n_rows = static_cast<long long>(rows->n_seq) * rows->rows_per_seq;
  if (n_rows == 0) return QSA_OK;
  if (!k_new || !v_new || !idx_k_new || !aligned16(k_new) || !aligned16(v_new) || !aligned16(idx_k_new))
    return QSA_ERR_INVALID_ARG;
  if ((rc = check_mrope_call(pre, nullptr, rows, cache)) != QSA_OK) return rc;
  if ((rc = host_capacity_check(rows, cache, cfg->page_size)) != QSA_OK) return rc;
  const Shape sh = make_shape(cfg);
  const PreArgs pa = pre_args(pre, nullptr, nullptr, rows, cache);
  cudaError_t e = launch_append(sh, rows->n_seq, rows->rows_per_seq, rows->seq_ids, rows->pos0,
                                cache->page_table, cache->max_pages, cache->num_pages,
                                cache->k_pool, cache->v_pool, cache->idxraw_pool, cache->idxblk_pool,
                                cache->ingested, k_new, v_new, idx_k_new, status, false, stream, &pa);
  if (e == cudaSuccess)
    e = launch_commit(rows->n_seq, rows->rows_per_seq, cache->max_pages * cfg->page_size,
                      rows->seq_ids, rows->pos0, cache->ingested, rows->advance, false, stream);
  return cuda_status(e);
}

int qsa_pre_index_q(const qsa_config *cfg, const qsa_pre_indexer *pre, const qsa_rows *rows,
                    const qsa_bf16 *q_idx, qsa_bf16 *q_out, cudaStream_t stream) {
  int rc;
  if ((rc = check_cfg(cfg)) != QSA_OK) return rc;
  if ((rc = check_pre(cfg, pre, true, false)) != QSA_OK) return rc;
  if ((rc = check_rows(rows)) != QSA_OK) return rc;
  if (static_cast<long long>(rows->n_seq) * rows->rows_per_seq == 0) return QSA_OK;
  if (!q_idx || !q_out) return QSA_ERR_INVALID_ARG;
  if (q_idx == q_out) return QSA_ERR_INVALID_ARG;  // not in place
  if ((rc = check_mrope_call(pre, nullptr, rows, nullptr)) != QSA_OK) return rc;
  const Shape sh = make_shape(cfg);
  return cuda_status(launch_pre_index_q(sh, rows->n_seq, rows->rows_per_seq, rows->pos0,
                                        pre_args(pre, nullptr, nullptr, rows, nullptr), q_idx, q_out, false,
                                        stream));
}

int qsa_decode_pre(const qsa_config *cfg, const qsa_pre_indexer *pre, const qsa_rows *rows,
                   const qsa_cache *cache, const qsa_bf16 *k_new, const qsa_bf16 *v_new,
                   const qsa_bf16 *idx_k_new, const qsa_bf16 *q_idx, const float *w, const qsa_bf16 *q,
                   int32_t *sel_out, int32_t *n_sel_out, qsa_bf16 *out, void *ws, size_t ws_bytes,
                   int32_t *status, cudaStream_t stream) {
  int rc;
  if ((rc = check_cfg(cfg)) != QSA_OK) return rc;
  if ((rc = check_pre(cfg, pre, true, true)) != QSA_OK) return rc;
  return decode_impl(cfg, pre, nullptr, rows, cache, k_new, v_new, idx_k_new, q_idx, w, q, sel_out, n_sel_out, out,
                     ws, ws_bytes, status, stream);
}

size_t qsa_workspace_bytes_ex(const qsa_config *cfg, int max_rows, int max_blocks_per_row) {
  if (check_cfg(cfg) != QSA_OK || max_rows < 0 || max_blocks_per_row < 0) return 0;
  const Shape sh = make_shape(cfg);
  const WsLayout L = ws_layout(sh, max_rows, ld_for(max_blocks_per_row));
  return L.total + round_up(q_prep_bytes(sh, max_rows), 256) + round_up(q_main_bytes(sh, max_rows), 256);
}

int qsa_append_ex(const qsa_config *cfg, const qsa_pre_indexer *pre, const qsa_attn_options *attn,
                  const qsa_rows *rows, const qsa_cache *cache, const qsa_bf16 *k_new, const qsa_bf16 *v_new,
                  const qsa_bf16 *idx_k_new, int32_t *status, cudaStream_t stream) {
  int rc;
  if ((rc = check_cfg(cfg)) != QSA_OK) return rc;
  if (pre && (rc = check_pre(cfg, pre, false, true)) != QSA_OK) return rc;
  if ((rc = check_attn(attn)) != QSA_OK) return rc;
  if ((rc = check_rows(rows)) != QSA_OK) return rc;
  if ((rc = check_cache(cache, true, true)) != QSA_OK) return rc;
  if (!cache->ingested || !status) return QSA_ERR_INVALID_ARG;
  const long long n_rows = static_cast<long long>(rows->n_seq) * rows->rows_per_seq;
  if (n_rows == 0) return QSA_OK;
  if (!k_new || !v_new || !idx_k_new || !aligned16(k_new) || !aligned16(v_new) || !aligned16(idx_k_new))
    return QSA_ERR_INVALID_ARG;
  if ((rc = check_mrope_call(pre, attn, rows, cache)) != QSA_OK) return rc;
  if ((rc = host_capacity_check(rows, cache, cfg->page_size)) != QSA_OK) return rc;
  const Shape sh = make_shape(cfg);
  PreArgs pa;
  if (pre) pa = pre_args(pre, nullptr, nullptr, rows, cache);
  AttnPrep ap;
  if (attn) ap = attn_prep(attn, nullptr, nullptr, rows);  // keys only
  cudaError_t e = launch_append(sh, rows->n_seq, rows->rows_per_seq, rows->seq_ids, rows->pos0,
                                cache->page_table, cache->max_pages, cache->num_pages,
                                cache->k_pool, cache->v_pool, cache->idxraw_pool, cache->idxblk_pool,
                                cache->ingested, k_new, v_new, idx_k_new, status, false, stream, &pa,
                                attn ? &ap : nullptr);
  if (e == cudaSuccess)
    e = launch_commit(rows->n_seq, rows->rows_per_seq, cache->max_pages * cfg->page_size,
                      rows->seq_ids, rows->pos0, cache->ingested, rows->advance, false, stream);
  return cuda_status(e);
}

int qsa_decode_ex(const qsa_config *cfg, const qsa_pre_indexer *pre, const qsa_attn_options *attn,
                  const qsa_rows *rows, const qsa_cache *cache, const qsa_bf16 *k_new, const qsa_bf16 *v_new,
                  const qsa_bf16 *idx_k_new, const qsa_bf16 *q_idx, const float *w, const qsa_bf16 *q,
                  int32_t *sel_out, int32_t *n_sel_out, qsa_bf16 *out, void *ws, size_t ws_bytes,
                  int32_t *status, cudaStream_t stream) {
  int rc;
  if ((rc = check_cfg(cfg)) != QSA_OK) return rc;
  if (pre && (rc = check_pre(cfg, pre, true, true)) != QSA_OK) return rc;
  if ((rc = check_attn(attn)) != QSA_OK) return rc;
  return decode_impl(cfg, pre, attn, rows, cache, k_new, v_new, idx_k_new, q_idx, w, q, sel_out, n_sel_out, out,
                     ws, ws_bytes, status, stream);
}

int qsa_gather_attn_reuse(const qsa_config *cfg, const qsa_rows *rows, const qsa_cache *cache,
                          const qsa_bf16 *q, const int32_t *sel, const int32_t *n_sel,
                          const int32_t *sel_pos, qsa_bf16 *out, void *ws, size_t ws_bytes,
                          int32_t *status, cudaStream_t stream) {
  int rc;
  if ((rc = check_cfg(cfg)) != QSA_OK) return rc;
  if ((rc = check_rows(rows)) != QSA_OK) return rc;
  if ((rc = check_cache(cache, true, false)) != QSA_OK) return rc;
  const int n_rows = rows->n_seq * rows->rows_per_seq;
  if (n_rows == 0) return QSA_OK;
  if (!q || !sel || !n_sel || !sel_pos || !out || !ws || !aligned16(q) || !aligned16(out) || !aligned16(ws))
    return QSA_ERR_INVALID_ARG;
  const Shape sh = make_shape(cfg);
  if (ws_bytes < attn_partial_bytes(sh, n_rows)) return QSA_ERR_WORKSPACE;
  return cuda_status(launch_attn(sh, rows->n_seq, rows->rows_per_seq, rows->seq_ids, rows->pos0,
                                 view(cache), q, sel, n_sel, out, ws, status, false, CommitArgs{},
                                 stream, sel_pos));
}

int qsa_decode_reuse(const qsa_config *cfg, const qsa_rows *rows, const qsa_cache *cache,
                     const qsa_bf16 *k_new, const qsa_bf16 *v_new, const qsa_bf16 *idx_k_new,
                     const qsa_bf16 *q, const int32_t *sel, const int32_t *n_sel,
                     const int32_t *sel_pos, qsa_bf16 *out, void *ws, size_t ws_bytes,
                     int32_t *status, cudaStream_t stream) {
  int rc;
  if ((rc = check_cfg(cfg)) != QSA_OK) return rc;
  if ((rc = check_rows(rows)) != QSA_OK) return rc;
  if ((rc = check_cache(cache, true, true)) != QSA_OK) return rc;
  if (!cache->ingested || !status) return QSA_ERR_INVALID_ARG;
  const int n_rows = rows->n_seq * rows->rows_per_seq;
  if (n_rows == 0) return QSA_OK;
  if (!k_new || !v_new || !idx_k_new || !q || !sel || !n_sel || !sel_pos || !out || !ws)
    return QSA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(idx_k_new) || !aligned16(q) ||
      !aligned16(out) || !aligned16(ws))
    return QSA_ERR_INVALID_ARG;
  if ((rc = host_capacity_check(rows, cache, cfg->page_size)) != QSA_OK) return rc;
  const Shape sh = make_shape(cfg);
  const int cap_tokens = cache->max_pages * cfg->page_size;
  const WsLayout L = ws_layout(sh, n_rows, ld_for(cap_tokens / cfg->ratio));
  if (ws_bytes < L.total) return QSA_ERR_WORKSPACE;
  const int R = rows->rows_per_seq;
  cudaError_t e = launch_append(sh, rows->n_seq, R, rows->seq_ids, rows->pos0, cache->page_table,
                                cache->max_pages, cache->num_pages, cache->k_pool, cache->v_pool,
                                cache->idxraw_pool, cache->idxblk_pool, cache->ingested, k_new,
                                v_new, idx_k_new, status, true, stream);
  CommitArgs commit;
  commit.n_seq = rows->n_seq;
  commit.R = R;
  commit.capacity = cap_tokens;
  commit.advance = rows->advance;
  commit.seq_ids = rows->seq_ids;
  commit.pos0 = rows->pos0;
  commit.ingested = cache->ingested;
  if (e == cudaSuccess)
    e = launch_attn(sh, rows->n_seq, R, rows->seq_ids, rows->pos0, view(cache), q, sel, n_sel, out,
                    static_cast<uint8_t *>(ws) + L.partials, status, true, commit, stream, sel_pos);
  return cuda_status(e);
}

int qsa_stage_in(void *dst, const void *src, size_t bytes, cudaStream_t stream) {
  if (!dst || !src || !aligned16(dst) || !aligned16(src) || bytes % 16 != 0) return QSA_ERR_INVALID_ARG;
  if (bytes == 0) return QSA_OK;
  // the device's address of the host buffer (the same pointer under unified
  // addressing); a buffer the device cannot reach is refused before any launch
  void *dev_src = nullptr;
  if (cudaHostGetDevicePointer(&dev_src, const_cast<void *>(src), 0) != cudaSuccess || !dev_src) {
    cudaGetLastError();  // the failed lookup leaves no error behind
    return QSA_ERR_INVALID_ARG;
  }
  const size_t n16 = bytes / 16;
  // enough CTAs to keep the C2C link busy, a few pieces each
  const size_t want = (n16 + 4 * kStageThreads - 1) / (4 * kStageThreads);
  const unsigned grid = static_cast<unsigned>(want < 256 ? (want > 0 ? want : 1) : 256);
  return cuda_status(launch_kernel(true, stage_in_kernel, dim3(grid), dim3(kStageThreads), 0, stream,
                                   static_cast<uint4 *>(dst), static_cast<const uint4 *>(dev_src), n16));
}

}  // extern "C"
