// Internal definitions shared by the libqsa translation units.
//
// Layouts (all row-major, bf16 as 16-bit patterns):
//   k_pool, v_pool  [num_pages][P][Hkv][D]     a token's K (or V) row for all
//                                                KV heads is Hkv*D*2 contiguous bytes
//   idxraw_pool     [num_pages][P][d_I]
//   idxblk_pool     [num_pages][P/ratio * d_I]  shares the page table at 1/ratio density;
//                                                rows tiled in 8 x 8 core matrices (blk_elem_offset)
//                   MXFP8: [num_pages][bpp * (d_I + d_I/32)] bytes, E4M3 elements in
//                   8 x 16-byte core matrices (fp8_elem_offset), then E8M0 scales
//   page_table      [n_slots][max_pages] int32
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/qsa.h"

namespace qsa {

constexpr int kMaxTopK = 2048;
constexpr int kMaxLocalWindow = 16384;  // always-kept local window, tokens
constexpr int kHeadDim = 128;

// Device-side status codes go through a first-error-wins CAS.
__device__ __forceinline__ void report(int32_t *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Offset (in elements) of element (rr, d) of a block-pool page: rows in tiles of
// G = min(blocks per page, 8) rows x 8 values, tiles ordered row-group major,
// then 8-value chunk; inside a tile row-major. For 8 or more blocks per page a
// page is a run of the tensor cores' K-major core matrices (8 rows x 16 bytes).
__host__ __device__ __forceinline__ int blk_elem_offset(int rr, int d, int bpp, int d_idx) {
  const int g = bpp < 8 ? bpp : 8;
  return ((rr / g) * (d_idx >> 3) + (d >> 3)) * (g << 3) + (rr % g) * 8 + (d & 7);
}

// --- pre-indexer ------------------------------------------------------------
// Gemma RMSNorm (gain 1 + gamma, fp32 accumulation) and NeoX RoPE of the index
// queries and of every compressed key ("Agentic shootout", "Flash-Next support:
// vLLM vs Atlas", (a) item 6 and its fused pre-indexer kernel). q_in / q_out:
// when set, the append kernel also pre-indexes the step's query rows.
// half_turns[i]: the frequency of rotary pair i, theta^(-2i/rot), in half-turns
// per position (divided by pi), computed once per call on the host in double.
// Kernels take the block as a __grid_constant__ parameter, so indexing the
// table reads the parameter bank directly.
constexpr int kMaxHalfRot = 64;  // rotary pairs of a head, at most (d_I = 128)
// Interleaved MRoPE (same report, the fused pre-indexer notes: temporal,
// height and width rotary pairs interleave by pair index modulo 3, bounded by
// the height and width sections). A token's position is a triple (t, h, w);
// plain RoPE is the case sec_h = sec_w = 0 with t = the token's position.
struct Mrope {
  bool on = false;               // position triples in use (a section was given)
  int sec_h = 0, sec_w = 0;      // pairs of the height and width sections
  const int32_t *pos = nullptr;  // device [rows][3]: the call's (t, h, w) per row; nullptr: (p, p, p)
};

struct PreArgs {
  const float *gamma_q = nullptr;
  const float *gamma_k = nullptr;
  float eps = 0.f;
  int rot = 0;  // rotary dims: 0, 64 or d_I
  const uint16_t *q_in = nullptr;
  uint16_t *q_out = nullptr;
  Mrope mr;
  int32_t *blkpos = nullptr;  // device [num_pages][P/ratio][4]: (t, h, w) of each block's first token
  double half_turns[kMaxHalfRot] = {};
};

// --- main-attention options -------------------------------------------------
// GemmaRMSNorm + NeoX RoPE of the attention's q heads (into q_out, read by the
// attention kernel) and of the appended k heads (before they enter the K pool),
// over D = 128 ("Agentic shootout", "Flash-Next support: vLLM vs Atlas", (a)
// item 6, Dataflow bullet: GemmaRMSNorm q/k heads, fused QK-norm + RoPE + gate).
// half_turns as in PreArgs (the main attention's own rotary dims).
struct AttnPrep {
  const float *gamma_q = nullptr;
  const float *gamma_k = nullptr;
  float eps = 0.f;
  int rot = 0;
  const uint16_t *q_in = nullptr;
  uint16_t *q_out = nullptr;
  Mrope mr;
  double half_turns[kMaxHalfRot] = {};
};

// --- launch parameter blocks ---------------------------------------------

struct CacheView {
  const int32_t *page_table;
  int max_pages;
  int num_pages;
  const uint16_t *k_pool;
  const uint16_t *v_pool;
  const uint16_t *idxraw_pool;
  const void *idxblk_pool;  // bf16 tiles, or an MX byte plane
};

struct Shape {
  int ratio, budget, topk, h_idx, d_idx, hq, hkv, d, page;
  int log2_ratio, log2_page;
  int idx_fp8;  // compressed keys in an MX plane (index queries rounded through it)
  int idx_fp4;  // ... and that plane is MXFP4 (E2M1 elements) rather than MXFP8
  int window;   // always-kept local window: the last `window` tokens of every row (0: none)
};

// --- MXFP8 block-pool pages --------------------------------------------------
// A page holds bpp = P/ratio blocks (bpp >= 8): bpp * d_I E4M3 bytes, element
// (rr, d) at fp8_elem_offset (core matrices of 8 blocks x 16 bytes, the K-major
// order of an 8-bit operand), then bpp * d_I/32 E8M0 scale bytes, scale (rr, c)
// at bpp * d_I + rr * d_I/32 + c.
__host__ __device__ __forceinline__ int fp8_elem_offset(int rr, int d, int d_idx) {
  return ((rr >> 3) * (d_idx >> 4) + (d >> 4)) * 128 + (rr & 7) * 16 + (d & 15);
}
__host__ __device__ __forceinline__ int fp8_page_bytes(int bpp, int d_idx) { return bpp * (d_idx + d_idx / 32); }

// MXFP4 pages: bpp * d_I / 2 bytes of E2M1 pairs (element d in the low nibble
// when d is even), 32 elements (one MX block) per 16-byte run, runs in 8-block
// groups: element (rr, d) in byte fp4_byte_offset, then the E8M0 scales, scale
// (rr, c) at bpp * d_I / 2 + rr * d_I/32 + c.
__host__ __device__ __forceinline__ int fp4_byte_offset(int rr, int d, int d_idx) {
  return ((rr >> 3) * (d_idx >> 5) + (d >> 5)) * 128 + (rr & 7) * 16 + ((d & 31) >> 1);
}
__host__ __device__ __forceinline__ int fp4_page_bytes(int bpp, int d_idx) { return bpp * (d_idx / 2 + d_idx / 32); }

// 2^e as fp32 for e in [-149, 127] (subnormal below -126): an E8M0 scale byte u
// is 2^(u - 127).
__device__ __forceinline__ float exp2_int(int e) {
  return e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23) : __uint_as_float(1u << (e + 149));
}

// MX scale exponent of a block of 32 values with largest magnitude amax:
// floor(log2 amax) - 8 (8: exponent of E4M3's top binade), at least -127; -127
// when amax is zero or below 2^-126. Read off amax's exponent field.
__device__ __forceinline__ int mx_scale_exp(float amax) {
  const int biased = static_cast<int>(__float_as_uint(amax) >> 23);
  return biased == 0 ? -127 : max(biased - 127 - 8, -127);
}

// E4M3 code of v: nearest-even, magnitudes past 448 saturate to 448.
__device__ __forceinline__ uint32_t e4m3_code(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(v));
  return r & 0xFFu;
}

// Value of an E4M3 code (exact in f16, then fp32).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(code)));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

// x through MXFP8 and back at scale 2^e, in the value domain (FMA-pipe
// arithmetic only): a = |x| / 2^e is below 512 by the scale rule; E4M3's
// quantum is 2^(floor(log2 a) - 3) from 2^-6 up and 2^-9 below it (the
// subnormals); a / quantum (< 16) rounds half to even by adding and removing
// 2^23, and the result clamps to 448 (satfinite). Equal, bit for bit, to
// e4m3_value(e4m3_code(x / 2^e)) * 2^e.
__device__ __forceinline__ float mx_round(float x, int e) {
  const float a = fabsf(x) * exp2_int(-e);
  // exponent field below 3: the difference wraps to a negative float, and fmaxf keeps 2^-9
  const float q = fmaxf(__uint_as_float((__float_as_uint(a) & 0x7F800000u) - (3u << 23)), 0x1p-9f);
  const float inv_q = __uint_as_float((254u << 23) - __float_as_uint(q));
  const float r = __fadd_rn(__fadd_rn(a * inv_q, 0x1p23f), -0x1p23f);
  return copysignf(fminf(r * q, 448.f) * exp2_int(e), x);
}

// MXFP4: scale exponent floor(log2 amax) - 2 (2: E2M1's top binade).
__device__ __forceinline__ int mx4_scale_exp(float amax) {
  const int biased = static_cast<int>(__float_as_uint(amax) >> 23);
  return biased == 0 ? -127 : max(biased - 127 - 2, -127);
}

// E2M1 code (sign << 3 | magnitude code 0..7) of v: nearest-even on
// {0, 0.5, 1, 1.5, 2, 3, 4, 6}, magnitudes past 6 clamped. Each midpoint goes to
// the even code: <= 0.25 -> 0, < 0.75 -> 1, <= 1.25 -> 2, < 1.75 -> 3,
// <= 2.5 -> 4, < 3.5 -> 5, <= 5 -> 6, else 7.
__device__ __forceinline__ uint32_t e2m1_code(float v) {
  const float a = fabsf(v);
  const uint32_t m = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) + (a > 5.f);
  return ((__float_as_uint(v) >> 31) << 3) | m;  // the sign kept, a zero's too
}

// Value of an E2M1 magnitude code 0..7 (with the sign bit 8).
__device__ __forceinline__ float e2m1_value(uint32_t code) {
  const uint32_t m = code & 7u;
  const float mag = m < 2 ? 0.5f * m : __uint_as_float(static_cast<uint32_t>(126 + (m >> 1)) << 23) * (1.f + 0.5f * (m & 1));
  return code & 8u ? -mag : mag;
}

// x through MXFP4 and back, given its block's scale exponent e (exact in bf16).
// x through MXFP4 and back at scale 2^e, in the value domain (no code):
// a = |x| / 2^e is below 8 by the scale rule; the E2M1 quantum is 0.5 below 2,
// 1 in [2, 4) and 2 above, so rintf's ties-to-even land on the even code at
// every midpoint; magnitudes past 6 clamp to 6. Equal, bit for bit and sign of
// zero included, to e2m1_value(e2m1_code(x / 2^e)) * 2^e.
__device__ __forceinline__ float mx4_round(float x, int e) {
  const float a = fabsf(x) * exp2_int(-e);
  const float q = a < 2.f ? 0.5f : (a < 4.f ? 1.f : 2.f);
  const float inv_q = a < 2.f ? 2.f : (a < 4.f ? 1.f : 0.5f);
  return copysignf(fminf(rintf(a * inv_q) * q, 6.f) * exp2_int(e), x);
}

// --- PTX wrappers ---------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy global -> shared; src_bytes = 0 fills the 16 bytes with zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
// L2 policy for data read once per step (the gathered K/V rows, the compressed
// keys): evicted first, so that what the step re-reads (page tables, scores,
// selections, split partials) and the kernels' code stay in L2 across steps.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
  return p;
}
__device__ __forceinline__ void cp_async16_stream(uint32_t dst, const void *src, int src_bytes,
                                                  uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                          uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose an 8x8 b16 matrix held in the standard fragment layout
// (thread t holds row t/4, columns 2*(t%4), 2*(t%4)+1).
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(a));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Order-preserving map of an fp32 score to uint32 (larger score -> larger key);
// -0 is folded onto +0 first so that the two compare equal.
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(s + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// --- programmatic dependent launch ----------------------------------------
// Inside the fused step every kernel is launched with programmatic stream
// serialization: it may start while its predecessor is still draining, runs its
// independent prologue, and waits (griddepcontrol.wait) before reading anything
// its predecessor writes. A kernel lets its successor launch only after its own
// wait has returned, so a prologue may read what the kernel two back wrote (the
// score kernel's prologue reads the positions the previous step's merge
// committed), and a kernel never overlaps one that is two back. Outside a
// programmatic launch the wait returns at once.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  // every kernel of the library asks for the largest shared-memory carveout, so an
  // SM that runs one of them can take a CTA of the next without first draining
  // to change its L1 / shared-memory split
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// The same with a thread-block cluster of cluster_x CTAs along x (grid.x a
// multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_cluster(bool pdl, int cluster_x, void (*kern)(KArgs...), dim3 grid, dim3 block,
                                  size_t smem, cudaStream_t st, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster_x;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// --- launchers (defined in the .cu files, called by the C entry points) ----
// pdl: launch as a programmatic dependent of the previous kernel on the stream

cudaError_t launch_append(const Shape &sh, int n_seq, int R, const int32_t *seq_ids,
                          const int32_t *pos0, const int32_t *page_table, int max_pages,
                          int num_pages, uint16_t *k_pool, uint16_t *v_pool,
                          uint16_t *idxraw_pool, void *idxblk_pool, const int32_t *ingested,
                          const uint16_t *k_new, const uint16_t *v_new,
                          const uint16_t *idx_k_new, int32_t *status, bool pdl, cudaStream_t st,
                          const PreArgs *pre = nullptr, const AttnPrep *att = nullptr);
// query rows [rows, H_I, d_I] -> RoPE(GemmaRMSNorm) at each row's position
cudaError_t launch_pre_index_q(const Shape &sh, int n_seq, int R, const int32_t *pos0, const PreArgs &pre,
                               const uint16_t *q_in, uint16_t *q_out, bool pdl, cudaStream_t st);
cudaError_t launch_commit(int n_seq, int R, int capacity, const int32_t *seq_ids,
                          int32_t *pos0, int32_t *ingested, int advance, bool pdl, cudaStream_t st);
cudaError_t launch_rewind(int n_seq, const int32_t *seq_ids, const int32_t *n_drop,
                          int32_t *ingested, int32_t *status, cudaStream_t st);
cudaError_t launch_score(const Shape &sh, int n_seq, int R, const int32_t *seq_ids,
                         const int32_t *pos0, const CacheView &cv, const uint16_t *q_idx,
                         const float *w, float *scores, int ld_scores, int32_t *status, bool pdl,
                         cudaStream_t st, bool q_in_step = false);
bool score_tc_supported(const Shape &sh);
cudaError_t launch_score_tc(const Shape &sh, int n_seq, int R, const int32_t *seq_ids,
                            const int32_t *pos0, const CacheView &cv, const uint16_t *q_idx,
                            const float *w, float *scores, int ld, int32_t *status, bool pdl,
                            cudaStream_t st, bool q_in_step = false);
cudaError_t launch_select(const Shape &sh, int n_seq, int R, const int32_t *pos0,
                          const float *scores, int ld_scores, int32_t *sel, int32_t *n_sel,
                          int max_blocks, int cap_tokens, int32_t *status, bool pdl,
                          cudaStream_t st);
int attn_splits(const Shape &sh, int rows);
size_t attn_partial_bytes(const Shape &sh, int rows);
// The step's counter commit, folded into the last kernel of the fused step
// (n_seq == 0: nothing to commit).
struct CommitArgs {
  int n_seq = 0;
  int R = 0;
  int capacity = 0;
  int advance = 0;
  const int32_t *seq_ids = nullptr;
  int32_t *pos0 = nullptr;
  int32_t *ingested = nullptr;
};
// sel_pos (optional, device [rows]): the selection is reused from the row at that
// position (its tail starts at that position's block boundary)
cudaError_t launch_attn(const Shape &sh, int n_seq, int R, const int32_t *seq_ids,
                        const int32_t *pos0, const CacheView &cv, const uint16_t *q,
                        const int32_t *sel, const int32_t *n_sel, uint16_t *out, void *partials,
                        int32_t *status, bool pdl, const CommitArgs &commit, cudaStream_t st,
                        const int32_t *sel_pos = nullptr, const uint16_t *gate = nullptr);
// tokens a row's attention can take (splits x split length)
int attn_max_tokens(const Shape &sh);

// Host-side argument checks and conversions of the entry points
// (qsa_api.cu), shared so that every entry point validates alike.
bool aligned16(const void *p);
int check_cfg(const qsa_config *c);
Shape make_shape(const qsa_config *c);
int check_rows(const qsa_rows *r);
int check_cache(const qsa_cache *c, bool need_kv, bool need_idx);
CacheView view(const qsa_cache *c);
// QSA_OK, QSA_ERR_CUDA (a non-sticky error, cleared) or QSA_ERR_CUDA_FATAL
// (a sticky error: the context is lost).
int cuda_status(cudaError_t e);

}  // namespace qsa
