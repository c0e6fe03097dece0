// Append, commit and rewind: the per-sequence indexer state.
//
// Append writes the new tokens' K/V rows into the paged KV pools and their raw
// index keys into the raw-key pool, and pools every block the new tokens
// complete ("Agentic shootout", "Flash-Next support: vLLM vs Atlas", (a) item
// 6: one compressed key per complete group of compress_ratio tokens,
// mean-pooled; its page mapping follows the main KV cache). The ingested
// counter is checked before anything is written and advanced by a separate
// commit kernel afterwards, so every CTA of a long append reads the same
// pre-append value ("Atlas Flash-Next defect investigations", Report A,
// Defect 1: decode at pos requires pos == ingested; rewind subtracts the
// dropped tokens).
#include <cuda_fp16.h>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kAppendTokensPerCta = 32;
constexpr int kAppendThreads = 256;
constexpr int kQPrepCtas = 8 * 152;  // query pre-indexing CTAs of one launch, at most

// cos / sin of the RoPE angle pos * theta^(-2i/rot) of pair i. The angle is formed
// in half-turns in double (pos times the pair's frequency from the host) and
// brought to [-1, 1] by subtracting the nearest even integer, which is exact in
// double; only the sine and cosine of that small angle are taken in fp32, so the
// angle itself carries no fp32 rounding at large positions.
__device__ __forceinline__ float2 rope_cs(int pos, int i, const double *half_turns) {
  const double t = static_cast<double>(pos) * half_turns[i];
  const double red = t - 2.0 * rint(0.5 * t);
  float sn, cs;
  sincospif(static_cast<float>(red), &sn, &cs);
  return make_float2(cs, sn);
}

// Interleaved MRoPE: the position NeoX pair ip of a token at (t, h, w) = tp
// turns by: h when ip % 3 == 1 and ip < 3 * sec_h, w when ip % 3 == 2 and
// ip < 3 * sec_w, else t. Plain RoPE is tp = (p, p, p).
__device__ __forceinline__ int pair_pos(int3 tp, int ip, int sec_h, int sec_w) {
  const int m = ip % 3;
  return (m == 1 && ip < 3 * sec_h) ? tp.y : ((m == 2 && ip < 3 * sec_w) ? tp.z : tp.x);
}

// The triple of the call's row `row`, a token at position pos: from the call's
// array with MRoPE on, else (pos, pos, pos) (a text token, or plain RoPE).
__device__ __forceinline__ int3 row_triple(const Mrope &mr, size_t row, int pos) {
  if (!mr.on || !mr.pos) return make_int3(pos, pos, pos);
  const int32_t *p = mr.pos + row * 3;
  return make_int3(p[0], p[1], p[2]);
}

// One warp, one d_I-vector held as lane L: dims L + 32m (m < D32). Gemma RMSNorm
// (gain 1 + gamma, fp32 sum of squares in a fixed shuffle order), then the NeoX
// rotation of pairs (i, i + rot/2), i < rot/2; with rot/2 a multiple of 32 a
// pair lives in one lane. cs(i) gives the pair's (cos, sin).
template <int D32, typename CS>
__device__ __forceinline__ void pre_index_lanes(float (&x)[D32], const float *__restrict__ gamma, float eps,
                                                int rot, int d_idx, int lane, CS cs) {
  float ss = 0.f;
#pragma unroll
  for (int m = 0; m < D32; ++m) ss += x[m] * x[m];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float inv = 1.0f / sqrtf(ss / static_cast<float>(d_idx) + eps);
#pragma unroll
  for (int m = 0; m < D32; ++m) x[m] = x[m] * inv * (1.0f + gamma[lane + 32 * m]);
  const int hm = rot >> 6;  // pairs per lane: (rot / 2) / 32
#pragma unroll
  for (int m = 0; m < D32 / 2; ++m) {
    if (m < hm) {
      const float2 c = cs(lane + 32 * m);
      const float x1 = x[m], x2 = x[m + hm];
      x[m] = x1 * c.x - x2 * c.y;
      x[m + hm] = x2 * c.x + x1 * c.y;
    }
  }
}

// ---- MX planes (OCP MX v1.0: E4M3 or E2M1 elements, one E8M0 scale per 32 values) ----

// One warp holding a d_I vector as lane L: dims L + 32m, so register m across
// the warp is exactly MX block m. x must already be bf16 values. Returns each
// lane's codes (E4M3, or E2M1 with FP4) and every block's scale exponent.
template <int D32, bool FP4 = false>
__device__ __forceinline__ void mx_quantize_lanes(const float (&x)[D32], uint32_t (&code)[D32], int (&ex)[D32]) {
#pragma unroll
  for (int m = 0; m < D32; ++m) {
    const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(x[m]))));
    ex[m] = FP4 ? mx4_scale_exp(amax) : mx_scale_exp(amax);
    const float sc = x[m] * exp2_int(-ex[m]);  // exact power-of-two scaling
    code[m] = FP4 ? e2m1_code(sc) : e4m3_code(sc);
  }
}

// bf16 value of x (round to nearest even) as fp32.
__device__ __forceinline__ float round_bf16(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// One warp, one vector of 32 * D32 values at in[base] -> out[base]: RoPE(Gemma
// RMSNorm) at the triple tp when gamma is set, rounded to bf16, then the MX
// round trip (mx: 1 MXFP8, 2 MXFP4, 0 none).
template <int D32>
__device__ __forceinline__ void prep_vector(const uint16_t *__restrict__ in, uint16_t *__restrict__ out,
                                            size_t base, int3 tp, const Mrope &mr, const float *gamma, float eps,
                                            int rot, const double *half_turns, int mx, int lane) {
  float x[D32];
#pragma unroll
  for (int m = 0; m < D32; ++m) x[m] = bf16_bits_to_float(in[base + lane + 32 * m]);
  if (gamma) {
    pre_index_lanes<D32>(x, gamma, eps, rot, 32 * D32, lane,
                         [&](int ip) { return rope_cs(pair_pos(tp, ip, mr.sec_h, mr.sec_w), ip, half_turns); });
#pragma unroll
    for (int m = 0; m < D32; ++m) x[m] = round_bf16(x[m]);
  }
  if (mx == 1) {
    uint32_t code[D32];
    int ex[D32];
    mx_quantize_lanes<D32>(x, code, ex);
#pragma unroll
    for (int m = 0; m < D32; ++m) x[m] = e4m3_value(code[m]) * exp2_int(ex[m]);  // exact in bf16
  } else if (mx == 2) {
    uint32_t code[D32];
    int ex[D32];
    mx_quantize_lanes<D32, true>(x, code, ex);
#pragma unroll
    for (int m = 0; m < D32; ++m) x[m] = e2m1_value(code[m]) * exp2_int(ex[m]);  // exact in bf16
  }
#pragma unroll
  for (int m = 0; m < D32; ++m) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x[m]);
    out[base + lane + 32 * m] = *reinterpret_cast<const uint16_t *>(&h);
  }
}

// The step's query vectors of sequence i, one warp per vector: first the index
// query heads (pre.q_out set: RoPE(GemmaRMSNorm) with pre.gamma_q, then with the
// MX plane that plane's round trip), then the main query heads (att.q_out set:
// RoPE(GemmaRMSNorm) with att.gamma_q over D). Index vector v is row i*R + v / H_I
// at position p0 + v / H_I; main vectors likewise with Hq. A CTA takes vectors
// slot*8 + warp, striding by n_slots*8, so a decode step's heads spread over CTAs.
__device__ void prep_queries(const Shape &sh, const PreArgs &pre, const AttnPrep &att, int i, int R, int p0,
                             int slot, int n_slots) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, n_warps = blockDim.x >> 5;
  const int n_idx = pre.q_out ? R * sh.h_idx : 0;
  const int n_vec = n_idx + (att.q_out ? R * sh.hq : 0);
  for (int v = slot * n_warps + warp; v < n_vec; v += n_slots * n_warps) {
    if (v < n_idx) {
      const int t = v / sh.h_idx;
      const size_t base = (static_cast<size_t>(i) * R * sh.h_idx + v) * sh.d_idx;
      const int mx = sh.idx_fp8 ? (sh.idx_fp4 ? 2 : 1) : 0;
      const int3 tp = row_triple(pre.mr, static_cast<size_t>(i) * R + t, p0 + t);
      if (sh.d_idx == 128)
        prep_vector<4>(pre.q_in, pre.q_out, base, tp, pre.mr, pre.gamma_q, pre.eps, pre.rot, pre.half_turns, mx,
                       lane);
      else
        prep_vector<2>(pre.q_in, pre.q_out, base, tp, pre.mr, pre.gamma_q, pre.eps, pre.rot, pre.half_turns, mx,
                       lane);
    } else {
      const int vm = v - n_idx;
      const int t = vm / sh.hq;
      const size_t base = (static_cast<size_t>(i) * R * sh.hq + vm) * kHeadDim;
      const int3 tp = row_triple(att.mr, static_cast<size_t>(i) * R + t, p0 + t);
      prep_vector<kHeadDim / 32>(att.q_in, att.q_out, base, tp, att.mr, att.gamma_q, att.eps, att.rot,
                                 att.half_turns, 0, lane);
    }
  }
}

// Query-prep CTAs of one sequence for R rows of n_seq sequences with `heads`
// vectors per row: 8 vectors (one per warp) each, capped so a launch holds at
// most kQPrepCtas of them.
int q_prep_ctas(int heads, int n_seq, int R) {
  const long long want = (static_cast<long long>(R) * heads + 7) / 8;
  const long long cap = kQPrepCtas / n_seq > 1 ? kQPrepCtas / n_seq : 1;
  return static_cast<int>(want < cap ? want : cap);
}

// One warp: the compressed key of block b. Raw keys are summed in position
// order in fp32 (as in the plain pooling), then scaled by 1/r; through the
// pre-indexer when pre.gamma_k is set; rounded to bf16; stored as bf16 tiles or,
// with an MX plane, quantised into it.
template <int D32>
__device__ void pool_block_warp(const Shape &sh, const PreArgs &pre, int b, int i, int R, int p0,
                                const int32_t *__restrict__ ptab, int num_pages,
                                const uint16_t *__restrict__ raw_pool, void *__restrict__ blk_pool,
                                const uint16_t *__restrict__ idx_new, float inv_r, int bpp, int lane,
                                int32_t *status) {
  const int r = sh.ratio, P = sh.page;
  float x[D32];
#pragma unroll
  for (int m = 0; m < D32; ++m) x[m] = 0.f;
  for (int jj = 0; jj < r; ++jj) {
    const int pos = b * r + jj;
    const uint16_t *src;
    if (pos >= p0) {
      src = idx_new + (static_cast<size_t>(i) * R + (pos - p0)) * sh.d_idx;
    } else {
      const int page = ptab[pos >> sh.log2_page];
      if (page < 0 || page >= num_pages) {
        if (lane == 0) report(status, QSA_ERR_PAGE);
        return;
      }
      src = raw_pool + (static_cast<size_t>(page) * P + (pos & (P - 1))) * sh.d_idx;
    }
#pragma unroll
    for (int m = 0; m < D32; ++m) x[m] += bf16_bits_to_float(src[lane + 32 * m]);
  }
  const int page_b = ptab[(b * r) >> sh.log2_page];
  if (page_b < 0 || page_b >= num_pages) {
    if (lane == 0) report(status, QSA_ERR_PAGE);
    return;
  }
#pragma unroll
  for (int m = 0; m < D32; ++m) x[m] *= inv_r;
  const int first = b * r;
  const int rr = b & (bpp - 1);
  if (pre.gamma_k) {
    // RoPE at the block's first token: its triple comes with this call's rows,
    // or was stored beside the page when an earlier call appended it
    int3 tp = make_int3(first, first, first);
    if (pre.mr.on) {
      if (first >= p0) {
        tp = row_triple(pre.mr, static_cast<size_t>(i) * R + (first - p0), first);
      } else if (pre.blkpos) {  // the host requires the pool with an MRoPE section
        const int4 q = reinterpret_cast<const int4 *>(pre.blkpos)[static_cast<size_t>(page_b) * bpp + rr];
        tp = make_int3(q.x, q.y, q.z);
      }
    }
    pre_index_lanes<D32>(x, pre.gamma_k, pre.eps, pre.rot, sh.d_idx, lane, [&](int ip) {
      return rope_cs(pair_pos(tp, ip, pre.mr.sec_h, pre.mr.sec_w), ip, pre.half_turns);
    });
  }
  if (sh.idx_fp4) {
#pragma unroll
    for (int m = 0; m < D32; ++m) x[m] = round_bf16(x[m]);
    uint32_t code[D32];
    int ex[D32];
    mx_quantize_lanes<D32, true>(x, code, ex);
    uint8_t *pg = static_cast<uint8_t *>(blk_pool) + static_cast<size_t>(page_b) * fp4_page_bytes(bpp, sh.d_idx);
#pragma unroll
    for (int m = 0; m < D32; ++m) {
      // dims lane and lane + 1 share a byte: the even lane stores both nibbles
      const uint32_t hi = __shfl_down_sync(0xffffffffu, code[m], 1);
      if ((lane & 1) == 0)
        pg[fp4_byte_offset(rr, lane + 32 * m, sh.d_idx)] = static_cast<uint8_t>(code[m] | (hi << 4));
    }
    if (lane == 0) {
#pragma unroll
      for (int m = 0; m < D32; ++m)
        pg[bpp * sh.d_idx / 2 + rr * (sh.d_idx / 32) + m] = static_cast<uint8_t>(ex[m] + 127);
    }
    return;
  }
  if (sh.idx_fp8) {
#pragma unroll
    for (int m = 0; m < D32; ++m) x[m] = round_bf16(x[m]);
    uint32_t code[D32];
    int ex[D32];
    mx_quantize_lanes<D32>(x, code, ex);
    uint8_t *pg = static_cast<uint8_t *>(blk_pool) + static_cast<size_t>(page_b) * fp8_page_bytes(bpp, sh.d_idx);
#pragma unroll
    for (int m = 0; m < D32; ++m) pg[fp8_elem_offset(rr, lane + 32 * m, sh.d_idx)] = static_cast<uint8_t>(code[m]);
    if (lane == 0) {
#pragma unroll
      for (int m = 0; m < D32; ++m)
        pg[bpp * sh.d_idx + rr * (sh.d_idx / 32) + m] = static_cast<uint8_t>(ex[m] + 127);
    }
    return;
  }
  uint16_t *dst = static_cast<uint16_t *>(blk_pool) + static_cast<size_t>(page_b) * bpp * sh.d_idx;
#pragma unroll
  for (int m = 0; m < D32; ++m) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x[m]);
    dst[blk_elem_offset(rr, lane + 32 * m, bpp, sh.d_idx)] = *reinterpret_cast<const uint16_t *>(&h);
  }
}

__global__ void __launch_bounds__(kAppendThreads)
append_kernel(Shape sh, int R, const int32_t *__restrict__ seq_ids,
              const int32_t *__restrict__ pos0, const int32_t *__restrict__ page_table,
              int max_pages, int num_pages, uint16_t *__restrict__ k_pool,
              uint16_t *__restrict__ v_pool, uint16_t *__restrict__ raw_pool,
              void *__restrict__ blk_pool, const int32_t *__restrict__ ingested,
              const uint16_t *__restrict__ k_new, const uint16_t *__restrict__ v_new,
              const uint16_t *__restrict__ idx_new, int32_t *status, int n_chunks,
              const __grid_constant__ PreArgs pre, const __grid_constant__ AttnPrep att) {
  // the previous step's commit (ingested, pos0) when launched as a dependent; only
  // then may the score kernel start: its prologue reads the positions
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x;
  const int p0 = pos0[i];
  if (static_cast<int>(blockIdx.y) >= n_chunks) {
    // the step's query vectors: index queries (pre.q_out set) and main queries
    // (att.q_out set)
    prep_queries(sh, pre, att, i, R, p0, blockIdx.y - n_chunks, gridDim.y - n_chunks);
    return;
  }
  const int s = seq_ids[i];
  const int P = sh.page;
  const int cap = max_pages * P;
  const bool lead = (threadIdx.x == 0 && blockIdx.y == 0);
  if (ingested[s] != p0) {
    if (lead) report(status, QSA_ERR_DESYNC);
    return;
  }
  if (p0 < 0 || p0 + R > cap) {
    if (lead) report(status, QSA_ERR_CAPACITY);
    return;
  }
  const int32_t *ptab = page_table + static_cast<size_t>(s) * max_pages;
  const int t_begin = blockIdx.y * kAppendTokensPerCta;
  const int t_end = min(R, t_begin + kAppendTokensPerCta);
  if (t_begin >= t_end) return;

  // 1. copy rows: per token, Hkv*D/8 uint4 of K, the same of V, d_I/8 of raw key
  // (K rows that go through the q/k norm are written in 1b instead)
  const int kv16 = sh.hkv * sh.d / 8;
  const int ix16 = sh.d_idx / 8;
  const int per_tok = 2 * kv16 + ix16;
  const int n_work = (t_end - t_begin) * per_tok;
  for (int e = threadIdx.x; e < n_work; e += blockDim.x) {
    const int tl = e / per_tok;
    const int c = e - tl * per_tok;
    if (att.gamma_k && c < kv16) continue;
    const int j = t_begin + tl;
    const int pos = p0 + j;
    const int page = ptab[pos >> sh.log2_page];
    if (page < 0 || page >= num_pages) {
      report(status, QSA_ERR_PAGE);
      continue;
    }
    const size_t slot = static_cast<size_t>(page) * P + (pos & (P - 1));
    const size_t row = static_cast<size_t>(i) * R + j;
    const uint4 *src;
    uint4 *dst;
    if (c < kv16) {
      src = reinterpret_cast<const uint4 *>(k_new + row * kv16 * 8) + c;
      dst = reinterpret_cast<uint4 *>(k_pool + slot * kv16 * 8) + c;
    } else if (c < 2 * kv16) {
      src = reinterpret_cast<const uint4 *>(v_new + row * kv16 * 8) + (c - kv16);
      dst = reinterpret_cast<uint4 *>(v_pool + slot * kv16 * 8) + (c - kv16);
    } else {
      src = reinterpret_cast<const uint4 *>(idx_new + row * ix16 * 8) + (c - 2 * kv16);
      dst = reinterpret_cast<uint4 *>(raw_pool + slot * ix16 * 8) + (c - 2 * kv16);
    }
    *dst = __ldg(src);
  }
  if (pre.mr.on && pre.blkpos) {
    // the triple of every block's first token, beside its page, for the call
    // that completes the block (it may come later)
    const int bpp = P >> sh.log2_ratio;
    for (int j = t_begin + threadIdx.x; j < t_end; j += blockDim.x) {
      const int pos = p0 + j;
      if (pos & (sh.ratio - 1)) continue;
      const int page = ptab[pos >> sh.log2_page];
      if (page < 0 || page >= num_pages) continue;  // reported by the copy above
      const int3 tp = row_triple(pre.mr, static_cast<size_t>(i) * R + j, pos);
      reinterpret_cast<int4 *>(pre.blkpos)[static_cast<size_t>(page) * bpp + ((pos & (P - 1)) >> sh.log2_ratio)] =
          make_int4(tp.x, tp.y, tp.z, 0);
    }
  }

  // 1b. key heads through GemmaRMSNorm + RoPE at the token's position (its
  // triple with MRoPE), one warp per (token, KV head)
  if (att.gamma_k) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, n_warps = blockDim.x >> 5;
    for (int v = warp; v < (t_end - t_begin) * sh.hkv; v += n_warps) {
      const int tl = v / sh.hkv, h = v - tl * sh.hkv;
      const int j = t_begin + tl;
      const int pos = p0 + j;
      const int page = ptab[pos >> sh.log2_page];
      if (page < 0 || page >= num_pages) {
        if (lane == 0) report(status, QSA_ERR_PAGE);
        continue;
      }
      const size_t src = ((static_cast<size_t>(i) * R + j) * sh.hkv + h) * kHeadDim;
      float x[kHeadDim / 32];
#pragma unroll
      for (int m = 0; m < kHeadDim / 32; ++m) x[m] = bf16_bits_to_float(k_new[src + lane + 32 * m]);
      const int3 tp = row_triple(att.mr, static_cast<size_t>(i) * R + j, pos);
      pre_index_lanes<kHeadDim / 32>(x, att.gamma_k, att.eps, att.rot, kHeadDim, lane, [&](int ip) {
        return rope_cs(pair_pos(tp, ip, att.mr.sec_h, att.mr.sec_w), ip, att.half_turns);
      });
      uint16_t *dst = k_pool + ((static_cast<size_t>(page) * P + (pos & (P - 1))) * sh.hkv + h) * kHeadDim;
#pragma unroll
      for (int m = 0; m < kHeadDim / 32; ++m) {
        const __nv_bfloat16 hb = __float2bfloat16_rn(x[m]);
        dst[lane + 32 * m] = *reinterpret_cast<const uint16_t *>(&hb);
      }
    }
  }

  // 2. pool the blocks whose last token is one of this CTA's tokens: block b
  // completes at position b*r + r - 1, so b in [first/r, last/r).
  const int r = sh.ratio;
  const int first_pos = p0 + t_begin;
  const int last_pos = p0 + t_end;
  const int b_lo = first_pos >> sh.log2_ratio;
  const int b_hi = last_pos >> sh.log2_ratio;
  const int half = sh.d_idx / 2;
  const int bpp = P >> sh.log2_ratio;  // blocks per page
  const float inv_r = 1.0f / static_cast<float>(r);
  if (pre.gamma_k || sh.idx_fp8) {
    // one warp per block: mean-pool, (Gemma RMSNorm, RoPE at the block's first
    // position), store as bf16 or into the MX plane
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, n_warps = blockDim.x >> 5;
    for (int bb = warp; bb < b_hi - b_lo; bb += n_warps) {
      const int b = b_lo + bb;
      if (sh.d_idx == 128)
        pool_block_warp<4>(sh, pre, b, i, R, p0, ptab, num_pages, raw_pool, blk_pool, idx_new, inv_r, bpp, lane, status);
      else
        pool_block_warp<2>(sh, pre, b, i, R, p0, ptab, num_pages, raw_pool, blk_pool, idx_new, inv_r, bpp, lane, status);
    }
    return;
  }
  for (int e = threadIdx.x; e < (b_hi - b_lo) * half; e += blockDim.x) {
    const int b = b_lo + e / half;
    const int d2 = (e % half) * 2;
    float s0 = 0.f, s1 = 0.f;
    bool ok = true;
    for (int jj = 0; jj < r; ++jj) {
      const int pos = b * r + jj;
      const uint16_t *src;
      if (pos >= p0) {
        src = idx_new + (static_cast<size_t>(i) * R + (pos - p0)) * sh.d_idx + d2;
      } else {
        const int page = ptab[pos >> sh.log2_page];
        if (page < 0 || page >= num_pages) {
          ok = false;
          break;
        }
        src = raw_pool + (static_cast<size_t>(page) * P + (pos & (P - 1))) * sh.d_idx + d2;
      }
      const uint32_t two = *reinterpret_cast<const uint32_t *>(src);
      s0 += bf16_bits_to_float(static_cast<uint16_t>(two & 0xFFFF));
      s1 += bf16_bits_to_float(static_cast<uint16_t>(two >> 16));
    }
    const int page_b = ptab[(b * r) >> sh.log2_page];
    if (!ok || page_b < 0 || page_b >= num_pages) {
      report(status, QSA_ERR_PAGE);
      continue;
    }
    // d2 is even, so (d2, d2 + 1) are adjacent in the tiled page layout
    uint16_t *dst = static_cast<uint16_t *>(blk_pool) + static_cast<size_t>(page_b) * bpp * sh.d_idx +
                    blk_elem_offset(b & (bpp - 1), d2, bpp, sh.d_idx);
    *reinterpret_cast<uint32_t *>(dst) = pack_bf16(s0 * inv_r, s1 * inv_r);
  }
}

// Standalone query pre-indexing: CTA (i, y) takes query vectors y*8 .. of
// sequence i, striding by gridDim.y*8.
__global__ void __launch_bounds__(kAppendThreads)
pre_index_q_kernel(Shape sh, int R, const int32_t *__restrict__ pos0, const __grid_constant__ PreArgs pre) {
  pdl_wait();  // positions
  pdl_trigger();
  const int i = blockIdx.x;
  const int p0 = pos0 ? pos0[i] : 0;  // no positions: MX round trip only
  prep_queries(sh, pre, AttnPrep{}, i, R, p0, blockIdx.y, gridDim.y);
}

__global__ void commit_kernel(int n_seq, int R, int capacity, const int32_t *__restrict__ seq_ids,
                              int32_t *__restrict__ pos0, int32_t *__restrict__ ingested,
                              int advance) {
  pdl_wait();  // every earlier kernel of the step reads pos0 / ingested
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_seq) return;
  const int s = seq_ids[i];
  const int p0 = pos0[i];
  if (ingested[s] == p0 && p0 >= 0 && p0 + R <= capacity) {
    ingested[s] = p0 + R;
    if (advance) pos0[i] = p0 + R;
  }
}

__global__ void rewind_kernel(int n_seq, const int32_t *__restrict__ seq_ids,
                              const int32_t *__restrict__ n_drop, int32_t *__restrict__ ingested,
                              int32_t *status) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_seq) return;
  const int s = seq_ids[i];
  const int n = n_drop[i];
  const int cur = ingested[s];
  if (n < 0 || n > cur) {
    report(status, QSA_ERR_REWIND);
    return;
  }
  ingested[s] = cur - n;
}

}  // namespace

cudaError_t launch_append(const Shape &sh, int n_seq, int R, const int32_t *seq_ids,
                          const int32_t *pos0, const int32_t *page_table, int max_pages,
                          int num_pages, uint16_t *k_pool, uint16_t *v_pool,
                          uint16_t *idxraw_pool, void *idxblk_pool, const int32_t *ingested,
                          const uint16_t *k_new, const uint16_t *v_new,
                          const uint16_t *idx_k_new, int32_t *status, bool pdl, cudaStream_t st,
                          const PreArgs *pre, const AttnPrep *att) {
  if (n_seq == 0 || R == 0) return cudaSuccess;
  const int n_chunks = (R + kAppendTokensPerCta - 1) / kAppendTokensPerCta;
  const int q_heads = (pre && pre->q_out ? sh.h_idx : 0) + (att && att->q_out ? sh.hq : 0);
  const int n_q = q_heads > 0 ? q_prep_ctas(q_heads, n_seq, R) : 0;
  dim3 grid(n_seq, n_chunks + n_q);
  return launch_kernel(pdl, append_kernel, grid, dim3(kAppendThreads), 0, st, sh, R, seq_ids, pos0, page_table,
                       max_pages, num_pages, k_pool, v_pool, idxraw_pool, idxblk_pool, ingested, k_new, v_new,
                       idx_k_new, status, n_chunks, pre ? *pre : PreArgs{}, att ? *att : AttnPrep{});
}

cudaError_t launch_pre_index_q(const Shape &sh, int n_seq, int R, const int32_t *pos0, const PreArgs &pre,
                               const uint16_t *q_in, uint16_t *q_out, bool pdl, cudaStream_t st) {
  if (n_seq == 0 || R == 0) return cudaSuccess;
  PreArgs p = pre;
  p.q_in = q_in;
  p.q_out = q_out;
  dim3 grid(n_seq, q_prep_ctas(sh.h_idx, n_seq, R));
  return launch_kernel(pdl, pre_index_q_kernel, grid, dim3(kAppendThreads), 0, st, sh, R, pos0, p);
}

cudaError_t launch_commit(int n_seq, int R, int capacity, const int32_t *seq_ids,
                          int32_t *pos0, int32_t *ingested, int advance, bool pdl, cudaStream_t st) {
  if (n_seq == 0 || R == 0) return cudaSuccess;
  return launch_kernel(pdl, commit_kernel, dim3((n_seq + 127) / 128), dim3(128), 0, st, n_seq, R,
                       capacity, seq_ids, pos0, ingested, advance);
}

cudaError_t launch_rewind(int n_seq, const int32_t *seq_ids, const int32_t *n_drop,
                          int32_t *ingested, int32_t *status, cudaStream_t st) {
  if (n_seq == 0) return cudaSuccess;
  rewind_kernel<<<(n_seq + 127) / 128, 128, 0, st>>>(n_seq, seq_ids, n_drop, ingested, status);
  return cudaGetLastError();
}

}  // namespace qsa
