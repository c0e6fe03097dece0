// Sparse GQA attention over the gathered token set, split across CTAs, and
// the merge of the splits ("Agentic shootout", "Flash-Next support: vLLM vs
// Atlas", (a) item 6: sparse paged GQA over the selected token indices, read
// straight from the cache pages; "Flash-Next support: llama.cpp vs Atlas",
// (a) item 3: the incomplete tail block is always visible, and (e) risk 1:
// flash-decode over scattered slots needs a gather + flash pass).
//
// Token set of a row with V visible tokens, n_blk = V/ratio complete blocks
// and n_sel selected blocks (ascending ids in sel): the selected tokens before
// run0, then the run [run0, V), where run0 = n_blk*ratio (the tail), or with an
// always-kept local window of W tokens ("Flash-Next support: llama.cpp vs
// Atlas", (d) adoption plan, phase 2, item 6: the last 128 tokens are kept, a
// union with the top-k set) run0 = min(n_blk*ratio, V - W):
//   slot j <  n_body : token sel[j/ratio]*ratio + j%ratio
//   slot j >= n_body : token run0 + (j - n_body)
// n_body = the selected tokens before run0 (whole blocks, plus the part of a
// selected block that run0 cuts); n_slots = n_body + V - run0 <=
// budget + W + ratio - 1.
//
// A unit of work is one split (a fixed range of kSplitSlots slots) of one row.
// A CTA takes up to kMaxUnitsPerCta units (u = blockIdx.x + k * gridDim.x),
// resolves the slots of all of them to cache rows once, and streams their
// chunks through one pipeline, so the loads of the next unit are in flight
// while the current one finishes. Each stage gathers the K and V rows of kChunk
// slots for all KV heads with 16-byte cp.async (3-stage pipeline) into an
// XOR-swizzled shared tile. Warp w owns KV head
// w % Hkv and a 16-slot sub-tile. Per sub-tile:
//   S^T[16 tok x 8 heads] = K[16 x 128] . Q^T   (tokens on M: m16n8k16 x8)
//   online softmax per head column (exp2, scale folded with log2 e)
//   P^T -> B operand via movmatrix.trans; P split as bf16 hi + bf16 lo so the
//   weights keep ~16 significant bits
//   O^T[128 x 8] += V^T . P^T                   (ldmatrix.trans of V, x16)
// The split writes (m, l, acc) in fp32; the merge kernel combines the splits in
// split order and rounds o = acc / l to bf16.
#include <algorithm>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kAttnThreads = 128;
constexpr int kAttnWarps = 4;
constexpr int kStages = 3;
constexpr int kSplitSlots = 112;  // 7 stages of 16 slots
constexpr int kMaxUnitsPerCta = 4;
// page-table entries a CTA copies to shared memory: one region per distinct
// sequence among its units (two decode rows' 32k-token tables); kept small so
// that two attention CTAs fit on an SM beside a select CTA
constexpr int kPageCache = 1040;
constexpr float kLog2e = 1.4426950408889634f;

template <int HKV>
struct AttnGeom {
  static constexpr int kWarpsPerHead = kAttnWarps / HKV;
  static constexpr int kChunk = 16 * kWarpsPerHead;           // slots per stage
  static constexpr int kThreadsPerSlot = kAttnThreads / kChunk;
  static constexpr int kRowBytes = kHeadDim * 2;              // 256
  static constexpr int kHalfStage = kChunk * HKV * kRowBytes;  // K (or V) bytes per stage
  static constexpr int kStageBytes = 2 * kHalfStage;
};

__device__ __forceinline__ int slot_token(int j, int n_body, int log2r, int r, int run0,
                                          const int32_t *sel_row) {
  return j < n_body ? sel_row[j >> log2r] * r + (j & (r - 1)) : run0 + (j - n_body);
}

// One unit: split `sp` of row `row`, its slot range and token-set layout, and
// where its sequence's page-table row sits in the CTA's page cache (-1: read
// from global memory).
struct AttnUnit {
  int row, sp, seq, visible, n_blk, n_body, run0, slot_lo, slot_hi, n_chunks, pc_off, pc_len;
};

template <int HKV>
__global__ void __launch_bounds__(kAttnThreads)
attn_kernel(Shape sh, int R, int n_units, int n_split, int split_len, const int32_t *__restrict__ seq_ids,
            const int32_t *__restrict__ pos0, CacheView cv, const uint16_t *__restrict__ q,
            const int32_t *__restrict__ sel, const int32_t *__restrict__ n_sel_arr,
            float *__restrict__ part_m, float *__restrict__ part_l, float *__restrict__ part_acc,
            int32_t *status, const int32_t *__restrict__ sel_pos) {
  using G = AttnGeom<HKV>;
  static_assert(kSplitSlots <= kAttnThreads, "one slot-table entry per thread and unit");
  extern __shared__ __align__(128) uint8_t smem[];
  // after the stage buffers: per unit, the cache row (page * P + offset) of
  // every slot of its split, or -1; the page cache; the scratch of the warp
  // combine
  const int table = (split_len + G::kChunk - 1) / G::kChunk * G::kChunk;
  int32_t *slot_row = reinterpret_cast<int32_t *>(smem + kStages * G::kStageBytes);
  int32_t *page_cache = slot_row + kMaxUnitsPerCta * table;
  float *red = reinterpret_cast<float *>(page_cache + kPageCache);
  __shared__ AttnUnit s_unit[kMaxUnitsPerCta];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = warp % HKV;            // KV head of this warp
  const int sub = warp / HKV;          // 16-slot sub-tile of the stage
  const int smem_u = smem_u32(smem);
  const int r = sh.ratio;
  const int P = sh.page;
  const int group = sh.hq / HKV;
  const int nu = min(kMaxUnitsPerCta, (n_units - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                                          static_cast<int>(gridDim.x));

  // ---- before the wait, everything the select kernel does not write: the
  // units' rows and positions, their sequences' page-table rows (copied to the
  // page cache) and the loads of the first unit's query
  if (tid < nu) {
    AttnUnit U;
    const int u = blockIdx.x + tid * gridDim.x;
    U.row = u / n_split;
    U.sp = u - U.row * n_split;
    const int i = U.row / R;
    U.seq = seq_ids[i];
    U.visible = pos0[i] + (U.row - i * R) + 1;
    const bool row_ok = U.visible >= 1 && U.visible <= cv.max_pages * P;
    if (!row_ok && U.sp == 0) report(status, QSA_ERR_CAPACITY);
    U.n_blk = row_ok ? (U.visible >> sh.log2_ratio) : -1;  // -1: nothing to attend
    U.pc_off = -1;
    U.pc_len = 0;
    s_unit[tid] = U;
  }
  __syncthreads();
  if (tid == 0) {  // page-cache room, one region per sequence (its units' longest need), while it lasts
    int used = 0;
    for (int k = 0; k < nu; ++k) {
      if (s_unit[k].n_blk < 0) continue;
      int j = 0;
      while (j < k && !(s_unit[j].n_blk >= 0 && s_unit[j].seq == s_unit[k].seq)) ++j;
      if (j < k) {  // an earlier unit of the same sequence holds the region
        s_unit[k].pc_off = s_unit[j].pc_off;
        continue;
      }
      int need = 0;
      for (int m = k; m < nu; ++m)
        if (s_unit[m].n_blk >= 0 && s_unit[m].seq == s_unit[k].seq)
          need = max(need, (s_unit[m].visible + P - 1) >> sh.log2_page);
      if (used + need <= kPageCache) {
        s_unit[k].pc_off = used;
        s_unit[k].pc_len = need;
        used += need;
      }
    }
  }
  __syncthreads();
  for (int k = 0; k < nu; ++k) {
    const AttnUnit &U = s_unit[k];
    if (U.pc_len == 0) continue;  // not a region's owner
    const int32_t *src = cv.page_table + static_cast<size_t>(U.seq) * cv.max_pages;
    for (int e = tid; e < U.pc_len; e += kAttnThreads) page_cache[U.pc_off + e] = src[e];
  }
  // Q^T fragments (B operand of S^T = K Q^T) of a unit for the warp's 8 heads.
  // The loads are unconditional (a lane past the group reads the group's first
  // head) and mask_q zeroes those lanes' fragments later, so nothing waits on
  // the loads where they are issued.
  auto load_q = [&](int row, uint32_t (&qf)[8][2]) {
    const int hl = lane >> 2;
    const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
        q + (static_cast<size_t>(row) * sh.hq + g * group + (hl < group ? hl : 0)) * kHeadDim);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qf[ks][0] = qrow[ks * 8 + (lane & 3)];
      qf[ks][1] = qrow[ks * 8 + 4 + (lane & 3)];
    }
  };
  auto mask_q = [&](uint32_t (&qf)[8][2]) {
    if ((lane >> 2) >= group) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) qf[ks][0] = qf[ks][1] = 0u;
    }
  };
  uint32_t qf[8][2];
  load_q(s_unit[0].row, qf);

  // ---- the units' slot ranges. A reused selection (sel_pos given) was made by
  // the row at sel_pos[row]: its blocks are complete at that position, and the
  // tail runs from that block boundary to the row ("Flash-Next support: vLLM vs
  // Atlas", (a) item 6, MTP skip_topk; "Flash-Next support: llama.cpp vs Atlas",
  // (a) item 3, shared indexer layers).
  // One warp per unit (every lane computes the same values; lane 0 stores them).
  // Without a local window the ranges read nothing the select kernel writes (the
  // count of a fused step needs no load; a loaded count or a reused selection
  // was written before this step), so they are set before the dependency wait;
  // a window's cut reads the selection, so it waits.
  auto unit_ranges = [&]() {
    if (warp < nu) {
      AttnUnit &U = s_unit[warp];
      bool row_ok = U.n_blk >= 0;
      int n_blk = row_ok ? U.n_blk : 0;
      if (row_ok && sel_pos) {
        const int ps = sel_pos[U.row];
        if (ps < 0 || ps >= U.visible) {
          if (U.sp == 0 && lane == 0) report(status, QSA_ERR_REUSE);
          row_ok = false;
          n_blk = 0;
        } else {
          n_blk = (ps + 1) >> sh.log2_ratio;
        }
      }
      // n_sel_arr == nullptr: the selection was made by this step's select kernel,
      // which takes min(n_blk, K) blocks of every row inside the page table, so
      // the count needs no load (the stores of sel are the only wait)
      const int cap_sel = min(n_blk, sh.topk);
      const int n_sel = row_ok ? (n_sel_arr ? min(max(n_sel_arr[U.row], 0), cap_sel) : cap_sel) : 0;
      int n_body = n_sel * r;
      int run0 = n_blk * r;
      if (row_ok && sh.window > 0 && U.visible - sh.window < run0) {
        run0 = max(U.visible - sh.window, 0);
        // selected blocks starting at or after run0 are a suffix of the ascending
        // list: count them 32 at a time from the end
        const int32_t *sel_row = sel + static_cast<size_t>(U.row) * sh.topk;
        int keep = n_sel;
        for (int top = n_sel - 1; top >= 0; top -= 32) {
          const int idx = top - lane;
          const unsigned late = __ballot_sync(0xffffffffu, idx >= 0 && sel_row[idx] * r >= run0);
          keep -= __popc(late);
          if (late != 0xffffffffu) break;
        }
        n_body = keep * r;
        if (keep > 0) {  // run0 may cut the last selected block before it
          const int b0 = sel_row[keep - 1] * r;
          if (b0 + r > run0) n_body = (keep - 1) * r + (run0 - b0);
        }
      }
      int n_slots = row_ok ? n_body + (U.visible - run0) : 0;
      if (n_slots > n_split * split_len) {  // a reused selection too old for the split plan
        if (U.sp == 0 && lane == 0) report(status, QSA_ERR_REUSE);
        n_slots = n_split * split_len;
      }
      __syncwarp();
      if (lane == 0) {
        U.n_body = n_body;
        U.run0 = run0;
        U.slot_lo = min(n_slots, U.sp * split_len);  // fixed cut: independent of the batch
        U.slot_hi = min(n_slots, U.slot_lo + split_len);
        U.n_chunks = (U.slot_hi - U.slot_lo + G::kChunk - 1) / G::kChunk;
      }
    }
  };
  const bool ranges_early = sh.window == 0;
  if (ranges_early) {
    unit_ranges();
    __syncthreads();
  }
  pdl_wait();  // sel (and a window's cut) come from the select kernel
  pdl_trigger();
  if (!ranges_early) {
    unit_ranges();
    __syncthreads();
  }

  // ---- resolve every slot of every unit to its cache row, all in parallel:
  // the stage loads below need no global lookups. Entries past a split's end
  // (the table covers whole stages) are -1.
  {
    int tok[kMaxUnitsPerCta];
#pragma unroll
    for (int k = 0; k < kMaxUnitsPerCta; ++k) {
      tok[k] = -1;
      if (k < nu && tid < table) {
        const AttnUnit &U = s_unit[k];
        const int j = U.slot_lo + tid;
        if (j < U.slot_hi)
          tok[k] = slot_token(j, U.n_body, sh.log2_ratio, r, U.run0, sel + static_cast<size_t>(U.row) * sh.topk);
      }
    }
#pragma unroll
    for (int k = 0; k < kMaxUnitsPerCta; ++k) {
      if (k < nu && tid < table) {
        const AttnUnit &U = s_unit[k];
        const int j = U.slot_lo + tid;
        int rowidx = -1;
        if (j < U.slot_hi) {
          const int t = tok[k];
          int page = -1;
          if (t >= 0 && t < U.visible)
            page = U.pc_off >= 0 ? page_cache[U.pc_off + (t >> sh.log2_page)]
                                 : cv.page_table[static_cast<size_t>(U.seq) * cv.max_pages + (t >> sh.log2_page)];
          if (page >= 0 && page < cv.num_pages)
            rowidx = page * P + (t & (P - 1));
          else
            report(status, QSA_ERR_PAGE);
        }
        slot_row[k * table + tid] = rowidx;
      }
    }
  }
  __syncthreads();

  // ---- gather of one stage: thread -> (slot, 16 of its 32*HKV 16-byte pieces)
  const uint64_t stream_policy = l2_evict_first();
  const int my_slot = tid / G::kThreadsPerSlot;
  const int my_part = tid % G::kThreadsPerSlot;
  auto load_stage = [&](int unit, int chunk_idx, int buf) {
    const int rowidx = slot_row[unit * table + chunk_idx * G::kChunk + my_slot];
    const uint16_t *kbase = cv.k_pool, *vbase = cv.v_pool;
    int bytes = 0;
    if (rowidx >= 0) {
      const size_t off = static_cast<size_t>(rowidx) * HKV * kHeadDim;
      kbase = cv.k_pool + off;
      vbase = cv.v_pool + off;
      bytes = 16;
    }
    const uint32_t stage = smem_u + buf * G::kStageBytes;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int piece = my_part + G::kThreadsPerSlot * u;  // in [0, 32*HKV)
      const int kv = piece / (16 * HKV);
      const int rem = piece % (16 * HKV);
      const int gg = rem >> 4, c16 = rem & 15;
      const uint16_t *src = (kv ? vbase : kbase) + (bytes ? gg * kHeadDim + c16 * 8 : 0);
      const uint32_t dst = stage + kv * G::kHalfStage + (gg * G::kChunk + my_slot) * G::kRowBytes +
                           ((c16 ^ (my_slot & 7)) << 4);
      cp_async16_stream(dst, src, bytes, stream_policy);
    }
  };
  // the load cursor runs kStages - 1 chunks ahead of the compute, across units
  int lk = 0, lc = 0;
  auto issue_next = [&](int buf) {
    while (lk < nu && lc >= s_unit[lk].n_chunks) {
      ++lk;
      lc = 0;
    }
    if (lk < nu) {
      load_stage(lk, lc, buf);
      ++lc;
    }
  };
#pragma unroll
  for (int st = 0; st < kStages - 1; ++st) {
    issue_next(st);
    cp_async_commit();
  }

  const float scale = kLog2e * rsqrtf(static_cast<float>(kHeadDim));
  int gidx = 0;  // chunks computed so far (all units)
  for (int k = 0; k < nu; ++k) {
    const AttnUnit U = s_unit[k];
    if (k > 0) load_q(U.row, qf);
    mask_q(qf);
    float acc[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[mt][c] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};

    for (int c = 0; c < U.n_chunks; ++c, ++gidx) {
      cp_async_wait<kStages - 2>();
      __syncthreads();
      issue_next((gidx + kStages - 1) % kStages);
      cp_async_commit();
      const int buf = gidx % kStages;
      const uint32_t kt = smem_u + buf * G::kStageBytes + (g * G::kChunk + sub * 16) * G::kRowBytes;
      const uint32_t vt = kt + G::kHalfStage;

      // S^T = K . Q^T
      float sa[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int rr = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int cc = 2 * ks + (lane >> 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kt + rr * G::kRowBytes + ((cc ^ (rr & 7)) << 4), a0, a1, a2, a3);
        mma_bf16(sa, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
      }
      // mask slots past the split's end, scale to the log2 domain
      const int j0 = U.slot_lo + c * G::kChunk + sub * 16 + (lane >> 2);
      const bool v0 = j0 < U.slot_hi, v1 = (j0 + 8) < U.slot_hi;
      float s0 = v0 ? sa[0] * scale : -INFINITY;
      float s1 = v0 ? sa[1] * scale : -INFINITY;
      float s2 = v1 ? sa[2] * scale : -INFINITY;
      float s3 = v1 ? sa[3] * scale : -INFINITY;
      float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
      const float ref0 = mn0 == -INFINITY ? 0.f : mn0;
      const float ref1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = exp2f(m_run[0] - ref0), al1 = exp2f(m_run[1] - ref1);
      const float p0 = exp2f(s0 - ref0), p1 = exp2f(s1 - ref1);
      const float p2 = exp2f(s2 - ref0), p3 = exp2f(s3 - ref1);
      l_run[0] = l_run[0] * al0 + p0 + p2;
      l_run[1] = l_run[1] * al1 + p1 + p3;
      m_run[0] = mn0;
      m_run[1] = mn1;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        acc[mt][0] *= al0;
        acc[mt][1] *= al1;
        acc[mt][2] *= al0;
        acc[mt][3] *= al1;
      }
      // P^T as B operand, hi + lo bf16
      const uint32_t hi_top = pack_bf16(p0, p1), hi_bot = pack_bf16(p2, p3);
      const __nv_bfloat162 ht = *reinterpret_cast<const __nv_bfloat162 *>(&hi_top);
      const __nv_bfloat162 hb = *reinterpret_cast<const __nv_bfloat162 *>(&hi_bot);
      const uint32_t lo_top = pack_bf16(p0 - __low2float(ht), p1 - __high2float(ht));
      const uint32_t lo_bot = pack_bf16(p2 - __low2float(hb), p3 - __high2float(hb));
      const uint32_t bh0 = movmatrix_t(hi_top), bh1 = movmatrix_t(hi_bot);
      const uint32_t bl0 = movmatrix_t(lo_top), bl1 = movmatrix_t(lo_bot);
      // O^T += V^T . P^T
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int tok = (lane & 7) + ((lane >> 4) << 3);
        const int cc = 2 * mt + ((lane >> 3) & 1);
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(vt + tok * G::kRowBytes + ((cc ^ (tok & 7)) << 4), a0, a1, a2, a3);
        mma_bf16(acc[mt], a0, a1, a2, a3, bh0, bh1);
        mma_bf16(acc[mt], a0, a1, a2, a3, bl0, bl1);
      }
    }

#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], o);
      l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], o);
    }

    // ---- combine warps that share a KV head (Hkv < 4), then write the split
    if constexpr (G::kWarpsPerHead > 1) {
      __syncthreads();  // the previous unit's combine has finished reading `red`
      // per warp: m[8], l[8], acc[8 heads][128 dims]
      float *mine = red + warp * (16 + 8 * kHeadDim);
      if (lane < 4) {
        mine[2 * lane] = m_run[0];
        mine[2 * lane + 1] = m_run[1];
        mine[8 + 2 * lane] = l_run[0];
        mine[8 + 2 * lane + 1] = l_run[1];
      }
      __syncthreads();
      float mx[2], scl[2], lsum[2] = {0.f, 0.f};
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const int col = 2 * (lane & 3) + c2;
        float m = -INFINITY;
        for (int w2 = g; w2 < kAttnWarps; w2 += HKV) m = fmaxf(m, red[w2 * (16 + 8 * kHeadDim) + col]);
        mx[c2] = m;
        const float ref = m == -INFINITY ? 0.f : m;
        for (int w2 = g; w2 < kAttnWarps; w2 += HKV) {
          const float *o = red + w2 * (16 + 8 * kHeadDim);
          lsum[c2] += o[8 + col] * exp2f(o[col] - ref);
        }
        scl[c2] = exp2f((c2 ? m_run[1] : m_run[0]) - ref);
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int d0 = mt * 16 + (lane >> 2);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int col = 2 * (lane & 3) + (c & 1);
          const int d = d0 + (c >> 1) * 8;
          mine[16 + col * kHeadDim + d] = acc[mt][c] * scl[c & 1];
        }
      }
      __syncthreads();
      if (sub == 0) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const int d0 = mt * 16 + (lane >> 2);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int col = 2 * (lane & 3) + (c & 1);
            const int d = d0 + (c >> 1) * 8;
            float v = 0.f;
            for (int w2 = g; w2 < kAttnWarps; w2 += HKV) v += red[w2 * (16 + 8 * kHeadDim) + 16 + col * kHeadDim + d];
            acc[mt][c] = v;
          }
        }
        m_run[0] = mx[0];
        m_run[1] = mx[1];
        l_run[0] = lsum[0];
        l_run[1] = lsum[1];
      }
    }
    const size_t base = (static_cast<size_t>(U.row) * n_split + U.sp) * sh.hq + g * group;
    if (sub == 0) {
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const int col = 2 * (lane & 3) + c2;
        if (lane < 4 && col < group) {
          part_m[base + col] = m_run[c2];
          part_l[base + col] = l_run[c2];
        }
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int d0 = mt * 16 + (lane >> 2);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int col = 2 * (lane & 3) + (c & 1);
          if (col < group) part_acc[(base + col) * kHeadDim + d0 + (c >> 1) * 8] = acc[mt][c];
        }
      }
    }
  }
  cp_async_wait<0>();
}

// Split merge: one CTA per (row, KV head), one warp per query head of the KV
// head's group; lane t owns dims 4t .. 4t+3. Up to 32 splits, every load is
// issued before any arithmetic (lane j fetches the running max m and sum l of
// split j, and every lane fetches its dims of all split outputs), so the merge
// costs one memory round trip; the weights 2^(m_s - max) then reach every lane
// by shuffle. More splits are taken 32 at a time. The sums run in split order,
// so the result does not depend on how the splits were scheduled. In the fused
// step the CTA (0, 0) also commits the step (advances ingested, and pos0 when
// asked): every earlier kernel of the step, including the attention kernel this
// one waits for, has finished reading them.
constexpr int kMergeThreads = 256;

__global__ void __launch_bounds__(kMergeThreads)
merge_kernel(int hq, int hkv, int n_split, const float *__restrict__ part_m,
             const float *__restrict__ part_l, const float *__restrict__ part_acc,
             uint16_t *__restrict__ out, CommitArgs cm, const uint16_t *__restrict__ gate) {
  const int row = blockIdx.x, g = blockIdx.y, t = threadIdx.x;
  // the commit's first reads go out before the wait: no kernel of this step
  // writes seq_ids, pos0 or ingested before the commit itself
  const bool committer = cm.n_seq > 0 && row == 0 && g == 0;
  int c_s = 0, c_p = 0, c_ing = 0;
  if (committer && t < cm.n_seq) {
    c_s = cm.seq_ids[t];
    c_p = cm.pos0[t];
    c_ing = cm.ingested[c_s];
  }
  pdl_wait();  // the split partials come from the attention kernel
  pdl_trigger();
  if (committer) {
    if (t < cm.n_seq && c_ing == c_p && c_p >= 0 && c_p + cm.R <= cm.capacity) {
      cm.ingested[c_s] = c_p + cm.R;
      if (cm.advance) cm.pos0[t] = c_p + cm.R;
    }
    for (int i = t + kMergeThreads; i < cm.n_seq; i += kMergeThreads) {
      const int s = cm.seq_ids[i];
      const int p0 = cm.pos0[i];
      if (cm.ingested[s] == p0 && p0 >= 0 && p0 + cm.R <= cm.capacity) {
        cm.ingested[s] = p0 + cm.R;
        if (cm.advance) cm.pos0[i] = p0 + cm.R;
      }
    }
  }
  const int group = hq / hkv;
  const int hl = t >> 5, lane = t & 31;
  if (hl >= group) return;
  const int h = g * group + hl;
  const size_t b0 = static_cast<size_t>(row) * n_split * hq + h;
  const float *acc_base = part_acc + b0 * kHeadDim + lane * 4;
  const size_t acc_step = static_cast<size_t>(hq) * kHeadDim;
  // the first 32 splits' loads all go out before anything waits on them
  float4 v[32];
  int cnt = min(32, n_split);
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (j < cnt) v[j] = __ldg(reinterpret_cast<const float4 *>(acc_base + j * acc_step));
  float m_mine = -INFINITY, l_mine = 0.f;
  if (lane < cnt) {
    m_mine = __ldg(&part_m[b0 + static_cast<size_t>(lane) * hq]);
    l_mine = __ldg(&part_l[b0 + static_cast<size_t>(lane) * hq]);
  }
  float m = m_mine;
  for (int s = lane + 32; s < n_split; s += 32) m = fmaxf(m, __ldg(&part_m[b0 + static_cast<size_t>(s) * hq]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float ref = m == -INFINITY ? 0.f : m;
  float l = 0.f;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < n_split; s0 += 32) {
    if (s0 > 0) {
      cnt = min(32, n_split - s0);
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < cnt) v[j] = __ldg(reinterpret_cast<const float4 *>(acc_base + (s0 + j) * acc_step));
      m_mine = -INFINITY;
      l_mine = 0.f;
      if (lane < cnt) {
        m_mine = __ldg(&part_m[b0 + static_cast<size_t>(s0 + lane) * hq]);
        l_mine = __ldg(&part_l[b0 + static_cast<size_t>(s0 + lane) * hq]);
      }
    }
    const float w = lane < cnt ? exp2f(m_mine - ref) : 0.f;
    l += w * l_mine;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float wj = __shfl_sync(0xffffffffu, w, j);
      if (j < cnt) {
        a.x += wj * v[j].x;
        a.y += wj * v[j].y;
        a.z += wj * v[j].z;
        a.w += wj * v[j].w;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  const float inv = l > 0.f ? 1.f / l : 0.f;
  float4 o = make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
  const size_t off = (static_cast<size_t>(row) * hq + h) * kHeadDim + lane * 4;
  if (gate) {
    // sigmoid output gate, elementwise, before the bf16 rounding ("Flash-Next
    // support: vLLM vs Atlas", (a) item 6, Dataflow bullet)
    const uint2 g = *reinterpret_cast<const uint2 *>(gate + off);
    auto sig = [](uint32_t bits) { return 1.f / (1.f + expf(-__uint_as_float(bits))); };
    o.x *= sig(g.x << 16);
    o.y *= sig(g.x & 0xFFFF0000u);
    o.z *= sig(g.y << 16);
    o.w *= sig(g.y & 0xFFFF0000u);
  }
  uint2 packed;
  packed.x = pack_bf16(o.x, o.y);
  packed.y = pack_bf16(o.z, o.w);
  *reinterpret_cast<uint2 *>(out + off) = packed;
}

struct SplitPlan {
  int n_split, split_len;
};

// Every row is cut into splits of kSplitSlots slots whatever the batch shape, so
// the reduction order of a row (and hence its bf16 output) is the same in
// decode, verify and chunked-prefill form: chunked and single-shot prefill agree
// bit for bit.
SplitPlan plan_splits(const Shape &sh, int rows) {
  (void)rows;
  const int max_slots = sh.budget + sh.window + sh.ratio - 1;
  return {(max_slots + kSplitSlots - 1) / kSplitSlots, kSplitSlots};
}

// Resident CTAs of the attention kernel on the current device (the grid is at
// least this many CTAs when there are enough units, so every CTA stays busy).
template <int HKV>
int attn_resident_ctas(size_t smem) {
  int dev = 0, sms = 0, occ = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, attn_kernel<HKV>, kAttnThreads, smem) != cudaSuccess)
    return 0;
  return sms * occ;
}

template <int HKV>
cudaError_t launch_attn_t(const Shape &sh, int n_seq, int R, const int32_t *seq_ids,
                          const int32_t *pos0, const CacheView &cv, const uint16_t *q,
                          const int32_t *sel, const int32_t *n_sel, uint16_t *out, void *partials,
                          int32_t *status, bool pdl, const CommitArgs &commit, cudaStream_t st,
                          const int32_t *sel_pos, const uint16_t *gate) {
  const int rows = n_seq * R;
  const SplitPlan pl = plan_splits(sh, rows);
  const size_t n_part = static_cast<size_t>(rows) * pl.n_split * sh.hq;
  float *pm = static_cast<float *>(partials);
  float *pl_ = pm + n_part;
  float *pa = pl_ + n_part;
  // per unit a slot table covering whole stages; the page cache; the
  // warp-combine scratch when several warps share a KV head
  const int table = (pl.split_len + AttnGeom<HKV>::kChunk - 1) / AttnGeom<HKV>::kChunk * AttnGeom<HKV>::kChunk;
  const size_t red_bytes = AttnGeom<HKV>::kWarpsPerHead > 1 ? kAttnWarps * (16 + 8 * kHeadDim) * sizeof(float) : 0;
  const size_t smem = kStages * AttnGeom<HKV>::kStageBytes + (kMaxUnitsPerCta * table + kPageCache) * sizeof(int32_t) +
                      red_bytes;
  auto kern = attn_kernel<HKV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long n_units = static_cast<long long>(rows) * pl.n_split;
  long long grid = (n_units + kMaxUnitsPerCta - 1) / kMaxUnitsPerCta;
  grid = std::max<long long>(grid, attn_resident_ctas<HKV>(smem));
  grid = std::min(grid, n_units);
  if (n_units > 0x7fffffff) return cudaErrorInvalidValue;
  e = launch_kernel(pdl, kern, dim3(static_cast<unsigned>(grid)), dim3(kAttnThreads), smem, st, sh, R,
                    static_cast<int>(n_units), pl.n_split, pl.split_len, seq_ids, pos0, cv, q, sel, n_sel, pm,
                    pl_, pa, status, sel_pos);
  if (e != cudaSuccess) return e;
  // The merge always launches as a programmatic dependent: its predecessor is
  // the attention kernel above, whatever launched that, and it reads nothing
  // before its wait that the attention writes, so its launch overlaps the
  // attention's tail instead of following it.
  return launch_kernel(true, merge_kernel, dim3(rows, sh.hkv), dim3(kMergeThreads), 0, st, sh.hq, sh.hkv,
                       pl.n_split, static_cast<const float *>(pm), static_cast<const float *>(pl_),
                       static_cast<const float *>(pa), out, commit, gate);
}

}  // namespace

int attn_splits(const Shape &sh, int rows) { return plan_splits(sh, rows).n_split; }

int attn_max_tokens(const Shape &sh) {
  const SplitPlan pl = plan_splits(sh, 1);
  return pl.n_split * pl.split_len;
}

size_t attn_partial_bytes(const Shape &sh, int rows) {
  // split partials (m, l, acc) of every row
  const size_t parts = static_cast<size_t>(rows) * plan_splits(sh, rows).n_split;
  return parts * sh.hq * (kHeadDim + 2) * sizeof(float);
}

cudaError_t launch_attn(const Shape &sh, int n_seq, int R, const int32_t *seq_ids,
                        const int32_t *pos0, const CacheView &cv, const uint16_t *q,
                        const int32_t *sel, const int32_t *n_sel, uint16_t *out, void *partials,
                        int32_t *status, bool pdl, const CommitArgs &commit, cudaStream_t st,
                        const int32_t *sel_pos, const uint16_t *gate) {
  if (n_seq == 0 || R == 0) return cudaSuccess;
  switch (sh.hkv) {
    case 1: return launch_attn_t<1>(sh, n_seq, R, seq_ids, pos0, cv, q, sel, n_sel, out, partials, status, pdl, commit, st, sel_pos, gate);
    case 2: return launch_attn_t<2>(sh, n_seq, R, seq_ids, pos0, cv, q, sel, n_sel, out, partials, status, pdl, commit, st, sel_pos, gate);
    case 4: return launch_attn_t<4>(sh, n_seq, R, seq_ids, pos0, cv, q, sel, n_sel, out, partials, status, pdl, commit, st, sel_pos, gate);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qsa
