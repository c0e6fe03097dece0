// Top-K block selection ("Agentic shootout", "Flash-Next support: vLLM vs
// Atlas", (a) item 6: block top-k of budget/compress_ratio groups; "PR 16
// review ... (Claude's review)", (a): top-512 + tail, inert below
// budget + ratio - 1 visible tokens).
//
// Scores become order-preserving uint32 keys (-0 folded onto +0), each taken
// relative to the row's smallest key so that the radix digits span exactly the
// range the row covers. Digits are 11 bits, most significant first: a pass
// histograms the keys that match the prefix fixed so far and a block-wide
// suffix scan finds the digit that holds the K-th largest key. Once the chosen
// digit holds at most 128 keys, they are gathered into a candidate list that
// all warps rank at once. The K-th largest key T is then exact, and so is the
// number of ties at T that must be taken. A stable compaction emits, in
// ascending block order, every block with key > T and the lowest-indexed blocks
// with key == T: exactly the top-K under (score desc, index asc).
//
// Layouts, by the longest row of a launch:
//   * one CTA per row, keys in registers (each thread a run of consecutive
//     blocks, plus one block of the row's tail just past a layout's size), up to
//     16k blocks; further digits by passes over each thread's own keys;
//   * past 9216 blocks, when they fit on the GPU at once, a thread-block cluster
//     of 2 or 4 CTAs per row, each holding a part of the row in registers and
//     exchanging ranges, histograms and candidates through distributed shared
//     memory;
//   * one CTA per row with runs of 32 keys (16 in registers, 16 in a padded
//     shared-memory copy of the row) up to 32k blocks;
//   * longer rows staged in shared memory (or, past that, read from global
//     memory) with candidate lists refined by passes over the list.
// The selection stays on the device, so a step that contains it can be
// captured in a CUDA graph.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;  // <= 32: the scan keeps one total per lane
constexpr int kMaxSmemKeys = 48 * 1024 - 4096;  // keys held on chip (176 KB) ...
constexpr int kCandMax = 4096;                   // ... plus the candidate list (16 KB)
constexpr int kDirectMax = 128;  // candidate lists this short are ranked directly
static_assert(kDirectMax <= 4 * kSelWarps && kDirectMax <= 4 * 32, "each warp ranks 4 candidates, each lane holds 4");
constexpr int kDigit = 11;
constexpr int kBins = 1 << kDigit;
constexpr int kBinsPerThread = kBins / kSelThreads;
constexpr int kBatch = 8;  // keys a thread loads before it histograms them

// Inclusive prefix sum over a warp.
__device__ __forceinline__ int warp_incl_scan_sel(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// Exclusive prefix sums over the CTA, with one barrier: each warp scans its
// lanes with shuffles and takes the sum of the warp totals below it with one
// warp reduction (and, when `total` is given, the CTA's sum with another), so
// no warp rescans the totals. Two calls must be separated by a barrier (the
// next call overwrites `tmp`).
__device__ __forceinline__ int block_exclusive_scan1(int v, int *tmp, int *total = nullptr) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int x = warp_incl_scan_sel(v, lane);
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  const int t = lane < kSelWarps ? tmp[lane] : 0;
  const int before = __reduce_add_sync(0xffffffffu, lane < warp ? t : 0);
  if (total) *total = __reduce_add_sync(0xffffffffu, t);
  return before + x - v;
}

// The same for a pair of counts.
__device__ __forceinline__ int2 block_exclusive_scan2(int2 v, int2 *tmp, int2 *total = nullptr) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int2 x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int yx = __shfl_up_sync(0xffffffffu, x.x, o);
    const int yy = __shfl_up_sync(0xffffffffu, x.y, o);
    if (lane >= o) {
      x.x += yx;
      x.y += yy;
    }
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  const int2 t = lane < kSelWarps ? tmp[lane] : make_int2(0, 0);
  const int2 before = make_int2(__reduce_add_sync(0xffffffffu, lane < warp ? t.x : 0),
                                __reduce_add_sync(0xffffffffu, lane < warp ? t.y : 0));
  if (total) *total = make_int2(__reduce_add_sync(0xffffffffu, t.x), __reduce_add_sync(0xffffffffu, t.y));
  return make_int2(before.x + x.x - v.x, before.y + x.y - v.y);
}

// After a histogram pass (hist filled, then a barrier): the digit that holds
// the remaining-th largest key. Thread t owns the kBinsPerThread digits below
// kBins - kBinsPerThread * t; a suffix scan from the top digit finds it. Updates
// prefix / mask / remaining, leaves the digit's key count in s_res[2] and `hist`
// all zero.
__device__ __forceinline__ void digit_search(int shift, uint32_t dmask, uint32_t &prefix, uint32_t &mask,
                                             int &remaining, int *hist, int2 *scan_tmp, int *s_res) {
  const int top_bin = kBins - 1 - kBinsPerThread * threadIdx.x;
  int c[kBinsPerThread];
  int sum = 0;
#pragma unroll
  for (int j = 0; j < kBinsPerThread; ++j) {
    c[j] = hist[top_bin - j];
    hist[top_bin - j] = 0;  // only this thread reads these bins
    sum += c[j];
  }
  int above = block_exclusive_scan1(sum, reinterpret_cast<int *>(scan_tmp));
#pragma unroll
  for (int j = 0; j < kBinsPerThread; ++j) {
    if (above < remaining && remaining <= above + c[j]) {
      s_res[0] = top_bin - j;
      s_res[1] = above;
      s_res[2] = c[j];
    }
    above += c[j];
  }
  __syncthreads();
  prefix |= static_cast<uint32_t>(s_res[0]) << shift;
  mask |= dmask << shift;
  remaining -= s_res[1];
}

// The remaining-th largest of a short candidate list (nc <= kDirectMax keys in
// shared memory): warp w ranks candidates w, w + 32, ... against the whole list
// (each lane holding up to four of its entries), so the ranking costs one pass
// over four registers and a warp reduction. The candidate that has fewer than
// `remaining` entries above it and at least that many at or above it is the
// threshold; equal candidates agree, so any of their warps may write it. Ends
// with a barrier; returns the threshold and the ties at it to take.
__device__ __forceinline__ void rank_candidates(const uint32_t *cand, int nc, uint32_t &thr, int &remaining,
                                                int *s_res) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t v[4];
  bool ok[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    ok[k] = lane + 32 * k < nc;
    v[k] = ok[k] ? cand[lane + 32 * k] : 0u;
  }
#pragma unroll
  for (int i = 0; i < kDirectMax / kSelWarps; ++i) {
    const int ci = warp + kSelWarps * i;  // warp-uniform
    if (ci < nc) {
      const uint32_t c = cand[ci];
      int ge = 0;  // (entries above c) << 16 | (entries equal to c); both <= 128
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (ok[k]) ge += (v[k] > c ? 0x10000 : 0) + (v[k] == c ? 1 : 0);
      ge = __reduce_add_sync(0xffffffffu, ge);
      const int g = ge >> 16, e = ge & 0xffff;
      if (lane == 0 && g < remaining && remaining <= g + e) {
        s_res[0] = static_cast<int>(c);
        s_res[1] = remaining - g;
      }
    }
  }
  __syncthreads();
  thr = static_cast<uint32_t>(s_res[0]);
  remaining = s_res[1];
}

// Key sources. Every key is taken relative to the row's smallest key, so the
// radix digits cover the range the row's keys actually span: scores of one row
// share sign and exponent bits, and digits of the raw key would pile most of the
// row into a few histogram bins.
struct SmemKeys {  // keys staged in shared memory
  const uint32_t *p;
  uint32_t base;
  __device__ __forceinline__ uint32_t operator()(int x) const { return p[x] - base; }
  // four keys from a 16-byte aligned position (x a multiple of 4)
  __device__ __forceinline__ uint4 get4(int x) const {
    uint4 v = *reinterpret_cast<const uint4 *>(p + x);
    return make_uint4(v.x - base, v.y - base, v.z - base, v.w - base);
  }
};
struct GlobalScores {  // fp32 scores read from global memory (rows too long for shared memory)
  const float *p;
  uint32_t base;
  __device__ __forceinline__ uint32_t operator()(int x) const { return score_key(p[x]) - base; }
  __device__ __forceinline__ uint4 get4(int x) const {
    const float4 v = *reinterpret_cast<const float4 *>(p + x);
    return make_uint4(score_key(v.x) - base, score_key(v.y) - base, score_key(v.z) - base,
                      score_key(v.w) - base);
  }
};

// One radix pass over a list of keys: histogram of the digit (k >> shift) & dmask
// of the keys matching `prefix` under `mask`, then the digit that holds the
// remaining-th largest key. Updates prefix / mask / remaining. `hist` is all
// zero on entry and is left all zero.
template <typename Src>
__device__ __forceinline__ void radix_pass(Src list, int m, int shift, uint32_t dmask,
                                           uint32_t &prefix, uint32_t &mask, int &remaining,
                                           int *hist, int2 *scan_tmp, int *s_res) {
  const int tid = threadIdx.x;
  for (int base = 0; base < m; base += kBatch * kSelThreads) {  // warp-uniform trip count
    uint32_t k[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int x = base + b * kSelThreads + tid;
      k[b] = x < m ? list(x) : 0u;
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int x = base + b * kSelThreads + tid;
      if (x < m && (k[b] & mask) == prefix) atomicAdd(&hist[(k[b] >> shift) & dmask], 1);
    }
  }
  __syncthreads();
  digit_search(shift, dmask, prefix, mask, remaining, hist, scan_tmp, s_res);
}

// Selection for one row whose keys (relative to the row minimum) span
// [0, range]: the exact K-th largest key, then the stable compaction.
template <typename Src>
__device__ __forceinline__ void select_row(Src src, int n, int K, uint32_t range, uint32_t *cand,
                                           int32_t *out, int *hist, int2 *scan_tmp, int *s_res,
                                           int *s_ncand) {
  const int tid = threadIdx.x, lane = tid & 31;
  int top = range ? 31 - __clz(range) : -1;  // highest bit any key of the row sets
  const uint32_t low_bits = (top >= 31) ? 0xffffffffu : (top >= 0 ? ((2u << top) - 1u) : 0u);
  uint32_t prefix = 0u;
  uint32_t mask = ~low_bits;
  int remaining = K;  // how many of the still-undecided keys must be taken
  if (top >= 0) {
    // first pass over every key of the row
    int width = min(kDigit, top + 1);
    int shift = top + 1 - width;
    radix_pass(src, n, shift, (1u << width) - 1u, prefix, mask, remaining, hist, scan_tmp, s_res);
    top = shift - 1;
    if (top >= 0) {
      // the keys of the chosen digit become a short candidate list (when they fit)
      for (int base = 0; base < n; base += kSelThreads) {
        const int x = base + tid;
        const uint32_t k = x < n ? src(x) : 0u;
        const bool c = x < n && (k & mask) == prefix;
        const unsigned bal = __ballot_sync(0xffffffffu, c);
        int off = 0;
        if (lane == 0 && bal) off = atomicAdd(s_ncand, __popc(bal));
        off = __shfl_sync(0xffffffffu, off, 0);
        const int pos = off + __popc(bal & ((1u << lane) - 1u));
        if (c && pos < kCandMax) cand[pos] = k;
      }
      __syncthreads();
      const int nc = *s_ncand;
      if (nc <= kDirectMax) {
        rank_candidates(cand, nc, prefix, remaining, s_res);
      } else if (nc <= kCandMax) {
        while (top >= 0) {
          width = min(kDigit, top + 1);
          shift = top + 1 - width;
          radix_pass(SmemKeys{cand, 0u}, nc, shift, (1u << width) - 1u, prefix, mask, remaining,
                     hist, scan_tmp, s_res);
          top = shift - 1;
        }
      } else {
        while (top >= 0) {
          width = min(kDigit, top + 1);
          shift = top + 1 - width;
          radix_pass(src, n, shift, (1u << width) - 1u, prefix, mask, remaining, hist, scan_tmp,
                     s_res);
          top = shift - 1;
        }
      }
    }
  }
  const uint32_t thr = prefix;  // the K-th largest key
  const int need = remaining;   // ties at thr to take (>= 1)

  // stable compaction: thread t scans a contiguous chunk (a multiple of 4 keys,
  // read 4 at a time); one scan gives both the keys above thr and the ties
  // before the chunk
  const int chunk = ((n + kSelThreads - 1) / kSelThreads + 3) & ~3;
  const int lo = min(n, tid * chunk), hi = min(n, lo + chunk);
  int gt = 0, eq = 0;
  for (int x = lo; x < hi; x += 4) {
    const uint4 v = src.get4(x);
    const uint32_t d[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (x + j < hi) {
        gt += d[j] > thr;
        eq += d[j] == thr;
      }
    }
  }
  const int2 pre = block_exclusive_scan2(make_int2(gt, eq), scan_tmp);
  int o = pre.x + min(pre.y, need);  // blocks emitted by the chunks before this one
  int tie_rank = pre.y;
  for (int x = lo; x < hi; x += 4) {
    const uint4 v = src.get4(x);
    const uint32_t d[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (x + j >= hi) continue;
      if (d[j] > thr) {
        if (o < K) out[o] = x + j;
        ++o;
      } else if (d[j] == thr) {
        if (tie_rank < need) {
          if (o < K) out[o] = x + j;
          ++o;
        }
        ++tie_rank;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Rows of at most (4 * NV + E) * kSelThreads blocks: thread t holds the keys of
// the 4 * NV consecutive blocks 4NV*t .. 4NV*t + 4NV - 1 in registers for the
// whole selection and, when E = 1, one more block from the row's tail, M + t
// (M = 4 * NV * kSelThreads), so that a row just past a multiple of 4096 blocks
// costs one key more per thread instead of four. Warp reductions use
// redux.sync; while the chosen digit holds more than kDirectMax keys, a further
// pass over the thread's own keys under the prefix fixed so far takes the next
// digit; then the chosen keys are gathered with a shared atomic per thread that
// holds any and ranked by all warps at once; the compaction is one block scan of
// each thread's counts above and at the threshold (packed 16:16; a second word
// for the tail),
// after which every thread writes its own selected blocks in index order (no
// bitmaps, no atomics). Barriers: range 1, histogram 1, digit search 2,
// candidates 1, ranking 1, compaction scan 1.
// ---------------------------------------------------------------------------
template <int NV, int E>
__device__ __forceinline__ void select_in_registers(const float *__restrict__ srow, int n, int K,
                                                    int32_t *__restrict__ out, uint32_t *cand, int *hist, int2 *scan_tmp, int *s_res,
                                                    int *s_ncand, uint32_t *red_min, uint32_t *red_max) {
  static_assert(E == 0 || E == 1, "at most one tail key per thread");
  constexpr int NR = 4 * NV;   // keys of the contiguous run
  constexpr int NK = NR + E;   // keys held
  constexpr int M = NR * kSelThreads;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int x0 = NR * tid;  // first block of this thread's run
  // 16-byte loads: ld is a multiple of 4, so a group that starts below n lies in the row
  const float4 *s4 = reinterpret_cast<const float4 *>(srow) + NV * tid;
  uint32_t d[NK];
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
    if (x0 + 4 * v < n) f = s4[v];
    d[4 * v] = score_key(f.x);
    d[4 * v + 1] = score_key(f.y);
    d[4 * v + 2] = score_key(f.z);
    d[4 * v + 3] = score_key(f.w);
  }
  if (E == 1) d[NK - 1] = M + tid < n ? score_key(srow[M + tid]) : 0u;
  // the block index of key j
  auto blk = [&](int j) { return j < NR ? x0 + j : M + tid; };
  auto valid = [&](int j) { return blk(j) < n; };
  uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
  for (int j = 0; j < NK; ++j)
    if (valid(j)) {
      kmin = min(kmin, d[j]);
      kmax = max(kmax, d[j]);
    }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0) {
    red_min[warp] = kmin;
    red_max[warp] = kmax;
  }
  __syncthreads();
  kmin = __reduce_min_sync(0xffffffffu, lane < kSelWarps ? red_min[lane] : 0xffffffffu);
  kmax = __reduce_max_sync(0xffffffffu, lane < kSelWarps ? red_max[lane] : 0u);
#pragma unroll
  for (int j = 0; j < NK; ++j) d[j] -= kmin;  // invalid entries are never read

  const uint32_t range = kmax - kmin;
  int top = range ? 31 - __clz(range) : -1;
  const uint32_t low_bits = (top >= 31) ? 0xffffffffu : (top >= 0 ? ((2u << top) - 1u) : 0u);
  uint32_t prefix = 0u;
  uint32_t mask = ~low_bits;
  int remaining = K;
  while (top >= 0) {
    // a pass over the keys under the prefix: histogram of the next digit
    const int width = min(kDigit, top + 1);
    const int shift = top + 1 - width;
    const uint32_t dmask = (1u << width) - 1u;
#pragma unroll
    for (int j = 0; j < NK; ++j)
      if (valid(j) && (d[j] & mask) == prefix) atomicAdd(&hist[(d[j] >> shift) & dmask], 1);
    __syncthreads();
    digit_search(shift, dmask, prefix, mask, remaining, hist, scan_tmp, s_res);  // leaves hist zero
    top = shift - 1;
    if (top < 0) break;  // the prefix is the whole key: the threshold
    if (s_res[2] <= kDirectMax) {
      // the keys of the chosen digit, in any order (only their values are
      // ranked): usually a few threads hold one or two, so each of those
      // reserves its slots with its own shared atomic
      uint32_t member = 0u;
#pragma unroll
      for (int j = 0; j < NK; ++j)
        if (valid(j) && (d[j] & mask) == prefix) member |= 1u << j;
      if (member) {
        int pos = atomicAdd(s_ncand, __popc(member));
#pragma unroll
        for (int j = 0; j < NK; ++j)
          if ((member >> j) & 1u) cand[pos++] = d[j];
      }
      __syncthreads();
      rank_candidates(cand, *s_ncand, prefix, remaining, s_res);
      break;
    }
  }
  const uint32_t thr = prefix;  // the K-th largest key
  const int need = remaining;   // ties at thr to take (>= 1)

  // ---- compaction, in index order: the runs (segment 0), then the tail keys
  // (segment 1, in thread order). The blocks before a key emit the keys above
  // thr before it and the ties before it, capped at `need`. Per thread and
  // segment the counts above and at thr are packed as above | at << 16 (each
  // at most 16 * kSelThreads < 2^16 over the row).
  uint32_t c0 = 0u, c1 = 0u;
#pragma unroll
  for (int j = 0; j < NK; ++j)
    if (valid(j)) {
      const uint32_t c = (d[j] > thr ? 1u : 0u) + (d[j] == thr ? 0x10000u : 0u);
      if (j < NR)
        c0 += c;
      else
        c1 += c;
    }
  uint32_t p0, p1 = 0u;
  if (E == 0) {
    p0 = static_cast<uint32_t>(block_exclusive_scan1(static_cast<int>(c0), reinterpret_cast<int *>(scan_tmp)));
  } else {
    int2 tot;
    const int2 pre = block_exclusive_scan2(make_int2(static_cast<int>(c0), static_cast<int>(c1)), scan_tmp, &tot);
    p0 = static_cast<uint32_t>(pre.x);
    p1 = static_cast<uint32_t>(pre.y) + static_cast<uint32_t>(tot.x);  // after every run
  }
  int o = static_cast<int>(p0 & 0xffffu) + min(static_cast<int>(p0 >> 16), need);
  int tie_rank = static_cast<int>(p0 >> 16);
#pragma unroll
  for (int j = 0; j < NK; ++j) {
    if (j == NR) {  // the tail key: its own place in segment 1
      o = static_cast<int>(p1 & 0xffffu) + min(static_cast<int>(p1 >> 16), need);
      tie_rank = static_cast<int>(p1 >> 16);
    }
    if (!valid(j)) continue;
    if (d[j] > thr) {
      if (o < K) out[o] = blk(j);
      ++o;
    } else if (d[j] == thr) {
      if (tie_rank < need) {
        if (o < K) out[o] = blk(j);
        ++o;
      }
      ++tie_rank;
    }
  }
}

// ---------------------------------------------------------------------------
// Rows of at most (4 * NV + NS) * kSelThreads blocks: thread t holds the run of
// 4 * NV + NS = 32 consecutive blocks starting at 32 t, the first 4 * NV keys in
// registers and the other NS in the row's copy in shared memory (padded so that
// a warp's accesses fall in distinct banks). The selection is the
// register path's: the range, a histogram pass over the top digit, and, while
// the chosen digit holds more than kDirectMax keys, further passes over the
// thread's own keys under the prefix fixed so far; then the chosen keys are
// ranked by all warps and one block scan compacts. The shared-memory keys stay
// raw and are taken relative to the row minimum as they are read.
// ---------------------------------------------------------------------------
template <int NV, int NS>
__device__ __forceinline__ void select_in_runs(const float *__restrict__ srow, int n, int K,
                                               int32_t *__restrict__ out, uint32_t *keys, uint32_t *cand,
                                               int *hist, int2 *scan_tmp, int *s_res, int *s_ncand,
                                               uint32_t *red_min, uint32_t *red_max) {
  constexpr int NR = 4 * NV;  // keys in registers
  constexpr int RUN = NR + NS;
  static_assert(RUN == 32, "a run is one 32-key row of the padded staging layout");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int x0 = RUN * tid;
  // The row goes to shared memory first, read with lane-contiguous 16-byte
  // loads (each thread reading its own run would spread a warp's load over 32
  // lines), at index b + b / 32: thread t's run is then words 33 t .. 33 t + 31,
  // so a warp reading key j of every run touches 32 distinct banks. ld is a
  // multiple of 4, so the 16-byte groups that start below n lie in the row.
  {
    const float4 *r4 = reinterpret_cast<const float4 *>(srow);
    for (int i = tid; 4 * i < n; i += kSelThreads) {
      const float4 f = r4[i];
      const int b = 4 * i;
      keys[b + (b >> 5)] = score_key(f.x);  // b .. b + 3 share one 32-block row
      keys[b + 1 + (b >> 5)] = score_key(f.y);
      keys[b + 2 + (b >> 5)] = score_key(f.z);
      keys[b + 3 + (b >> 5)] = score_key(f.w);
    }
  }
  __syncthreads();
  const uint32_t *ks = keys + 33 * tid;  // this thread's run
  uint32_t d[NR];
  // (only words of the staged row are read: x0 + j < n)
#pragma unroll
  for (int j = 0; j < NR; ++j) d[j] = x0 + j < n ? ks[j] : 0u;
  ks += NR;  // the run's keys kept in shared memory
  auto valid = [&](int j) { return x0 + j < n; };
  uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
  for (int j = 0; j < NR; ++j)
    if (valid(j)) {
      kmin = min(kmin, d[j]);
      kmax = max(kmax, d[j]);
    }
#pragma unroll 4
  for (int j = 0; j < NS; ++j)
    if (valid(NR + j)) {
      const uint32_t k = ks[j];
      kmin = min(kmin, k);
      kmax = max(kmax, k);
    }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0) {
    red_min[warp] = kmin;
    red_max[warp] = kmax;
  }
  __syncthreads();
  kmin = __reduce_min_sync(0xffffffffu, lane < kSelWarps ? red_min[lane] : 0xffffffffu);
  kmax = __reduce_max_sync(0xffffffffu, lane < kSelWarps ? red_max[lane] : 0u);
#pragma unroll
  for (int j = 0; j < NR; ++j) d[j] -= kmin;  // invalid entries are never read
  auto skey = [&](int j) { return ks[j] - kmin; };

  const uint32_t range = kmax - kmin;
  int top = range ? 31 - __clz(range) : -1;
  const uint32_t low_bits = (top >= 31) ? 0xffffffffu : (top >= 0 ? ((2u << top) - 1u) : 0u);
  uint32_t prefix = 0u;
  uint32_t mask = ~low_bits;
  int remaining = K;
  while (top >= 0) {
    // a pass over the keys under the prefix: histogram of the next digit
    const int width = min(kDigit, top + 1);
    const int shift = top + 1 - width;
    const uint32_t dmask = (1u << width) - 1u;
#pragma unroll
    for (int j = 0; j < NR; ++j)
      if (valid(j) && (d[j] & mask) == prefix) atomicAdd(&hist[(d[j] >> shift) & dmask], 1);
#pragma unroll 4
    for (int j = 0; j < NS; ++j) {
      if (!valid(NR + j)) continue;
      const uint32_t k = skey(j);
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & dmask], 1);
    }
    __syncthreads();
    digit_search(shift, dmask, prefix, mask, remaining, hist, scan_tmp, s_res);  // leaves hist zero
    top = shift - 1;
    if (top < 0) break;  // the prefix is the whole key: the threshold
    if (s_res[2] <= kDirectMax) {
      // the keys under the prefix: few, ranked by all warps at once
      int pos = -1;
      uint32_t member = 0u;
#pragma unroll
      for (int j = 0; j < NR; ++j)
        if (valid(j) && (d[j] & mask) == prefix) member |= 1u << j;
      int extra = 0;
#pragma unroll 4
      for (int j = 0; j < NS; ++j) extra += (valid(NR + j) && (skey(j) & mask) == prefix) ? 1 : 0;
      const int mine = __popc(member) + extra;
      if (mine) pos = atomicAdd(s_ncand, mine);
#pragma unroll
      for (int j = 0; j < NR; ++j)
        if ((member >> j) & 1u) cand[pos++] = d[j];
      if (extra) {
        for (int j = 0; j < NS; ++j) {
          if (!valid(NR + j)) continue;
          const uint32_t k = skey(j);
          if ((k & mask) == prefix) cand[pos++] = k;
        }
      }
      __syncthreads();
      rank_candidates(cand, *s_ncand, prefix, remaining, s_res);
      break;
    }
  }
  const uint32_t thr = prefix;  // the K-th largest key
  const int need = remaining;   // ties at thr to take (>= 1)

  // ---- compaction: the blocks before this thread's emit the keys above thr
  // before it and the ties before it, capped at `need` (counts packed 16:16)
  uint32_t c0 = 0u;
#pragma unroll
  for (int j = 0; j < NR; ++j)
    if (valid(j)) c0 += (d[j] > thr ? 1u : 0u) + (d[j] == thr ? 0x10000u : 0u);
#pragma unroll 4
  for (int j = 0; j < NS; ++j)
    if (valid(NR + j)) {
      const uint32_t k = skey(j);
      c0 += (k > thr ? 1u : 0u) + (k == thr ? 0x10000u : 0u);
    }
  const uint32_t p0 =
      static_cast<uint32_t>(block_exclusive_scan1(static_cast<int>(c0), reinterpret_cast<int *>(scan_tmp)));
  int o = static_cast<int>(p0 & 0xffffu) + min(static_cast<int>(p0 >> 16), need);
  int tie_rank = static_cast<int>(p0 >> 16);
  auto emit = [&](uint32_t k, int blk) {
    if (k > thr) {
      if (o < K) out[o] = blk;
      ++o;
    } else if (k == thr) {
      if (tie_rank < need) {
        if (o < K) out[o] = blk;
        ++o;
      }
      ++tie_rank;
    }
  };
#pragma unroll
  for (int j = 0; j < NR; ++j)
    if (valid(j)) emit(d[j], x0 + j);
  for (int j = 0; j < NS; ++j)
    if (valid(NR + j)) emit(skey(j), x0 + NR + j);
}

// Longer rows: keys staged in shared memory (or read from global memory when
// the row does not fit there either).
__device__ __noinline__ void select_general(const float *__restrict__ srow, int n, int K,
                                            int32_t *__restrict__ out, uint32_t *keys, uint32_t *cand,
                                            int smem_keys, int *hist, int2 *scan_tmp, int *s_res,
                                            int *s_ncand, uint32_t *red_min, uint32_t *red_max) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool on_chip = n <= smem_keys;
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  {
    // 16-byte loads: ld is a multiple of 4, so the row start is 16-byte aligned
    const float4 *s4 = reinterpret_cast<const float4 *>(srow);
    const int n4 = n >> 2;
    for (int x = tid; x < n4; x += kSelThreads) {
      const float4 v = s4[x];
      const uint32_t k0 = score_key(v.x), k1 = score_key(v.y), k2 = score_key(v.z), k3 = score_key(v.w);
      if (on_chip) *reinterpret_cast<uint4 *>(keys + 4 * x) = make_uint4(k0, k1, k2, k3);
      kmin = min(kmin, min(min(k0, k1), min(k2, k3)));
      kmax = max(kmax, max(max(k0, k1), max(k2, k3)));
    }
    for (int x = 4 * n4 + tid; x < n; x += kSelThreads) {
      const uint32_t k = score_key(srow[x]);
      if (on_chip) keys[x] = k;
      kmin = min(kmin, k);
      kmax = max(kmax, k);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if (lane == 0) {
    red_min[warp] = kmin;
    red_max[warp] = kmax;
  }
  __syncthreads();
  kmin = lane < kSelWarps ? red_min[lane] : 0xffffffffu;
  kmax = lane < kSelWarps ? red_max[lane] : 0u;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if (on_chip)
    select_row(SmemKeys{keys, kmin}, n, K, kmax - kmin, cand, out, hist, scan_tmp, s_res, s_ncand);
  else
    select_row(GlobalScores{srow, kmin}, n, K, kmax - kmin, cand, out, hist, scan_tmp, s_res, s_ncand);
}

__global__ void __launch_bounds__(kSelThreads)
select_kernel(Shape sh, int R, const int32_t *__restrict__ pos0, const float *__restrict__ scores,
              int ld, int32_t *__restrict__ sel, int32_t *__restrict__ n_sel, int smem_keys,
              int cap_tokens, int32_t *status) {
  // [smem_keys] row keys, then [kCandMax] candidates
  extern __shared__ __align__(16) uint32_t keys[];
  __shared__ int hist[kBins];
  __shared__ int2 scan_tmp[kSelWarps];
  __shared__ uint32_t red_min[kSelWarps], red_max[kSelWarps];
  __shared__ int s_res[3], s_ncand;

  const int row = blockIdx.x;
  const int i = row / R;
  const int visible = pos0[i] + (row - i * R) + 1;
  const int n = visible >> sh.log2_ratio;
  const int K = sh.topk;
  int32_t *out = sel + static_cast<size_t>(row) * K;
  const int tid = threadIdx.x;

  if (visible < 1 || visible > cap_tokens || n > ld) {
    pdl_wait();
    pdl_trigger();
    for (int x = tid; x < K; x += kSelThreads) out[x] = -1;
    if (tid == 0) {
      n_sel[row] = 0;
      report(status, QSA_ERR_CAPACITY);
    }
    return;
  }
  if (n <= K) {  // every block is selected: exactly dense attention
    pdl_wait();
    pdl_trigger();
    for (int x = tid; x < K; x += kSelThreads) out[x] = x < n ? x : -1;
    if (tid == 0) n_sel[row] = n;
    return;
  }

#pragma unroll
  for (int j = 0; j < kBinsPerThread; ++j) hist[kBinsPerThread * tid + j] = 0;
  if (tid == 0) s_ncand = 0;
  pdl_wait();  // scores come from the score kernel
  pdl_trigger();
  uint32_t *cand = keys + smem_keys;
  const float *srow = scores + static_cast<size_t>(row) * ld;
  // rows up to 16k blocks (64k tokens at ratio 4) keep their keys in registers
  // (a thread's run of 4 NV keys plus E tail keys; the smallest layout that holds the row)
  if (n <= 4 * kSelThreads) {
    select_in_registers<1, 0>(srow, n, K, out, cand, hist, scan_tmp, s_res, &s_ncand, red_min, red_max);
  } else if (n <= 8 * kSelThreads) {
    select_in_registers<2, 0>(srow, n, K, out, cand, hist, scan_tmp, s_res, &s_ncand, red_min, red_max);
  } else if (n <= 9 * kSelThreads) {
    select_in_registers<2, 1>(srow, n, K, out, cand, hist, scan_tmp, s_res, &s_ncand, red_min, red_max);
  } else if (n <= 12 * kSelThreads) {
    select_in_registers<3, 0>(srow, n, K, out, cand, hist, scan_tmp, s_res, &s_ncand, red_min, red_max);
  } else if (n <= 16 * kSelThreads) {
    select_in_registers<4, 0>(srow, n, K, out, cand, hist, scan_tmp, s_res, &s_ncand, red_min, red_max);
  } else if (n <= 32 * kSelThreads) {  // runs of 32: 16 keys in registers, 16 in shared memory
    select_in_runs<4, 16>(srow, n, K, out, keys, cand, hist, scan_tmp, s_res, &s_ncand, red_min, red_max);
  } else {
    select_general(srow, n, K, out, keys, cand, smem_keys, hist, scan_tmp, s_res, &s_ncand, red_min, red_max);
  }
  if (tid == 0) n_sel[row] = K;
}

// ---------------------------------------------------------------------------
// Long rows on a thread-block cluster of C CTAs (1024 threads each) per row.
// CTA rank c holds the consecutive blocks [c * per, (c + 1) * per) of the row
// (per a multiple of 4) in the register layout of per blocks (runs of 4 NV keys
// per thread), so a row of 16k blocks costs 8 keys per thread on 2 SMs instead
// of 16 on one. The CTAs share what each phase needs through distributed
// shared memory: the row's range (each CTA's min and max), each radix pass's
// histograms (every CTA sums the cluster's into its own copy and runs the same
// digit search, so all reach the same digit; the search also counts the keys
// above the digit held by lower-ranked CTAs) and the final short candidate list
// (every CTA copies the cluster's lists in rank order and ranks the merged
// list, counting the lower-ranked CTAs' candidates above and at the threshold).
// Those lower-rank counts are where a CTA's selected blocks start in the output,
// so the compaction is a local block scan. A CTA reads another's shared memory
// only after a cluster barrier that follows the owner's last write of it, and a
// split barrier (arrive after the last remote read, wait before exit) keeps
// every CTA resident while another may still read from it. The histograms are
// double-buffered: a buffer is cleared only after the next cluster barrier.
// ---------------------------------------------------------------------------

// Distributed shared memory: the address of p's counterpart in cluster CTA
// `rank`, loads from such an address, and the cluster barrier.
__device__ __forceinline__ uint32_t cluster_addr(const void *p, int rank) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint2 ld_cluster_v2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared::cluster.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ int4 ld_cluster_v4(uint32_t addr) {
  int4 v;
  asm volatile("ld.shared::cluster.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync() {
  cluster_arrive();
  cluster_wait();
}

// After a cluster barrier that follows every CTA's histogram of this pass (hb:
// the pass's buffer, at the same offset in every CTA): the digit that holds the
// remaining-th largest key of the row. The C histograms are summed into hsum
// (all CTAs) and hlow (CTAs ranked below crank), each thread reading runs of 4
// bins, so a warp's remote reads are contiguous; then thread t owns the
// kBinsPerThread digits below kBins - kBinsPerThread * t. Leaves in s_res: [0]
// the digit, [1] the row's keys above it, [2] the row's keys in it, [3] and [4]
// the same two counts over the lower-ranked CTAs.
template <int C>
__device__ __forceinline__ void cluster_digit_search(int remaining, int crank, const int *hb, int *hsum, int *hlow,
                                                     int2 *scan_tmp, int *s_res) {
  const int tid = threadIdx.x;
  static_assert(kBins / 4 <= kSelThreads, "a thread reads at most one run of 4 bins");
  if (tid < kBins / 4) {
    const int b = 4 * tid;
    int4 s = make_int4(0, 0, 0, 0), l = make_int4(0, 0, 0, 0);
#pragma unroll
    for (int r = 0; r < C; ++r) {
      const int4 v = ld_cluster_v4(cluster_addr(hb + b, r));
      s.x += v.x;
      s.y += v.y;
      s.z += v.z;
      s.w += v.w;
      if (r < crank) {
        l.x += v.x;
        l.y += v.y;
        l.z += v.z;
        l.w += v.w;
      }
    }
    *reinterpret_cast<int4 *>(hsum + b) = s;
    *reinterpret_cast<int4 *>(hlow + b) = l;
  }
  __syncthreads();
  const int top_bin = kBins - 1 - kBinsPerThread * tid;
  int c_all[kBinsPerThread], c_low[kBinsPerThread];
  int s_all = 0, s_low = 0;
#pragma unroll
  for (int j = 0; j < kBinsPerThread; ++j) {
    c_all[j] = hsum[top_bin - j];
    c_low[j] = hlow[top_bin - j];
    s_all += c_all[j];
    s_low += c_low[j];
  }
  int2 above = block_exclusive_scan2(make_int2(s_all, s_low), scan_tmp);
#pragma unroll
  for (int j = 0; j < kBinsPerThread; ++j) {
    if (above.x < remaining && remaining <= above.x + c_all[j]) {
      s_res[0] = top_bin - j;
      s_res[1] = above.x;
      s_res[2] = c_all[j];
      s_res[3] = above.y;
      s_res[4] = c_low[j];
    }
    above.x += c_all[j];
    above.y += c_low[j];
  }
  __syncthreads();
}

template <int C, int NV>
__device__ __forceinline__ void select_cluster_row(const float *__restrict__ srow, int n, int K, int crank,
                                                   int32_t *__restrict__ out, int (*hist)[kBins], int *hsum,
                                                   int *hlow, uint32_t *cand, uint32_t *mcand, int2 *scan_tmp,
                                                   int *s_res, int *s_ncand, uint32_t *red_min, uint32_t *red_max,
                                                   uint2 *s_mm) {
  constexpr int NK = 4 * NV;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = ((n + 4 * C - 1) / (4 * C)) * 4;  // blocks per CTA, a multiple of 4
  const int lo = crank * per;
  const int hi = min(n, lo + per);
  const int x0 = lo + NK * tid;  // this thread's first block
  // 16-byte loads: ld and x0 are multiples of 4, so a group that starts below n lies in the row
  const float4 *s4 = reinterpret_cast<const float4 *>(srow + x0);
  uint32_t d[NK];
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
    if (x0 + 4 * v < hi) f = s4[v];
    d[4 * v] = score_key(f.x);
    d[4 * v + 1] = score_key(f.y);
    d[4 * v + 2] = score_key(f.z);
    d[4 * v + 3] = score_key(f.w);
  }
  auto valid = [&](int j) { return x0 + j < hi; };

  // ---- the row's range: every CTA publishes its min and max, then reads all
  uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
  for (int j = 0; j < NK; ++j)
    if (valid(j)) {
      kmin = min(kmin, d[j]);
      kmax = max(kmax, d[j]);
    }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0) {
    red_min[warp] = kmin;
    red_max[warp] = kmax;
  }
  __syncthreads();
  if (warp == 0) {
    kmin = __reduce_min_sync(0xffffffffu, lane < kSelWarps ? red_min[lane] : 0xffffffffu);
    kmax = __reduce_max_sync(0xffffffffu, lane < kSelWarps ? red_max[lane] : 0u);
    if (lane == 0) *s_mm = make_uint2(kmin, kmax);
  }
  // the first cluster barrier: every CTA has started and published its range
  cluster_sync();
  kmin = 0xffffffffu;
  kmax = 0u;
#pragma unroll
  for (int r = 0; r < C; ++r) {
    const uint2 m = ld_cluster_v2(cluster_addr(s_mm, r));
    kmin = min(kmin, m.x);
    kmax = max(kmax, m.y);
  }
#pragma unroll
  for (int j = 0; j < NK; ++j) d[j] -= kmin;  // invalid entries are never read

  const uint32_t range = kmax - kmin;
  int top = range ? 31 - __clz(range) : -1;
  const uint32_t low_bits = (top >= 31) ? 0xffffffffu : (top >= 0 ? ((2u << top) - 1u) : 0u);
  uint32_t prefix = 0u;
  uint32_t mask = ~low_bits;
  int remaining = K;
  int gt_low = 0;  // keys above the threshold held by lower-ranked CTAs
  int eq_low = 0;  // keys at the threshold held by lower-ranked CTAs
  if (top < 0) {
    // every key of the row is equal: the threshold is that key
#pragma unroll
    for (int r = 0; r < C; ++r)
      if (r < crank) eq_low += max(0, min(n, (r + 1) * per) - r * per);
  }
  for (int pass = 0; top >= 0; ++pass) {
    // a pass over the keys under the prefix: histogram of the next digit
    const int width = min(kDigit, top + 1);
    const int shift = top + 1 - width;
    const uint32_t dmask = (1u << width) - 1u;
    int *hb = hist[pass & 1];
    if (pass >= 2) {  // this buffer's remote readers passed the previous pass's barrier
      for (int b = tid; b < kBins; b += kSelThreads) hb[b] = 0;
      __syncthreads();
    }
#pragma unroll
    for (int j = 0; j < NK; ++j)
      if (valid(j) && (d[j] & mask) == prefix) atomicAdd(&hb[(d[j] >> shift) & dmask], 1);
    cluster_sync();
    cluster_digit_search<C>(remaining, crank, hb, hsum, hlow, scan_tmp, s_res);
    prefix |= static_cast<uint32_t>(s_res[0]) << shift;
    mask |= dmask << shift;
    remaining -= s_res[1];
    gt_low += s_res[3];
    top = shift - 1;
    if (top < 0) {  // the prefix is the whole key: the threshold
      eq_low = s_res[4];
      break;
    }
    if (s_res[2] <= kDirectMax) {
      // the keys under the prefix (at most kDirectMax over the row): each CTA
      // lists its own, then every CTA copies the cluster's lists in rank order
      // (CTA r's entries at offs[r]) and ranks the merged list
      uint32_t member = 0u;
#pragma unroll
      for (int j = 0; j < NK; ++j)
        if (valid(j) && (d[j] & mask) == prefix) member |= 1u << j;
      if (member) {
        int pos = atomicAdd(s_ncand, __popc(member));
#pragma unroll
        for (int j = 0; j < NK; ++j)
          if ((member >> j) & 1u) cand[pos++] = d[j];
      }
      cluster_sync();
      int cnt[C], offs[C + 1];
      offs[0] = 0;
#pragma unroll
      for (int r = 0; r < C; ++r) {
        cnt[r] = static_cast<int>(ld_cluster_u32(cluster_addr(s_ncand, r)));
        offs[r + 1] = offs[r] + cnt[r];
      }
      const int nc = offs[C];
      int my_off = 0;  // the lower-ranked CTAs' entries (static indices only: no local memory)
#pragma unroll
      for (int q = 0; q < C; ++q)
        if (q < crank) my_off += cnt[q];
      if (tid < nc) {
        int r = 0, base = 0;
#pragma unroll
        for (int q = 1; q < C; ++q)
          if (tid >= offs[q]) {
            r = q;
            base = offs[q];
          }
        mcand[tid] = ld_cluster_u32(cluster_addr(cand + (tid - base), r));
      }
      __syncthreads();
      rank_candidates(mcand, nc, prefix, remaining, s_res);
      // the lower-ranked CTAs' candidates above and at the threshold: the
      // merged list holds them first, my_off of them
      if (warp == 0) {
        int g = 0, e = 0;
        for (int i = lane; i < my_off; i += 32) {
          g += mcand[i] > prefix ? 1 : 0;
          e += mcand[i] == prefix ? 1 : 0;
        }
        g = __reduce_add_sync(0xffffffffu, g);
        e = __reduce_add_sync(0xffffffffu, e);
        if (lane == 0) {
          s_res[3] = g;
          s_res[4] = e;
        }
      }
      __syncthreads();
      gt_low += s_res[3];
      eq_low = s_res[4];
      break;
    }
  }
  // every remote access of this CTA is done: the others may leave once all
  // have arrived here
  cluster_arrive();
  const uint32_t thr = prefix;  // the K-th largest key
  const int need = remaining;   // ties at thr to take (>= 1)

  // ---- compaction: the blocks before this thread's emit gt_low plus the keys
  // above thr before it in this CTA, and min(eq_low + the ties before it, need)
  // ties; its own blocks follow in index order (counts packed 16:16)
  uint32_t c0 = 0u;
#pragma unroll
  for (int j = 0; j < NK; ++j)
    if (valid(j)) c0 += (d[j] > thr ? 1u : 0u) + (d[j] == thr ? 0x10000u : 0u);
  const uint32_t p0 =
      static_cast<uint32_t>(block_exclusive_scan1(static_cast<int>(c0), reinterpret_cast<int *>(scan_tmp)));
  int tie_rank = eq_low + static_cast<int>(p0 >> 16);
  int o = gt_low + static_cast<int>(p0 & 0xffffu) + min(tie_rank, need);
#pragma unroll
  for (int j = 0; j < NK; ++j) {
    if (!valid(j)) continue;
    if (d[j] > thr) {
      if (o < K) out[o] = x0 + j;
      ++o;
    } else if (d[j] == thr) {
      if (tie_rank < need) {
        if (o < K) out[o] = x0 + j;
        ++o;
      }
      ++tie_rank;
    }
  }
  cluster_wait();
}

template <int C>
__global__ void __launch_bounds__(kSelThreads)
select_cluster_kernel(Shape sh, int R, const int32_t *__restrict__ pos0, const float *__restrict__ scores, int ld,
                      int32_t *__restrict__ sel, int32_t *__restrict__ n_sel, int cap_tokens, int32_t *status) {
  __shared__ __align__(16) int hist[2][kBins];
  __shared__ __align__(16) int hsum[kBins];
  __shared__ __align__(16) int hlow[kBins];
  __shared__ uint32_t cand[kDirectMax], mcand[kDirectMax];
  __shared__ int2 scan_tmp[kSelWarps];
  __shared__ uint32_t red_min[kSelWarps], red_max[kSelWarps];
  __shared__ uint2 s_mm;
  __shared__ int s_res[5], s_ncand;

  uint32_t crank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(crank));
  const int row = blockIdx.x / C;
  const int i = row / R;
  const int visible = pos0[i] + (row - i * R) + 1;
  const int n = visible >> sh.log2_ratio;
  const int K = sh.topk;
  int32_t *out = sel + static_cast<size_t>(row) * K;
  const int tid = threadIdx.x;

  // rows that need no ranking are written by rank 0 alone, with no cluster
  // barrier (the same branch in every CTA of the cluster: n is the row's)
  if (visible < 1 || visible > cap_tokens || n > ld || n > 4 * 4 * kSelThreads * C) {
    pdl_wait();
    pdl_trigger();
    if (crank != 0) return;
    for (int x = tid; x < K; x += kSelThreads) out[x] = -1;
    if (tid == 0) {
      n_sel[row] = 0;
      report(status, QSA_ERR_CAPACITY);
    }
    return;
  }
  if (n <= K) {  // every block is selected: exactly dense attention
    pdl_wait();
    pdl_trigger();
    if (crank != 0) return;
    for (int x = tid; x < K; x += kSelThreads) out[x] = x < n ? x : -1;
    if (tid == 0) n_sel[row] = n;
    return;
  }

  for (int b = tid; b < 2 * kBins; b += kSelThreads) (&hist[0][0])[b] = 0;
  if (tid == 0) s_ncand = 0;
  pdl_wait();  // scores come from the score kernel
  pdl_trigger();
  const float *srow = scores + static_cast<size_t>(row) * ld;
  const int per = ((n + 4 * C - 1) / (4 * C)) * 4;
  const int r = static_cast<int>(crank);
  if (per <= 4 * kSelThreads)
    select_cluster_row<C, 1>(srow, n, K, r, out, hist, hsum, hlow, cand, mcand, scan_tmp, s_res, &s_ncand, red_min,
                             red_max, &s_mm);
  else if (per <= 8 * kSelThreads)
    select_cluster_row<C, 2>(srow, n, K, r, out, hist, hsum, hlow, cand, mcand, scan_tmp, s_res, &s_ncand, red_min,
                             red_max, &s_mm);
  else if (per <= 12 * kSelThreads)
    select_cluster_row<C, 3>(srow, n, K, r, out, hist, hsum, hlow, cand, mcand, scan_tmp, s_res, &s_ncand, red_min,
                             red_max, &s_mm);
  else
    select_cluster_row<C, 4>(srow, n, K, r, out, hist, hsum, hlow, cand, mcand, scan_tmp, s_res, &s_ncand, red_min,
                             red_max, &s_mm);
  if (crank == 0 && tid == 0) n_sel[row] = K;
}

int sm_count() {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      sms = v;
  }
  return sms;
}

}  // namespace

cudaError_t launch_select(const Shape &sh, int n_seq, int R, const int32_t *pos0,
                          const float *scores, int ld_scores, int32_t *sel, int32_t *n_sel,
                          int max_blocks, int cap_tokens, int32_t *status, bool pdl,
                          cudaStream_t st) {
  if (n_seq == 0 || R == 0) return cudaSuccess;
  // Rows past 9216 blocks (beyond the one-CTA layouts of at most 9 keys per
  // thread) go to a cluster of C CTAs per row when the launch's C * rows CTAs
  // fit on the GPU at once (1024 threads at 64 registers: one CTA per SM) and
  // every row fits C CTAs' register runs of at most 16 keys
  const long long rows = static_cast<long long>(n_seq) * R;
  const int sms = sm_count();
  if (max_blocks > 9 * kSelThreads && sms > 0) {
    const int c = (rows * 4 <= sms && max_blocks <= 4 * 16 * kSelThreads) ? 4
                  : (rows * 2 <= sms && max_blocks <= 2 * 16 * kSelThreads) ? 2 : 1;
    if (c == 4)
      return launch_kernel_cluster(pdl, 4, select_cluster_kernel<4>, dim3(static_cast<unsigned>(rows * 4)),
                                   dim3(kSelThreads), 0, st, sh, R, pos0, scores, ld_scores, sel, n_sel, cap_tokens,
                                   status);
    if (c == 2)
      return launch_kernel_cluster(pdl, 2, select_cluster_kernel<2>, dim3(static_cast<unsigned>(rows * 2)),
                                   dim3(kSelThreads), 0, st, sh, R, pos0, scores, ld_scores, sel, n_sel, cap_tokens,
                                   status);
  }
  // rows of more than kMaxSmemKeys blocks read their scores from global memory;
  // runs of 32 take their row padded by one word per 32 blocks
  int want = max_blocks + max_blocks / 32 + 1;
  if (max_blocks > 16 * kSelThreads && want < 33 * kSelThreads) want = 33 * kSelThreads;
  const int cap = want < kMaxSmemKeys ? want : kMaxSmemKeys;
  const size_t smem = (static_cast<size_t>(cap) + kCandMax) * 4;
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_kernel(pdl, select_kernel, dim3(n_seq * R), dim3(kSelThreads), smem, st, sh, R, pos0,
                       scores, ld_scores, sel, n_sel, cap, cap_tokens, status);
}

}  // namespace qsa
