// Top-K block selection ("Agentic shootout", "Flash-Next support: vLLM vs
// Atlas", (a) item 6: block top-k of budget/compress_ratio groups; "PR 16
// review ... (Claude's review)", (a): top-512 + tail, inert below
// budget + ratio - 1 visible tokens).
//
// One CTA per row. Scores become order-preserving uint32 keys (-0 folded onto
// +0) held in shared memory. The keys of a row share their high bits (same
// sign and exponent), so the radix digits are taken from the window of bits in
// which the row's smallest and largest keys differ, 11 bits at a time, most
// significant first: each pass histograms the keys that match the prefix fixed
// so far and a block-wide suffix scan finds the digit that holds the K-th
// largest key. After at most three passes the K-th largest key T is exact, and
// so is the number of ties at T that must be taken. A stable compaction then
// emits, in ascending block order, every block with key > T and the
// lowest-indexed blocks with key == T: exactly the top-K under (score desc,
// index asc). The selection stays on the device, so a step that contains it can
// be captured in a CUDA graph.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kMaxSmemKeys = 48 * 1024;  // 192 KB of keys held on chip
constexpr int kDigit = 11;
constexpr int kBins = 1 << kDigit;       // 2048: two bins per thread

// Exclusive prefix sum over the CTA; `tmp` holds kSelWarps ints.
__device__ __forceinline__ int block_exclusive_scan(int v, int *tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = tmp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    tmp[lane] = t;  // inclusive totals per warp
  }
  __syncthreads();
  const int before = warp > 0 ? tmp[warp - 1] : 0;
  __syncthreads();
  return before + x - v;
}

// Histogram update; a warp whose active lanes all hold the same digit (a run of
// equal scores) makes one atomic instead of 32 that would serialise.
__device__ __forceinline__ void hist_add(int *hist, uint32_t digit, bool active) {
  const unsigned act = __ballot_sync(0xffffffffu, active);
  if (!active) return;
  const int leader = __ffs(act) - 1;
  const uint32_t d0 = __shfl_sync(act, digit, leader);
  if (__all_sync(act, digit == d0)) {
    if ((threadIdx.x & 31) == leader) atomicAdd(&hist[digit], __popc(act));
  } else {
    atomicAdd(&hist[digit], 1);
  }
}

__global__ void __launch_bounds__(kSelThreads)
select_kernel(Shape sh, int R, const int32_t *__restrict__ pos0, const float *__restrict__ scores,
              int ld, int32_t *__restrict__ sel, int32_t *__restrict__ n_sel, int smem_keys,
              int cap_tokens, int32_t *status) {
  extern __shared__ uint32_t keys[];
  __shared__ int hist[kBins];
  __shared__ int scan_tmp[kSelWarps];
  __shared__ uint32_t red_min[kSelWarps], red_max[kSelWarps];
  __shared__ int s_digit, s_above;

  const int row = blockIdx.x;
  const int i = row / R;
  const int visible = pos0[i] + (row - i * R) + 1;
  const int n = visible >> sh.log2_ratio;
  const int K = sh.topk;
  int32_t *out = sel + static_cast<size_t>(row) * K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

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

  pdl_wait();  // scores come from the score kernel
  pdl_trigger();
  const float *srow = scores + static_cast<size_t>(row) * ld;
  const bool cached = n <= smem_keys;
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  if (cached) {
    // 16-byte loads: ld is a multiple of 4, so the row start is 16-byte aligned
    const float4 *s4 = reinterpret_cast<const float4 *>(srow);
    const int n4 = n >> 2;
    for (int x = tid; x < n4; x += kSelThreads) {
      const float4 v = s4[x];
      const uint32_t k0 = score_key(v.x), k1 = score_key(v.y), k2 = score_key(v.z), k3 = score_key(v.w);
      keys[4 * x] = k0;
      keys[4 * x + 1] = k1;
      keys[4 * x + 2] = k2;
      keys[4 * x + 3] = k3;
      kmin = min(kmin, min(min(k0, k1), min(k2, k3)));
      kmax = max(kmax, max(max(k0, k1), max(k2, k3)));
    }
    for (int x = 4 * n4 + tid; x < n; x += kSelThreads) {
      const uint32_t k = score_key(srow[x]);
      keys[x] = k;
      kmin = min(kmin, k);
      kmax = max(kmax, k);
    }
  } else {
    for (int x = tid; x < n; x += kSelThreads) {
      const uint32_t k = score_key(srow[x]);
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
  kmin = red_min[lane];
  kmax = red_max[lane];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  auto key_at = [&](int x) -> uint32_t { return cached ? keys[x] : score_key(srow[x]); };

  // bits above the window are common to every key of the row
  const uint32_t diff = kmin ^ kmax;
  int top = diff ? 31 - __clz(diff) : -1;  // highest differing bit
  const uint32_t low_bits = (top >= 31) ? 0xffffffffu : (top >= 0 ? ((2u << top) - 1u) : 0u);
  uint32_t prefix = kmax & ~low_bits;
  uint32_t mask = ~low_bits;
  int remaining = K;  // how many of the still-undecided keys must be taken
  const int n_iter = (n + kSelThreads - 1) / kSelThreads;
#pragma unroll 1
  while (top >= 0) {
    const int width = min(kDigit, top + 1);
    const int shift = top + 1 - width;
    const uint32_t dmask = (1u << width) - 1u;
    hist[2 * tid] = 0;
    hist[2 * tid + 1] = 0;
    __syncthreads();
    for (int it = 0; it < n_iter; ++it) {  // warp-uniform trip count
      const int x = it * kSelThreads + tid;
      const uint32_t k = x < n ? key_at(x) : 0u;
      const bool act = x < n && (k & mask) == prefix;
      hist_add(hist, (k >> shift) & dmask, act);
    }
    __syncthreads();
    // thread t owns digits (kBins-1-2t) and (kBins-2-2t): a suffix scan from the
    // top digit finds the digit that holds the remaining-th largest key
    const int c_hi = hist[kBins - 1 - 2 * tid], c_lo = hist[kBins - 2 - 2 * tid];
    const int above = block_exclusive_scan(c_hi + c_lo, scan_tmp);
    if (above < remaining && remaining <= above + c_hi) {
      s_digit = kBins - 1 - 2 * tid;
      s_above = above;
    } else if (above + c_hi < remaining && remaining <= above + c_hi + c_lo) {
      s_digit = kBins - 2 - 2 * tid;
      s_above = above + c_hi;
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(s_digit) << shift;
    mask |= dmask << shift;
    remaining -= s_above;
    top = shift - 1;
    __syncthreads();
  }
  const uint32_t thr = prefix;  // the K-th largest key
  const int need = remaining;   // ties at thr to take (>= 1)

  // stable compaction over contiguous per-thread chunks
  const int chunk = (n + kSelThreads - 1) / kSelThreads;
  const int lo = min(n, tid * chunk), hi = min(n, lo + chunk);
  int gt = 0, eq = 0;
  for (int x = lo; x < hi; ++x) {
    const uint32_t k = key_at(x);
    gt += k > thr;
    eq += k == thr;
  }
  const int tie_base = block_exclusive_scan(eq, scan_tmp);
  const int take_eq = min(max(need - tie_base, 0), eq);
  int o = block_exclusive_scan(gt + take_eq, scan_tmp);
  int tie_rank = tie_base;
  for (int x = lo; x < hi; ++x) {
    const uint32_t k = key_at(x);
    if (k > thr) {
      if (o < K) out[o] = x;
      ++o;
    } else if (k == thr) {
      if (tie_rank < need) {
        if (o < K) out[o] = x;
        ++o;
      }
      ++tie_rank;
    }
  }
  if (tid == 0) n_sel[row] = K;
}

}  // namespace

cudaError_t launch_select(const Shape &sh, int n_seq, int R, const int32_t *pos0,
                          const float *scores, int ld_scores, int32_t *sel, int32_t *n_sel,
                          int max_blocks, int cap_tokens, int32_t *status, bool pdl,
                          cudaStream_t st) {
  if (n_seq == 0 || R == 0) return cudaSuccess;
  const int cap = max_blocks < kMaxSmemKeys ? max_blocks : kMaxSmemKeys;
  const size_t smem = static_cast<size_t>(cap) * 4;
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_kernel(pdl, select_kernel, dim3(n_seq * R), dim3(kSelThreads), smem, st, sh, R, pos0,
                       scores, ld_scores, sel, n_sel, cap, cap_tokens, status);
}

}  // namespace qsa
