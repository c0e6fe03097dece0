// Top-K block selection ("Agentic shootout", "Flash-Next support: vLLM vs
// Atlas", (a) item 6: block top-k of budget/compress_ratio groups; "PR 16
// review ... (Claude's review)", (a): top-512 + tail, inert below
// budget + ratio - 1 visible tokens).
//
// One CTA per row. Scores become order-preserving uint32 keys (-0 folded onto
// +0) held in shared memory. A 4-pass MSB-first radix select (8-bit digits,
// shared-memory histograms) finds the K-th largest key T exactly and the
// number of ties at T that must be taken. A stable compaction then emits, in
// ascending block order, every block with key > T and the lowest-indexed
// blocks with key == T: exactly the top-K under (score desc, index asc).
// The selection stays on the device, so a step that contains it can be
// captured in a CUDA graph.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kMaxSmemKeys = 50 * 1024;  // 200 KB of keys held on chip

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

__global__ void __launch_bounds__(kSelThreads)
select_kernel(Shape sh, int R, const int32_t *__restrict__ pos0, const float *__restrict__ scores,
              int ld, int32_t *__restrict__ sel, int32_t *__restrict__ n_sel, int smem_keys,
              int cap_tokens, int32_t *status) {
  extern __shared__ uint32_t keys[];
  __shared__ int hist[256];
  __shared__ int scan_tmp[kSelWarps];
  __shared__ int s_digit, s_above;

  const int row = blockIdx.x;
  const int i = row / R;
  const int visible = pos0[i] + (row - i * R) + 1;
  const int n = visible >> sh.log2_ratio;
  const int K = sh.topk;
  int32_t *out = sel + static_cast<size_t>(row) * K;
  const int tid = threadIdx.x;

  if (visible < 1 || visible > cap_tokens || n > ld) {
    for (int x = tid; x < K; x += kSelThreads) out[x] = -1;
    if (tid == 0) {
      n_sel[row] = 0;
      report(status, QSA_ERR_CAPACITY);
    }
    return;
  }
  if (n <= K) {  // every block is selected: exactly dense attention
    for (int x = tid; x < K; x += kSelThreads) out[x] = x < n ? x : -1;
    if (tid == 0) n_sel[row] = n;
    return;
  }

  const float *srow = scores + static_cast<size_t>(row) * ld;
  const bool cached = n <= smem_keys;
  if (cached)
    for (int x = tid; x < n; x += kSelThreads) keys[x] = score_key(srow[x]);
  __syncthreads();
  auto key_at = [&](int x) -> uint32_t { return cached ? keys[x] : score_key(srow[x]); };

  uint32_t prefix = 0, mask = 0;
  int remaining = K;  // how many of the still-undecided keys must be taken
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    if (tid < 256) hist[tid] = 0;
    if (tid == 0) {
      s_digit = 0;
      s_above = 0;
    }
    __syncthreads();
    for (int x = tid; x < n; x += kSelThreads) {
      const uint32_t k = key_at(x);
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 0xFF], 1);
    }
    __syncthreads();
    if (tid < 32) {
      // lane L owns digits [255-8L-7, 255-8L]; scan from the top digit down
      int local[8];
      int sum = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        local[q] = hist[255 - 8 * tid - q];
        sum += local[q];
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += y;
      }
      int above = incl - sum;  // keys in higher digit groups
      if (above < remaining && remaining <= incl) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (above < remaining && remaining <= above + local[q]) {
            s_digit = 255 - 8 * tid - q;
            s_above = above;
          }
          above += local[q];
        }
      }
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(s_digit) << shift;
    mask |= 0xFFu << shift;
    remaining -= s_above;
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
                          int max_blocks, int cap_tokens, int32_t *status, cudaStream_t st) {
  if (n_seq == 0 || R == 0) return cudaSuccess;
  const int cap = max_blocks < kMaxSmemKeys ? max_blocks : kMaxSmemKeys;
  const size_t smem = static_cast<size_t>(cap) * 4;
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  select_kernel<<<n_seq * R, kSelThreads, smem, st>>>(sh, R, pos0, scores, ld_scores, sel, n_sel, cap,
                                                      cap_tokens, status);
  return cudaGetLastError();
}

}  // namespace qsa
