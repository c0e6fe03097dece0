// Index score: s_b = sum_h w_h * max(0, q_I,h . k_b) for every complete block
// b of a row ("Agentic shootout", "PR 16 review: qwen4exp serving in Atlas
// (Claude's review)", (a): relu-score over 4-token mean-pooled blocks;
// "Flash-Next support: vLLM vs Atlas", (a) item 6: the query is scored
// against the compressed keys).
//
// One CTA scores a tile of 128 consecutive blocks of one row. The contraction
// runs on the tensor cores with the blocks on the MMA's M dimension and the
// index heads on N (m16n8k16, bf16 in, fp32 accumulate), so each accumulator
// row is one block and the ReLU * w reduction over heads is a sum inside a
// thread plus two lane shuffles. Keys are gathered through the page table with
// 16-byte cp.async into an XOR-swizzled shared tile (conflict-free ldmatrix).
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kTileBlocks = 128;
constexpr int kScoreThreads = 128;

template <int DI, int NH>
__global__ void __launch_bounds__(kScoreThreads)
score_kernel(Shape sh, int R, const int32_t *__restrict__ seq_ids,
             const int32_t *__restrict__ pos0, CacheView cv, const uint16_t *__restrict__ q_idx,
             const float *__restrict__ w, float *__restrict__ scores, int ld, int32_t *status) {
  constexpr int CPR = DI / 8;     // 16-byte chunks per key row
  constexpr int KS = DI / 16;     // MMA k-steps
  constexpr int NT = NH / 8;      // n-tiles of 8 heads
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *keys = smem;                                   // [128][DI] bf16, swizzled
  uint8_t *qs = smem + kTileBlocks * DI * 2;              // [NH][DI] bf16, swizzled
  float *ws = reinterpret_cast<float *>(qs + NH * DI * 2);  // [NH]

  pdl_wait();  // the compressed keys come from the append kernel
  pdl_trigger();
  const int row = blockIdx.y;
  const int i = row / R;
  const int visible = pos0[i] + (row - i * R) + 1;
  if (visible < 1 || visible > cv.max_pages * sh.page) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(status, QSA_ERR_CAPACITY);
    return;
  }
  const int n_blk = visible >> sh.log2_ratio;
  if (n_blk <= sh.topk) return;                           // dense row: nothing to score
  const int b0 = blockIdx.x * kTileBlocks;
  if (b0 >= n_blk) return;
  const int s = seq_ids[i];
  const int32_t *ptab = cv.page_table + static_cast<size_t>(s) * cv.max_pages;
  const int bpp_log2 = sh.log2_page - sh.log2_ratio;      // blocks per page (log2)
  const int tid = threadIdx.x;

  // keys of the tile
  for (int e = tid; e < kTileBlocks * CPR; e += kScoreThreads) {
    const int r = e / CPR, c = e % CPR;
    const int b = b0 + r;
    const void *src = cv.idxblk_pool;
    int bytes = 0;
    if (b < n_blk) {
      const int page = ptab[b >> bpp_log2];
      if (page >= 0 && page < cv.num_pages) {
        src = static_cast<const uint16_t *>(cv.idxblk_pool) + (static_cast<size_t>(page) << bpp_log2) * DI +
              blk_elem_offset(b & ((1 << bpp_log2) - 1), c * 8, 1 << bpp_log2, DI);
        bytes = 16;
      } else {
        report(status, QSA_ERR_PAGE);
      }
    }
    cp_async16(smem_u32(keys + r * DI * 2 + ((c ^ (r & 7)) * 16)), src, bytes);
  }
  // query heads of the row (heads >= H_I are zero)
  for (int e = tid; e < NH * CPR; e += kScoreThreads) {
    const int h = e / CPR, c = e % CPR;
    const bool ok = h < sh.h_idx;
    const void *src = ok ? static_cast<const void *>(q_idx + (static_cast<size_t>(row) * sh.h_idx + h) * DI + c * 8)
                         : static_cast<const void *>(q_idx);
    cp_async16(smem_u32(qs + h * DI * 2 + ((c ^ (h & 7)) * 16)), src, ok ? 16 : 0);
  }
  if (tid < NH) ws[tid] = tid < sh.h_idx ? w[static_cast<size_t>(row) * sh.h_idx + tid] : 0.f;
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();

  const int warp = tid >> 5, lane = tid & 31;
  float acc[2][NT][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[mt][nt][c] = 0.f;

  const uint32_t keys_u = smem_u32(keys), qs_u = smem_u32(qs);
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    uint32_t a[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const int r = warp * 32 + mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
      const int c = 2 * ks + (lane >> 4);
      ldsm_x4(keys_u + r * DI * 2 + ((c ^ (r & 7)) * 16), a[mt][0], a[mt][1], a[mt][2], a[mt][3]);
    }
#pragma unroll
    for (int np = 0; np < NT / 2; ++np) {
      const int h = (2 * np + (lane >> 4)) * 8 + (lane & 7);
      const int c = 2 * ks + ((lane >> 3) & 1);
      uint32_t b00, b01, b10, b11;
      ldsm_x4(qs_u + h * DI * 2 + ((c ^ (h & 7)) * 16), b00, b01, b10, b11);
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        mma_bf16(acc[mt][2 * np], a[mt][0], a[mt][1], a[mt][2], a[mt][3], b00, b01);
        mma_bf16(acc[mt][2 * np + 1], a[mt][0], a[mt][1], a[mt][2], a[mt][3], b10, b11);
      }
    }
  }

  // epilogue: w * ReLU summed over the thread's heads, then over the quad
  float* srow = scores + static_cast<size_t>(row) * ld;
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float v = 0.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int h = nt * 8 + 2 * (lane & 3);
        v += ws[h] * fmaxf(acc[mt][nt][2 * half], 0.f);
        v += ws[h + 1] * fmaxf(acc[mt][nt][2 * half + 1], 0.f);
      }
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      const int b = b0 + warp * 32 + mt * 16 + (lane >> 2) + half * 8;
      if ((lane & 3) == 0 && b < n_blk) srow[b] = v;
    }
  }
}

template <int DI, int NH>
cudaError_t launch_score_t(const Shape &sh, int n_seq, int R, const int32_t *seq_ids,
                           const int32_t *pos0, const CacheView &cv, const uint16_t *q_idx,
                           const float *w, float *scores, int ld, int32_t *status, bool pdl,
                           cudaStream_t st) {
  const size_t smem = kTileBlocks * DI * 2 + NH * DI * 2 + NH * 4;
  auto kern = score_kernel<DI, NH>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid((ld + kTileBlocks - 1) / kTileBlocks, n_seq * R);
  return launch_kernel(pdl, kern, grid, dim3(kScoreThreads), smem, st, sh, R, seq_ids, pos0, cv, q_idx,
                       w, scores, ld, status);
}

}  // namespace

cudaError_t launch_score(const Shape &sh, int n_seq, int R, const int32_t *seq_ids,
                         const int32_t *pos0, const CacheView &cv, const uint16_t *q_idx,
                         const float *w, float *scores, int ld_scores, int32_t *status, bool pdl,
                         cudaStream_t st, bool q_in_step) {
  if (n_seq == 0 || R == 0) return cudaSuccess;
  // tcgen05 path whenever the TMA page boxes fit (8..32 blocks per page);
  // the mma.sync kernel below covers the remaining shapes (ratio 16, bf16 keys only)
  if (sh.idx_fp8 && !score_tc_supported(sh)) return cudaErrorInvalidValue;
  if (score_tc_supported(sh))
    return launch_score_tc(sh, n_seq, R, seq_ids, pos0, cv, q_idx, w, scores, ld_scores, status, pdl, st,
                           q_in_step);
  const int nh = sh.h_idx <= 16 ? 16 : (sh.h_idx <= 32 ? 32 : 64);
  if (sh.d_idx == 128) {
    if (nh == 16) return launch_score_t<128, 16>(sh, n_seq, R, seq_ids, pos0, cv, q_idx, w, scores, ld_scores, status, pdl, st);
    if (nh == 32) return launch_score_t<128, 32>(sh, n_seq, R, seq_ids, pos0, cv, q_idx, w, scores, ld_scores, status, pdl, st);
    return launch_score_t<128, 64>(sh, n_seq, R, seq_ids, pos0, cv, q_idx, w, scores, ld_scores, status, pdl, st);
  }
  if (nh == 16) return launch_score_t<64, 16>(sh, n_seq, R, seq_ids, pos0, cv, q_idx, w, scores, ld_scores, status, pdl, st);
  if (nh == 32) return launch_score_t<64, 32>(sh, n_seq, R, seq_ids, pos0, cv, q_idx, w, scores, ld_scores, status, pdl, st);
  return launch_score_t<64, 64>(sh, n_seq, R, seq_ids, pos0, cv, q_idx, w, scores, ld_scores, status, pdl, st);
}

}  // namespace qsa
