// Index score on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// s_b = sum_h w_h * max(0, q_I,h . k_b) for every complete block b of a row
// ("Agentic shootout", "PR 16 review: qwen4exp serving in Atlas (Claude's
// review)", (a): relu-score over mean-pooled blocks; "Flash-Next support: vLLM
// vs Atlas", (a) item 6: the query is scored against the compressed keys).
//
// One CTA scores one tile of 128 consecutive blocks for a group of G <= 4
// consecutive rows of one sequence (decode: G = 1; verify and prefill rows of a
// sequence share the key tile). The contraction is
//     D[128 blocks, N] = K_tile[128, d_I] . Q_group^T[d_I, N],  N = G * H_I
// with blocks on M, so each TMEM lane holds one block and the ReLU * w head sum
// is a reduction inside one thread.
//   * The compressed-key pool stores each page as the tensor cores' K-major
//     core matrices (8 blocks x 16 bytes), so the tile is gathered with one bulk
//     copy per page (cp.async.bulk, 4 KB at ratio 4, d_I = 128) straight into an
//     MMA-ready, unswizzled K-major layout: core matrices adjacent in K are 128 B
//     apart, 8-block groups d_I * 16 B apart. The query rows of the group come
//     in by TMA (cp.async.bulk.tensor, 128B swizzle), one box per 64 dims.
//   * One thread issues d_I/16 tcgen05.mma (kind::f16, bf16 in, fp32 accumulate
//     in TMEM) and commits them to an mbarrier.
//   * With an MX plane -- MXFP8 (E4M3 elements, pages of bpp * (d_I + d_I/32)
//     bytes) or MXFP4 (E2M1 pairs, bpp * (d_I/2 + d_I/32) bytes), E8M0 scales
//     per 32 values -- two producers copy those pages into two byte rings, and
//     8 converter warps rebuild each tile as bf16 straight into tensor memory
//     (a block row per thread, tcgen05.st; every MX value is exact in bf16);
//     the MMA reads that A operand from TMEM, the epilogue is the bf16 one. The
//     HBM stream is 132 or 68 bytes per block instead of 256, and shared memory
//     holds only copies, so the rings run deep. The converter warps also round
//     each group's query tile to the plane's format in place, in the value
//     domain (the MMA waits for that), so the queries load as early as in the
//     bf16 path.
//   * 4 * G epilogue warps, one per (row of the group, TMEM lane quarter), read
//     their 32 lanes with tcgen05.ld: the warp holds its row's head columns in
//     registers, hands the TMEM buffer back at once, and reduces them with
//     paired fp32 FMAs (fma.rn.f32x2) in four independent chains combined in a
//     fixed order -- the same for every group size, so a row's score does not
//     depend on the batch shape. TMEM holds up to four accumulators (as many as
//     fit), so the MMAs of the next tiles run while a tile's epilogue reads.
// Every mbarrier wait is bounded in time; on expiry the CTA records
// QSA_ERR_TIMEOUT, waits (bounded) for its own copies, frees its TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <atomic>
#include <mutex>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kTcTileBlocks = 128;
constexpr int kTcMaxGroup = 4;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s: the default limit of every wait

// ---- PTX wrappers (tcgen05 / mbarrier / TMA) --------------------------------

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// Test for the completion of the phase with the given parity; while it is not
// complete the thread may be suspended (not polling) until it completes or
// suspend_ns pass.
constexpr uint32_t kSuspendNs = 100000;  // 100 us, at most
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t suspend_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(suspend_ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// Contiguous global -> shared bulk copy completing on an mbarrier, with an L2
// cache policy. Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                               uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// K-major, SWIZZLE_128B shared-memory matrix descriptor: start address, LBO
// (unused for swizzled K-major, set to 16 B), SBO = 1024 B between 8-row groups,
// descriptor version 1, layout type 2 (128B swizzle).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFF) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// K-major, unswizzled shared-memory matrix descriptor: start address, LBO = byte
// distance between core matrices adjacent in K, SBO = byte distance between
// 8-row groups, descriptor version 1, layout type 0 (no swizzle).
__device__ __forceinline__ uint64_t smem_desc_interleave(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFF) >> 4);
  d |= static_cast<uint64_t>((lbo & 0x3FFFF) >> 4) << 16;
  d |= static_cast<uint64_t>((sbo & 0x3FFFF) >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
// The same MMA with the A operand in tensor memory: lane = row of A, 32-bit
// column c = K elements 2c (low half) and 2c + 1.
__device__ __forceinline__ void tc_mma_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// N consecutive 32-bit columns of this thread's TMEM lane from registers (N = 16 or 32).
template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const uint32_t *r) {
  if constexpr (N == 32) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
  } else {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::
            "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
  }
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// (d0, d1) += (a0 * b0, a1 * b1), each a fused multiply-add rounded to nearest.
__device__ __forceinline__ void ffma2(float &d0, float &d1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rd, {%0, %1};\n fma.rn.f32x2 rd, ra, rb, rd;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

struct TcArgs {
  Shape sh;
  int R;               // rows per sequence
  int G;               // rows per group
  int groups_per_seq;  // ceil(R / G)
  int npad;            // MMA N (multiple of 16, <= 256)
  int hp;              // TMEM columns per row of the group (H_I, or npad when G == 1)
  int ncols;           // TMEM columns of one accumulator (power of two >= 32)
  int acc_log2;        // log2 of the accumulators in TMEM (2 or 4)
  int tmem_cols;       // TMEM columns allocated: the accumulators (+ MX: the A stages), a power of two
  int bpp_log2;        // log2(blocks per page)
  const int32_t *seq_ids;
  const int32_t *pos0;
  const int32_t *page_table;
  int max_pages;
  int num_pages;
  const uint8_t *keys;   // compressed-key pool (tiled pages: bf16, or the MXFP8 plane)
  const float *w;
  float *scores;
  int ld;
  int32_t *status;
  unsigned long long wait_limit_ns;  // limit of every mbarrier wait (qsa_set_wait_limit_ns)
  int n_groups;        // groups of rows (n_seq * groups_per_seq)
  int q_in_step;       // the queries are written by this step's first kernel: load them only
                       // after the dependency wait
};

constexpr int kMaxEpiWarps = 4 * kTcMaxGroup;  // one per (row of the group, TMEM lane quarter)
// warp 0: producer, warp 1: MMA issuer, then epilogue warps (bf16: up to 4 x 4);
// MXFP8: then 8 converter warps and a second producer warp, with G <= 2
constexpr int kMaxThreads = 64 + 32 * kMaxEpiWarps;       // bf16 keys
constexpr int kMaxThreadsFp8 = 64 + 32 * 8 + 32 * 8 + 32;  // MXFP8 keys
constexpr int kMaxStages = 12;     // producer ring (bf16 keys: at most kMaxStagesBf16)
constexpr int kMaxStagesBf16 = 6;
constexpr int kMaxCStages = 4;     // MXFP8: bf16 A stages in TMEM filled by the converter warps
constexpr int kConvWarps = 8;      // MXFP8: converter warps, 4 per copy ring, a block row per thread
constexpr int kRowCols = 64;  // head columns of one row, at most
// shared memory of the epilogue: per warp the weights of its row in two
// buffers [2][kRowCols] (the current group's, and the next one's fetched ahead)
constexpr int kEpiFloats = kMaxEpiWarps * 2 * kRowCols;
constexpr int kMaxAcc = 4;  // TMEM accumulators, at most
constexpr int kNumBars = 2 * kMaxStages + 4 + 2 * kMaxAcc + 2 * kMaxCStages + 2;  // MX keys
constexpr int kNumBarsBf16 = 2 * kMaxStagesBf16 + 4 + 2 * kMaxAcc;               // bf16 keys

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Bounded wait that also gives up when another role has aborted the CTA.
// limit_ns: the wait's time limit (kWaitLimitNs unless a test shortened it); the
// suspend hint stays well below it, so an expired wait is noticed in time.
__device__ __forceinline__ bool mbar_wait_or_abort(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                                   int32_t *status, unsigned long long limit_ns) {
  const uint32_t hint = static_cast<uint32_t>(limit_ns / 4 < kSuspendNs ? limit_ns / 4 : kSuspendNs);
  if (mbar_try_wait(bar, parity, hint)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity, hint)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      report(status, QSA_ERR_TIMEOUT);
      return false;
    }
  }
}

// The same wait taken by a whole warp (every lane polls): the verdict is made
// warp-uniform, so a lane that saw the phase complete cannot run on while
// another lane gave up (the warp's later full-mask shuffles and syncs would
// then never complete).
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                               int32_t *status, unsigned long long limit_ns) {
  return __all_sync(0xffffffffu, mbar_wait_or_abort(bar, parity, abort_flag, status, limit_ns));
}

// Tiles of 128 blocks that group g needs, its sequence's pos0 being p0 (0 when
// its last row is dense or its position is outside the page table; the select
// kernel reports the latter).
__device__ __forceinline__ int group_tiles(const TcArgs &a, int g, int p0) {
  const int i = g / a.groups_per_seq;
  const int j0 = (g - i * a.groups_per_seq) * a.G;
  const int g_rows = min(a.G, a.R - j0);
  const int vis_last = p0 + j0 + g_rows;
  if (p0 + j0 + 1 < 1 || vis_last > a.max_pages * a.sh.page) return 0;
  const int nb = vis_last >> a.sh.log2_ratio;
  return nb > a.sh.topk ? (nb + kTcTileBlocks - 1) / kTcTileBlocks : 0;
}

// 32 consecutive groups held by a warp, one per lane: the group's tile count,
// and its sequence's pos0 and slot. Every role walks its items through such a
// chunk, so moving from one group to the next is a shuffle, not a global load;
// a new chunk costs one round trip (pos0 and seq_ids load side by side).
struct GroupChunk {
  int base = -1;  // first group of the chunk
  int tiles = 0, p0 = 0, seq = 0;
};

__device__ __forceinline__ void chunk_load(GroupChunk &c, const TcArgs &a, int base, int lane) {
  c.base = base;
  const int g = base + lane;
  c.tiles = 0;
  c.p0 = 0;
  c.seq = 0;
  if (g < a.n_groups) {
    const int i = g / a.groups_per_seq;
    c.p0 = a.pos0[i];
    c.seq = a.seq_ids[i];
    c.tiles = group_tiles(a, g, c.p0);
  }
}

// Warp-collective: moves the chunk to group g's 32 groups when needed; then
// group g's entries are lane g - c.base's.
__device__ __forceinline__ int chunk_lane(GroupChunk &c, const TcArgs &a, int g, int lane) {
  if (g < c.base || g >= c.base + 32) chunk_load(c, a, g & ~31, lane);
  return g - c.base;
}
__device__ __forceinline__ int chunk_tiles(GroupChunk &c, const TcArgs &a, int g, int lane) {
  const int src = chunk_lane(c, a, g, lane);
  return __shfl_sync(0xffffffffu, c.tiles, src);
}
__device__ __forceinline__ int chunk_p0(GroupChunk &c, const TcArgs &a, int g, int lane) {
  const int src = chunk_lane(c, a, g, lane);
  return __shfl_sync(0xffffffffu, c.p0, src);
}
__device__ __forceinline__ int chunk_seq(GroupChunk &c, const TcArgs &a, int g, int lane) {
  const int src = chunk_lane(c, a, g, lane);
  return __shfl_sync(0xffffffffu, c.seq, src);
}

// The work of a CTA is a contiguous range of the (group, tile) items in
// group-major order; every role walks the same range independently.
struct Walker {
  int g, t, tiles, left;
};

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// Warp-collective: total items, then this CTA's first item; leaves the chunk
// of that item's group loaded.
__device__ __forceinline__ Walker walker_start(const TcArgs &a, GroupChunk &c, int lane) {
  const int n_groups = a.n_groups;
  int total = 0;
  for (int g0 = 0; g0 < n_groups; g0 += 32) {
    if (c.base != g0) chunk_load(c, a, g0, lane);
    total += __shfl_sync(0xffffffffu, warp_incl_scan(c.tiles, lane), 31);
  }
  const long long first = static_cast<long long>(total) * blockIdx.x / gridDim.x;
  const long long last = static_cast<long long>(total) * (blockIdx.x + 1) / gridDim.x;
  Walker w{n_groups, 0, 0, static_cast<int>(last - first)};
  if (w.left <= 0) return w;
  int base = 0;
  for (int g0 = 0; g0 < n_groups; g0 += 32) {
    if (c.base != g0) chunk_load(c, a, g0, lane);
    const int incl = warp_incl_scan(c.tiles, lane);
    const int tot = __shfl_sync(0xffffffffu, incl, 31);
    if (base + tot > first) {
      const unsigned m = __ballot_sync(0xffffffffu, base + incl > first);
      const int src = __ffs(m) - 1;
      const int tl_s = __shfl_sync(0xffffffffu, c.tiles, src);
      const int incl_s = __shfl_sync(0xffffffffu, incl, src);
      w.g = g0 + src;
      w.tiles = tl_s;
      w.t = static_cast<int>(first - (base + incl_s - tl_s));
      return w;
    }
    base += tot;
  }
  return w;
}

// Warp-collective: the next item.
__device__ __forceinline__ void walker_next(Walker &w, const TcArgs &a, GroupChunk &c, int lane) {
  --w.left;
  if (++w.t < w.tiles) return;
  w.t = 0;
  do {
    ++w.g;
    w.tiles = w.g < a.n_groups ? chunk_tiles(c, a, w.g, lane) : 0;
  } while (w.g < a.n_groups && w.tiles == 0 && w.left > 0);
  if (w.g >= a.n_groups) w.left = 0;
}

// Warp-collective: the first group after g with tiles to score in g's chunk
// (-1 if none there): the group whose inputs a role may fetch ahead.
__device__ __forceinline__ int chunk_next_group(const GroupChunk &c, int g, int lane) {
  const unsigned m = __ballot_sync(0xffffffffu, c.base + lane > g && c.tiles > 0);
  return m ? c.base + __ffs(m) - 1 : -1;
}

// A batch of up to 32 / pages_in_tile consecutive tiles of one group, as the
// producer warp sees it: lane L holds the page id of page L of the batch.
struct Batch {
  int nb = 0;        // tiles in the batch
  int row0 = 0;      // first row of the group
  int nblk_old = 0;  // blocks of the sequence complete before this step's appends
  int pg = 0;        // this lane's page id (fetch_page_id)
  bool have = false; // this lane's page holds a visible block
  const int32_t *pid = nullptr;  // where this lane's page id is
};

// Warp-collective. The group's first row, the blocks visible to its last row
// and its sequence's page-table row come from the chunk; the page id itself is
// fetched by fetch_page_id, one load per lane, a batch ahead of its use.
__device__ __forceinline__ Batch load_batch(const TcArgs &a, const Walker &w, GroupChunk &c, int lane,
                                            int per_batch, int pages_in_tile, int bpp) {
  const int i = w.g / a.groups_per_seq;
  const int j0 = (w.g - i * a.groups_per_seq) * a.G;
  const int g_rows = min(a.G, a.R - j0);
  const int p0 = chunk_p0(c, a, w.g, lane);
  const int seq = chunk_seq(c, a, w.g, lane);
  const int nblk_last = (p0 + j0 + g_rows) >> a.sh.log2_ratio;
  const int32_t *ptab = a.page_table + static_cast<size_t>(seq) * a.max_pages;
  Batch b;
  b.row0 = i * a.R + j0;
  b.nblk_old = p0 >> a.sh.log2_ratio;
  b.nb = min(min(per_batch, w.tiles - w.t), w.left);
  const int pidx = w.t * pages_in_tile + lane;
  b.have = lane < b.nb * pages_in_tile && pidx * bpp < nblk_last;
  b.pid = ptab + pidx;
  return b;
}

// The page id of a batch's lane: a predicated load straight into b.pg, issued
// after any merge of Batch values. A page id merged with another value by a
// select (a batch or an empty one) would be waited for at the select, not where
// it is first used (a batch later), and hold up the current batch's copies by a
// memory round trip.
__device__ __forceinline__ void fetch_page_id(Batch &b) {
  b.pg = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %2, 0;\n\t@p ld.global.b32 %0, [%1];\n}"
      : "+r"(b.pg)
      : "l"(b.pid), "r"(static_cast<unsigned>(b.have))
      : "memory");
}

// Two E4M3 bytes of w (moved by prmt selector SEL into bytes 1 and 3) -> a
// bf16 pair, times the block scale 2^e. With an E4M3 byte as the high byte of a
// 16-bit half, its sign is already the bf16 sign; its exponent and mantissa
// bits, shifted right by 4, become a bf16's low exponent bits and top mantissa
// bits, which read as a bf16 of value x * 2^-120 -- for subnormal E4M3 too (as a
// bf16 subnormal) -- so one exact bf16 multiply by 2^(120 + e) finishes it:
// prmt, shift, lop3, mul.bf16x2, no conversion instructions. sc2 holds
// 2^(120 + e) in both halves (e <= 7), or 2^120 with a second multiply by 2^e
// (sc2b) for larger scales.
template <uint32_t SEL>
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t w, uint32_t sc2, uint32_t sc2b, bool two_step) {
  uint32_t y, r;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(y) : "r"(w), "n"(SEL));
  const uint32_t t = (y & 0x80008000u) | ((y >> 4) & 0x07F007F0u);
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(t), "r"(sc2));
  if (two_step) asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(r), "r"(sc2b));
  return r;
}

// Byte K of w (two E2M1 codes: the low nibble the even element) -> a bf16 pair,
// times the block scale 2^e. An E2M1 code's magnitude bits placed as a bf16's
// low exponent bits and top mantissa bit, its sign as the bf16 sign, read as
// x * 2^-126 (the subnormal code 0.5 too), so one exact bf16 multiply by
// 2^(126 + e) finishes it (sc2; e <= 1, else 2^126 and then 2^e in sc2b).
// w_hi = w >> 4 holds byte K's high nibble in its byte K's low bits, so one
// prmt (byte K of w into byte 0, byte K of w_hi into byte 2) puts the low
// nibble at bits 0-3 and the high nibble at 16-19; the other bits are masked.
template <int K>
__device__ __forceinline__ uint32_t e2m1x2_to_bf16x2(uint32_t w, uint32_t w_hi, uint32_t sc2, uint32_t sc2b,
                                                     bool two_step) {
  uint32_t y;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(y) : "r"(w), "r"(w_hi), "n"(K | (K << 4) | ((4 + K) << 8) | ((4 + K) << 12)));
  const uint32_t t = ((y & 0x00070007u) << 6) | ((y & 0x00080008u) << 12);
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(t), "r"(sc2));
  if (two_step) asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(r), "r"(sc2b));
  return r;
}

// bf16 bits of 2^e (e in [-126, 127]), in both halves of a word.
__device__ __forceinline__ uint32_t bf16x2_pow2(int e) {
  const uint32_t h = static_cast<uint32_t>(e + 127) << 7;
  return h | (h << 16);
}

// Shared memory (1024-aligned):
//   bf16 keys:  [A stages: S x tile][B slots][epilogue][barriers][tmem address][abort flag]
//   MXFP8 keys: [B slots][byte ring: S x 128 blocks of d_I + d_I/32 bytes][epilogue]
//               [barriers][tmem address][abort flag]; the bf16 A tiles live in TMEM
// A tile is 128 rows x d_I bf16 in the K-major core-matrix layout; a B slot is
// DI/64 halves x npad rows x 128 B (128B swizzle). TMEM: 2 or 4 accumulators
// of ncols columns, then (MX planes) kMaxCStages A tiles of d_I / 2 columns.
template <int DI, bool FP8, bool FP4 = false>
__global__ void __launch_bounds__(FP8 ? kMaxThreadsFp8 : kMaxThreads, 1)
score_tc_kernel(const __grid_constant__ CUtensorMap tm_q, TcArgs a, int n_stages) {
  // FP8: an MX plane (the converter path); FP4: that plane is MXFP4, else MXFP8
  static_assert(!FP4 || FP8, "MXFP4 runs on the MX path");
  constexpr int HALVES = DI / 64;
  constexpr int A_STAGE = kTcTileBlocks * DI * 2;  // one tile of keys, tiled pages back to back
  constexpr int R_STAGE = FP4 ? kTcTileBlocks * (DI / 2 + DI / 32)
                              : (FP8 ? kTcTileBlocks * (DI + DI / 32) : A_STAGE);  // one tile as copied
  constexpr int N_OP = FP8 ? kMaxCStages : 0;      // operand stages besides the copy ring
  constexpr int N_OPD = FP8 ? kMaxCStages : 1;     // the same as a divisor (bf16: unused)
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  const uint32_t base_u = (raw_u + 1023u) & ~1023u;
  uint8_t *base = smem_raw + (base_u - raw_u);
  const int S = n_stages;
  // copy rings: MXFP8 keeps one per producer warp (even and odd tiles), each with
  // its own converter warps, so a late page copy holds up only its own ring; bf16
  // keeps one ring, filled by the one producer and drained by the MMA
  constexpr int NR = FP8 ? 2 : 1;
  const int S_R = S / NR;
  const uint32_t a_u = base_u;  // bf16: the copy ring holds the MMA's A tiles
  const uint32_t b_half = a.npad * 128;
  const uint32_t b_slot = HALVES * b_half;
  const uint32_t b_u = FP8 ? base_u : a_u + S * A_STAGE;
  const uint32_t r_u = FP8 ? b_u + 2 * b_slot : a_u;  // where the producers' copies land
  float *ws = reinterpret_cast<float *>(base + (FP8 ? 2 * b_slot + S * R_STAGE : S * A_STAGE + 2 * b_slot));
  // barriers: MS copy stages (full, then empty), 2 B slots (full, empty), 2 TMEM
  // buffers (full, empty), then (MXFP8) the A stages (full, empty) and 2 query slots
  constexpr int MS = FP8 ? kMaxStages : kMaxStagesBf16;
  constexpr int NBARS = FP8 ? kNumBars : kNumBarsBf16;
  const uint32_t bars = smem_u32(ws + kEpiFloats);
  // barrier addresses
  auto a_full = [&](int s) { return bars + 8u * s; };
  auto a_empty = [&](int s) { return bars + 8u * (MS + s); };
  auto b_full = [&](int s) { return bars + 8u * (2 * MS + s); };
  auto b_empty = [&](int s) { return bars + 8u * (2 * MS + 2 + s); };
  auto t_full = [&](int s) { return bars + 8u * (2 * MS + 4 + s); };
  auto t_empty = [&](int s) { return bars + 8u * (2 * MS + 4 + kMaxAcc + s); };
  constexpr int CB = 2 * MS + 4 + 2 * kMaxAcc;  // first MX barrier
  auto c_full = [&](int s) { return bars + 8u * (CB + s); };
  auto c_empty = [&](int s) { return bars + 8u * (CB + kMaxCStages + s); };
  auto q_ready = [&](int s) { return bars + 8u * (CB + 2 * kMaxCStages + s); };
  // TMEM accumulators: tile k accumulates into buffer k % n_acc
  const int n_acc = 1 << a.acc_log2, acc_mask = n_acc - 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ws + kEpiFloats + 2 * NBARS);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const Shape &sh = a.sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_groups = a.n_groups;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(a_full(s), 1);
      mbar_init(a_empty(s), FP8 ? kConvWarps / NR : 1);  // the ring's converter warps, or the MMA's commit
    }
    for (int s = 0; s < N_OP; ++s) {
      mbar_init(c_full(s), kConvWarps / NR);  // the converter warps of the tile's ring
      mbar_init(c_empty(s), 1);
    }
    if (FP8)
      for (int s = 0; s < 2; ++s) mbar_init(q_ready(s), kConvWarps);  // the group's queries MX-rounded
    for (int s = 0; s < 2; ++s) {
      mbar_init(b_full(s), 1);
      mbar_init(b_empty(s), 1);
    }
    for (int s = 0; s < n_acc; ++s) {
      mbar_init(t_full(s), 1);
      mbar_init(t_empty(s), 32 * 4 * a.G);  // every epilogue thread
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), a.tmem_cols);
  const int bpp = 1 << a.bpp_log2;
  const int pages_in_tile = kTcTileBlocks >> a.bpp_log2;
  const uint32_t page_bytes = FP4 ? static_cast<uint32_t>(fp4_page_bytes(bpp, DI))
                              : (FP8 ? static_cast<uint32_t>(fp8_page_bytes(bpp, DI)) : static_cast<uint32_t>(bpp) * DI * 2);
  // MXFP8: a second producer warp (the last one) for the second copy ring
  const int prod2 = FP8 ? static_cast<int>(blockDim.x >> 5) - 1 : -1;
  const int per_batch = 32 / pages_in_tile;
  // Every role's first item, and the producers' first page ids, before the
  // block barrier: these two round trips (positions and slots side by side,
  // then the page ids) overlap the barrier set-up and the TMEM allocation.
  GroupChunk chunk;
  const Walker w0 = walker_start(a, chunk, lane);
  Batch cur0;
  if ((warp == 0 || warp == prod2) && w0.left > 0) cur0 = load_batch(a, w0, chunk, lane, per_batch, pages_in_tile, bpp);
  fetch_page_id(cur0);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp == 0 || warp == prod2) {
    // ---------------- producers ----------------
    // MXFP8: two producer warps issue alternate tiles (warp 0 the even ones and
    // every query load), each into its own ring: one in-order stream of random
    // page copies tops out near 1.3 G pages/s on this part, two independent
    // ones carry nearly 1.8. Both walk the same (group, tile) sequence.
    // Tiles are issued in batches of consecutive tiles of one group: lane L
    // holds the page id of page L of the batch. The next batch is worked out
    // (walker, page ids) once the current batch's copies are out, so its
    // page-id loads overlap the ring's draining rather than delaying the
    // current copies (worked out first, the next batch held the current one's
    // copies back by about 0.8 us per step). Tiles whose blocks were all complete before this step
    // (pooled by earlier steps) need nothing from the append kernel: up to a
    // ring's worth of them is issued before the dependency wait, so their HBM
    // latency overlaps the append.
    const int par = warp == 0 ? 0 : 1;
    Walker w = w0;
    const uint64_t stream_policy = l2_evict_first();
    Batch cur = cur0;
    int cur_g = -1, gseq = -1, k = 0;
    bool ok = true, waited = false;
    // a query load held back until the dependency wait (queries written this step)
    bool pend = false;
    int pend_bs = 0, pend_row0 = 0;
    auto wait_now = [&]() {
      pdl_wait();  // blocks completed by this step come from the append kernel
      pdl_trigger();
      waited = true;
      if (pend && lane == 0) {
        mbar_arrive_expect_tx(b_full(pend_bs), b_slot);
#pragma unroll
        for (int hh = 0; hh < HALVES; ++hh)
          tma_load_2d(b_u + pend_bs * b_slot + hh * b_half, &tm_q, b_full(pend_bs), hh * 64, pend_row0 * sh.h_idx);
      }
      pend = false;
    };
    while (ok && w.left > 0) {
      if (par == 0 && w.g != cur_g) {
        ++gseq;
        const int bs = gseq & 1;
        // at most the first group's query load waits for the dependency wait
        if (a.q_in_step && !waited && gseq >= 1) wait_now();
        if (gseq >= 2 && !mbar_wait_warp(b_empty(bs), ((gseq >> 1) - 1) & 1, abort_flag, a.status, a.wait_limit_ns)) break;
        if (a.q_in_step && !waited) {
          pend = true;
          pend_bs = bs;
          pend_row0 = cur.row0;
        } else if (lane == 0) {
          mbar_arrive_expect_tx(b_full(bs), b_slot);
#pragma unroll
          for (int hh = 0; hh < HALVES; ++hh)
            tma_load_2d(b_u + bs * b_slot + hh * b_half, &tm_q, b_full(bs), hh * 64, cur.row0 * sh.h_idx);
        }
        cur_g = w.g;
      }
      // a page id outside the pool is reported and not copied (its blocks score garbage)
      const bool bad_page = cur.have && (cur.pg < 0 || cur.pg >= a.num_pages);
      if (bad_page) report(a.status, QSA_ERR_PAGE);
      const bool load = cur.have && !bad_page;
      const unsigned have_mask = __ballot_sync(0xffffffffu, load);
      for (int it = 0; it < cur.nb; ++it, ++k) {
        // tile k: ring k % NR, that ring's tile kr = k / NR, stage kr % S_R of the ring
        const int kr = k / NR;
        const int s = (k % NR) * S_R + kr % S_R;
        if (!waited && (kr >= S_R || (w.t + it + 1) * kTcTileBlocks > cur.nblk_old)) wait_now();
        if (NR == 2 && (k & 1) != par) continue;  // the other producer's tile
        if (kr >= S_R && !mbar_wait_warp(a_empty(s), ((kr / S_R) - 1) & 1, abort_flag, a.status, a.wait_limit_ns)) {
          ok = false;
          break;
        }
        const unsigned mine = (pages_in_tile == 32 ? 0xffffffffu : ((1u << pages_in_tile) - 1u))
                              << (it * pages_in_tile);
        const int n_load = __popc(have_mask & mine);
        if (lane == 0) mbar_arrive_expect_tx(a_full(s), static_cast<uint32_t>(n_load) * page_bytes);
        __syncwarp();
        if (load && ((mine >> lane) & 1u)) {
          const int slot = lane - it * pages_in_tile;
          bulk_load_hint(r_u + s * R_STAGE + slot * page_bytes, a.keys + static_cast<size_t>(cur.pg) * page_bytes,
                         page_bytes, a_full(s), stream_policy);
        }
      }
      // the next batch, once this one's copies are out: its page ids arrive
      // while the ring drains
      for (int it = 0; it < cur.nb; ++it) walker_next(w, a, chunk, lane);
      cur = w.left > 0 ? load_batch(a, w, chunk, lane, per_batch, pages_in_tile, bpp) : Batch{};
      fetch_page_id(cur);
    }
    if (!waited) wait_now();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    Walker w = w0;
    int cur_g = -1, gseq = -1;
    const uint32_t idesc = idesc_bf16_f32(kTcTileBlocks, a.npad);
    for (int k = 0; w.left > 0; ++k) {
      const int s = FP8 ? k % N_OPD : k % S;  // operand stage
      const int buf = k & acc_mask;
      bool ok = true;
      if (lane == 0)
        ok = FP8 ? mbar_wait_or_abort(c_full(s), (k / N_OPD) & 1, abort_flag, a.status, a.wait_limit_ns)
                 : mbar_wait_or_abort(a_full(s), (k / S) & 1, abort_flag, a.status, a.wait_limit_ns);
      int bs = gseq & 1;
      if (w.g != cur_g) {
        ++gseq;
        bs = gseq & 1;
        if (lane == 0 && ok)
          ok = mbar_wait_or_abort(FP8 ? q_ready(bs) : b_full(bs), (gseq >> 1) & 1, abort_flag, a.status, a.wait_limit_ns);
        cur_g = w.g;
      }
      if (lane == 0 && ok && k >= n_acc)
        ok = mbar_wait_or_abort(t_empty(buf), ((k >> a.acc_log2) - 1) & 1, abort_flag, a.status, a.wait_limit_ns);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (lane == 0) {
        tc_fence_after();
        const uint32_t d = tmem + buf * a.ncols;
#pragma unroll
        for (int kk = 0; kk < DI / 16; ++kk) {
          const int hh = kk >> 2, k4 = kk & 3;
          const uint64_t bd = smem_desc_sw128(b_u + bs * b_slot + hh * b_half + k4 * 32);
          if (FP8) {
            // K step kk: columns 8kk .. 8kk+7 of the A tile in TMEM
            tc_mma_ta(d, tmem + n_acc * a.ncols + s * (DI / 2) + kk * 8, bd, idesc, kk > 0 ? 1u : 0u);
          } else {
            // K step kk: core matrices 2kk and 2kk+1 along K
            const uint64_t ad = smem_desc_interleave(a_u + s * A_STAGE + kk * 256, 128, DI * 16);
            tc_mma(d, ad, bd, idesc, kk > 0 ? 1u : 0u);
          }
        }
        tc_commit(FP8 ? c_empty(s) : a_empty(s));
        tc_commit(t_full(buf));
      }
      walker_next(w, a, chunk, lane);
      if (lane == 0 && (w.left <= 0 || w.g != cur_g)) tc_commit(b_empty(bs));
    }
  } else if (FP8 && warp >= 2 + 4 * a.G) {
    // ---------------- MX converters (warps 2 + 4G .. 2 + 4G + 7) ----------------
    // Converter warps 0-3 drain ring 0 (even tiles), 4-7 ring 1 (odd tiles).
    // Thread t of converter warp w rebuilds block row b = 32 (w % 4) + t of its
    // ring's tiles -- the TMEM lane quarter w % 4 is the one the warp may write --
    // reading page slot b / bpp, row rr = b % bpp of that page (lanes 0-7 read
    // one 128-byte run: no bank conflicts), and stores the bf16 values as d_I / 2
    // columns of its lane, half a row per tcgen05.st. The A stage of tile k is
    // k % kMaxCStages, so each A stage belongs to one ring.
    const int cw = warp - 2 - 4 * a.G;
    const int q = warp & 3, rc = cw >> 2;
    const int b = q * 32 + lane;
    const int slot = b >> a.bpp_log2, rr = b & (bpp - 1);
    // a 16-byte run of the row: 16 E4M3 elements, or 32 E2M1 (one MX block)
    const uint32_t src_row = slot * page_bytes + ((rr >> 3) * (FP4 ? DI / 32 : DI / 16)) * 128 + (rr & 7) * 16;
    const uint32_t scl_off = slot * page_bytes + bpp * (FP4 ? DI / 2 : DI) + rr * (DI / 32);
    const uint32_t a_lane = tmem + (static_cast<uint32_t>(q * 32) << 16) + n_acc * a.ncols;
    Walker w = w0;
    int cur_gq = -1, gq = -1;
    for (int k = 0; w.left > 0; ++k) {
      if (w.g != cur_gq) {
        // a new group: its query tile (TMA, 128B swizzle) is MX-rounded in
        // place before the MMA may use it. Thread unit u = (row r, 32-value
        // block): the block's 4 chunks of 16 bytes sit at chunk positions
        // (c ^ (r % 8)) of the row's 128-byte line in half c / 8 of the slot.
        ++gq;
        const int bs = gq & 1;
        if (!mbar_wait_warp(b_full(bs), (gq >> 1) & 1, abort_flag, a.status, a.wait_limit_ns)) break;
        const int units = a.npad * (DI / 32);
        for (int u = cw * 32 + lane; u < units; u += kConvWarps * 32) {
          const int r = u / (DI / 32), blk = u - r * (DI / 32);
          const uint32_t line = b_u + bs * b_slot + (blk >> 1) * b_half + r * 128;
          uint32_t v[16];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v[4 * i]), "=r"(v[4 * i + 1]), "=r"(v[4 * i + 2]), "=r"(v[4 * i + 3])
                         : "r"(line + ((((blk & 1) * 4 + i) ^ (r & 7)) << 4)));
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(v[i] << 16)), fabsf(__uint_as_float(v[i] & 0xFFFF0000u))));
          const int e = FP4 ? mx4_scale_exp(amax) : mx_scale_exp(amax);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float xl = __uint_as_float(v[i] << 16), xh = __uint_as_float(v[i] & 0xFFFF0000u);
            const float lo = FP4 ? mx4_round(xl, e) : mx_round(xl, e);
            const float hi = FP4 ? mx4_round(xh, e) : mx_round(xh, e);
            v[i] = (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xFFFF0000u);  // exact in bf16
          }
#pragma unroll
          for (int i = 0; i < 4; ++i)
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(line + ((((blk & 1) * 4 + i) ^ (r & 7)) << 4)),
                         "r"(v[4 * i]), "r"(v[4 * i + 1]), "r"(v[4 * i + 2]), "r"(v[4 * i + 3])
                         : "memory");
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the MMA reads through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(q_ready(bs));
        cur_gq = w.g;
      }
      if ((k & 1) != rc) {  // the other ring's tile
        walker_next(w, a, chunk, lane);
        continue;
      }
      const int kr = k >> 1;
      const int s = rc * S_R + kr % S_R, c = k % N_OPD;
      if (!mbar_wait_warp(a_full(s), (kr / S_R) & 1, abort_flag, a.status, a.wait_limit_ns)) break;
      if (k >= N_OPD && !mbar_wait_warp(c_empty(c), ((k / N_OPD) - 1) & 1, abort_flag, a.status, a.wait_limit_ns)) break;
      const uint32_t src = r_u + s * R_STAGE;
      uint32_t scl;
      if (DI == 128)
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(scl) : "r"(src + scl_off));
      else {
        uint16_t s16;
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(s16) : "r"(src + scl_off));
        scl = s16;
      }
      if constexpr (FP4) {
#pragma unroll
        for (int hf = 0; hf < DI / 64; ++hf) {
          uint32_t o[32];  // 64 dims (two MX blocks) as bf16 pairs: 32 TMEM columns
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const int j = hf * 2 + jj;  // MX block j: dims 32j .. 32j+31, one 16-byte run
            uint32_t v0, v1, v2, v3;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
                         : "r"(src + src_row + j * 128));
            // scale 2^e: one multiply by 2^(126 + e) when that is a normal bf16
            // (e <= 1), else 2^126 then 2^e
            const int e = static_cast<int>((scl >> (8 * j)) & 0xFFu) - 127;
            const bool two = e > 1;
            const uint32_t sc2 = bf16x2_pow2(two ? 126 : 126 + e);
            const uint32_t sc2b = bf16x2_pow2(two ? e : 0);
            uint32_t *oj = o + jj * 16;  // byte k of the run: dims 32j + 2k, 32j + 2k + 1
            oj[0] = e2m1x2_to_bf16x2<0>(v0, v0 >> 4, sc2, sc2b, two);
            oj[1] = e2m1x2_to_bf16x2<1>(v0, v0 >> 4, sc2, sc2b, two);
            oj[2] = e2m1x2_to_bf16x2<2>(v0, v0 >> 4, sc2, sc2b, two);
            oj[3] = e2m1x2_to_bf16x2<3>(v0, v0 >> 4, sc2, sc2b, two);
            oj[4] = e2m1x2_to_bf16x2<0>(v1, v1 >> 4, sc2, sc2b, two);
            oj[5] = e2m1x2_to_bf16x2<1>(v1, v1 >> 4, sc2, sc2b, two);
            oj[6] = e2m1x2_to_bf16x2<2>(v1, v1 >> 4, sc2, sc2b, two);
            oj[7] = e2m1x2_to_bf16x2<3>(v1, v1 >> 4, sc2, sc2b, two);
            oj[8] = e2m1x2_to_bf16x2<0>(v2, v2 >> 4, sc2, sc2b, two);
            oj[9] = e2m1x2_to_bf16x2<1>(v2, v2 >> 4, sc2, sc2b, two);
            oj[10] = e2m1x2_to_bf16x2<2>(v2, v2 >> 4, sc2, sc2b, two);
            oj[11] = e2m1x2_to_bf16x2<3>(v2, v2 >> 4, sc2, sc2b, two);
            oj[12] = e2m1x2_to_bf16x2<0>(v3, v3 >> 4, sc2, sc2b, two);
            oj[13] = e2m1x2_to_bf16x2<1>(v3, v3 >> 4, sc2, sc2b, two);
            oj[14] = e2m1x2_to_bf16x2<2>(v3, v3 >> 4, sc2, sc2b, two);
            oj[15] = e2m1x2_to_bf16x2<3>(v3, v3 >> 4, sc2, sc2b, two);
          }
          tmem_st<32>(a_lane + c * (DI / 2) + hf * 32, o);
        }
      } else {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
      uint32_t o[DI / 4];  // half a row as bf16 pairs: d_I / 4 TMEM columns
#pragma unroll
      for (int jj = 0; jj < DI / 32; ++jj) {
        const int j = hf * (DI / 32) + jj;  // the half's 16-byte chunks of the row
        uint32_t v0, v1, v2, v3;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
                     : "r"(src + src_row + j * 128));
        // the block's scale 2^e, e = byte - 127 in [-127, 127]: one multiply by
        // 2^(120 + e) when that is a normal bf16 (e <= 7), else 2^120 then 2^e
        const int e = static_cast<int>((scl >> (8 * (j >> 1))) & 0xFFu) - 127;
        const bool two = e > 7;
        const uint32_t sc2 = bf16x2_pow2(two ? 120 : 120 + e);
        const uint32_t sc2b = bf16x2_pow2(two ? e : 0);
        // prmt 0x1404: bytes 0, 1 of the word into bytes 1 and 3 (zeros below);
        // 0x3424: bytes 2, 3
        uint32_t *oj = o + jj * 8;  // dims 16j .. 16j+15 of the row
        oj[0] = e4m3x2_to_bf16x2<0x1404>(v0, sc2, sc2b, two);
        oj[1] = e4m3x2_to_bf16x2<0x3424>(v0, sc2, sc2b, two);
        oj[2] = e4m3x2_to_bf16x2<0x1404>(v1, sc2, sc2b, two);
        oj[3] = e4m3x2_to_bf16x2<0x3424>(v1, sc2, sc2b, two);
        oj[4] = e4m3x2_to_bf16x2<0x1404>(v2, sc2, sc2b, two);
        oj[5] = e4m3x2_to_bf16x2<0x3424>(v2, sc2, sc2b, two);
        oj[6] = e4m3x2_to_bf16x2<0x1404>(v3, sc2, sc2b, two);
        oj[7] = e4m3x2_to_bf16x2<0x3424>(v3, sc2, sc2b, two);
      }
      tmem_st<DI / 4>(a_lane + c * (DI / 2) + hf * (DI / 4), o);
      }
      }
      // the MMA may read the stage once every store has landed
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(c_full(c));
        mbar_arrive(a_empty(s));
      }
      walker_next(w, a, chunk, lane);
    }
  } else {
    // ---------------- epilogue (warps 2 .. 2 + 4G) ----------------
    // Warp 2 + e reads TMEM lane quarter q = warp % 4 (its own 32 lanes) and
    // reduces row j = e / 4 of the group over all head columns of that row.
    const int e = warp - 2;
    const int q = warp & 3;
    const int j = e >> 2;  // < G: the block has 4G epilogue warps
    Walker w = w0;
    const int n16 = a.hp >> 4;  // 16-column TMEM loads of the row (hp a multiple of 16, <= 64)
    // The head weights of this warp's row in a group, copied into one of the
    // warp's two weight buffers with 4-byte cp.async (zero past H_I or past the
    // group's last row); the next group's copy runs while the current group's
    // tiles are scored, so a group change costs no global round trip.
    float *wbuf = ws + e * 2 * kRowCols;
    auto fetch_weights = [&](int g, int half) {
      const uint32_t dst = smem_u32(wbuf + half * kRowCols);
      int i = 0, row = 0;
      bool any = false;
      if (g >= 0) {
        i = g / a.groups_per_seq;
        const int jj0 = (g - i * a.groups_per_seq) * a.G;
        any = j < min(a.G, a.R - jj0);
        row = i * a.R + jj0 + j;
      }
      for (int c = lane; c < kRowCols; c += 32) {
        const bool ok = any && c < sh.h_idx;
        const float *src = ok ? a.w + static_cast<size_t>(row) * sh.h_idx + c : a.w;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst + 4u * c), "l"(src), "r"(ok ? 4 : 0)
                     : "memory");
      }
      cp_async_commit();
    };
    int cur_half = 0;                   // buffer of the current group's weights
    int nw_g = w.left > 0 ? w.g : -1;   // group whose weights sit (or land) in the other buffer
    fetch_weights(nw_g, 1);
    const float *wrow = wbuf;
    int cur_g = -1, j0 = 0, g_rows = 0, row0 = 0, p0 = 0;
    for (int k = 0; w.left > 0; ++k) {
      const int buf = k & acc_mask;
      if (w.g != cur_g) {
        const int i = w.g / a.groups_per_seq;
        j0 = (w.g - i * a.groups_per_seq) * a.G;
        g_rows = min(a.G, a.R - j0);
        row0 = i * a.R + j0;
        p0 = chunk_p0(chunk, a, w.g, lane);
        __syncwarp();  // every lane is done with the buffers' previous contents
        if (nw_g != w.g) {  // not fetched ahead (the group lies past the chunk)
          cp_async_wait<0>();
          nw_g = w.g;
          fetch_weights(nw_g, cur_half ^ 1);
        }
        cp_async_wait<0>();
        __syncwarp();
        cur_half ^= 1;
        wrow = wbuf + cur_half * kRowCols;
        cur_g = w.g;
        nw_g = chunk_next_group(chunk, w.g, lane);
        fetch_weights(nw_g, cur_half ^ 1);
      }
      if (!mbar_wait_warp(t_full(buf), (k >> a.acc_log2) & 1, abort_flag, a.status, a.wait_limit_ns)) break;
      tc_fence_after();
      const uint32_t lane_addr =
          tmem + buf * a.ncols + (static_cast<uint32_t>(q * 32) << 16) + j * a.hp;
      // the row's head columns in two halves of 32 (fewer live registers); the
      // FMA chains take the columns in the same order either way
      const float4 *w4 = reinterpret_cast<const float4 *>(wrow);
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int hf = 0; hf < kRowCols / 32; ++hf) {
        float v[32];
#pragma unroll
        for (int c = 0; c < 2; ++c)
          if (2 * hf + c < n16) tmem_ld16(lane_addr + (2 * hf + c) * 16, v + c * 16);
        tmem_ld_wait();
        if (hf == kRowCols / 32 - 1) {
          // the row is in registers: hand the TMEM buffer back to the MMA warp
          tc_fence_before();
          mbar_arrive(t_empty(buf));
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int cc = 4 * hf + c;  // 8-column group of the row
          if (cc < 2 * n16) {
            const float4 wa = w4[2 * cc], wb = w4[2 * cc + 1];
            ffma2(acc[0], acc[1], wa.x, wa.y, fmaxf(v[8 * c], 0.f), fmaxf(v[8 * c + 1], 0.f));
            ffma2(acc[2], acc[3], wa.z, wa.w, fmaxf(v[8 * c + 2], 0.f), fmaxf(v[8 * c + 3], 0.f));
            ffma2(acc[4], acc[5], wb.x, wb.y, fmaxf(v[8 * c + 4], 0.f), fmaxf(v[8 * c + 5], 0.f));
            ffma2(acc[6], acc[7], wb.z, wb.w, fmaxf(v[8 * c + 6], 0.f), fmaxf(v[8 * c + 7], 0.f));
          }
        }
      }
      const float sc = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
      if (j < g_rows) {
        const int nb = (p0 + j0 + j + 1) >> sh.log2_ratio;  // blocks visible to row j
        const int blk = w.t * kTcTileBlocks + q * 32 + lane;
        if (nb > sh.topk && blk < nb) a.scores[static_cast<size_t>(row0 + j) * a.ld + blk] = sc;
      }
      walker_next(w, a, chunk, lane);
    }
    cp_async_wait<0>();  // a weight prefetch may still be in flight
  }
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) {
    // give this CTA's own copies and MMAs time to land before its shared memory
    // and TMEM are released (bounded)
    const unsigned long long t0 = global_ns();
    while (global_ns() - t0 < 2000000ull) {
    }
  }
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, a.tmem_cols);
}

// The limit every mbarrier wait of the scorer gives up after (1 s by default);
// qsa_set_wait_limit_ns lets a test shorten it to make a wait expire.
std::atomic<unsigned long long> g_wait_limit_ns{kWaitLimitNs};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2D bf16 tensor map [rows][cols] (row stride cols*2 bytes), box box_cols x box_rows,
// 128-byte swizzle.
bool encode_2d(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
               uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

}  // namespace

bool score_tc_supported(const Shape &sh) {
  const int bpp = sh.page >> sh.log2_ratio;
  return bpp >= 8 && bpp <= 32 && (sh.d_idx == 64 || sh.d_idx == 128) && sh.h_idx <= 64;
}

cudaError_t launch_score_tc(const Shape &sh, int n_seq, int R, const int32_t *seq_ids,
                            const int32_t *pos0, const CacheView &cv, const uint16_t *q_idx,
                            const float *w, float *scores, int ld, int32_t *status, bool pdl,
                            cudaStream_t st, bool q_in_step) {
  if (n_seq == 0 || R == 0) return cudaSuccess;
  TcArgs a;
  a.q_in_step = q_in_step ? 1 : 0;
  a.sh = sh;
  a.R = R;
  // with the MXFP8 plane 8 converter warps and a second producer join, so at most
  // 2 rows share a tile (64 + 128 G + 256 + 32 threads within kMaxThreadsFp8)
  const int g_max = sh.idx_fp8 ? (kMaxThreadsFp8 - 96 - 32 * kConvWarps) / 128 : kTcMaxGroup;
  a.G = (sh.h_idx % 16 == 0) ? min(min(R, g_max), 256 / sh.h_idx) : 1;
  a.groups_per_seq = (R + a.G - 1) / a.G;
  a.npad = (a.G * sh.h_idx + 15) / 16 * 16;
  a.hp = (a.G == 1) ? a.npad : sh.h_idx;
  a.ncols = pow2_at_least(a.npad);
  // as many accumulators (4, else 2) as fit in the SM's 512 TMEM columns beside
  // the MX A stages: the MMA then runs further ahead of the epilogue and frees
  // its copy-ring stages sooner
  const int mx_cols = sh.idx_fp8 ? kMaxCStages * sh.d_idx / 2 : 0;
  a.acc_log2 = kMaxAcc * a.ncols + mx_cols <= 512 ? 2 : 1;
  a.tmem_cols = pow2_at_least((1 << a.acc_log2) * a.ncols + mx_cols);
  if (a.tmem_cols > 512) return cudaErrorInvalidValue;
  a.bpp_log2 = sh.log2_page - sh.log2_ratio;
  a.seq_ids = seq_ids;
  a.pos0 = pos0;
  a.page_table = cv.page_table;
  a.max_pages = cv.max_pages;
  a.num_pages = cv.num_pages;
  a.keys = static_cast<const uint8_t *>(cv.idxblk_pool);
  a.w = w;
  a.scores = scores;
  a.ld = ld;
  a.status = status;
  a.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);

  CUtensorMap tm_q;
  const long long total_rows = static_cast<long long>(n_seq) * R;
  if (!encode_2d(&tm_q, q_idx, sh.d_idx, static_cast<uint64_t>(total_rows) * sh.h_idx, 64, a.npad))
    return cudaErrorInvalidValue;

  a.n_groups = n_seq * a.groups_per_seq;
  const int halves = sh.d_idx / 64;
  const bool fp8 = sh.idx_fp8 != 0;
  const size_t a_stage = static_cast<size_t>(kTcTileBlocks) * sh.d_idx * 2;
  const bool fp4 = sh.idx_fp4 != 0;
  const size_t r_stage = fp4 ? static_cast<size_t>(kTcTileBlocks) * (sh.d_idx / 2 + sh.d_idx / 32)
                             : (fp8 ? static_cast<size_t>(kTcTileBlocks) * (sh.d_idx + sh.d_idx / 32) : a_stage);
  const size_t b_slots = 2ull * halves * a.npad * 128;
  const size_t fixed = 1024 + b_slots + kEpiFloats * 4 + 8 * (fp8 ? kNumBars : kNumBarsBf16) + 16;
  const size_t smem_cap = 227 * 1024;
  int stages = static_cast<int>((smem_cap - fixed) / r_stage);
  const int max_stages = fp8 ? kMaxStages : kMaxStagesBf16;
  if (stages > max_stages) stages = max_stages;
  if (fp8) stages &= ~1;  // two rings of equal depth
  if (stages < (fp8 ? 4 : 2)) return cudaErrorInvalidValue;
  size_t smem = fixed + stages * r_stage;
  // TMEM: resident CTAs x tmem_cols must stay within the SM's 512 columns so
  // tcgen05.alloc never waits on another CTA; raise the shared memory request
  // until at most 512 / tmem_cols CTAs fit on an SM.
  const size_t sm_smem = 233472;  // shared memory per SM (228 KB)
  const int max_ctas = 512 / a.tmem_cols;
  const size_t min_smem = sm_smem / (max_ctas + 1) - 1024 + 1;
  if (smem < min_smem) smem = min_smem;
  auto kern = fp4 ? (sh.d_idx == 128 ? score_tc_kernel<128, true, true> : score_tc_kernel<64, true, true>)
                  : fp8 ? (sh.d_idx == 128 ? score_tc_kernel<128, true> : score_tc_kernel<64, true>)
                        : (sh.d_idx == 128 ? score_tc_kernel<128, false> : score_tc_kernel<64, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int threads = 64 + 128 * a.G + (fp8 ? 32 * kConvWarps + 32 : 0);  // MXFP8: converters, second producer
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem)) != cudaSuccess)
    return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  if (per_sm > max_ctas) per_sm = max_ctas;
  return launch_kernel(pdl, kern, dim3(sms * per_sm), dim3(threads), smem, st, tm_q, a, stages);
  return cudaGetLastError();
}

}  // namespace qsa

// Test hook for the failure path: the limit of the scorer's mbarrier waits, in
// nanoseconds (0 restores the default of 1 s; other values are clamped to
// [1 us, 10 s]). Read when a launch is issued; returns the previous limit.
extern "C" unsigned long long qsa_set_wait_limit_ns(unsigned long long ns) {
  unsigned long long v = ns == 0 ? qsa::kWaitLimitNs : ns;
  if (v < 1000ull) v = 1000ull;
  if (v > 10000000000ull) v = 10000000000ull;
  return qsa::g_wait_limit_ns.exchange(v);
}
