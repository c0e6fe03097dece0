// qsa_gather_attn_static: gather attention with library-owned scratch.
//
// Some callers cannot hand the library a workspace: a plugin that receives only
// the input and output tensors from a host framework that owns every device
// allocation and offers no allocation hook, or a latency-critical loop where a
// cudaMalloc (which can synchronise the device) is not allowed. For them this
// entry point keeps the split-K partial results in a fixed array compiled into
// the library instead of a caller-provided workspace. Nothing here allocates:
// no cudaMalloc, cudaFree or allocating library call.
//
// Costs and rules of the shared array:
//   * Every GPU that loads the library holds QSA_STATIC_SCRATCH_BYTES (32 MiB) of
//     device memory for the array until the process exits.
//   * All calls on a device share the one array, and it keeps whatever the last
//     call left in it. Calls whose kernels overlap on the GPU (different
//     streams, or different host threads without ordering) race on it and give
//     wrong results; serialise them on one stream.
//   * The attention kernel writes every partial (m, l, acc) it later reads, on
//     every call, so nothing in the array has to start at zero.
//   * The array's device address is looked up once per device, with that device
//     current, on the first call made on it (cudaGetSymbolAddress). Make that
//     first call on each device before any stream capture begins.
#include <mutex>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr size_t kStaticScratchBytes = QSA_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_attn_scratch[kStaticScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_attn_scratch on the current device (looked up once).
cudaError_t scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace qsa

using namespace qsa;

extern "C" int qsa_gather_attn_static(const qsa_config *cfg, const qsa_rows *rows,
                                      const qsa_cache *cache, const qsa_bf16 *q,
                                      const int32_t *sel, const int32_t *n_sel, qsa_bf16 *out,
                                      int32_t *status, cudaStream_t stream) {
  // the same checks as qsa_gather_attn, bar the workspace
  int rc;
  if ((rc = check_cfg(cfg)) != QSA_OK) return rc;
  if ((rc = check_rows(rows)) != QSA_OK) return rc;
  if ((rc = check_cache(cache, true, false)) != QSA_OK) return rc;
  const int n_rows = rows->n_seq * rows->rows_per_seq;
  if (n_rows == 0) return QSA_OK;
  if (!q || !sel || !n_sel || !out || !aligned16(q) || !aligned16(out)) return QSA_ERR_INVALID_ARG;
  const Shape sh = make_shape(cfg);
  // the partials of this many rows must fit the fixed array
  if (attn_partial_bytes(sh, n_rows) > kStaticScratchBytes) return QSA_ERR_WORKSPACE;

  void *scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e == cudaErrorInvalidDevice) return QSA_ERR_INVALID_ARG;
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_attn(sh, rows->n_seq, rows->rows_per_seq, rows->seq_ids, rows->pos0, view(cache), q,
                                 sel, n_sel, out, scratch, status, false, CommitArgs{}, stream));
}
