// kda_chunk_fwd_noalloc: the prefill for callers that cannot allocate device
// memory themselves.
//
// Some callers have no way to get a workspace: a plain C host program that
// only holds the tensors another component gave it, a serving loop that must
// not call cudaMalloc on its hot path (cudaMalloc can synchronise the whole
// device and its latency is unbounded), or code whose memory is owned by a
// framework allocator it cannot reach.  kda_chunk_fwd needs a workspace only
// for its segment-parallel scan of long sequences with few (sequence, head)
// chains; this entry point gives that path a fixed scratch area instead: a
// file-scope device array of KDA_NOALLOC_WORKSPACE_BYTES that every GPU
// loading the library holds until the process exits.
//
// The host cannot use the array's name as a device address.  On its first
// call on a device (with that device current) the entry point asks the
// runtime for the array's device address with cudaGetSymbolAddress, checks
// the result and keeps it for later calls on that device; make that first
// call before any stream capture starts.  Nothing here calls cudaMalloc,
// cudaFree or any allocating library routine.
//
// All calls on a device share the one array and it keeps whatever the last
// call left there.  The scan writes every workspace element before reading
// it, so nothing has to be cleared between calls; but two calls that overlap
// on the GPU (different streams, no ordering between them) would overwrite
// each other's scratch: keep such calls ordered.
#include <mutex>

#include "kda_common.cuh"

namespace kda {

bool chunk_fwd_takes_scan(unsigned pre, const int32_t *cu_seqlens, const int64_t *snap_offsets,
                          int n_seq, int64_t total_tokens, int H, int dk, int dv, int chunk,
                          size_t *scan_bytes);
int chunk_fwd_run(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v, const kda_bf16 *z,
                  const kda_bf16 *beta, const float *A, float gmin, const int32_t *cu_seqlens,
                  int n_seq, int64_t total_tokens, int H, int dk, int dv, int chunk, unsigned pre,
                  const float *S0, kda_bf16 *o, float *S_final, float *snaps,
                  const int64_t *snap_offsets, void *workspace, size_t workspace_bytes,
                  kda_stream_t stream, bool allow_scan);

namespace {

static __device__ __align__(256) unsigned char g_noalloc_workspace[KDA_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
void *g_workspace_ptr[kMaxDevices] = {};
std::mutex g_workspace_mutex;

// Device address of the scratch array on the current device (set up once per
// device), or nullptr if the runtime could not provide it.
void *noalloc_workspace() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_workspace_mutex);
  if (!g_workspace_ptr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_workspace) != cudaSuccess || !ptr) return nullptr;
    g_workspace_ptr[dev] = ptr;
  }
  return g_workspace_ptr[dev];
}

}  // namespace

}  // namespace kda

extern "C" int kda_chunk_fwd_noalloc(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                                     const kda_bf16 *z, const kda_bf16 *beta, const float *A,
                                     float gmin, const int32_t *cu_seqlens, int n_seq,
                                     int64_t total_tokens, int H, int dk, int dv, int chunk,
                                     const float *S0, kda_bf16 *o, float *S_final, float *snaps,
                                     const int64_t *snap_offsets, kda_stream_t stream) {
  // Only the segment-parallel scan needs scratch, and whether a call takes it
  // is decided by the same rule kda_chunk_fwd applies; every other call gets
  // no workspace and so runs the single-pass kernel, which needs none.  A scan
  // whose scratch does not fit the fixed array runs on the single-pass kernel
  // too (the same results up to rounding, without the scan's parallelism).
  size_t need = 0;
  if (!kda::chunk_fwd_takes_scan(0u, cu_seqlens, snap_offsets, n_seq, total_tokens, H, dk, dv,
                                 chunk, &need))
    need = 0;
  const bool scan = need > 0 && need <= KDA_NOALLOC_WORKSPACE_BYTES;
  void *ws = nullptr;
  if (scan) {
    ws = kda::noalloc_workspace();
    if (!ws) return KDA_ERR_CUDA;
  }
  return kda::chunk_fwd_run(q, k, v, z, beta, A, gmin, cu_seqlens, n_seq, total_tokens, H, dk,
                            dv, chunk, 0u, S0, o, S_final, snaps, snap_offsets, ws,
                            scan ? need : 0, stream, scan);
}
