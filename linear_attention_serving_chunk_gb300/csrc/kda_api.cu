// C ABI of the KDA library: host-side argument checks and launches.
// Every entry point validates what the host can see, enqueues its kernels on
// the caller's stream and returns; nothing here allocates or synchronises
// (except kda_device_status, which says so).
#include <math.h>

#include "kda_common.cuh"

namespace kda {

// Device status word.  Kernels with bounded waits get its address as an
// argument and record KDA_ERR_TIMEOUT there instead of hanging.
__device__ int g_status = 0;

cudaError_t decode_step_launch(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                               const kda_bf16 *z, const kda_bf16 *beta, const float *A,
                               float gmin, float *pool, const int32_t *slots, int n, int H,
                               int dk, int dv, kda_bf16 *o, cudaStream_t stream);
cudaError_t snapshot_restore_launch(const float *snaps, const int64_t *src_idx, float *pool,
                                    const int32_t *dst_slots, int n, int H, int dk, int dv,
                                    cudaStream_t stream);
cudaError_t prefill_simt_launch(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                                const kda_bf16 *z, const kda_bf16 *beta, const float *A,
                                float gmin, const int32_t *cu_seqlens, int n_seq,
                                int64_t fixed_len, int H, int dk, int dv, const float *S0,
                                kda_bf16 *o, float *S_final, float *snaps,
                                const int64_t *snap_offsets, cudaStream_t stream);

bool prefill_tc_supported(int dk, int dv, int64_t total_tokens);
cudaError_t prefill_tc_launch(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                              const kda_bf16 *z, const kda_bf16 *beta, const float *A, float gmin,
                              const int32_t *cu_seqlens, int n_seq, int64_t total_tokens,
                              int64_t fixed_len, int H, const float *S0, kda_bf16 *o,
                              float *S_final, float *snaps, const int64_t *snap_offsets,
                              int *status, cudaStream_t stream);

namespace {

int *status_word() {
  void *p = nullptr;
  return cudaGetSymbolAddress(&p, g_status) == cudaSuccess ? static_cast<int *>(p) : nullptr;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool dim_ok(int d) { return d == 64 || d == 128; }

// gmin must keep exp(-16 gmin) (the largest sub-tile rescaling factor) well
// inside the fp32/bf16 range; the report's value is -5.
bool gmin_ok(float gmin) { return isfinite(gmin) && gmin <= 0.f && gmin >= -5.5f; }

}  // namespace

}  // namespace kda

using namespace kda;

extern "C" {

const char *kda_status_string(int status) {
  switch (status) {
    case KDA_OK: return "ok";
    case KDA_ERR_NULL: return "null pointer";
    case KDA_ERR_SHAPE: return "inconsistent sizes";
    case KDA_ERR_ALIGN: return "pointer not 16-byte aligned";
    case KDA_ERR_UNSUPPORTED: return "unsupported dk/dv/chunk/gmin";
    case KDA_ERR_WORKSPACE: return "workspace missing or too small";
    case KDA_ERR_CUDA: return "CUDA error";
    case KDA_ERR_TIMEOUT: return "bounded device wait timed out";
    default: return "unknown status";
  }
}

int kda_version(void) { return 100; }

size_t kda_chunk_fwd_workspace_bytes(int n_seq, int64_t total_tokens, int H, int dk, int dv,
                                     int chunk) {
  (void)n_seq; (void)total_tokens; (void)H; (void)dk; (void)dv; (void)chunk;
  return 0;
}

int kda_chunk_fwd(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v, const kda_bf16 *z,
                  const kda_bf16 *beta, const float *A, float gmin, const int32_t *cu_seqlens,
                  int n_seq, int64_t total_tokens, int H, int dk, int dv, int chunk,
                  const float *S0, kda_bf16 *o, float *S_final, float *snaps,
                  const int64_t *snap_offsets, void *workspace, size_t workspace_bytes,
                  kda_stream_t stream) {
  if (n_seq < 0 || total_tokens < 0 || H <= 0 || H > 65535) return KDA_ERR_SHAPE;
  if (!dim_ok(dk) || !dim_ok(dv) || chunk != kChunk || !gmin_ok(gmin))
    return KDA_ERR_UNSUPPORTED;
  if (n_seq == 0) return total_tokens == 0 ? KDA_OK : KDA_ERR_SHAPE;
  if (n_seq > 65535) return KDA_ERR_SHAPE;
  if (!A) return KDA_ERR_NULL;
  if (total_tokens > 0 && (!q || !k || !v || !z || !beta || !o)) return KDA_ERR_NULL;
  int64_t fixed_len = 0;
  if (!cu_seqlens) {
    if (total_tokens % n_seq != 0) return KDA_ERR_SHAPE;
    fixed_len = total_tokens / n_seq;
  } else if (snaps && !snap_offsets) {
    return KDA_ERR_NULL;
  }
  const void *ptrs[] = {q, k, v, z, beta, A, S0, o, S_final, snaps, snap_offsets, cu_seqlens};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return KDA_ERR_ALIGN;
  const size_t need = kda_chunk_fwd_workspace_bytes(n_seq, total_tokens, H, dk, dv, chunk);
  if (need > 0 && (!workspace || workspace_bytes < need)) return KDA_ERR_WORKSPACE;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (prefill_tc_supported(dk, dv, total_tokens)) {
    int *status = status_word();
    if (!status) return KDA_ERR_CUDA;
    err = prefill_tc_launch(q, k, v, z, beta, A, gmin, cu_seqlens, n_seq, total_tokens, fixed_len,
                            H, S0, o, S_final, snaps, snap_offsets, status, st);
  } else {
    err = prefill_simt_launch(q, k, v, z, beta, A, gmin, cu_seqlens, n_seq, fixed_len, H, dk, dv,
                              S0, o, S_final, snaps, snap_offsets, st);
  }
  return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_decode_step(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v, const kda_bf16 *z,
                    const kda_bf16 *beta, const float *A, float gmin, float *state_pool,
                    const int32_t *slots, int n, int H, int dk, int dv, kda_bf16 *o,
                    kda_stream_t stream) {
  if (n < 0 || H <= 0) return KDA_ERR_SHAPE;
  if (!dim_ok(dk) || !dim_ok(dv) || !gmin_ok(gmin)) return KDA_ERR_UNSUPPORTED;
  if (n == 0) return KDA_OK;
  if (static_cast<int64_t>(n) * H > 0x7fffffffLL) return KDA_ERR_SHAPE;
  if (!q || !k || !v || !z || !beta || !A || !state_pool || !o) return KDA_ERR_NULL;
  const void *ptrs[] = {q, k, v, z, beta, A, state_pool, slots, o};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return KDA_ERR_ALIGN;
  const cudaError_t err = decode_step_launch(q, k, v, z, beta, A, gmin, state_pool, slots, n, H,
                                             dk, dv, o, reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_state_snapshot(const float *snaps, const int64_t *src_idx, float *state_pool,
                       const int32_t *dst_slots, int n, int H, int dk, int dv,
                       kda_stream_t stream) {
  if (n < 0 || H <= 0 || H > 65535) return KDA_ERR_SHAPE;
  if (!dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED;
  if (n == 0) return KDA_OK;
  if (!snaps || !src_idx || !state_pool || !dst_slots) return KDA_ERR_NULL;
  const void *ptrs[] = {snaps, src_idx, state_pool, dst_slots};
  for (const void *p : ptrs)
    if (!aligned16(p)) return KDA_ERR_ALIGN;
  const cudaError_t err = snapshot_restore_launch(snaps, src_idx, state_pool, dst_slots, n, H, dk,
                                                  dv, reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_device_status(int reset) {
  int value = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return KDA_ERR_CUDA;
  if (cudaMemcpyFromSymbol(&value, g_status, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
  if (reset) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
  }
  return value == 0 ? KDA_OK : value;
}

}  // extern "C"
