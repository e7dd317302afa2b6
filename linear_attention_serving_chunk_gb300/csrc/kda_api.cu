// C ABI of the KDA library: host-side argument checks and launches.
// Every entry point validates what the host can see, enqueues its kernels on
// the caller's stream and returns; nothing here allocates or synchronises
// (except kda_device_status, which says so).
#include <math.h>

#include <mutex>

#include "kda_common.cuh"

namespace kda {

// Device status word.  Kernels get its address as an argument and OR into it
// what only the GPU can see: KDA_ERR_TIMEOUT (a bounded wait gave up instead
// of hanging), KDA_ERR_SHAPE (a malformed device-side index, skipped),
// KDA_ERR_RANGE (an fp16 operand overflowed).
__device__ int g_status = 0;

cudaError_t decode_step_launch(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                               const kda_bf16 *z, const kda_bf16 *beta, const float *A,
                               float gmin, float *pool, const int32_t *slots, int n_slots,
                               int n, int H, int dk, int dv, kda_bf16 *o, unsigned pre,
                               int *status, cudaStream_t stream);
cudaError_t decode_tokens_launch(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                                 const kda_bf16 *z, const kda_bf16 *beta, const float *A,
                                 float gmin, float *pool, const int32_t *slots, int n_slots,
                                 const int32_t *cu_seqlens, int n, int64_t total, int H, int dk,
                                 int dv, kda_bf16 *o, unsigned pre, int commit, int *status,
                                 int n_sms, cudaStream_t stream);
cudaError_t snapshot_restore_launch(const float *snaps, int64_t n_rows, const int64_t *src_idx,
                                    float *pool, int n_slots, const int32_t *dst_slots, int n,
                                    int H, int dk, int dv, int *status, cudaStream_t stream);
bool prefill_tc_supported(int dk, int dv, int64_t total_tokens);
cudaError_t prefill_tc_launch(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                              const kda_bf16 *z, const kda_bf16 *beta, const float *A, float gmin,
                              const int32_t *cu_seqlens, int n_seq, int64_t total_tokens,
                              int64_t fixed_len, int H, int dk, int dv, const float *S0,
                              kda_bf16 *o, float *S_final, float *snaps,
                              const int64_t *snap_offsets, int *status, int zero_v,
                              int s0_identity, const int32_t *slots, int n_slots, unsigned pre,
                              int test_stall, cudaStream_t stream);
cudaError_t chunk_prep_launch(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                              const kda_bf16 *z, const kda_bf16 *beta, const float *A, float gmin,
                              const int32_t *cu_seqlens, const int32_t *chunk_start,
                              const int2 *chunk_info, int n_seq,
                              int64_t total_tokens, int64_t fixed_len, int H, int dk, int dv,
                              int h0, int hg, int64_t max_tasks, uint8_t *rec, int *status,
                              unsigned pre, int n_ctas, cudaStream_t stream);
cudaError_t state_pass_launch(const uint8_t *rec, const int32_t *cu_seqlens,
                              const int32_t *chunk_start, int n_seq, int64_t fixed_len,
                              int64_t total_tokens, int H, int dk, int dv, int h0, int hg,
                              const float *S0, kda_bf16 *o, float *S_final, float *snaps,
                              const int64_t *snap_offsets, int *status, const int32_t *slots,
                              int n_slots, int zero_u, int s0_identity, float *S_final2,
                              const int32_t *order, cudaStream_t stream);
cudaError_t chunk_start_launch(const int32_t *cu_seqlens, int n_seq, int64_t total_tokens,
                               int32_t *chunk_start, int2 *chunk_info, int32_t *order,
                               int *status, cudaStream_t stream);
cudaError_t segment_combine_launch(const float *M, const float *N, const float *S0,
                                   float *S_start, float *S_final, int n_seq, int n_segs, int H,
                                   cudaStream_t stream);

namespace {

// Segment-parallel scan plan for equal-length sequences with few (sequence,
// head) chains: split each sequence into n_segs segments of seg_len tokens so
// that about kScanTargetChains segment chains run at once.  Without the scan
// a chain walks its chunks one after another and most SMs sit idle.
constexpr int kSMs = 152;
constexpr int kScanTargetChains = 4 * kSMs;
constexpr int64_t kScanMinSegment = 4096;
struct ScanPlan {
  int n_segs;
  int64_t seg_len;
};

bool plan_scan(int n_seq, int64_t total_tokens, int H, int dk, int dv, ScanPlan *plan) {
  // segment_combine_kernel chains 128 x 128 states
  if (dk != 128 || dv != 128 || n_seq <= 0 || total_tokens <= 0) return false;
  if (total_tokens % n_seq != 0) return false;
  const int64_t T = total_tokens / n_seq;
  const int64_t chains = static_cast<int64_t>(n_seq) * H;
  // The scan does about three times the work of one sequential pass, so it
  // pays only when the sequential pass would fill less than a quarter of the SMs.
  if (chains * 4 > kSMs) return false;
  int n_segs = 1;
  while (chains * n_segs < kScanTargetChains && T % (2 * n_segs) == 0 &&
         (T / (2 * n_segs)) % 64 == 0 && T / (2 * n_segs) >= kScanMinSegment)
    n_segs *= 2;
  if (n_segs < 4) return false;
  plan->n_segs = n_segs;
  plan->seg_len = T / n_segs;
  return true;
}

size_t scan_workspace_bytes(int n_seq, int H, const ScanPlan &plan) {
  // M, N and the segment start states: three [n_seq * n_segs, H, 128, 128] fp32 arrays
  return 3 * static_cast<size_t>(n_seq) * plan.n_segs * H * 128 * 128 * sizeof(float);
}

// The scan on the two-pass kernels: the three arrays, then one record per
// (chunk, head) of the whole batch.
size_t scan_records_bytes(int n_seq, int64_t total_tokens, int H) {
  return static_cast<size_t>((total_tokens / n_seq + 63) / 64) * n_seq * H * (73 * 1024);
}

// Two-pass prefill: a chunk-preparation pass over every
// (chunk, head) of a group of hg heads, then the state pass over that group's
// chains.  Workspace: the varlen tables (the chunk start of every sequence,
// the first token and length of every chunk, the state pass's order of the
// sequences; 1 KiB granules), then one record per (chunk, head of the group).  The chunk count is bounded by
// ceil(total / 64) + n_seq, which covers any split of the tokens.
constexpr size_t kRecordBytes = 73 * 1024;  // kRecBytes of kda_split.cuh

int64_t split_max_chunks(int n_seq, int64_t total_tokens) {
  return (total_tokens + 63) / 64 + n_seq;
}

size_t round_kib(size_t b) { return (b + 1023) / 1024 * 1024; }

size_t chunk_start_bytes(int n_seq) {
  return round_kib((static_cast<size_t>(n_seq) + 1) * sizeof(int32_t));
}

size_t chunk_info_bytes(int n_seq, int64_t total_tokens) {
  return round_kib(static_cast<size_t>(split_max_chunks(n_seq, total_tokens)) * sizeof(int2));
}

// [chunk_start | chunk_info | state-pass order of the sequences], then the records
size_t split_table_bytes(int n_seq, int64_t total_tokens) {
  return chunk_start_bytes(n_seq) + chunk_info_bytes(n_seq, total_tokens) +
         round_kib(static_cast<size_t>(n_seq) * sizeof(int32_t));
}

size_t split_workspace_bytes(int n_seq, int64_t total_tokens, int hg) {
  return split_table_bytes(n_seq, total_tokens) +
         static_cast<size_t>(split_max_chunks(n_seq, total_tokens)) * hg * kRecordBytes;
}

// Largest head group whose records fit in `bytes` (0: none fits).
int split_heads(int n_seq, int64_t total_tokens, int H, size_t bytes) {
  const size_t table = split_table_bytes(n_seq, total_tokens);
  if (bytes <= table) return 0;
  const size_t per_head =
      static_cast<size_t>(split_max_chunks(n_seq, total_tokens)) * kRecordBytes;
  const size_t hg = (bytes - table) / per_head;
  return static_cast<int>(hg < static_cast<size_t>(H) ? hg : static_cast<size_t>(H));
}

// Per-stream status words.  A caller that binds a device int to a stream has
// every call on that stream record into it instead of the device word: calls
// on different streams are told apart, and the caller can read its word with
// a copy ordered on its own stream, without synchronising the device.
constexpr int kMaxStatusBindings = 64;
struct StatusBinding {
  cudaStream_t stream;
  int *word;
};
std::mutex g_bind_mu;
StatusBinding g_bind[kMaxStatusBindings];
int g_n_bind = 0;

int *bound_status_word(cudaStream_t st) {
  std::lock_guard<std::mutex> lock(g_bind_mu);
  for (int i = 0; i < g_n_bind; ++i)
    if (g_bind[i].stream == st) return g_bind[i].word;
  return nullptr;
}

// The word the kernels of a call on stream st record into.
int *status_word(cudaStream_t st) {
  if (int *w = bound_status_word(st)) return w;
  void *p = nullptr;
  return cudaGetSymbolAddress(&p, g_status) == cudaSuccess ? static_cast<int *>(p) : nullptr;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool dim_ok(int d) { return d == 64 || d == 128; }

// gmin must keep exp(-16 gmin) (the largest sub-tile rescaling factor) well
// inside the fp32/bf16 range; the report's value is -5.
bool gmin_ok(float gmin) { return isfinite(gmin) && gmin <= 0.f && gmin >= -5.5f; }

bool pre_ok(unsigned pre) { return (pre & ~(KDA_PRE_L2NORM_QK | KDA_PRE_SIGMOID_BETA)) == 0; }

constexpr unsigned kPassFlags = KDA_PASS_PREPARE | KDA_PASS_STATE;

// kda_decode_tokens with at most this many tokens per sequence on average runs
// the token-by-token kernel on the state in registers (one state read, one
// write); longer runs take the chunked single-pass kernel.
constexpr int64_t kDecodeTokensRun = 16;

}  // namespace

// The one rule for whether a kda_chunk_fwd call takes the segment-parallel
// scan (shared with kda_chunk_fwd_noalloc): equal-length sequences given
// without cu_seqlens and without snap_offsets, no split-phase flag, and a
// plan that pays (few long chains).
bool chunk_fwd_takes_scan(unsigned pre, const int32_t *cu_seqlens, const int64_t *snap_offsets,
                          int n_seq, int64_t total_tokens, int H, int dk, int dv, int chunk,
                          size_t *scan_bytes) {
  ScanPlan plan;
  if ((pre & (kPassFlags | KDA_TEST_STALL)) || cu_seqlens || snap_offsets || chunk != kChunk ||
      H <= 0 || n_seq <= 0 || total_tokens <= 0 || !prefill_tc_supported(dk, dv, total_tokens) ||
      !plan_scan(n_seq, total_tokens, H, dk, dv, &plan))
    return false;
  if (scan_bytes) *scan_bytes = scan_workspace_bytes(n_seq, H, plan);
  return true;
}

}  // namespace kda

using namespace kda;

extern "C" {

const char *kda_status_string(int status) {
  switch (status) {
    case KDA_OK: return "ok";
    case KDA_ERR_NULL: return "null pointer";
    case KDA_ERR_SHAPE: return "inconsistent sizes or a malformed device-side index";
    case KDA_ERR_ALIGN: return "pointer not 16-byte aligned";
    case KDA_ERR_UNSUPPORTED: return "unsupported dk/dv/chunk/gmin";
    case KDA_ERR_WORKSPACE: return "workspace missing or too small";
    case KDA_ERR_CUDA: return "CUDA error";
    case KDA_ERR_TIMEOUT: return "bounded device wait timed out";
    case KDA_ERR_RANGE: return "value beyond the fp16 range of a tensor-core operand";
    default: return "unknown status";
  }
}

int kda_version(void) { return 200; }

size_t kda_chunk_fwd_workspace_bytes(int n_seq, int64_t total_tokens, int H, int dk, int dv,
                                     int chunk) {
  if (chunk != kChunk || H <= 0 || n_seq <= 0 || total_tokens <= 0) return 0;
  ScanPlan plan;
  if (plan_scan(n_seq, total_tokens, H, dk, dv, &plan))
    return scan_workspace_bytes(n_seq, H, plan) + scan_records_bytes(n_seq, total_tokens, H);
  if (!prefill_tc_supported(dk, dv, total_tokens)) return 0;
  return split_workspace_bytes(n_seq, total_tokens, H);
}

int kda_chunk_fwd(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v, const kda_bf16 *z,
                  const kda_bf16 *beta, const float *A, float gmin, const int32_t *cu_seqlens,
                  int n_seq, int64_t total_tokens, int H, int dk, int dv, int chunk,
                  const float *S0, kda_bf16 *o, float *S_final, float *snaps,
                  const int64_t *snap_offsets, void *workspace, size_t workspace_bytes,
                  kda_stream_t stream) {
  return kda_chunk_fwd_ex(q, k, v, z, beta, A, gmin, cu_seqlens, n_seq, total_tokens, H, dk, dv,
                          chunk, 0u, S0, o, S_final, snaps, snap_offsets, workspace,
                          workspace_bytes, stream);
}

}  // extern "C"

namespace kda {

// kda_chunk_fwd_ex; allow_scan = false runs a call that would take the
// segment-parallel scan on the single-pass kernel instead (which needs no
// scratch): the allocation-free entry point's fallback when its fixed scratch
// is too small for the scan.
int chunk_fwd_run(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v, const kda_bf16 *z,
                  const kda_bf16 *beta, const float *A, float gmin, const int32_t *cu_seqlens,
                  int n_seq, int64_t total_tokens, int H, int dk, int dv, int chunk, unsigned pre,
                  const float *S0, kda_bf16 *o, float *S_final, float *snaps,
                  const int64_t *snap_offsets, void *workspace, size_t workspace_bytes,
                  kda_stream_t stream, bool allow_scan) {
  if (n_seq < 0 || total_tokens < 0 || H <= 0 || H > 65535) return KDA_ERR_SHAPE;
  const unsigned passes = pre & kPassFlags;
  const bool stall = (pre & KDA_TEST_STALL) != 0;
  const unsigned ops = pre & ~(kPassFlags | KDA_TEST_STALL);
  if (!dim_ok(dk) || !dim_ok(dv) || chunk != kChunk || !gmin_ok(gmin) || !pre_ok(ops))
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
  if (total_tokens > 0 && !prefill_tc_supported(dk, dv, total_tokens)) return KDA_ERR_SHAPE;
  if (stall && (passes || total_tokens == 0)) return KDA_ERR_UNSUPPORTED;
  if (passes) {
    // one of the two passes on its own: all heads in one group, so the
    // records of the whole call sit in the workspace between the calls
    if (passes == kPassFlags || total_tokens == 0) return KDA_ERR_UNSUPPORTED;
    if (!workspace || !aligned16(workspace) ||
        split_heads(n_seq, total_tokens, H, workspace_bytes) < H)
      return KDA_ERR_WORKSPACE;
  }
  size_t need = 0;
  const bool scan = allow_scan && chunk_fwd_takes_scan(pre, cu_seqlens, snap_offsets, n_seq,
                                                       total_tokens, H, dk, dv, chunk, &need);
  if (scan) {
    if (!workspace || workspace_bytes < need) return KDA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return KDA_ERR_ALIGN;
  }
  // every host-side check is done: from here on the call launches work
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int *status = status_word(st);
  if (!status) return KDA_ERR_CUDA;
  if (stall) {  // test hook: the single-pass kernel gives up on an unarmed wait
    const cudaError_t err = prefill_tc_launch(
        q, k, v, z, beta, A, gmin, cu_seqlens, n_seq, total_tokens, fixed_len, H, dk, dv, S0, o,
        S_final, snaps, snap_offsets, status, 0, 0, nullptr, n_seq, ops, 1, st);
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
  }
  if (total_tokens == 0) {
    // nothing to run but the final states: S_final = S0 (or zero)
    if (S_final) {
      const size_t bytes = static_cast<size_t>(n_seq) * H * dk * dv * sizeof(float);
      const cudaError_t err = S0 ? cudaMemcpyAsync(S_final, S0, bytes, cudaMemcpyDeviceToDevice, st)
                                 : cudaMemsetAsync(S_final, 0, bytes, st);
      return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
    }
    return KDA_OK;
  }
  if (scan) {
    ScanPlan plan;
    plan_scan(n_seq, total_tokens, H, dk, dv, &plan);
    const int n2 = n_seq * plan.n_segs;
    const size_t arr = static_cast<size_t>(n2) * H * 128 * 128;
    float *Mb = static_cast<float *>(workspace), *Nb = Mb + arr, *Ss = Nb + arr;
    if (workspace_bytes >= need + scan_records_bytes(n_seq, total_tokens, H)) {
      // On the two-pass kernels: every chunk's record once, then the state
      // pass over the segments twice: N (from zero) and M (from the identity
      // with v = 0) as the two chains of one paired pass, then the outputs
      // from the true segment starts.  The records are laid out by global
      // chunk, which is also what the segment view (n2 sequences of seg_len
      // tokens) addresses.
      uint8_t *rec = static_cast<uint8_t *>(workspace) + need;
      const int64_t cps = (fixed_len + 63) / 64;
      cudaError_t err = chunk_prep_launch(q, k, v, z, beta, A, gmin, nullptr, nullptr, nullptr, n_seq,
                                          total_tokens, fixed_len, H, dk, dv, 0, H,
                                          n_seq * cps * H, rec, status, ops, kSMs, st);
      if (err == cudaSuccess)
        err = state_pass_launch(rec, nullptr, nullptr, n2, plan.seg_len, total_tokens, H, dk, dv,
                                0, H, nullptr, nullptr, Nb, nullptr, nullptr, status, nullptr, 0,
                                0, 0, Mb, nullptr, st);
      if (err == cudaSuccess)
        err = segment_combine_launch(Mb, Nb, S0, Ss, S_final, n_seq, plan.n_segs, H, st);
      if (err == cudaSuccess)
        err = state_pass_launch(rec, nullptr, nullptr, n2, plan.seg_len, total_tokens, H, dk, dv,
                                0, H, Ss, o, nullptr, snaps, nullptr, status, nullptr, 0, 0, 0,
                                nullptr, nullptr, st);
      return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
    }
    // 1. every segment from a zero state (N) and its transition from S0 = I with v = 0 (M)
    cudaError_t err = prefill_tc_launch(q, k, v, z, beta, A, gmin, nullptr, n2, total_tokens,
                                        plan.seg_len, H, dk, dv, nullptr, nullptr, Nb, nullptr,
                                        nullptr, status, 0, 0, nullptr, 0, ops, 0, st);
    if (err == cudaSuccess)
      err = prefill_tc_launch(q, k, v, z, beta, A, gmin, nullptr, n2, total_tokens, plan.seg_len,
                              H, dk, dv, nullptr, nullptr, Mb, nullptr, nullptr, status, 1, 1,
                              nullptr, 0, ops, 0, st);
    // 2. chain the segments: start states and the final state
    if (err == cudaSuccess)
      err = segment_combine_launch(Mb, Nb, S0, Ss, S_final, n_seq, plan.n_segs, H, st);
    // 3. outputs and snapshots from the true start state of every segment
    if (err == cudaSuccess)
      err = prefill_tc_launch(q, k, v, z, beta, A, gmin, nullptr, n2, total_tokens, plan.seg_len,
                              H, dk, dv, Ss, o, nullptr, snaps, nullptr, status, 0, 0, nullptr,
                              0, ops, 0, st);
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
  }
  cudaError_t err;
  const int hg = workspace && aligned16(workspace)
                     ? split_heads(n_seq, total_tokens, H, workspace_bytes)
                     : 0;
  if (hg > 0) {
    // two passes per group of hg heads: chunk preparation, then the state pass
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *chunk_start = nullptr, *order = nullptr;
    int2 *chunk_info = nullptr;
    err = cudaSuccess;
    const bool run_prep = passes != KDA_PASS_STATE, run_state = passes != KDA_PASS_PREPARE;
    if (cu_seqlens) {
      chunk_start = reinterpret_cast<int32_t *>(ws);
      chunk_info = reinterpret_cast<int2 *>(ws + chunk_start_bytes(n_seq));
      order = reinterpret_cast<int32_t *>(ws + chunk_start_bytes(n_seq) +
                                          chunk_info_bytes(n_seq, total_tokens));
      if (run_prep)
        err = chunk_start_launch(cu_seqlens, n_seq, total_tokens, chunk_start, chunk_info, order,
                                 status, st);
    }
    uint8_t *rec = ws + split_table_bytes(n_seq, total_tokens);
    const int64_t max_chunks = cu_seqlens ? split_max_chunks(n_seq, total_tokens)
                                          : static_cast<int64_t>(n_seq) * ((fixed_len + 63) / 64);
    for (int h0 = 0; h0 < H && err == cudaSuccess; h0 += hg) {
      const int g = H - h0 < hg ? H - h0 : hg;
      if (run_prep)
        err = chunk_prep_launch(q, k, v, z, beta, A, gmin, cu_seqlens, chunk_start, chunk_info, n_seq,
                                total_tokens, fixed_len, H, dk, dv, h0, g, max_chunks * g, rec,
                                status, ops, kSMs, st);
      if (err == cudaSuccess && run_state)
        err = state_pass_launch(rec, cu_seqlens, chunk_start, n_seq, fixed_len, total_tokens, H,
                                dk, dv, h0, g, S0, o, S_final, snaps, snap_offsets, status,
                                nullptr, 0, 0, 0, nullptr, order, st);
    }
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
  }
  err = prefill_tc_launch(q, k, v, z, beta, A, gmin, cu_seqlens, n_seq, total_tokens, fixed_len, H,
                          dk, dv, S0, o, S_final, snaps, snap_offsets, status, 0, 0, nullptr,
                          n_seq, ops, 0, st);
  return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda

extern "C" {

int kda_chunk_fwd_ex(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v, const kda_bf16 *z,
                     const kda_bf16 *beta, const float *A, float gmin,
                     const int32_t *cu_seqlens, int n_seq, int64_t total_tokens, int H, int dk,
                     int dv, int chunk, unsigned pre, const float *S0, kda_bf16 *o,
                     float *S_final, float *snaps, const int64_t *snap_offsets, void *workspace,
                     size_t workspace_bytes, kda_stream_t stream) {
  return kda::chunk_fwd_run(q, k, v, z, beta, A, gmin, cu_seqlens, n_seq, total_tokens, H, dk,
                            dv, chunk, pre, S0, o, S_final, snaps, snap_offsets, workspace,
                            workspace_bytes, stream, true);
}

int kda_decode_step(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v, const kda_bf16 *z,
                    const kda_bf16 *beta, const float *A, float gmin, float *state_pool,
                    int n_slots, const int32_t *slots, int n, int H, int dk, int dv, kda_bf16 *o,
                    kda_stream_t stream) {
  return kda_decode_step_ex(q, k, v, z, beta, A, gmin, state_pool, n_slots, slots, n, H, dk, dv,
                            0u, o, stream);
}

int kda_decode_step_ex(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                       const kda_bf16 *z, const kda_bf16 *beta, const float *A, float gmin,
                       float *state_pool, int n_slots, const int32_t *slots, int n, int H,
                       int dk, int dv, unsigned pre, kda_bf16 *o, kda_stream_t stream) {
  if (n < 0 || H <= 0 || n_slots < 0) return KDA_ERR_SHAPE;
  if (!dim_ok(dk) || !dim_ok(dv) || !gmin_ok(gmin) || !pre_ok(pre)) return KDA_ERR_UNSUPPORTED;
  if (n == 0) return KDA_OK;
  if (static_cast<int64_t>(n) * H > 0x7fffffffLL) return KDA_ERR_SHAPE;
  if (!slots && n > n_slots) return KDA_ERR_SHAPE;
  if (!q || !k || !v || !z || !beta || !A || !state_pool || !o) return KDA_ERR_NULL;
  const void *ptrs[] = {q, k, v, z, beta, A, state_pool, slots, o};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return KDA_ERR_ALIGN;
  int *status = status_word(reinterpret_cast<cudaStream_t>(stream));
  if (!status) return KDA_ERR_CUDA;
  const cudaError_t err = decode_step_launch(q, k, v, z, beta, A, gmin, state_pool, slots,
                                             n_slots, n, H, dk, dv, o, pre, status,
                                             reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_decode_tokens(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                      const kda_bf16 *z, const kda_bf16 *beta, const float *A, float gmin,
                      const int32_t *cu_seqlens, int n, int64_t total_tokens, int H, int dk,
                      int dv, unsigned pre, float *state_pool, int n_slots, const int32_t *slots,
                      int commit, kda_bf16 *o, kda_stream_t stream) {
  if (n < 0 || total_tokens < 0 || H <= 0 || H > 65535 || n > 65535 || n_slots < 0)
    return KDA_ERR_SHAPE;
  if (!dim_ok(dk) || !dim_ok(dv) || !gmin_ok(gmin) || !pre_ok(pre)) return KDA_ERR_UNSUPPORTED;
  if (n == 0) return total_tokens == 0 ? KDA_OK : KDA_ERR_SHAPE;
  if (!A || !state_pool || !slots || !cu_seqlens) return KDA_ERR_NULL;
  if (total_tokens > 0 && (!q || !k || !v || !z || !beta || !o)) return KDA_ERR_NULL;
  const void *ptrs[] = {q, k, v, z, beta, A, state_pool, slots, cu_seqlens, o};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return KDA_ERR_ALIGN;
  if (total_tokens == 0) return KDA_OK;  // no token: every state stays as it is
  if (!prefill_tc_supported(dk, dv, total_tokens)) return KDA_ERR_SHAPE;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  float *S_final = commit ? state_pool : nullptr;
  int *status = status_word(st);
  if (!status) return KDA_ERR_CUDA;
  if (total_tokens <= kDecodeTokensRun * static_cast<int64_t>(n) &&
      static_cast<int64_t>(n_slots) * H <= 0x7fffffffLL) {
    // short runs: the tokens one after another on the state in registers
    const cudaError_t err =
        decode_tokens_launch(q, k, v, z, beta, A, gmin, state_pool, slots, n_slots, cu_seqlens, n,
                             total_tokens, H, dk, dv, o, pre, commit, status, kSMs, st);
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
  }
  const cudaError_t err =
      prefill_tc_launch(q, k, v, z, beta, A, gmin, cu_seqlens, n, total_tokens, 0, H, dk, dv,
                        state_pool, o, S_final, nullptr, nullptr, status, 0, 0, slots, n_slots,
                        pre, 0, st);
  return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_state_snapshot(const float *snaps, int64_t n_rows, const int64_t *src_idx,
                       float *state_pool, int n_slots, const int32_t *dst_slots, int n, int H,
                       int dk, int dv, kda_stream_t stream) {
  if (n < 0 || H <= 0 || H > 65535 || n_rows < 0 || n_slots < 0) return KDA_ERR_SHAPE;
  if (!dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED;
  if (n == 0) return KDA_OK;
  if (!snaps || !src_idx || !state_pool || !dst_slots) return KDA_ERR_NULL;
  const void *ptrs[] = {snaps, src_idx, state_pool, dst_slots};
  for (const void *p : ptrs)
    if (!aligned16(p)) return KDA_ERR_ALIGN;
  int *status = status_word(reinterpret_cast<cudaStream_t>(stream));
  if (!status) return KDA_ERR_CUDA;
  const cudaError_t err =
      snapshot_restore_launch(snaps, n_rows, src_idx, state_pool, n_slots, dst_slots, n, H, dk,
                              dv, status, reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_stream_status_bind(kda_stream_t stream, int *device_word) {
  if (device_word && (reinterpret_cast<uintptr_t>(device_word) & 3u)) return KDA_ERR_ALIGN;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_bind_mu);
  for (int i = 0; i < g_n_bind; ++i)
    if (g_bind[i].stream == st) {
      if (device_word)
        g_bind[i].word = device_word;
      else
        g_bind[i] = g_bind[--g_n_bind];
      return KDA_OK;
    }
  if (!device_word) return KDA_OK;  // nothing was bound: nothing to undo
  if (g_n_bind == kMaxStatusBindings) return KDA_ERR_SHAPE;
  g_bind[g_n_bind++] = StatusBinding{st, device_word};
  return KDA_OK;
}

int kda_stream_status(kda_stream_t stream, int reset) {
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int *w = bound_status_word(st);
  if (!w) return KDA_ERR_NULL;
  int value = 0;
  if (cudaMemcpyAsync(&value, w, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return KDA_ERR_CUDA;
  if (reset && cudaMemsetAsync(w, 0, sizeof(int), st) != cudaSuccess) return KDA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return KDA_ERR_CUDA;
  return value == 0 ? KDA_OK : value;
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
