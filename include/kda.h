/*
 * kda.h - C ABI of the GB300 (sm_103a) Kimi Delta Attention (KDA) library.
 *
 * KDA is the gated delta rule with a channel-wise, lower-bounded decay.  Per
 * sequence and head, with a dk x dv fp32 state S (row = key channel i,
 * column = value channel j):
 *
 *   g_t = gmin * sigmoid(exp(A_h) * z_t)                (vector over dk, gmin = -5)
 *   S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T
 *   o_t = S_t^T q_t
 *
 * Sources: "Kimi K3 Technical Report - Open Frontier Intelligence", Key
 * claims and Method (sec. 2.1 chunkwise-parallel form; sec. 2.1.1 and Fig. 3,
 * the scaled-sigmoid log-decay bounded below at gmin = -5 with a learnable
 * per-head A; sec. 2.1.2, channel-wise gating), and "How a Frontier Model Gets
 * Built, Read from the Kimi K3 Report", Technical Details (a fixed-size
 * running state replaces the KV cache).  The update itself is not printed on
 * those pages; the recurrence above is the reading this library implements.
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers of the current CUDA device,
 *    row-major (C order), 16-byte aligned.  bf16 tensors are passed as raw
 *    16-bit patterns (kda_bf16).
 *  - The caller owns all memory.  The library allocates nothing, frees
 *    nothing and never synchronises: work is enqueued on `stream` (a
 *    cudaStream_t; NULL = the legacy default stream) and the call returns.
 *  - Arguments the host can check are checked before anything is launched;
 *    a rejected call returns a non-zero kda_status and enqueues nothing.
 *    A launch failure returns KDA_ERR_CUDA.  Nothing aborts, traps or throws.
 *  - Values only the GPU sees (cu_seqlens, snap_offsets, slot and row
 *    indices) are checked by the kernels before they are used: a malformed
 *    entry is skipped (no memory outside the caller's arrays is touched) and
 *    KDA_ERR_SHAPE is recorded in the device status word (kda_device_status);
 *    the outputs of the skipped sequence or row are then undefined.
 *  - Value range: the tensor-core prefill (dk = dv = 128) carries the state
 *    and the chunk terms U = T diag(beta) V and W = U - Wk S through fp16
 *    operands (fp32 accumulation).  Entries whose magnitude would exceed the
 *    fp16 maximum 65504 are detected and recorded as KDA_ERR_RANGE in the
 *    device status word (the outputs are then undefined, never silently
 *    inf).  With unit q, k rows and beta in (0, 1), |v| <= 1024 and
 *    |S0| <= 1024 stay well inside that range.
 *  - Supported sizes: dk, dv in {64, 128}; chunk = 64; -5.5 <= gmin <= 0.
 *    The chunkwise prefill rescales 16-token sub-tiles by factors up to
 *    exp(-16 * gmin); the bound keeps them inside the bf16/fp32 range
 *    (sec. 2.1.1, Fig. 3 of the report page).
 *
 * Layouts (total = sum of sequence lengths; n = sequences or decode rows):
 *   q, k, z       [total, H, dk] bf16        v, o   [total, H, dv] bf16
 *   beta          [total, H] bf16            A      [H] fp32 (per head)
 *   states        [n, H, dk, dv] fp32 (dv contiguous)
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t kda_bf16;                 /* raw bfloat16 bit pattern */

/* Input pre-ops fused into the kernels (the `pre` flags of kda_chunk_fwd_ex,
 * kda_decode_step_ex and kda_decode_tokens; 0 = inputs used as given).  The
 * recurrence expects unit-norm q, k rows and beta in (0, 1); with these flags
 * the caller passes the projections' raw outputs and the kernels form
 *   q <- q / ||q||_2, k <- k / ||k||_2   per (token, head) row, in fp32
 *                                         (an all-zero row stays zero), and
 *   beta <- 1 / (1 + exp(-beta)),
 * right after loading them, before any other use.  The normalised rows are
 * kept in fp32 until they are combined with the decay factors (rounding them
 * to bf16 first would move the outputs by about 2.4e-2 RMS). */
#define KDA_PRE_L2NORM_QK 1u
#define KDA_PRE_SIGMOID_BETA 2u

/* Split-phase calls of kda_chunk_fwd_ex (dk = dv = 128): with
 * KDA_PASS_PREPARE the call only runs the parallel chunk-preparation pass and
 * leaves every (chunk, head)'s record in the workspace; a later call with
 * KDA_PASS_STATE and the same workspace, sizes and cu_seqlens runs only the
 * state pass from those records (q, k, v, z, beta, A are not read; S0, o,
 * S_final, snaps are).  The workspace must hold the records of all heads
 * (kda_chunk_fwd_workspace_bytes(), else KDA_ERR_WORKSPACE); both flags at
 * once, or other shapes, give KDA_ERR_UNSUPPORTED.  Used to time the passes
 * separately or to run them on different streams (order them). */
#define KDA_PASS_PREPARE 0x100u
#define KDA_PASS_STATE 0x200u

/* Test hook of kda_chunk_fwd_ex (dk = dv = 128, no workspace): the kernel
 * first waits, with a small poll limit, on an mbarrier that nothing arrives
 * on, before it issues any copy or MMA; the wait gives up, KDA_ERR_TIMEOUT
 * is recorded in the device status word and every CTA returns cleanly
 * without writing outputs.  It exercises the bounded-wait error path of the
 * tensor-core kernels; never set it otherwise. */
#define KDA_TEST_STALL 0x10000u

typedef struct CUstream_st *kda_stream_t;  /* same type as cudaStream_t */

typedef enum {
  KDA_OK = 0,
  KDA_ERR_NULL = 1,        /* a required pointer is NULL */
  KDA_ERR_SHAPE = 2,       /* inconsistent or negative sizes */
  KDA_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
  KDA_ERR_UNSUPPORTED = 4, /* dk/dv/chunk/gmin outside the supported set */
  KDA_ERR_WORKSPACE = 5,   /* workspace missing or too small */
  KDA_ERR_CUDA = 6,        /* a CUDA launch or runtime call failed */
  KDA_ERR_TIMEOUT = 7,     /* a bounded in-kernel wait gave up (device status) */
  KDA_ERR_RANGE = 8        /* an fp16 tensor-core operand overflowed (device status) */
} kda_status;

/* Human-readable name of a status code (static string, never NULL). */
const char *kda_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int kda_version(void);

/*
 * Workspace bytes for the fastest kda_chunk_fwd path at these sizes (0 when
 * that path needs none).  Pure host arithmetic; 0 for unsupported sizes.
 * The sizes assume cu_seqlens and snap_offsets are NULL when the call gives
 * them as NULL; a call with snap_offsets never takes the scan below.
 *  - Equal-length batches (cu_seqlens and snap_offsets NULL) with dk = dv = 128 whose
 *    (sequence, head) chains would fill under a quarter of the GPU (n_seq * H
 *    <= 38) and whose sequences are long run as a segment-parallel scan (each
 *    segment's zero-start state N and transition M, an fp32 chain
 *    S_start[g+1] = M_g S_start[g] + N_g, then a pass from the true segment
 *    starts).  The scan needs three [n_seq * n_segs, H, 128, 128] fp32 arrays
 *    and REQUIRES them (KDA_ERR_WORKSPACE otherwise); the value returned adds
 *    the two-pass records of every (chunk, head) (73 KiB each), with which
 *    the scan runs on the two-pass kernels (chunk preparation once, three
 *    state passes); with the arrays alone it runs on the single-pass kernel.
 *  - Other dk = dv = 128 calls run in two passes when the workspace allows:
 *    a parallel pass prepares every (chunk, head)'s state-independent part
 *    (73 KiB records), then one pass per (sequence, head) carries the state.
 *    The value returned holds the records of all heads for up to
 *    ceil(total_tokens / 64) + n_seq chunks (any split of the tokens), plus
 *    small tables (each sequence's first chunk, each chunk's first token and
 *    length, and the order in which the state pass takes the sequences:
 *    longest first; 1 KiB granules).  A smaller workspace makes the call run the heads in
 *    groups; one too small for a single head's records, or none, makes it
 *    run the single-pass kernel instead.  Either way the results are the same
 *    up to rounding.
 */
size_t kda_chunk_fwd_workspace_bytes(int n_seq, int64_t total_tokens, int H, int dk, int dv,
                                     int chunk);

/*
 * kda_chunk_fwd - chunkwise-parallel KDA prefill over a batch of sequences
 * (report page, sec. 2.1: chunkwise-parallel form; sec. 2.1.1/Fig. 3: every
 * causal tile, diagonal and off-diagonal, as a dense matmul).
 *
 *   q, k, v, z, beta, A  inputs in the layouts above; gmin = -5 for KDA.
 *   cu_seqlens  device int32 [n_seq + 1], token offsets of packed sequences
 *               (cu_seqlens[0] = 0, non-decreasing, cu_seqlens[n_seq] =
 *               total_tokens); NULL = n_seq sequences of equal length
 *               total_tokens / n_seq (must divide).  Chunks restart at each
 *               sequence start; a sequence's last chunk may be partial.
 *   S0          initial states [n_seq, H, dk, dv] fp32, or NULL for zero.
 *   o           output [total, H, dv] bf16 (round to nearest even).
 *   S_final     final states [n_seq, H, dk, dv] fp32, or NULL.
 *   snaps       chunk-boundary states for prefix caching, or NULL: the state
 *               after the first 64*j tokens of sequence s (j = 1 ..
 *               floor(L_s / 64)) is written to row snap_offsets[s] + j - 1 of
 *               a [rows, H, dk, dv] fp32 array.  S0 itself is not a snapshot.
 *   snap_offsets device int64 [n_seq + 1], prefix sums of floor(L_s / 64);
 *               may be NULL only when cu_seqlens is NULL (rows s * (T / 64)).
 *   workspace   device scratch, 16-byte aligned, of workspace_bytes bytes
 *               (see kda_chunk_fwd_workspace_bytes: required for the scan,
 *               optional otherwise; NULL allowed with 0 bytes); contents need
 *               not be zeroed and are garbage afterwards.  Calls sharing one
 *               workspace must not overlap on the GPU.
 *   Errors: KDA_ERR_NULL, _SHAPE, _ALIGN, _UNSUPPORTED, _WORKSPACE, _CUDA.
 */
int kda_chunk_fwd(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                  const kda_bf16 *z, const kda_bf16 *beta, const float *A, float gmin,
                  const int32_t *cu_seqlens, int n_seq, int64_t total_tokens, int H,
                  int dk, int dv, int chunk, const float *S0, kda_bf16 *o, float *S_final,
                  float *snaps, const int64_t *snap_offsets, void *workspace,
                  size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_chunk_fwd_ex - kda_chunk_fwd with input pre-ops: `pre` is a set of
 * KDA_PRE_* flags, optionally with one KDA_PASS_* flag (other bits:
 * KDA_ERR_UNSUPPORTED).  pre = 0 is exactly kda_chunk_fwd.  The pre-ops run inside the prefill kernels on every pass
 * (the scan's segment passes included); no normalised copy of q, k or beta is
 * written anywhere.
 */
int kda_chunk_fwd_ex(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                     const kda_bf16 *z, const kda_bf16 *beta, const float *A, float gmin,
                     const int32_t *cu_seqlens, int n_seq, int64_t total_tokens, int H,
                     int dk, int dv, int chunk, unsigned pre, const float *S0, kda_bf16 *o,
                     float *S_final, float *snaps, const int64_t *snap_offsets,
                     void *workspace, size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_chunk_fwd_noalloc - kda_chunk_fwd for callers that cannot allocate
 * device memory (no access to an allocator, or no cudaMalloc allowed on their
 * path because it can synchronise the device).  The pages have no
 * counterpart: this is a convenience of this library.
 *
 * Same arguments as kda_chunk_fwd without the workspace.  When the call
 * takes the segment-parallel scan (an equal-length batch with few long
 * chains: kda_chunk_fwd_workspace_bytes() then gives the scan's size) it
 * uses a fixed scratch array of KDA_NOALLOC_WORKSPACE_BYTES in device memory
 * that the library holds on every GPU that loads it; a scan needing more
 * runs on the single-pass kernel instead (same results up to rounding, less
 * parallel).  Every other call runs the single-pass kernel, which needs no
 * scratch.  The first call on a device
 * looks up the array's device address (with that device current); make it
 * before any stream capture.  All calls share the array: calls that overlap
 * on the GPU race.  Allocates nothing.
 */
#define KDA_NOALLOC_WORKSPACE_BYTES (32u << 20)

int kda_chunk_fwd_noalloc(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                          const kda_bf16 *z, const kda_bf16 *beta, const float *A, float gmin,
                          const int32_t *cu_seqlens, int n_seq, int64_t total_tokens, int H,
                          int dk, int dv, int chunk, const float *S0, kda_bf16 *o,
                          float *S_final, float *snaps, const int64_t *snap_offsets,
                          kda_stream_t stream);

/*
 * kda_decode_step - one token of the recurrence for n sequences on resident
 * fp32 states, updated in place (the fixed-size running state of "How a
 * Frontier Model Gets Built, Read from the Kimi K3 Report", Technical
 * Details).  Row b of q, k, v, z, beta ([n, H, ...]) is applied to state slot
 * slots[b] of state_pool [n_slots, H, dk, dv]; slots is a device int32 [n]
 * array, or NULL for slot b (then n <= n_slots).  Slots must be distinct (two
 * rows writing one slot race); a slot outside [0, n_slots) is skipped on the
 * device (its row of o is not written) and recorded as KDA_ERR_SHAPE in the
 * device status word.  o [n, H, dv] bf16 receives S_t^T q_t (the updated
 * state).
 *   Errors: KDA_ERR_NULL, _SHAPE, _ALIGN, _UNSUPPORTED, _CUDA.
 */
int kda_decode_step(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                    const kda_bf16 *z, const kda_bf16 *beta, const float *A, float gmin,
                    float *state_pool, int n_slots, const int32_t *slots, int n, int H, int dk,
                    int dv, kda_bf16 *o, kda_stream_t stream);

/* kda_decode_step_ex - kda_decode_step with KDA_PRE_* input pre-ops (pre = 0
 * is exactly kda_decode_step). */
int kda_decode_step_ex(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                       const kda_bf16 *z, const kda_bf16 *beta, const float *A, float gmin,
                       float *state_pool, int n_slots, const int32_t *slots, int n, int H,
                       int dk, int dv, unsigned pre, kda_bf16 *o, kda_stream_t stream);

/*
 * kda_decode_tokens - several tokens per sequence on resident states: the
 * serving step for multi-token decode and speculative verification (the
 * recurrence of the report page, sec. 2.1, applied to short runs on the
 * fixed-size running state).  Sequence b's tokens are rows [cu_seqlens[b],
 * cu_seqlens[b+1]) of q, k, v, z, beta (layouts as kda_chunk_fwd; any
 * lengths).  With at most 16 tokens per sequence on average the tokens are
 * applied one after another to the state held on chip (each state read once
 * and, with commit, written once); longer runs go through the chunkwise form
 * (chunks of 64).  Its state is slot slots[b] of state_pool
 * [n_slots, H, dk, dv].  o receives every token's output.  With commit != 0
 * the state after the last token is written back to the slot (in place);
 * with commit == 0 the pool is left unchanged (verify without accepting).
 * Slots must be distinct; a slot outside [0, n_slots) is skipped on the
 * device and recorded as KDA_ERR_SHAPE.  cu_seqlens (int32 [n + 1]) and
 * slots (int32 [n]) are device arrays.  pre: KDA_PRE_* input pre-ops (0 =
 * none).  The short-run kernel's copy waits are bounded: one that gives up
 * records KDA_ERR_TIMEOUT in the device status word.
 *   Errors: KDA_ERR_NULL, _SHAPE, _ALIGN, _UNSUPPORTED, _CUDA.
 */
int kda_decode_tokens(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                      const kda_bf16 *z, const kda_bf16 *beta, const float *A, float gmin,
                      const int32_t *cu_seqlens, int n, int64_t total_tokens, int H, int dk,
                      int dv, unsigned pre, float *state_pool, int n_slots,
                      const int32_t *slots, int commit,
                      kda_bf16 *o, kda_stream_t stream);

/*
 * kda_state_snapshot - restore chunk-boundary states for prefix caching
 * ("state-aware prefix caching", report page, Key claims / Infrastructure):
 * for b in [0, n) copy the H x dk x dv fp32 block at row src_idx[b] of snaps
 * ([n_rows, H, dk, dv], as written by kda_chunk_fwd) to slot dst_slots[b] of
 * state_pool ([n_slots, H, dk, dv]).  src_idx: device int64 [n]; dst_slots:
 * device int32 [n]; destinations must be distinct.  A pair with src_idx[b]
 * outside [0, n_rows) or dst_slots[b] outside [0, n_slots) is skipped on the
 * device and recorded as KDA_ERR_SHAPE.  After it, the slot is a valid S0
 * for kda_chunk_fwd on the suffix or a state for kda_decode_step.
 *   Errors: KDA_ERR_NULL, _SHAPE, _ALIGN, _UNSUPPORTED, _CUDA.
 */
int kda_state_snapshot(const float *snaps, int64_t n_rows, const int64_t *src_idx,
                       float *state_pool, int n_slots, const int32_t *dst_slots, int n, int H,
                       int dk, int dv, kda_stream_t stream);

/*
 * kda_device_status - read (and with reset != 0, clear) the library's
 * device-side status word on the current device.  Kernels record there what
 * only the GPU can see: KDA_ERR_TIMEOUT (a bounded wait gave up instead of
 * hanging), KDA_ERR_SHAPE (a malformed cu_seqlens / snap_offsets entry or an
 * out-of-range slot or row index, skipped), KDA_ERR_RANGE (an fp16 operand
 * overflowed).  The word is one per device and sticky: every call on the
 * device that runs on a stream with no word of its own (kda_stream_status_bind)
 * ORs into it until it is reset, so such calls on different streams are not
 * told apart.  This call synchronises the device.  Returns KDA_OK, the
 * recorded code(s) OR-ed together, or KDA_ERR_CUDA.
 */
int kda_device_status(int reset);

/*
 * kda_stream_status_bind - give a stream a status word of its own.  From this
 * call on, every library call issued on `stream` has its kernels OR their
 * device-side codes (the ones kda_device_status lists) into *device_word
 * instead of the device word; calls on other streams are unaffected.
 * device_word: one int in device memory (4-byte aligned), owned by the
 * caller, zeroed by the caller before first use and valid until it is
 * unbound; the library never allocates or frees it.  A call on the stream
 * captured into a CUDA graph keeps the word bound at capture time.
 * device_word == NULL removes the stream's binding (a no-op if it has none);
 * binding again replaces the word.  Host-side only: nothing is enqueued and
 * nothing synchronises.  Thread-safe.  At most 64 streams are bound at once.
 * Returns KDA_OK, KDA_ERR_ALIGN (a misaligned word) or KDA_ERR_SHAPE (64
 * streams are already bound).
 */
int kda_stream_status_bind(kda_stream_t stream, int *device_word);

/*
 * kda_stream_status - read (and with reset != 0, clear) the word bound to
 * `stream`: a copy ordered after the work already issued on that stream,
 * then a synchronisation of that stream only.  Returns KDA_OK, the recorded
 * code(s) OR-ed together, KDA_ERR_NULL (no word is bound to the stream) or
 * KDA_ERR_CUDA.
 */
int kda_stream_status(kda_stream_t stream, int reset);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
