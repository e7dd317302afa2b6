// Sequential state pass of the two-pass tensor-core prefill (dk, dv in
// {64, 128}, chunk C = 64).
//
// The chunkwise form ("Kimi K3 Technical Report - Open Frontier
// Intelligence", sec. 2.1) splits every chunk into a part that depends only
// on the chunk's own inputs (the gate, A_kk, T = (I + A_kk)^{-1}, Wk, U, P
// and the scaled Q~, K') and a part that carries the state:
//
//   W  = U - Wk S                       O = Q~ S + P W  (Q~ = Q e^G)
//   S' = Diag(gamma) S + K'^T W         gamma = e^{G_last}, K' = K e^{G_last - G}
//
// The first part has no order between chunks and runs for every (chunk,
// head) at once in the chunk-preparation pass, which leaves one record per
// (chunk, head) (layout in kda_split.cuh).  This kernel is the second part:
// one CTA per (sequence, head) chain walks its chunks in order with the fp32
// state in TMEM; per chunk it
//   - reads the state out of TMEM (fp16 copy for the MMA, snapshot of the
//     previous chunk's state, scaling by gamma in place),
//   - D1 = [-Wk ; -Q~] S_fp16        (rows 0..63: -Wk S, rows 64..127: -Q~ S)
//   - W = U + D1[0..63] -> fp16
//   - S += K'^T W,  D1[64..127] += -P W   (= -O)
//   - writes o.
// The records arrive by bulk async copies two chunks ahead (two stages), so
// the chain only waits on its own three MMAs.  Every wait is bounded; a wait
// that gives up records KDA_ERR_TIMEOUT and the CTA stops cleanly.
//
// Heads of 64 key channels carry zero state rows 64..127 (their records hold
// zero key channels); heads of 64 value channels run one CTA per chain.
// Packed batches are taken longest chain first (the chunk-table kernel's order
// table), so that no long chain starts in the last wave.  The chunk table, the
// chunk preparation and this pass are programmatic dependent launches: each
// waits on the device for the grids before it, and the next one's launch
// overlaps its run.
#include <string.h>

#include "kda_common.cuh"
#include "kda_pdl.cuh"
#include "kda_sm100.cuh"
#include "kda_split.cuh"
#include "kda_tc_common.cuh"

namespace kda {

namespace {

using namespace sm100;
using namespace tcx;

constexpr int SP_THREADS = 512;
constexpr int NC = 64;  // value columns of the state per CTA (two CTAs per chain)

// One stage holds one record, with only this CTA's half of U:
// A3 | KP | U half | P | gamma.  The M5 operand [X ; -P] (128 x 64, MN-major:
// two 64-row blocks 8 KiB apart) starts 8 KiB before P, so its first block X
// is the U half: it only feeds D1 rows 0..63, which nothing reads after M5
// (the next chunk's first MMA overwrites them).
constexpr uint32_t ST_A3 = 0;
constexpr uint32_t ST_KP = 32 * KiB;
constexpr uint32_t ST_U = 48 * KiB;
constexpr uint32_t ST_P = 56 * KiB;
constexpr uint32_t ST_A5 = ST_P - 8 * KiB;
constexpr uint32_t ST_G = 64 * KiB;
constexpr uint32_t ST_BYTES = 65 * KiB;
constexpr uint32_t SM_SBF = 2 * ST_BYTES;        // [dk x NC] S in fp16, MN-major
constexpr uint32_t SM_WBF = SM_SBF + 16 * KiB;   // [tok x NC] W in fp16, MN-major; o staging
constexpr uint32_t SM_SNAP = SM_WBF + 8 * KiB;   // snapshot staging: 2 boxes [128 rows][32 fp32], 128-byte swizzle
constexpr uint32_t SM_MISC = SM_SNAP + 32 * KiB;
constexpr uint32_t MS_BAR_FULL = SM_MISC;        // 2 mbarriers (records in)
constexpr uint32_t MS_BAR_MMA = SM_MISC + 16;
constexpr uint32_t MS_TMEM = SM_MISC + 32;
constexpr uint32_t SP_SMEM_BYTES = SM_MISC + 64;
static_assert(SP_SMEM_BYTES <= 232448, "shared memory budget");

constexpr uint32_t kRecInBytes = 32 * KiB + 16 * KiB + 8 * KiB + 8 * KiB + 512;

constexpr uint32_t TM_S = 0;    // fp32 state columns (row = key channel)
constexpr uint32_t TM_D1 = NC;  // -Wk S (rows 0..63); -O (rows 64..127)
constexpr uint32_t TM_COLS = 128;
// The segment scan's paired pass (`dual`) carries a second chain through the
// same records: the transition M (from the identity, v taken as zero) beside
// N (from zero, with v).  Its fp16 copy of the state and its W take the
// snapshot staging area (no snapshots in that pass), its TMEM columns follow.
constexpr uint32_t SM_SBF2 = SM_SNAP;
constexpr uint32_t SM_WBF2 = SM_SNAP + 16 * KiB;
constexpr uint32_t TM_S2 = 128;
constexpr uint32_t TM_D12 = 128 + NC;
constexpr uint32_t TM_COLS_DUAL = 256;

constexpr uint32_t kWaitPolls = 1u << 24;
constexpr int kCopyThread = 128;  // issues the record copies

constexpr uint32_t ID_KMN = idesc_mma(128, NC, kFmtF16, kFmtF16, 0, 1);   // K-major x MN
constexpr uint32_t ID_MNMN = idesc_mma(128, NC, kFmtF16, kFmtF16, 1, 1);  // MN x MN

struct SpParams {
  const uint8_t *rec;          // records [chunk][head in group]
  const int32_t *cu_seqlens;   // or NULL: equal lengths fixed_len
  const int32_t *chunk_start;  // first chunk of each sequence (varlen), or NULL
  int64_t fixed_len;
  int64_t total;               // tokens of the batch
  int n_seq;
  int H, h0, hg;               // heads h0 .. h0 + hg - 1 of H
  int dk, dv;                  // 64 or 128 each
  const float *S0;
  kda_bf16 *o;
  float *S_final;
  float *snaps;
  const int64_t *snap_offsets;
  int *status;
  const int32_t *slots;
  int n_slots;
  int zero_u;       // 1: v taken as zero (W = -Wk S; U is not loaded)
  int s0_identity;  // 1: every chain starts from S0 = I (dk = dv)
  float *S_final2;  // non-NULL: the paired pass -- chain 1 from zero with v
                    // (final state to S_final), chain 2 from the identity with
                    // v = 0 (final state to S_final2); no o, no snapshots
  const int32_t *order;  // varlen: the sequence of each grid row (longest first), or NULL
};

// One CTA per (sequence, head, half of the value columns): the columns of the
// state never mix, so each half runs on its own with the same records.
__global__ void __launch_bounds__(SP_THREADS, 1)
state_pass_kernel(const __grid_constant__ CUtensorMap tm_snap, const SpParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  const Smem S{smem, sb};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if ((sb & 1023u) != 0) {  // the swizzled layouts need 1024-byte alignment
    if (tid == 0) atomicOr(p.status, KDA_ERR_UNSUPPORTED);
    return;
  }
  grid_dependency_wait();  // the records, tables and S0 of the kernels before
  const int halves = p.dv / NC;  // CTAs per chain
  const int hh = blockIdx.x / halves, half = blockIdx.x - hh * halves;
  // grid rows in the chunk table's order, longest sequences first, so that the
  // long chains do not start in the last wave
  int s = blockIdx.y;
  if (p.order) {
    s = p.order[blockIdx.y];
    if (s < 0 || s >= p.n_seq) {
      if (tid == 0) atomicOr(p.status, KDA_ERR_SHAPE);
      return;
    }
  }
  const int H = p.H, h = p.h0 + hh;
  const int DK = p.dk, DV = p.dv;
  const int col0 = NC * half;

  bool shape_bad = false;
  int slot = s;
  if (p.slots) {
    slot = p.slots[s];
    if (slot < 0 || slot >= p.n_slots) {  // nothing of this sequence is touched
      if (tid == 0) atomicOr(p.status, KDA_ERR_SHAPE);
      return;
    }
  }
  int64_t t_begin, t_end, chunk0;
  if (p.cu_seqlens) {
    if (!seq_range(p.cu_seqlens, s, p.total, t_begin, t_end)) shape_bad = true;
    chunk0 = p.chunk_start[s];
    // a table that does not cover this sequence's chunks (chunk_start_kernel
    // zeroes it when cu_seqlens is malformed): read no record
    if (chunk0 < 0 || chunk0 + (t_end - t_begin + 63) / 64 > p.chunk_start[p.n_seq]) {
      t_end = t_begin;
      shape_bad = true;
    }
  } else {
    t_begin = static_cast<int64_t>(s) * p.fixed_len;
    t_end = t_begin + p.fixed_len;
    chunk0 = static_cast<int64_t>(s) * ((p.fixed_len + 63) / 64);
  }
  const int n_chunks = static_cast<int>((t_end - t_begin + 63) / 64);
  int64_t snap_row = 0;
  bool want_snaps = p.snaps != nullptr;
  if (want_snaps) {
    snap_row = p.snap_offsets ? snap_first_row(p.snap_offsets, s, p.n_seq, t_end - t_begin)
                              : static_cast<int64_t>(s) * (p.fixed_len / 64);
    if (snap_row < 0) {
      want_snaps = false;
      shape_bad = true;
    }
  }
  const size_t state_off = (static_cast<size_t>(slot) * H + h) * DK * DV;

  const uint32_t bar_full = sb + MS_BAR_FULL, bar_mma = sb + MS_BAR_MMA;
  if (tid == 0) {
    mbar_init(bar_full, 1);
    mbar_init(bar_full + 8, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  const bool dual = p.S_final2 != nullptr;
  const uint32_t tm_cols = dual ? TM_COLS_DUAL : TM_COLS;
  if (warp == 1) {
    tmem_alloc(sb + MS_TMEM, tm_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + MS_TMEM);

  // TMEM read-outs: a warp reaches the 32 lanes of its quadrant; the 16 warps
  // split the CTA's 64 columns in quarters of 16.
  const int quad = warp & 3, q4 = warp >> 2;
  const int trow = quad * 32 + lane;  // TMEM lane = matrix row
  const uint32_t t_lane = tmem + (static_cast<uint32_t>(quad * 32) << 16);
  const int cq = col0 + 16 * q4;      // first state column of this thread

  const bool row_in = trow < DK;
  {  // initial state -> TMEM (rows beyond dk are zero)
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      v[j] = p.s0_identity ? (trow == cq + j ? 1.f : 0.f)
             : (p.S0 && row_in) ? p.S0[state_off + static_cast<size_t>(trow) * DV + cq + j]
                                : 0.f;
    tmem_st16(t_lane + TM_S + 16 * q4, v);
    if (dual) {  // the transition chain starts from the identity
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = trow == cq + j ? 1.f : 0.f;
      tmem_st16(t_lane + TM_S2 + 16 * q4, v);
    }
    tmem_wait_st();
  }

  auto issue = [&](int n) {  // record of chunk n -> stage n & 1
    const uint32_t st = sb + static_cast<uint32_t>(n & 1) * ST_BYTES;
    const uint8_t *rec =
        p.rec + (static_cast<size_t>(chunk0 + n) * p.hg + hh) * static_cast<size_t>(kRecBytes);
    const uint32_t bar = bar_full + 8u * static_cast<uint32_t>(n & 1);
    mbar_expect_tx(bar, p.zero_u ? kRecInBytes - 8 * KiB : kRecInBytes);
    bulk_g2s(st + ST_A3, rec + kRecA3, 32 * KiB, bar);
    bulk_g2s(st + ST_KP, rec + kRecKP, 16 * KiB, bar);
    if (!p.zero_u) bulk_g2s(st + ST_U, rec + kRecU + half * 8 * KiB, 8 * KiB, bar);
    bulk_g2s(st + ST_P, rec + kRecP, 8 * KiB, bar);
    bulk_g2s(st + ST_G, rec + kRecG, 512, bar);
  };
  // bit b: stage b's record copy is in flight (a mask: an array indexed by
  // the stage would live in local memory)
  uint32_t full_pending = 0;
  bool mma_pending = false, aborted = false;
  if (tid == kCopyThread) {
    if (n_chunks > 0) issue(0);
    if (n_chunks > 1) issue(1);
  }
  full_pending = (n_chunks > 0 ? 1u : 0u) | (n_chunks > 1 ? 2u : 0u);
  uint32_t mma_phase = 0;
  int64_t snap_pending = -1;
  float range_max = 0.f;  // largest magnitude sent through an fp16 operand

  auto wait_mma = [&]() -> bool {
    const bool ok = mbar_wait_bounded(bar_mma, mma_phase, kWaitPolls);
    if (__syncthreads_or(ok ? 0 : 1)) {
      if (tid == 0) atomicOr(p.status, KDA_ERR_TIMEOUT);
      tc_fence_after();
      return false;
    }
    mma_phase ^= 1u;
    mma_pending = false;
    tc_fence_after();
    return true;
  };

  for (int n = 0; n < n_chunks; ++n) {
    const int stg = n & 1;
    const uint32_t st = sb + static_cast<uint32_t>(stg) * ST_BYTES;
    const int64_t t0 = t_begin + 64LL * n;
    const int L = static_cast<int>(min(static_cast<int64_t>(64), t_end - t0));
    // Each thread waits for the record on its own (no CTA barrier here, so the
    // previous chunk's o stores overlap this read-out); a wait that gives up
    // is agreed on at the barrier before the first MMA.
    const bool rec_ok = mbar_wait_bounded(bar_full + 8u * stg, (n >> 1) & 1, kWaitPolls);

    // ---- state read-out: fp16 copy for the MMA, S *= gamma in place ----------------------
    // The unscaled values stay in registers for the snapshot, which is
    // written while the first MMA runs; the TMEM store is waited for only
    // before the barrier ahead of S += K'^T W.
    float sv[16];
    tmem_ld16(t_lane + TM_S + 16 * q4, sv);
    tmem_wait_ld();
    {
#pragma unroll
      for (int j = 0; j < 16; ++j) range_max = fmaxf(range_max, fabsf(sv[j]));
      store_row16_f16(S, sb + SM_SBF, trow, q4, sv, 1.f);
      const float gam = S.f32(st + ST_G + 4 * trow);
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = sv[j] * gam;
      tmem_st16(t_lane + TM_S + 16 * q4, v);
      if (dual) {
        float s2[16];
        tmem_ld16(t_lane + TM_S2 + 16 * q4, s2);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) range_max = fmaxf(range_max, fabsf(s2[j]));
        store_row16_f16(S, sb + SM_SBF2, trow, q4, s2, 1.f);
#pragma unroll
        for (int j = 0; j < 16; ++j) s2[j] *= gam;
        tmem_st16(t_lane + TM_S2 + 16 * q4, s2);
      }
    }
    if (tid == kCopyThread) bulk_wait_read0();  // the last snapshot's stores have read the tile
    fence_proxy_async();
    tc_fence_before();
    if (__syncthreads_or(rec_ok ? 0 : 1)) {
      if (tid == 0) atomicOr(p.status, KDA_ERR_TIMEOUT);
      tmem_wait_st();
      aborted = true;
      break;
    }
    full_pending &= ~(1u << stg);

    // ---- D1 = [-Wk ; -Q~] S ------------------------------------------------------------
    if (tid == 0) {
      tc_fence_after();
      issue_mma(tmem + TM_D1, st + ST_A3, false, REG128, sb + SM_SBF, true, REG128, 8, ID_KMN, 0);
      if (dual)
        issue_mma(tmem + TM_D12, st + ST_A3, false, REG128, sb + SM_SBF2, true, REG128, 8, ID_KMN,
                  0);
      mma_commit(bar_mma);
    }
    mma_pending = true;
    if (snap_pending >= 0) {
      // The state after the previous (full) chunk, while the MMA runs: staged
      // as two [128 rows][32 fp32] boxes in the 128-byte-swizzled layout (so a
      // warp's 16-byte writes to 32 consecutive rows hit every bank once per
      // 8 rows) and stored by TMA after the next barrier.
      const uint32_t box = sb + SM_SNAP + static_cast<uint32_t>(q4 >> 1) * 16384u +
                           static_cast<uint32_t>(trow) * 128u;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        S.u128(box + (static_cast<uint32_t>(((q4 & 1) * 4 + j) ^ (trow & 7)) << 4)) =
            make_uint4(__float_as_uint(sv[4 * j]), __float_as_uint(sv[4 * j + 1]),
                       __float_as_uint(sv[4 * j + 2]), __float_as_uint(sv[4 * j + 3]));
      fence_proxy_async();
    }
    if (!wait_mma()) { tmem_wait_st(); aborted = true; break; }
    if (snap_pending >= 0) {
      if (tid == kCopyThread) {
        // box = 32 columns x dk rows of state (snapshot row, head) y
        const int y = static_cast<int>(snap_pending * H + h);
        tma_store_3d(&tm_snap, col0, 0, y, sb + SM_SNAP);
        tma_store_3d(&tm_snap, col0 + 32, 0, y, sb + SM_SNAP + 16384u);
        bulk_commit();
      }
      snap_pending = -1;
    }

    // ---- W = U - Wk S -> fp16 ----------------------------------------------------------------
    if (quad < 2) {
      float v[16];
      tmem_ld16(t_lane + TM_D1 + 16 * q4, v);
      tmem_wait_ld();
      if (!p.zero_u) add_row16_f16(S, st + ST_U, trow, q4, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) range_max = fmaxf(range_max, fabsf(v[j]));
      store_row16_f16(S, sb + SM_WBF, trow, q4, v, 1.f);
      if (dual) {  // W of the transition chain: v = 0
        tmem_ld16(t_lane + TM_D12 + 16 * q4, v);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) range_max = fmaxf(range_max, fabsf(v[j]));
        store_row16_f16(S, sb + SM_WBF2, trow, q4, v, 1.f);
      }
    }
    tmem_wait_st();  // the gamma-scaled state is in TMEM before S += K'^T W
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // ---- S += K'^T W;  D1 += [X ; -P] W (only when o is wanted) ---------------------------------
    if (tid == 0) {
      tc_fence_after();
      if (p.o) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {  // the two products interleaved
          issue_mma_step(tmem + TM_S, st + ST_KP, true, REG64, sb + SM_WBF, true, REG64, ks,
                         ID_MNMN, 1);
          issue_mma_step(tmem + TM_D1, st + ST_A5, true, REG64, sb + SM_WBF, true, REG64, ks,
                         ID_MNMN, 1);
        }
      } else {  // the segment scan's passes for N and M
        issue_mma(tmem + TM_S, st + ST_KP, true, REG64, sb + SM_WBF, true, REG64, 4, ID_MNMN, 1);
        if (dual)
          issue_mma(tmem + TM_S2, st + ST_KP, true, REG64, sb + SM_WBF2, true, REG64, 4, ID_MNMN,
                    1);
      }
      mma_commit(bar_mma);
    }
    mma_pending = true;
    if (!wait_mma()) { aborted = true; break; }
    // every reader of this stage is done: refill it with chunk n + 2
    if (tid == kCopyThread && n + 2 < n_chunks) issue(n + 2);
    if (n + 2 < n_chunks) full_pending |= 1u << stg;

    // ---- outputs: o = -D1 rows 64..127 -------------------------------------------------------
    // Each of the 8 warps holds 32 rows x 16 columns (32 bytes of bf16 per
    // row); it stages them in its 1 KiB slice of the W tile (free once the
    // MMAs above are done) and stores 16 rows x 32 bytes per instruction.
    if (quad >= 2 && p.o) {
      float v[16];
      tmem_ld16(t_lane + TM_D1 + 16 * q4, v);
      tmem_wait_ld();
      const uint32_t tile = sb + SM_WBF + static_cast<uint32_t>((quad - 2) * 4 + q4) * 1024u;
#pragma unroll
      for (int j = 0; j < 2; ++j)
        S.u128(tile + lane * 32u + (static_cast<uint32_t>(j ^ (lane & 1)) << 4)) =
            make_uint4(pack_bf16x2(-v[8 * j + 0], -v[8 * j + 1]),
                       pack_bf16x2(-v[8 * j + 2], -v[8 * j + 3]),
                       pack_bf16x2(-v[8 * j + 4], -v[8 * j + 5]),
                       pack_bf16x2(-v[8 * j + 6], -v[8 * j + 7]));
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int rl = 16 * i + (lane >> 1), c = lane & 1;  // row in the warp's 32, 16-byte piece
        const int r = (quad - 2) * 32 + rl;
        if (r < L) {
          const uint4 w = S.u128(tile + rl * 32u + (static_cast<uint32_t>(c ^ (rl & 1)) << 4));
          reinterpret_cast<uint4 *>(p.o + (static_cast<size_t>(t0 + r) * H + h) * DV + cq)[c] = w;
        }
      }
    }
    if (want_snaps && L == 64) snap_pending = snap_row;
    if (L == 64) ++snap_row;
    // the next chunk's first MMA overwrites D1 only after its state read-out
    // barrier, which every thread reaches after its o stores above
  }

  if (!aborted && (p.S_final || snap_pending >= 0)) {
    float v[16];
    tmem_ld16(t_lane + TM_S + 16 * q4, v);
    tmem_wait_ld();
    if (p.S_final && row_in) {
      float4 *dst = reinterpret_cast<float4 *>(p.S_final + state_off +
                                               static_cast<size_t>(trow) * DV + cq);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
    if (dual) {
      tmem_ld16(t_lane + TM_S2 + 16 * q4, v);
      tmem_wait_ld();
      if (row_in) {
        float4 *dst = reinterpret_cast<float4 *>(p.S_final2 + state_off +
                                                 static_cast<size_t>(trow) * DV + cq);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      }
    }
    if (snap_pending >= 0 && row_in) {
      float4 *dst = reinterpret_cast<float4 *>(
          p.snaps + (static_cast<size_t>(snap_pending) * H + h) * DK * DV +
          static_cast<size_t>(trow) * DV + cq);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        __stcs(dst + j, make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
    }
  }

  if (tid == kCopyThread) bulk_wait0();  // snapshot stores complete before the CTA ends
  // Drain anything still in flight (bounded) before TMEM and shared memory go.
  if (aborted && tid == 0) {
    if (mma_pending) mbar_wait_bounded(bar_mma, mma_phase, kWaitPolls);
  }
  if (aborted && tid == kCopyThread) {
    for (int b = 0; b < 2; ++b)
      if ((full_pending >> b) & 1u) mbar_wait_bounded(bar_full + 8 * b, 0, kWaitPolls) ||
                               mbar_wait_bounded(bar_full + 8 * b, 1, kWaitPolls);
  }
  tc_fence_before();
  if (__syncthreads_or(range_max > 65504.f ? 1 : 0) && tid == 0)
    atomicOr(p.status, KDA_ERR_RANGE);
  if (shape_bad && tid == 0) atomicOr(p.status, KDA_ERR_SHAPE);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tm_cols);
  }
}

}  // namespace

cudaError_t state_pass_launch(const uint8_t *rec, const int32_t *cu_seqlens,
                              const int32_t *chunk_start, int n_seq, int64_t fixed_len,
                              int64_t total_tokens, int H, int dk, int dv, int h0, int hg,
                              const float *S0, kda_bf16 *o, float *S_final, float *snaps,
                              const int64_t *snap_offsets, int *status, const int32_t *slots,
                              int n_slots, int zero_u, int s0_identity, float *S_final2,
                              const int32_t *order, cudaStream_t stream) {
  // Snapshots as a 3-D fp32 array [rows * H][dk][dv]; rows <= total_tokens / 64
  // (each snapshot follows a full chunk), which bounds the map's extent.  A
  // box is 32 value columns x dk key rows of one (row, head) state, so a
  // 64-row state never reaches the next one.
  CUtensorMap tm_snap;
  memset(&tm_snap, 0, sizeof(tm_snap));
  if (snaps) {
    const EncodeTiledFn encode = tensor_map_encoder();
    if (!encode) return cudaErrorInvalidValue;
    const uint64_t states = static_cast<uint64_t>(total_tokens / 64) * H;
    // TMA coordinates are 32-bit signed
    if (states == 0 || states > 0x7fffffffull) return cudaErrorInvalidValue;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(dv), static_cast<cuuint64_t>(dk),
                                static_cast<cuuint64_t>(states)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(dv) * 4,
                                   static_cast<cuuint64_t>(dk) * dv * 4};
    const cuuint32_t box[3] = {32, static_cast<cuuint32_t>(dk), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&tm_snap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, snaps, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const uint32_t smem = SP_SMEM_BYTES;
  cudaError_t err = cudaFuncSetAttribute(state_pass_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  SpParams prm{rec,     cu_seqlens, chunk_start, fixed_len, total_tokens, n_seq, H,
               h0,      hg,         dk,          dv,        S0,           o,     S_final,
               snaps,   snap_offsets, status,    slots,     n_slots,      zero_u, s0_identity,
               S_final2, order};
  const dim3 grid(static_cast<unsigned>((dv / NC) * hg), static_cast<unsigned>(n_seq));
  return launch_pdl(state_pass_kernel, grid, dim3(SP_THREADS), smem, stream, tm_snap, prm);
}

}  // namespace kda

namespace kda {

namespace {

// chunk_start[i] = sum over sequences j < i of ceil(len_j / 64), i = 0 .. n_seq:
// one CTA, a running prefix over blocks of 1024 sequences.  cu_seqlens is
// checked on the way (cu[0] = 0, non-decreasing, cu[n_seq] = total): if any
// entry is malformed the whole table is set to zero (no chunk-preparation
// task, no record read by the state pass) and KDA_ERR_SHAPE is recorded.
// Then, for every global chunk c of the batch, chunk_info[c] = (first token,
// tokens in the chunk): the chunk preparation resolves a task with one load.
// Sequences ranked by chunk count up to this many; beyond it the state pass
// takes them in batch order (its tail is then short against the whole pass).
constexpr int kOrderMax = 512;

__global__ void __launch_bounds__(1024) chunk_start_kernel(const int32_t *__restrict__ cu,
                                                           int n_seq, int64_t total,
                                                           int32_t *__restrict__ chunk_start,
                                                           int2 *__restrict__ chunk_info,
                                                           int32_t *__restrict__ order,
                                                           int *status) {
  __shared__ int32_t cnt[kOrderMax];
  grid_dependency_wait();
  grid_launch_dependents();  // the chunk preparation may set up meanwhile
  __shared__ int32_t warp_sum[32];
  __shared__ int32_t carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  int bad = 0;
  if (tid == 0 && (cu[0] != 0 || static_cast<int64_t>(cu[n_seq]) != total)) bad = 1;
  __syncthreads();
  for (int base = 0; base < n_seq; base += 1024) {
    const int i = base + tid;
    int c = 0;
    if (i < n_seq) {
      const int32_t a = cu[i], b = cu[i + 1];
      if (a < 0 || b < a || static_cast<int64_t>(b) > total) bad = 1;
      else c = (b - a + 63) / 64;
    }
    int x = c;  // inclusive scan inside the warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) warp_sum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = warp_sum[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, off);
        if (lane >= off) w += y;
      }
      warp_sum[lane] = w;
    }
    __syncthreads();
    if (i < n_seq) chunk_start[i] = carry + (warp > 0 ? warp_sum[warp - 1] : 0) + x - c;
    __syncthreads();
    if (tid == 0) carry += warp_sum[31];
    __syncthreads();
  }
  if (tid == 0) chunk_start[n_seq] = carry;
  if (__syncthreads_or(bad)) {
    for (int i = tid; i <= n_seq; i += 1024) chunk_start[i] = 0;
    for (int i = tid; i < n_seq; i += 1024) order[i] = i;
    if (tid == 0) atomicOr(status, KDA_ERR_SHAPE);
    return;
  }
  // state-pass order: descending chunk count, ties in batch order (a permutation)
  if (n_seq <= kOrderMax) {
    for (int i = tid; i < n_seq; i += 1024) cnt[i] = chunk_start[i + 1] - chunk_start[i];
    __syncthreads();
    for (int i = tid; i < n_seq; i += 1024) {
      const int ci = cnt[i];
      int rank = 0;
      for (int j = 0; j < n_seq; ++j) {
        const int cj = cnt[j];
        rank += (cj > ci || (cj == ci && j < i)) ? 1 : 0;
      }
      order[rank] = i;
    }
  } else {
    for (int i = tid; i < n_seq; i += 1024) order[i] = i;
  }
  // chunk c belongs to the last sequence s with chunk_start[s] <= c (an empty
  // sequence shares its start with the next one; the search skips it)
  const int32_t chunks = chunk_start[n_seq];
  for (int32_t c = tid; c < chunks; c += 1024) {
    int lo = 0, hi = n_seq - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (chunk_start[mid] <= c) lo = mid; else hi = mid - 1;
    }
    const int32_t j = c - chunk_start[lo];
    const int32_t t0 = cu[lo] + 64 * j;
    chunk_info[c] = make_int2(t0, min(64, cu[lo + 1] - t0));
  }
}

}  // namespace

cudaError_t chunk_start_launch(const int32_t *cu_seqlens, int n_seq, int64_t total_tokens,
                               int32_t *chunk_start, int2 *chunk_info, int32_t *order,
                               int *status, cudaStream_t stream) {
  return launch_pdl(chunk_start_kernel, dim3(1), dim3(1024), 0, stream, cu_seqlens, n_seq,
                    total_tokens, chunk_start, chunk_info, order, status);
}

}  // namespace kda
