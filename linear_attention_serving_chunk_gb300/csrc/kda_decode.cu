// Single-token recurrent decode step on resident fp32 states, in place.
//
// Per (sequence, head): a = exp(g), S' = Diag(a) S, p = S'^T k, u = S'^T q,
// delta = beta (v - p), S'' = S' + k delta^T, o = S''^T q = u + (k.q) delta.
// This equals S_t = (I - beta k k^T) Diag(exp(g)) S_{t-1} + beta k v^T and
// o_t = S_t^T q_t (the fixed-size running state of "How a Frontier Model Gets
// Built, Read from the Kimi K3 Report", Technical Details; gate from "Kimi K3
// Technical Report - Open Frontier Intelligence", sec. 2.1.1).
//
// The step is bound by HBM: each state (dk*dv*4 bytes) is read once and
// written once.  One 256-thread CTA owns one state; every thread keeps a
// (dk / row_groups) x 4 block of it in registers between the read and the
// write, so the state crosses HBM exactly twice.  Rows of S are read and
// written as 16-byte vectors, one 512-byte row per warp instruction (dv=128).
#include "kda_common.cuh"
#include "kda_tc_common.cuh"

namespace kda {

namespace {

constexpr int kDecodeThreads = 256;

template <int DK, int DV>
__global__ void __launch_bounds__(kDecodeThreads)
decode_step_kernel(const kda_bf16 *__restrict__ q, const kda_bf16 *__restrict__ k,
                   const kda_bf16 *__restrict__ v, const kda_bf16 *__restrict__ z,
                   const kda_bf16 *__restrict__ beta, const float *__restrict__ A,
                   float gmin, float *__restrict__ pool, const int32_t *__restrict__ slots,
                   int n_slots, int H, kda_bf16 *__restrict__ o, unsigned pre,
                   int *__restrict__ status) {
  constexpr int TPR = DV / 4;                // threads across one row (4 columns each)
  constexpr int RG = kDecodeThreads / TPR;   // row groups
  constexpr int RPT = DK / RG;               // rows per thread
  static_assert(RPT * RG == DK && TPR * RG == kDecodeThreads, "decode tiling");

  __shared__ float s_a[DK], s_k[DK], s_q[DK];
  __shared__ float s_red_p[RG][DV], s_red_u[RG][DV];
  __shared__ float s_delta[DV];
  __shared__ float s_part[3][DK / 32];  // per-warp sums of k.q, k.k, q.q

  const int row = blockIdx.x;  // b * H + h
  const int b = row / H, h = row - b * H;
  const int tid = threadIdx.x;
  const int cg = tid % TPR, rg = tid / TPR;
  const int slot = slots ? slots[b] : b;
  if (slot < 0 || slot >= n_slots) {  // a bad slot index: the row is skipped
    if (tid == 0) atomicOr(status, KDA_ERR_SHAPE);
    return;
  }
  float *S = pool + (static_cast<size_t>(slot) * H + h) * (DK * DV);

  // Issue the whole state read first; the gate below overlaps its latency.
  float4 s[RPT];
#pragma unroll
  for (int rr = 0; rr < RPT; ++rr)
    s[rr] = __ldcs(reinterpret_cast<const float4 *>(S + (rg * RPT + rr) * DV) + cg);

  if (tid < DK) {
    const size_t x = static_cast<size_t>(row) * DK + tid;
    const float kv = bf2f(k[x]), qv = bf2f(q[x]);
    s_a[tid] = decay_factor(gmin, expf(A[h]), bf2f(z[x]));
    s_k[tid] = kv;
    s_q[tid] = qv;
    float kq = kv * qv, kk = kv * kv, qq = qv * qv;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      kq += __shfl_xor_sync(0xffffffffu, kq, off);
      kk += __shfl_xor_sync(0xffffffffu, kk, off);
      qq += __shfl_xor_sync(0xffffffffu, qq, off);
    }
    if ((tid & 31) == 0) {
      s_part[0][tid >> 5] = kq;
      s_part[1][tid >> 5] = kk;
      s_part[2][tid >> 5] = qq;
    }
  }
  __syncthreads();
  // Raw q and k (pre-op flag): every read of k and q below takes the 1 / norm
  // factors ik, iq; otherwise both are 1.
  float ik = 1.f, iq = 1.f;
  if (pre & KDA_PRE_L2NORM_QK) {
    float kk = 0.f, qq = 0.f;
#pragma unroll
    for (int w = 0; w < DK / 32; ++w) {
      kk += s_part[1][w];
      qq += s_part[2][w];
    }
    ik = kk > 0.f ? rsqrtf(kk) : 0.f;
    iq = qq > 0.f ? rsqrtf(qq) : 0.f;
  }

  float p[4] = {0.f, 0.f, 0.f, 0.f}, u[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int rr = 0; rr < RPT; ++rr) {
    const int i = rg * RPT + rr;
    const float a = s_a[i], kv = s_k[i] * ik, qv = s_q[i] * iq;
    s[rr].x *= a; s[rr].y *= a; s[rr].z *= a; s[rr].w *= a;
    p[0] += s[rr].x * kv; p[1] += s[rr].y * kv; p[2] += s[rr].z * kv; p[3] += s[rr].w * kv;
    u[0] += s[rr].x * qv; u[1] += s[rr].y * qv; u[2] += s[rr].z * qv; u[3] += s[rr].w * qv;
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    s_red_p[rg][cg * 4 + c] = p[c];
    s_red_u[rg][cg * 4 + c] = u[c];
  }
  __syncthreads();

  if (tid < DV) {
    float pj = 0.f, uj = 0.f;
#pragma unroll
    for (int g = 0; g < RG; ++g) {
      pj += s_red_p[g][tid];
      uj += s_red_u[g][tid];
    }
    float kq = 0.f;
#pragma unroll
    for (int w = 0; w < DK / 32; ++w) kq += s_part[0][w];
    kq *= ik * iq;
    const size_t xv = static_cast<size_t>(row) * DV + tid;
    float bt = bf2f(beta[row]);
    if (pre & KDA_PRE_SIGMOID_BETA) bt = 1.f / (1.f + __expf(-bt));
    const float delta = bt * (bf2f(v[xv]) - pj);
    s_delta[tid] = delta;
    o[xv] = f2bf(uj + kq * delta);
  }
  __syncthreads();

  const float d0 = s_delta[cg * 4 + 0], d1 = s_delta[cg * 4 + 1];
  const float d2 = s_delta[cg * 4 + 2], d3 = s_delta[cg * 4 + 3];
#pragma unroll
  for (int rr = 0; rr < RPT; ++rr) {
    const float kv = s_k[rg * RPT + rr] * ik;
    s[rr].x += kv * d0; s[rr].y += kv * d1; s[rr].z += kv * d2; s[rr].w += kv * d3;
    __stcs(reinterpret_cast<float4 *>(S + (rg * RPT + rr) * DV) + cg, s[rr]);
  }
}

// Several tokens per (sequence, head) on its resident state: the state is
// read into registers once, the run's tokens are applied in order -- each one
// the step above -- and the state is written back once (only when
// committing).  Warp w owns value columns [w DV/8, (w+1) DV/8); its lanes split
// the key rows, so p = S^T k and u = S^T q are reduced by shuffles inside the
// warp and a token needs no barrier.  The tokens' inputs are staged in shared
// memory kTokBlock at a time (with the pre-ops and k.q per token, two warps a
// token); each row group of the staging arrays is padded to an odd number of
// 16-byte units, so a lane's float4 reads of the decay, k and q of its rows are
// conflict-free.  The arithmetic is packed fp32x2 over column pairs.
//
// Persistent CTAs, two per SM, each walking its (sequence, head) rows.  While
// a CTA applies one row's tokens from registers, the next row's state comes
// in by TMA (DV / 32 boxes of 32 columns x DK rows, 128-byte swizzle, on one
// mbarrier) and the raw bf16 k, q, z, v rows of its first kTokBlock tokens by
// asynchronous copies: the state read overlaps the arithmetic instead of
// preceding it.  Lane row group rl holds the state rows rl + RL rr, so the
// swizzle puts a warp's row groups on distinct banks when the state moves
// into registers.  Later blocks of a long run are loaded directly.  Every
// mbarrier wait is bounded; one that gives up records KDA_ERR_TIMEOUT, waits
// (bounded) for the copy in flight and stops the CTA.
constexpr int kTokBlock = 8;
constexpr int kTokCtasPerSm = 2;
constexpr uint32_t kTokPolls = 1u << 24;

// Padded length of a row group of RPT key channels in the staging arrays.
constexpr int tok_row_stride(int rpt) { return ((rpt / 4 + 1) & 1) ? rpt + 4 : rpt + 8; }

template <int DK, int DV>
struct TokTiling {
  static constexpr int NW = kDecodeThreads / 32;
  static constexpr int CQ = DV / (4 * NW);  // 4-column groups per warp
  static constexpr int RL = 32 / CQ;        // row groups per warp (lanes sharing columns)
  static constexpr int RPT = DK / RL;       // rows per lane
  static constexpr int RPS = tok_row_stride(RPT);  // row group stride (floats)
  static constexpr int KS = RL * RPS;              // one token's padded key channels
  static constexpr int TOKB = (3 * DK + DV) * 2;   // raw k, q, z, v of one token (bytes)
  static constexpr uint32_t SS = 0;                                   // next state, DV / 32 boxes
  static constexpr uint32_t RAW = SS + DK * DV * 4;                   // raw token rows
  static constexpr uint32_t STG = RAW + kTokBlock * TOKB;             // fp32 staging
  // (plus 1 KiB to align the swizzled boxes to 1024 bytes)
  static constexpr uint32_t BYTES =
      1024 + STG + (3 * kTokBlock * KS + kTokBlock * DV + 2 * kTokBlock) * 4;
  static_assert(CQ * RL == 32 && RPT * RL == DK && 4 * CQ * NW == DV, "decode tiling");
  static_assert(RPT % 4 == 0 && ((RPS / 4) & 1) == 1, "float4 rows, odd 16-byte stride");
  static_assert(DV % 32 == 0 && (DK * 128) % 1024 == 0, "whole 128-byte-swizzled boxes");
  static_assert(TOKB % 16 == 0 && STG % 16 == 0, "16-byte pieces");
};

struct TokRow {  // one (sequence, head) row of the work
  int64_t t0;    // first token
  int L;         // tokens (0: nothing to do, or a rejected row)
  int slot, h;
  bool bad;      // slot or cu_seqlens out of range
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// N (2 or 4) consecutive bf16 values from a 2N-byte-aligned address (shared or global)
template <int N>
__device__ __forceinline__ void load_bf16_row(const kda_bf16 *p, float (&out)[N]) {
  static_assert(N == 2 || N == 4, "2 or 4 channels a lane");
  uint32_t w[N / 2];
  if constexpr (N == 4) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    w[0] = u.x;
    w[1] = u.y;
  } else {
    w[0] = *reinterpret_cast<const uint32_t *>(p);
  }
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    out[2 * i] = __uint_as_float(w[i] << 16);
    out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

template <int DK, int DV>
__global__ void __launch_bounds__(kDecodeThreads, kTokCtasPerSm)
decode_tokens_kernel(const __grid_constant__ CUtensorMap tm_state,
                     const kda_bf16 *__restrict__ q, const kda_bf16 *__restrict__ k,
                     const kda_bf16 *__restrict__ v, const kda_bf16 *__restrict__ z,
                     const kda_bf16 *__restrict__ beta, const float *__restrict__ A,
                     float gmin, float *__restrict__ pool, const int32_t *__restrict__ slots,
                     int n_slots, const int32_t *__restrict__ cu_seqlens, int64_t total, int H,
                     int64_t rows, kda_bf16 *__restrict__ o, unsigned pre, int commit,
                     int *__restrict__ status) {
  using T = TokTiling<DK, DV>;
  constexpr int NW = T::NW, CQ = T::CQ, RL = T::RL, RPT = T::RPT, RPS = T::RPS, KS = T::KS;
  // key channel c = rl + RL rr of a token at rl RPS + rr
  auto kidx = [](int c) { return c % RL * RPS + c / RL; };
  extern __shared__ __align__(16) uint8_t tsm_raw[];
  __shared__ __align__(8) uint64_t load_bar;
  uint8_t *tsm = tsm_raw + ((1024u - (sm100::smem_u32(tsm_raw) & 1023u)) & 1023u);
  float(*s_a)[KS] = reinterpret_cast<float(*)[KS]>(tsm + T::STG);
  float(*s_k)[KS] = s_a + kTokBlock;
  float(*s_q)[KS] = s_k + kTokBlock;
  float(*s_v)[DV] = reinterpret_cast<float(*)[DV]>(s_q + kTokBlock);
  float *s_beta = reinterpret_cast<float *>(s_v + kTokBlock), *s_kq = s_beta + kTokBlock;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cq = lane % CQ, rl = lane / CQ;
  const int col = 4 * (warp * CQ + cq);  // this lane's first value column
  const uint32_t sbase = sm100::smem_u32(tsm), bar = sm100::smem_u32(&load_bar);
  if (tid == 0) {
    sm100::mbar_init(bar, 1);
    sm100::fence_mbar_init();
    sm100::prefetch_tensormap(&tm_state);
  }
  __syncthreads();

  auto row_of = [&](int64_t r) -> TokRow {
    TokRow w{0, 0, 0, 0, false};
    if (r >= rows) return w;
    const uint32_t r32 = static_cast<uint32_t>(r);  // rows = n H < 2^32
    const int b = static_cast<int>(r32 / static_cast<uint32_t>(H));
    w.h = static_cast<int>(r32 - static_cast<uint32_t>(b) * static_cast<uint32_t>(H));
    w.slot = slots[b];
    int64_t e = 0;
    if (w.slot < 0 || w.slot >= n_slots || !seq_range(cu_seqlens, b, total, w.t0, e)) {
      w.bad = true;
      return w;
    }
    w.L = static_cast<int>(e - w.t0);
    return w;
  };
  // the state of row w (TMA) and its first block's raw token rows; beta of
  // those tokens into a register of threads 0 .. nt - 1
  float beta_next = 0.f;
  auto prefetch = [&](const TokRow &w) {
    if (w.L == 0) return;
    if (tid == 0) {
      sm100::fence_proxy_async();
      sm100::mbar_expect_tx(bar, DK * DV * 4);
      const int st = w.slot * H + w.h;  // < 2^31, checked by the launch
#pragma unroll
      for (int b = 0; b < DV / 32; ++b)
        sm100::tma_load_3d(sbase + T::SS + b * DK * 128, &tm_state, 32 * b, 0, st, bar);
    }
    const int nt = min(w.L, kTokBlock);
    constexpr int P = T::TOKB / 16;  // 16-byte pieces per token
    for (int x = tid; x < nt * P; x += kDecodeThreads) {
      const int j = x / P, ob = (x - j * P) * 16;  // byte offset in the token's raw rows
      const size_t tok = static_cast<size_t>(w.t0 + j) * H + w.h;
      const uint8_t *src =
          ob < 2 * DK   ? reinterpret_cast<const uint8_t *>(k + tok * DK) + ob
          : ob < 4 * DK ? reinterpret_cast<const uint8_t *>(q + tok * DK) + (ob - 2 * DK)
          : ob < 6 * DK ? reinterpret_cast<const uint8_t *>(z + tok * DK) + (ob - 4 * DK)
                        : reinterpret_cast<const uint8_t *>(v + tok * DV) + (ob - 6 * DK);
      cp_async16(sbase + T::RAW + j * T::TOKB + ob, src);
    }
    cp_async_commit();
    if (tid < nt) beta_next = bf2f(beta[static_cast<size_t>(w.t0 + tid) * H + w.h]);
  };
  // Tokens 0 .. nt - 1 of a block into the fp32 staging area, from their bf16
  // rows: the raw rows in shared memory for a row's first block, global memory
  // for later ones.  Two warps per token, each lane on DK / 32 consecutive
  // channels: one warp takes k and q (the pre-op norms and k.q, reduced in the
  // warp), the other the decay of z and v.  Thread j < nt holds token j's beta.
  // The closing barrier also ends every read of the raw rows.
  auto stage = [&](int nt, bool from_raw, int64_t t0, int h) {
    constexpr int CK = DK / 32, CV = DV / 32;
    for (int t = warp; t < 2 * nt; t += NW) {
      const int j = t >> 1;
      const kda_bf16 *kr, *qr, *zr, *vr;
      if (from_raw) {
        kr = reinterpret_cast<const kda_bf16 *>(tsm + T::RAW + j * T::TOKB);
        qr = kr + DK;
        zr = kr + 2 * DK;
        vr = kr + 3 * DK;
      } else {
        const size_t tok = static_cast<size_t>(t0 + j) * H + h;
        kr = k + tok * DK;
        qr = q + tok * DK;
        zr = z + tok * DK;
        vr = v + tok * DV;
      }
      if ((t & 1) == 0) {
        float kv[CK], qv[CK];
        load_bf16_row<CK>(kr + CK * lane, kv);
        load_bf16_row<CK>(qr + CK * lane, qv);
        if (pre & KDA_PRE_L2NORM_QK) {
          float kk = 0.f, qq = 0.f;
#pragma unroll
          for (int e = 0; e < CK; ++e) {
            kk += kv[e] * kv[e];
            qq += qv[e] * qv[e];
          }
          kk = warp_sum(kk);
          qq = warp_sum(qq);
          const float ik = kk > 0.f ? rsqrtf(kk) : 0.f, iq = qq > 0.f ? rsqrtf(qq) : 0.f;
#pragma unroll
          for (int e = 0; e < CK; ++e) {
            kv[e] *= ik;
            qv[e] *= iq;
          }
        }
        float kq = 0.f;
#pragma unroll
        for (int e = 0; e < CK; ++e) kq += kv[e] * qv[e];
        kq = warp_sum(kq);
#pragma unroll
        for (int e = 0; e < CK; ++e) {
          const int ci = kidx(CK * lane + e);
          s_k[j][ci] = kv[e];
          s_q[j][ci] = qv[e];
        }
        if (lane == 0) s_kq[j] = kq;
      } else {
        const float eA = expf(A[h]);
        float zv[CK], vv[CV];
        load_bf16_row<CK>(zr + CK * lane, zv);
        load_bf16_row<CV>(vr + CV * lane, vv);
#pragma unroll
        for (int e = 0; e < CK; ++e) s_a[j][kidx(CK * lane + e)] = decay_factor(gmin, eA, zv[e]);
#pragma unroll
        for (int e = 0; e < CV; ++e) s_v[j][CV * lane + e] = vv[e];
      }
    }
    if (tid < nt)
      s_beta[tid] = (pre & KDA_PRE_SIGMOID_BETA) ? 1.f / (1.f + __expf(-beta_next)) : beta_next;
    __syncthreads();
  };

  const int64_t stride = gridDim.x;
  uint32_t phase = 0;
  TokRow cur = row_of(blockIdx.x);
  TokRow nxt = row_of(blockIdx.x + stride);
  prefetch(cur);
  for (int64_t r = blockIdx.x; r < rows; r += stride) {
    const TokRow after = row_of(r + 2 * stride);  // used one row later: its latency is hidden
    if (cur.bad && tid == 0) atomicOr(status, KDA_ERR_SHAPE);  // nothing of it is touched
    const int L = cur.L;
    float2 sl[RPT], sh[RPT];  // rows rl + RL rr; columns col, col + 1 (sl) and + 2, + 3 (sh)
    if (L > 0) {
      const bool ok = sm100::mbar_wait_bounded(bar, phase, kTokPolls);
      phase ^= 1u;
      cp_async_wait_all();
      if (__syncthreads_or(ok ? 0 : 1)) {  // also: every thread's raw token pieces are in
        if (tid == 0) {
          atomicOr(status, KDA_ERR_TIMEOUT);
          sm100::mbar_wait_bounded(bar, phase ^ 1u, kTokPolls);  // the copy in flight
        }
        return;
      }
      {
        const int b = col >> 5, chunk = (col & 31) >> 2;
#pragma unroll
        for (int rr = 0; rr < RPT; ++rr) {
          const int r = rl + RL * rr;
          const float4 t = *reinterpret_cast<const float4 *>(
              tsm + T::SS + b * DK * 128 + r * 128 + ((chunk ^ (r & 7)) << 4));
          sl[rr] = make_float2(t.x, t.y);
          sh[rr] = make_float2(t.z, t.w);
        }
      }
      stage(min(L, kTokBlock), true, cur.t0, cur.h);  // the first block's tokens
    }
    // the next row's state and tokens come in while this row's tokens are applied
    prefetch(nxt);

    for (int64_t t0 = cur.t0; t0 < cur.t0 + L; t0 += kTokBlock) {
      const int nt = static_cast<int>(min(static_cast<int64_t>(kTokBlock), cur.t0 + L - t0));
      if (t0 != cur.t0) {  // a long run's later block: straight from global memory
        __syncthreads();   // the previous block's tokens are done with the staging area
        const float keep = beta_next;  // threads 0 .. 7 hold the next row's beta
        if (tid < nt) beta_next = bf2f(beta[static_cast<size_t>(t0 + tid) * H + cur.h]);
        stage(nt, false, t0, cur.h);
        beta_next = keep;
      }
      for (int j = 0; j < nt; ++j) {
        float2 pl = make_float2(0.f, 0.f), ph = pl, ul = pl, uh = pl;  // p, u of the 4 columns
#pragma unroll
        for (int m = 0; m < RPT / 4; ++m) {
          const float4 a4 = *reinterpret_cast<const float4 *>(&s_a[j][rl * RPS + 4 * m]);
          const float4 k4 = *reinterpret_cast<const float4 *>(&s_k[j][rl * RPS + 4 * m]);
          const float4 q4 = *reinterpret_cast<const float4 *>(&s_q[j][rl * RPS + 4 * m]);
          const float av[4] = {a4.x, a4.y, a4.z, a4.w}, kv4[4] = {k4.x, k4.y, k4.z, k4.w},
                      qv4[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int rr = 4 * m + e;
            const float2 a2 = make_float2(av[e], av[e]), k2 = make_float2(kv4[e], kv4[e]),
                         q2 = make_float2(qv4[e], qv4[e]);
            sl[rr] = __fmul2_rn(sl[rr], a2);
            sh[rr] = __fmul2_rn(sh[rr], a2);
            pl = __ffma2_rn(sl[rr], k2, pl);
            ph = __ffma2_rn(sh[rr], k2, ph);
            ul = __ffma2_rn(sl[rr], q2, ul);
            uh = __ffma2_rn(sh[rr], q2, uh);
          }
        }
        // sums over the warp's row groups (lanes CQ apart): every lane gets its columns' p, u
#pragma unroll
        for (int off = CQ; off < 32; off <<= 1) {
          const float2 rpl = make_float2(__shfl_xor_sync(0xffffffffu, pl.x, off),
                                         __shfl_xor_sync(0xffffffffu, pl.y, off));
          const float2 rph = make_float2(__shfl_xor_sync(0xffffffffu, ph.x, off),
                                         __shfl_xor_sync(0xffffffffu, ph.y, off));
          const float2 rul = make_float2(__shfl_xor_sync(0xffffffffu, ul.x, off),
                                         __shfl_xor_sync(0xffffffffu, ul.y, off));
          const float2 ruh = make_float2(__shfl_xor_sync(0xffffffffu, uh.x, off),
                                         __shfl_xor_sync(0xffffffffu, uh.y, off));
          pl = __fadd2_rn(pl, rpl);
          ph = __fadd2_rn(ph, rph);
          ul = __fadd2_rn(ul, rul);
          uh = __fadd2_rn(uh, ruh);
        }
        const float bt = s_beta[j], kq = s_kq[j];
        const float4 v4 = *reinterpret_cast<const float4 *>(&s_v[j][col]);
        const float2 dl = make_float2(bt * (v4.x - pl.x), bt * (v4.y - pl.y));
        const float2 dh = make_float2(bt * (v4.z - ph.x), bt * (v4.w - ph.y));
        if (rl == 0) {
          uint2 w;
          w.x = static_cast<uint32_t>(f2bf(ul.x + kq * dl.x)) |
                (static_cast<uint32_t>(f2bf(ul.y + kq * dl.y)) << 16);
          w.y = static_cast<uint32_t>(f2bf(uh.x + kq * dh.x)) |
                (static_cast<uint32_t>(f2bf(uh.y + kq * dh.y)) << 16);
          *reinterpret_cast<uint2 *>(o + (static_cast<size_t>(t0 + j) * H + cur.h) * DV + col) = w;
        }
#pragma unroll
        for (int m = 0; m < RPT / 4; ++m) {
          const float4 k4 = *reinterpret_cast<const float4 *>(&s_k[j][rl * RPS + 4 * m]);
          const float kv4[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 k2 = make_float2(kv4[e], kv4[e]);
            sl[4 * m + e] = __ffma2_rn(k2, dl, sl[4 * m + e]);
            sh[4 * m + e] = __ffma2_rn(k2, dh, sh[4 * m + e]);
          }
        }
      }
    }
    if (L > 0 && commit) {
      float *S = pool + (static_cast<size_t>(cur.slot) * H + cur.h) * (DK * DV);
#pragma unroll
      for (int rr = 0; rr < RPT; ++rr)
        __stcs(reinterpret_cast<float4 *>(S + (rl + RL * rr) * DV + col),
               make_float4(sl[rr].x, sl[rr].y, sh[rr].x, sh[rr].y));
    }
    cur = nxt;
    nxt = after;
  }
  cp_async_wait_all();  // nothing may still be arriving when the CTA's shared memory goes
}

template <int DK, int DV>
cudaError_t launch_decode_tokens(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                                 const kda_bf16 *z, const kda_bf16 *beta, const float *A,
                                 float gmin, float *pool, const int32_t *slots, int n_slots,
                                 const int32_t *cu_seqlens, int n, int64_t total, int H,
                                 kda_bf16 *o, unsigned pre, int commit, int *status, int n_sms,
                                 cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(n) * H;
  const int64_t states = static_cast<int64_t>(n_slots) * H;  // TMA coordinates are 32-bit
  if (states <= 0 || states > 0x7fffffffLL) return cudaErrorInvalidValue;
  const tcx::EncodeTiledFn encode = tcx::tensor_map_encoder();
  if (!encode) return cudaErrorInvalidValue;
  CUtensorMap tm_state;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(DV), static_cast<cuuint64_t>(DK),
                              static_cast<cuuint64_t>(states)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(DV) * 4,
                                 static_cast<cuuint64_t>(DK) * DV * 4};
  const cuuint32_t box[3] = {32, static_cast<cuuint32_t>(DK), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (encode(&tm_state, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, pool, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int64_t slots_max = static_cast<int64_t>(kTokCtasPerSm) * n_sms;
  const int64_t ctas = rows < slots_max ? rows : slots_max;
  if (ctas <= 0) return cudaSuccess;
  const int smem = static_cast<int>(TokTiling<DK, DV>::BYTES);
  cudaError_t err = cudaFuncSetAttribute(decode_tokens_kernel<DK, DV>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  decode_tokens_kernel<DK, DV><<<static_cast<unsigned>(ctas), kDecodeThreads, smem, stream>>>(
      tm_state, q, k, v, z, beta, A, gmin, pool, slots, n_slots, cu_seqlens, total, H, rows, o,
      pre, commit, status);
  return cudaGetLastError();
}

template <int DK, int DV>
cudaError_t launch_decode(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                          const kda_bf16 *z, const kda_bf16 *beta, const float *A, float gmin,
                          float *pool, const int32_t *slots, int n_slots, int n, int H,
                          kda_bf16 *o, unsigned pre, int *status, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(n) * H;
  decode_step_kernel<DK, DV><<<static_cast<unsigned>(rows), kDecodeThreads, 0, stream>>>(
      q, k, v, z, beta, A, gmin, pool, slots, n_slots, H, o, pre, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t decode_tokens_launch(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                                 const kda_bf16 *z, const kda_bf16 *beta, const float *A,
                                 float gmin, float *pool, const int32_t *slots, int n_slots,
                                 const int32_t *cu_seqlens, int n, int64_t total, int H, int dk,
                                 int dv, kda_bf16 *o, unsigned pre, int commit, int *status,
                                 int n_sms, cudaStream_t stream) {
#define KDA_DT(DK_, DV_)                                                                        \
  if (dk == DK_ && dv == DV_)                                                                   \
    return launch_decode_tokens<DK_, DV_>(q, k, v, z, beta, A, gmin, pool, slots, n_slots,     \
                                          cu_seqlens, n, total, H, o, pre, commit, status,     \
                                          n_sms, stream);
  KDA_DT(128, 128)
  KDA_DT(64, 64)
  KDA_DT(128, 64)
  KDA_DT(64, 128)
#undef KDA_DT
  return cudaErrorInvalidValue;
}

cudaError_t decode_step_launch(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                               const kda_bf16 *z, const kda_bf16 *beta, const float *A,
                               float gmin, float *pool, const int32_t *slots, int n_slots,
                               int n, int H, int dk, int dv, kda_bf16 *o, unsigned pre,
                               int *status, cudaStream_t stream) {
  if (dk == 128 && dv == 128)
    return launch_decode<128, 128>(q, k, v, z, beta, A, gmin, pool, slots, n_slots, n, H, o,
                                    pre, status, stream);
  if (dk == 64 && dv == 64)
    return launch_decode<64, 64>(q, k, v, z, beta, A, gmin, pool, slots, n_slots, n, H, o,
                                    pre, status, stream);
  if (dk == 128 && dv == 64)
    return launch_decode<128, 64>(q, k, v, z, beta, A, gmin, pool, slots, n_slots, n, H, o,
                                    pre, status, stream);
  if (dk == 64 && dv == 128)
    return launch_decode<64, 128>(q, k, v, z, beta, A, gmin, pool, slots, n_slots, n, H, o,
                                    pre, status, stream);
  return cudaErrorInvalidValue;
}

}  // namespace kda
