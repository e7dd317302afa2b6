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
// warp and a token needs no CTA barrier.  The tokens' inputs are staged in
// shared memory kTokBlock at a time (with the pre-ops and k.q per token).
// A lane reads the decay, k and q of its RPT rows as float4s; each row group
// is padded to an odd number of 16-byte units, so the row groups of a warp
// fall on distinct banks and the loads are conflict-free.
constexpr int kTokBlock = 16;

// Padded length of a row group of RPT key channels in the staging arrays.
constexpr int tok_row_stride(int rpt) { return ((rpt / 4 + 1) & 1) ? rpt + 4 : rpt + 8; }

template <int DK, int DV>
__global__ void __launch_bounds__(kDecodeThreads)
decode_tokens_kernel(const kda_bf16 *__restrict__ q, const kda_bf16 *__restrict__ k,
                     const kda_bf16 *__restrict__ v, const kda_bf16 *__restrict__ z,
                     const kda_bf16 *__restrict__ beta, const float *__restrict__ A,
                     float gmin, float *__restrict__ pool, const int32_t *__restrict__ slots,
                     int n_slots, const int32_t *__restrict__ cu_seqlens, int64_t total, int H,
                     kda_bf16 *__restrict__ o, unsigned pre, int commit,
                     int *__restrict__ status) {
  constexpr int NW = kDecodeThreads / 32;
  constexpr int CQ = DV / (4 * NW);   // 4-column groups per warp
  constexpr int RL = 32 / CQ;         // row groups per warp (lanes sharing columns)
  constexpr int RPT = DK / RL;        // rows per lane
  static_assert(CQ * RL == 32 && RPT * RL == DK && 4 * CQ * NW == DV, "decode tiling");
  constexpr int RPS = tok_row_stride(RPT);  // row group stride (floats)
  constexpr int KS = RL * RPS;              // one token's padded key channels
  static_assert(RPT % 4 == 0 && ((RPS / 4) & 1) == 1, "float4 rows, odd 16-byte stride");
  // key channel c of a token at c / RPT * RPS + c % RPT
  auto kidx = [](int c) { return c / RPT * RPS + c % RPT; };

  __shared__ __align__(16) float s_a[kTokBlock][KS], s_k[kTokBlock][KS], s_q[kTokBlock][KS];
  __shared__ __align__(16) float s_v[kTokBlock][DV];
  __shared__ float s_beta[kTokBlock], s_kq[kTokBlock];

  const int row = blockIdx.x;  // b * H + h
  const int b = row / H, h = row - b * H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cq = lane % CQ, rl = lane / CQ;
  const int col = 4 * (warp * CQ + cq);  // this lane's first value column
  const int slot = slots[b];
  int64_t t_begin, t_end;
  if (slot < 0 || slot >= n_slots || !seq_range(cu_seqlens, b, total, t_begin, t_end)) {
    if (tid == 0) atomicOr(status, KDA_ERR_SHAPE);  // nothing of this sequence is touched
    return;
  }
  if (t_end == t_begin) return;  // no token: the state stays as it is
  float *S = pool + (static_cast<size_t>(slot) * H + h) * (DK * DV);
  // rows rl * RPT + rr, columns col, col + 1 (sl) and col + 2, col + 3 (sh):
  // column pairs for the packed fp32x2 arithmetic
  float2 sl[RPT], sh[RPT];
#pragma unroll
  for (int rr = 0; rr < RPT; ++rr) {
    const float4 t = __ldcs(reinterpret_cast<const float4 *>(S + (rl * RPT + rr) * DV + col));
    sl[rr] = make_float2(t.x, t.y);
    sh[rr] = make_float2(t.z, t.w);
  }
  const float eA = expf(A[h]);

  for (int64_t t0 = t_begin; t0 < t_end; t0 += kTokBlock) {
    const int nt = static_cast<int>(min(static_cast<int64_t>(kTokBlock), t_end - t0));
    __syncthreads();  // the previous block's tokens are done with the staging arrays
    for (int x = tid; x < nt * DK; x += kDecodeThreads) {
      const int j = x / DK, c = x - j * DK;
      const size_t g = (static_cast<size_t>(t0 + j) * H + h) * DK + c;
      const int ci = kidx(c);
      s_k[j][ci] = bf2f(k[g]);
      s_q[j][ci] = bf2f(q[g]);
      s_a[j][ci] = decay_factor(gmin, eA, bf2f(z[g]));
    }
    for (int x = tid; x < nt * DV; x += kDecodeThreads) {
      const int j = x / DV, c = x - j * DV;
      s_v[j][c] = bf2f(v[(static_cast<size_t>(t0 + j) * H + h) * DV + c]);
    }
    __syncthreads();
    // per token (one warp each): the pre-op norms applied to k and q in place,
    // then k.q; beta through the pre-op
    for (int j = warp; j < nt; j += NW) {
      if (pre & KDA_PRE_L2NORM_QK) {
        float kk = 0.f, qq = 0.f;
        for (int c = lane; c < DK; c += 32) {
          const int ci = kidx(c);
          kk += s_k[j][ci] * s_k[j][ci];
          qq += s_q[j][ci] * s_q[j][ci];
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          kk += __shfl_xor_sync(0xffffffffu, kk, off);
          qq += __shfl_xor_sync(0xffffffffu, qq, off);
        }
        const float ik = kk > 0.f ? rsqrtf(kk) : 0.f, iq = qq > 0.f ? rsqrtf(qq) : 0.f;
        for (int c = lane; c < DK; c += 32) {
          const int ci = kidx(c);
          s_k[j][ci] *= ik;
          s_q[j][ci] *= iq;
        }
        __syncwarp();
      }
      float kq = 0.f;
      for (int c = lane; c < DK; c += 32) kq += s_k[j][kidx(c)] * s_q[j][kidx(c)];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
      if (lane == 0) {
        float bt = bf2f(beta[static_cast<size_t>(t0 + j) * H + h]);
        if (pre & KDA_PRE_SIGMOID_BETA) bt = 1.f / (1.f + __expf(-bt));
        s_beta[j] = bt;
        s_kq[j] = kq;
      }
    }
    __syncthreads();
    for (int j = 0; j < nt; ++j) {
      float2 pl = make_float2(0.f, 0.f), ph = pl, ul = pl, uh = pl;  // p, u of the 4 columns
      float kr[RPT];  // this lane's k rows, kept for the update
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
          kr[rr] = kv4[e];
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
        *reinterpret_cast<uint2 *>(o + (static_cast<size_t>(t0 + j) * H + h) * DV + col) = w;
      }
#pragma unroll
      for (int rr = 0; rr < RPT; ++rr) {
        const float2 k2 = make_float2(kr[rr], kr[rr]);
        sl[rr] = __ffma2_rn(k2, dl, sl[rr]);
        sh[rr] = __ffma2_rn(k2, dh, sh[rr]);
      }
    }
  }
  if (commit) {
#pragma unroll
    for (int rr = 0; rr < RPT; ++rr)
      __stcs(reinterpret_cast<float4 *>(S + (rl * RPT + rr) * DV + col),
             make_float4(sl[rr].x, sl[rr].y, sh[rr].x, sh[rr].y));
  }
}

template <int DK, int DV>
cudaError_t launch_decode_tokens(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                                 const kda_bf16 *z, const kda_bf16 *beta, const float *A,
                                 float gmin, float *pool, const int32_t *slots, int n_slots,
                                 const int32_t *cu_seqlens, int n, int64_t total, int H,
                                 kda_bf16 *o, unsigned pre, int commit, int *status,
                                 cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(n) * H;
  decode_tokens_kernel<DK, DV><<<static_cast<unsigned>(rows), kDecodeThreads, 0, stream>>>(
      q, k, v, z, beta, A, gmin, pool, slots, n_slots, cu_seqlens, total, H, o, pre, commit,
      status);
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
                                 cudaStream_t stream) {
#define KDA_DT(DK_, DV_)                                                                        \
  if (dk == DK_ && dv == DV_)                                                                   \
    return launch_decode_tokens<DK_, DV_>(q, k, v, z, beta, A, gmin, pool, slots, n_slots,     \
                                          cu_seqlens, n, total, H, o, pre, commit, status,     \
                                          stream);
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
