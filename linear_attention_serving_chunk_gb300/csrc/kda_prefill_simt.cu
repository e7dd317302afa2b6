// Chunkwise-parallel KDA prefill, fp32 on the CUDA cores.
//
// The chunkwise form ("Kimi K3 Technical Report - Open Frontier Intelligence",
// sec. 2.1) for one chunk of C = 64 rows r with inclusive cumulative log-decay
// G_r = sum_{m<=r} g_m (per key channel c) and chunk-start state S:
//
//   A_kk[r,i] = beta_r sum_c k_r[c] k_i[c] e^{G_r[c]-G_i[c]}      (i < r)
//   T         = (I + A_kk)^{-1}                                  (unit lower)
//   W         = T diag(beta) (V - (K * e^G) S)
//   P[r,i]    = sum_c q_r[c] k_i[c] e^{G_r[c]-G_i[c]}              (i <= r)
//   O         = (Q * e^G) S + P W
//   S'        = Diag(e^{G_last}) S + (K * e^{G_last - G})^T W
//
// e^{G_r - G_i} is never formed per (r, i, c).  It is split into a row factor
// and a column factor that are both finite: the chunk is cut into four
// 16-row sub-tiles, and for a column i in sub-tile J the reference is the
// cumulative decay just before J.  The column factor e^{G_ref(J) - G_i} is at
// most e^{-16 gmin} = e^80, the row factor e^{G_r - G_ref(J)} is at most 1 for
// r in or below J.  That is what the lower bound gmin = -5 buys (sec. 2.1.1,
// Fig. 3): the diagonal sub-tiles are plain dot products, with no per-pair
// exponentials.  All factors are products of per-token decays exp(g), kept
// per sub-tile (forward and backward running products), so the only
// transcendental work is the gate itself.
//
// Work split: one CTA per (value-column slice of NS columns, head, sequence)
// runs that chain's chunks in order; columns of the state are independent.
// This kernel is the straightforward SIMT form of the algorithm; the
// tensor-core kernel computes the same quantities with tcgen05 matmuls.
#include "kda_common.cuh"

namespace kda {

namespace {

constexpr int kThreads = 256;

template <int DK, int NS>
struct SimtSmem {
  // Per element (r, c); transformed in place once per chunk:
  //   KE: k -> k * Ef        QE: q -> q * Ef
  //   KH: a -> Ef -> k * Eb / Lam[J]   KP: Eb -> k * Eb * Y[R]
  float KE[kChunk][DK + 1];
  float QE[kChunk][DK + 1];
  float KH[kChunk][DK + 1];
  float KP[kChunk][DK + 1];
  float lam_inv[kSubTiles][DK];
  float X[kSubTiles][kSubTiles][DK];  // X[R][J] = prod_{J <= M < R} Lam[M]
  float Y[kSubTiles][DK];             // Y[R] = prod_{M > R} Lam[M]
  float gam[DK];                      // prod_M Lam[M] = e^{G_last}
  float P[kChunk][kChunk + 1];
  float T[kChunk][kChunk + 1];
  float AW[kChunk][kChunk + 1];  // A_kk, then [R1 | W] (2 x C x NS)
  float S[DK][NS];
  float V[kChunk][NS];
  float beta[kChunk];
};

template <int DK, int NS>
__global__ void __launch_bounds__(kThreads, 1)
prefill_simt_kernel(const kda_bf16 *__restrict__ q, const kda_bf16 *__restrict__ k,
                    const kda_bf16 *__restrict__ v, const kda_bf16 *__restrict__ z,
                    const kda_bf16 *__restrict__ beta, const float *__restrict__ A, float gmin,
                    const int32_t *__restrict__ cu_seqlens, int64_t fixed_len, int H, int DV,
                    const float *S0, kda_bf16 *__restrict__ o,
                    float *S_final, float *__restrict__ snaps,
                    const int64_t *__restrict__ snap_offsets,
                    const int32_t *__restrict__ slots, unsigned pre) {
  static_assert(NS % 4 == 0 && (kChunk * 4) == kThreads, "row-major thread mapping");
  constexpr int JW = NS / 4;  // value columns per thread in the (row, column-group) mapping
  extern __shared__ float4 smem_raw[];
  SimtSmem<DK, NS> &sm = *reinterpret_cast<SimtSmem<DK, NS> *>(smem_raw);

  const int sl = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int j0 = sl * NS;
  const int tid = threadIdx.x;
  int64_t t_begin, t_end;
  if (cu_seqlens) {
    t_begin = cu_seqlens[s];
    t_end = cu_seqlens[s + 1];
  } else {
    t_begin = static_cast<int64_t>(s) * fixed_len;
    t_end = t_begin + fixed_len;
  }
  int64_t snap_row = 0;
  if (snaps) snap_row = snap_offsets ? snap_offsets[s] : static_cast<int64_t>(s) * (fixed_len / kChunk);
  const float eA = expf(A[h]);
  // S0 / S_final rows: the sequence itself, or its slot of a state pool
  const size_t state_off = (static_cast<size_t>(slots ? slots[s] : s) * H + h) * DK * DV;

  for (int x = tid; x < DK * NS; x += kThreads) {
    const int c = x / NS, j = x % NS;
    sm.S[c][j] = S0 ? S0[state_off + static_cast<size_t>(c) * DV + j0 + j] : 0.f;
  }

  // Thread mapping for the (row, value-column) products: row r, columns jb..jb+JW.
  const int mr = tid >> 2, mjb = (tid & 3) * JW;
  float *R1 = &sm.AW[0][0];
  float *W = R1 + kChunk * NS;

  for (int64_t t0 = t_begin; t0 < t_end; t0 += kChunk) {
    const int L = static_cast<int>(min(static_cast<int64_t>(kChunk), t_end - t0));
    __syncthreads();  // the previous chunk is done with shared memory

    // 1. load k, q, decay factors a = exp(g), v slice, beta; rows >= L are
    //    padding (k = q = v = 0, beta = 0, a = 1) and change nothing.
    for (int x = tid; x < kChunk * DK; x += kThreads) {
      const int r = x / DK, c = x % DK;
      float kv = 0.f, qv = 0.f, a = 1.f;
      if (r < L) {
        const size_t gi = (static_cast<size_t>(t0 + r) * H + h) * DK + c;
        kv = bf2f(k[gi]);
        qv = bf2f(q[gi]);
        a = decay_factor(gmin, eA, bf2f(z[gi]));
      }
      sm.KE[r][c] = kv;
      sm.QE[r][c] = qv;
      sm.KH[r][c] = a;
    }
    for (int x = tid; x < kChunk * NS; x += kThreads) {
      const int r = x / NS, j = x % NS;
      sm.V[r][j] = r < L ? bf2f(v[(static_cast<size_t>(t0 + r) * H + h) * DV + j0 + j]) : 0.f;
    }
    if (tid < kChunk) {
      float b = tid < L ? bf2f(beta[static_cast<size_t>(t0 + tid) * H + h]) : 0.f;
      if ((pre & KDA_PRE_SIGMOID_BETA) && tid < L) b = 1.f / (1.f + __expf(-b));
      sm.beta[tid] = b;
    }
    __syncthreads();
    if (pre & KDA_PRE_L2NORM_QK) {
      // raw q, k: unit L2 norm per row, four threads per row (DK / 4 channels each)
      const int r = tid >> 2, c0 = (tid & 3) * (DK / 4);
      float sk = 0.f, sq = 0.f;
      for (int c = c0; c < c0 + DK / 4; ++c) {
        sk += sm.KE[r][c] * sm.KE[r][c];
        sq += sm.QE[r][c] * sm.QE[r][c];
      }
#pragma unroll
      for (int off = 1; off < 4; off <<= 1) {
        sk += __shfl_xor_sync(0xffffffffu, sk, off);
        sq += __shfl_xor_sync(0xffffffffu, sq, off);
      }
      const float ik = sk > 0.f ? rsqrtf(sk) : 0.f, iq = sq > 0.f ? rsqrtf(sq) : 0.f;
      for (int c = c0; c < c0 + DK / 4; ++c) {
        sm.KE[r][c] *= ik;
        sm.QE[r][c] *= iq;
      }
      __syncthreads();
    }

    // 2. per (sub-tile R, channel c): backward products Eb[r] = prod_{m=r+1}^{end(R)} a_m
    //    into KP, forward products Ef[r] = prod_{m=start(R)}^{r} a_m in place in KH,
    //    sub-tile totals Lam[R] = Ef[end(R)].
    for (int x = tid; x < kSubTiles * DK; x += kThreads) {
      const int R = x / DK, c = x % DK;
      float acc = 1.f;
      for (int r = kSub * R + kSub - 1; r >= kSub * R; --r) {
        sm.KP[r][c] = acc;
        acc *= sm.KH[r][c];
      }
      float f = 1.f;
      for (int r = kSub * R; r < kSub * R + kSub; ++r) {
        f *= sm.KH[r][c];
        sm.KH[r][c] = f;
      }
    }
    __syncthreads();
    for (int c = tid; c < DK; c += kThreads) {
      float lam[kSubTiles];
#pragma unroll
      for (int R = 0; R < kSubTiles; ++R) {
        lam[R] = sm.KH[kSub * R + kSub - 1][c];
        sm.lam_inv[R][c] = 1.f / lam[R];
      }
#pragma unroll
      for (int R = 0; R < kSubTiles; ++R) {
        float xr = 1.f;
        sm.X[R][R][c] = 1.f;
        for (int J = R - 1; J >= 0; --J) {
          xr *= lam[J];
          sm.X[R][J][c] = xr;
        }
      }
      float y = 1.f;
#pragma unroll
      for (int R = kSubTiles - 1; R >= 0; --R) {
        sm.Y[R][c] = y;
        y *= lam[R];
      }
      sm.gam[c] = y;
    }
    __syncthreads();

    // 3. in-place element transform (each element reads and writes only itself).
    for (int x = tid; x < kChunk * DK; x += kThreads) {
      const int r = x / DK, c = x % DK, R = r / kSub;
      const float kv = sm.KE[r][c], qv = sm.QE[r][c], ef = sm.KH[r][c], eb = sm.KP[r][c];
      sm.KE[r][c] = kv * ef;
      sm.QE[r][c] = qv * ef;
      sm.KH[r][c] = kv * eb * sm.lam_inv[R][c];
      sm.KP[r][c] = kv * eb * sm.Y[R][c];
    }
    __syncthreads();

    // 4. A_kk (strictly lower, times beta_r) and P (lower incl.), sub-tile by sub-tile:
    //    e^{G_r - G_i} = [Ef_r X[R][J]] * [Eb_i / Lam_J].
    for (int p = tid; p < kChunk * kChunk; p += kThreads) {
      const int r = p / kChunk, i = p % kChunk;
      float sk = 0.f, sq = 0.f;
      if (i <= r) {
        const int R = r / kSub, J = i / kSub;
        for (int c = 0; c < DK; ++c) {
          const float kh = sm.KH[i][c] * sm.X[R][J][c];
          sk += sm.KE[r][c] * kh;
          sq += sm.QE[r][c] * kh;
        }
      }
      sm.AW[r][i] = (i < r) ? sm.beta[r] * sk : 0.f;
      sm.P[r][i] = sq;
    }
    __syncthreads();

    // 5. T = (I + A_kk)^{-1} by forward substitution, one column per thread.
    if (tid < kChunk) {
      const int i = tid;
      for (int r = 0; r < kChunk; ++r) sm.T[r][i] = (r == i) ? 1.f : 0.f;
      for (int r = i + 1; r < kChunk; ++r) {
        float acc = 0.f;
        for (int m = i; m < r; ++m) acc += sm.AW[r][m] * sm.T[m][i];
        sm.T[r][i] = -acc;
      }
    }
    __syncthreads();

    // 6. R1 = beta (V - (K * e^G) S)   [C x NS]; A_kk is no longer needed.
    {
      const int R = mr / kSub;
      float acc[JW];
#pragma unroll
      for (int jj = 0; jj < JW; ++jj) acc[jj] = 0.f;
      for (int c = 0; c < DK; ++c) {
        const float kt = sm.KE[mr][c] * sm.X[R][0][c];
#pragma unroll
        for (int jj = 0; jj < JW; ++jj) acc[jj] += kt * sm.S[c][mjb + jj];
      }
#pragma unroll
      for (int jj = 0; jj < JW; ++jj)
        R1[mr * NS + mjb + jj] = sm.beta[mr] * (sm.V[mr][mjb + jj] - acc[jj]);
    }
    __syncthreads();

    // 7. W = T R1.
    {
      float acc[JW];
#pragma unroll
      for (int jj = 0; jj < JW; ++jj) acc[jj] = 0.f;
      for (int i = 0; i <= mr; ++i) {
        const float t = sm.T[mr][i];
#pragma unroll
        for (int jj = 0; jj < JW; ++jj) acc[jj] += t * R1[i * NS + mjb + jj];
      }
#pragma unroll
      for (int jj = 0; jj < JW; ++jj) W[mr * NS + mjb + jj] = acc[jj];
    }
    __syncthreads();

    // 8. O = (Q * e^G) S + P W  -> bf16 output rows < L.
    {
      const int R = mr / kSub;
      float acc[JW];
#pragma unroll
      for (int jj = 0; jj < JW; ++jj) acc[jj] = 0.f;
      for (int c = 0; c < DK; ++c) {
        const float qt = sm.QE[mr][c] * sm.X[R][0][c];
#pragma unroll
        for (int jj = 0; jj < JW; ++jj) acc[jj] += qt * sm.S[c][mjb + jj];
      }
      for (int i = 0; i <= mr; ++i) {
        const float pv = sm.P[mr][i];
#pragma unroll
        for (int jj = 0; jj < JW; ++jj) acc[jj] += pv * W[i * NS + mjb + jj];
      }
      if (mr < L) {
        kda_bf16 *orow = o + (static_cast<size_t>(t0 + mr) * H + h) * DV + j0 + mjb;
#pragma unroll
        for (int jj = 0; jj < JW; ++jj) orow[jj] = f2bf(acc[jj]);
      }
    }
    __syncthreads();

    // 9. S' = Diag(e^{G_last}) S + (K * e^{G_last - G})^T W, each thread owns
    //    (DK * NS / kThreads) entries of S.
    {
      constexpr int PER = DK * NS / kThreads;
      constexpr int TPC = NS / PER;  // threads per state row
      const int c = tid / TPC, jb = (tid % TPC) * PER;
      float acc[PER];
#pragma unroll
      for (int jj = 0; jj < PER; ++jj) acc[jj] = sm.gam[c] * sm.S[c][jb + jj];
      for (int r = 0; r < kChunk; ++r) {
        const float kp = sm.KP[r][c];
#pragma unroll
        for (int jj = 0; jj < PER; ++jj) acc[jj] += kp * W[r * NS + jb + jj];
      }
#pragma unroll
      for (int jj = 0; jj < PER; ++jj) sm.S[c][jb + jj] = acc[jj];
      if (snaps && L == kChunk) {
        float *dst = snaps + (static_cast<size_t>(snap_row) * H + h) * DK * DV +
                     static_cast<size_t>(c) * DV + j0 + jb;
#pragma unroll
        for (int jj = 0; jj < PER; ++jj) dst[jj] = acc[jj];
      }
    }
    if (L == kChunk) ++snap_row;
  }
  __syncthreads();
  if (S_final) {
    for (int x = tid; x < DK * NS; x += kThreads) {
      const int c = x / NS, j = x % NS;
      S_final[state_off + static_cast<size_t>(c) * DV + j0 + j] = sm.S[c][j];
    }
  }
}

template <int DK, int NS>
cudaError_t launch_simt(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                        const kda_bf16 *z, const kda_bf16 *beta, const float *A, float gmin,
                        const int32_t *cu_seqlens, int n_seq, int64_t fixed_len, int H, int dv,
                        const float *S0, kda_bf16 *o, float *S_final, float *snaps,
                        const int64_t *snap_offsets, const int32_t *slots, unsigned pre,
                        cudaStream_t stream) {
  const size_t smem = sizeof(SimtSmem<DK, NS>);
  cudaError_t err = cudaFuncSetAttribute(prefill_simt_kernel<DK, NS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const dim3 grid(static_cast<unsigned>(dv / NS), static_cast<unsigned>(H),
                  static_cast<unsigned>(n_seq));
  prefill_simt_kernel<DK, NS><<<grid, kThreads, smem, stream>>>(
      q, k, v, z, beta, A, gmin, cu_seqlens, fixed_len, H, dv, S0, o, S_final, snaps,
      snap_offsets, slots, pre);
  return cudaGetLastError();
}

}  // namespace

cudaError_t prefill_simt_launch(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                                const kda_bf16 *z, const kda_bf16 *beta, const float *A,
                                float gmin, const int32_t *cu_seqlens, int n_seq,
                                int64_t fixed_len, int H, int dk, int dv, const float *S0,
                                kda_bf16 *o, float *S_final, float *snaps,
                                const int64_t *snap_offsets, const int32_t *slots,
                                unsigned pre, cudaStream_t stream) {
  if (dk == 128)
    return launch_simt<128, 32>(q, k, v, z, beta, A, gmin, cu_seqlens, n_seq, fixed_len, H, dv,
                                S0, o, S_final, snaps, snap_offsets, slots, pre, stream);
  if (dk == 64)
    return launch_simt<64, 32>(q, k, v, z, beta, A, gmin, cu_seqlens, n_seq, fixed_len, H, dv,
                               S0, o, S_final, snaps, snap_offsets, slots, pre, stream);
  return cudaErrorInvalidValue;
}

}  // namespace kda
