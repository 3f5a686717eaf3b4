// fp32 general matrix products for the pool's backward pass: strided batches
// of C = op(A) op(B) + beta C on row-major operands, computed with fp32 fused
// multiply-adds in this file's kernel (the backward's gradients are exact
// fp32 arithmetic; the tensor cores have no fp32 operand type).
//
// Tiling: a CTA computes a BM x BN tile of C, stepping K by BK = 8. The A and
// B slabs of the next step are loaded into registers while the current one,
// staged in shared memory (A k-major, B k-major, so that a thread's rows and
// columns are consecutive floats), is multiplied; each thread owns RM x RN
// blocks of 4 x 4 outputs spread across the tile (block r of rows at
// r * BM / RM), so that a warp's float4 reads of one k-row fall on distinct
// banks. Out-of-range rows, columns and k are zero-filled on load and skipped
// on store, so every shape is accepted; beta = 0 never reads C. Accumulating
// products (beta = 1) with few output tiles and a long K are split over K:
// each slice adds its partial tile to C with fp32 atomics (the order of the
// additions, and so the rounding of the sum, then varies from run to run).
#include "kernels.h"

namespace wm {
namespace {

constexpr int BK = 8;

template <int BM, int BN, int RM, int RN, bool TA, bool TB>
__global__ void __launch_bounds__((BM / (4 * RM)) * (BN / (4 * RN)), 2)
    sgemm_kernel(int M, int N, int K, const float* __restrict__ A, long long lda, long long sa,
                 const float* __restrict__ B, long long ldb, long long sb, float beta,
                 float* __restrict__ C, long long ldc, long long sc, int ksplit, int kchunk) {
  constexpr int TX = BN / (4 * RN), TY = BM / (4 * RM), NT = TX * TY;
  constexpr int LA = BM * BK / NT, LB = BN * BK / NT;  // elements each thread loads per step
  static_assert(LA * NT == BM * BK && LB * NT == BN * BK, "tile must divide among threads");
  __shared__ __align__(16) float As[2][BK][BM + 4];
  __shared__ __align__(16) float Bs[2][BK][BN + 4];
  const int tid = threadIdx.x, tx = tid % TX, ty = tid / TX;
  // blockIdx.z = batch entry * ksplit + K slice; slice z covers K columns
  // [z * kchunk, min(K, (z + 1) * kchunk)) and, when ksplit > 1, adds its
  // partial tile to C with atomics (C += A B: beta is 1)
  const long long b = blockIdx.z / ksplit;
  const int kz = (int)(blockIdx.z % ksplit);
  const int kbeg = kz * kchunk, kend = min(K, kbeg + kchunk);
  A += b * sa;
  B += b * sb;
  C += b * sc;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;

  float ra[LA], rb[LB];
  // element e of a slab: TA/TB pick the index that is contiguous in memory
  auto load = [&](int k0) {
#pragma unroll
    for (int i = 0; i < LA; ++i) {
      const int e = tid + i * NT;
      const int kk = TA ? e / BM : e % BK, mm = TA ? e % BM : e / BK;
      const int m = m0 + mm, k = k0 + kk;
      ra[i] = (m < M && k < kend) ? (TA ? A[(long long)k * lda + m] : A[(long long)m * lda + k]) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < LB; ++i) {
      const int e = tid + i * NT;
      const int kk = TB ? e % BK : e / BN, nn = TB ? e / BK : e % BN;
      const int n = n0 + nn, k = k0 + kk;
      rb[i] = (n < N && k < kend) ? (TB ? B[(long long)n * ldb + k] : B[(long long)k * ldb + n]) : 0.f;
    }
  };
  auto stage = [&](int s) {
#pragma unroll
    for (int i = 0; i < LA; ++i) {
      const int e = tid + i * NT;
      As[s][TA ? e / BM : e % BK][TA ? e % BM : e / BK] = ra[i];
    }
#pragma unroll
    for (int i = 0; i < LB; ++i) {
      const int e = tid + i * NT;
      Bs[s][TB ? e % BK : e / BN][TB ? e / BK : e % BN] = rb[i];
    }
  };

  float acc[RM * 4][RN * 4];
#pragma unroll
  for (int i = 0; i < RM * 4; ++i)
#pragma unroll
    for (int j = 0; j < RN * 4; ++j) acc[i][j] = 0.f;

  const int nk = (kend - kbeg + BK - 1) / BK;
  load(kbeg);
  stage(0);
  __syncthreads();
  for (int t = 0; t < nk; ++t) {
    const int s = t & 1;
    if (t + 1 < nk) load(kbeg + (t + 1) * BK);
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float av[RM * 4], bv[RN * 4];
#pragma unroll
      for (int r = 0; r < RM; ++r) {
        const float4 v = *reinterpret_cast<const float4*>(&As[s][kk][r * (BM / RM) + ty * 4]);
        av[4 * r] = v.x; av[4 * r + 1] = v.y; av[4 * r + 2] = v.z; av[4 * r + 3] = v.w;
      }
#pragma unroll
      for (int r = 0; r < RN; ++r) {
        const float4 v = *reinterpret_cast<const float4*>(&Bs[s][kk][r * (BN / RN) + tx * 4]);
        bv[4 * r] = v.x; bv[4 * r + 1] = v.y; bv[4 * r + 2] = v.z; bv[4 * r + 3] = v.w;
      }
#pragma unroll
      for (int i = 0; i < RM * 4; ++i)
#pragma unroll
        for (int j = 0; j < RN * 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    if (t + 1 < nk) stage(s ^ 1);
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < RM * 4; ++i) {
    const int m = m0 + (i / 4) * (BM / RM) + ty * 4 + (i % 4);
    if (m >= M) continue;
    float* cr = C + (long long)m * ldc;
#pragma unroll
    for (int j = 0; j < RN * 4; ++j) {
      const int n = n0 + (j / 4) * (BN / RN) + tx * 4 + (j % 4);
      if (n < N) {
        if (ksplit > 1) atomicAdd(cr + n, acc[i][j]);
        else cr[n] = beta == 0.f ? acc[i][j] : fmaf(beta, cr[n], acc[i][j]);
      }
    }
  }
}

template <int BM, int BN, int RM, int RN>
void launch_cfg(const SgemmArgs& g, int ksplit, int kchunk, cudaStream_t st) {
  constexpr int NT = (BM / (4 * RM)) * (BN / (4 * RN));
  const dim3 grid((unsigned)((g.N + BN - 1) / BN), (unsigned)((g.M + BM - 1) / BM),
                  (unsigned)(g.batch * ksplit));
#define WM_SGEMM_LAUNCH(TA_, TB_)                                                                 \
  sgemm_kernel<BM, BN, RM, RN, TA_, TB_><<<grid, NT, 0, st>>>(g.M, g.N, g.K, g.A, g.lda, g.sa, g.B,   \
                                                              g.ldb, g.sb, g.beta, g.C, g.ldc, g.sc, \
                                                              ksplit, kchunk)
  if (g.ta) {
    if (g.tb) WM_SGEMM_LAUNCH(true, true);
    else WM_SGEMM_LAUNCH(true, false);
  } else {
    if (g.tb) WM_SGEMM_LAUNCH(false, true);
    else WM_SGEMM_LAUNCH(false, false);
  }
#undef WM_SGEMM_LAUNCH
}

}  // namespace

cudaError_t sgemm_rm(const SgemmArgs& g, cudaStream_t st) {
  if (g.M < 0 || g.N < 0 || g.K < 0 || g.batch < 0) return cudaErrorInvalidValue;
  if (g.M == 0 || g.N == 0 || g.batch == 0) return cudaSuccess;
  // small products (the per-row mixing gradients) take 32 x 32 tiles of 64
  // threads; the rest 128 x 128 tiles of 256 threads
  const bool small = g.M <= 32 || g.N <= 32;
  if ((g.M + (small ? 31LL : 127LL)) / (small ? 32 : 128) > 65535) return cudaErrorInvalidValue;
  // Accumulating products (beta = 1) with few tiles and a long K split K
  // over CTAs that add their partial tiles with atomics, to about four
  // resident waves (two 256-thread CTAs per SM) with K slices of >= 512.
  int ksplit = 1;
  if (!small && g.beta == 1.f) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long ctas = ((g.N + 127LL) / 128) * ((g.M + 127LL) / 128) * g.batch;
    const long long want = 4LL * 2 * sms;
    while (ksplit < 16 && ctas * ksplit * 2 <= want && g.K / (ksplit * 2) >= 512) ksplit *= 2;
  }
  const int kchunk = ksplit > 1 ? ((g.K + ksplit - 1) / ksplit + BK - 1) / BK * BK : g.K;
  const int zmax = 65535 / ksplit;  // batch entries per launch (grid z = entries x slices)
  for (int b0 = 0; b0 < g.batch; b0 += zmax) {
    SgemmArgs c = g;
    c.batch = g.batch - b0 < zmax ? g.batch - b0 : zmax;
    c.A += b0 * g.sa;
    c.B += b0 * g.sb;
    c.C += b0 * g.sc;
    if (small) launch_cfg<32, 32, 1, 1>(c, 1, c.K, st);
    else launch_cfg<128, 128, 2, 2>(c, ksplit, kchunk, st);
  }
  return cudaGetLastError();
}

}  // namespace wm
