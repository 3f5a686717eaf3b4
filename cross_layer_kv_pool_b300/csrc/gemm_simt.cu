// CUDA-core GEMM with the library's epilogues. It is the engine of the fp32
// storage mode (whose 1e-4 tolerance rules out reduced-precision tensor-core
// inputs) and a debug engine for bf16 (WM_FLAG_SIMT_GEMM).
//   C[b][m][n] = epi( sum_k A[b][m][k] B[b][n][k] ),  fp32 accumulation.
#include "kernels.h"

namespace wm {

namespace {
constexpr int BM = 32, BN = 128, BK = 16, NT = 256;
}

// Writes one row's run of values through the epilogue. Shared by both modes
// below; v holds ``cnt`` consecutive values of row gm starting at column gn0.
template <typename S>
__device__ void epi_store_head(const Epi& e, int b, int gm, int gn0, float* v) {
  const int d = e.d;
  const int p = e.pos[gm];
  if (p < 0 || p >= e.Tmax) {
    atomicOr(e.flags, FLAG_BAD_POS);
    return;
  }
  if (e.mode == EPI_QNORM_ROPE) {
    head_norm_rope<S>(v, d, (const S*)e.gain, e.eps, e.rope + (long long)p * (d >> 1));
    S* c = (S*)e.C + (long long)gm * e.ldc + gn0;
    for (int t = 0; t < d; ++t) c[t] = from_f<S>(v[t]);
    return;
  }
  // EPI_KV: batch b is the channel j
  const int sq = e.seq[gm];
  if (sq < 0 || sq >= e.B) {
    atomicOr(e.flags, FLAG_BAD_SEQ);
    return;
  }
  if (e.chan_ss) {
    const float cs = chan_scale(e, gm, b);
    for (int t = 0; t < d; ++t) v[t] *= cs;
  }
  if (e.kv_branch == 0)
    head_norm_rope<S>(v, d, (const S*)e.gain + (long long)b * e.gain_bstride, e.eps,
                      e.rope + (long long)p * (d >> 1));
  const int h = gn0 / d;
  S* c = (S*)(e.kv_branch == 0 ? e.cache_k : e.cache_v) +
         ((((long long)sq * e.k + e.chan0 + b) * e.Hkv + h) * e.Tmax + p) * d;
  for (int t = 0; t < d; ++t) c[t] = from_f<S>(v[t]);
}

template <typename S, bool DUAL>
__global__ void __launch_bounds__(NT) gemm_simt_kernel(const GemmDesc g) {
  pdl_wait();
  pdl_trigger();
  __shared__ float As[BK][BM + 1];
  __shared__ float Bs[BK][BN + 4];
  __shared__ float B2s[DUAL ? BK : 1][BN + 4];
  __shared__ float Cs[BM][BN + 1];
  const int b = blockIdx.z;
  const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
  const S* A = (const S*)g.A + (long long)b * g.a_bstride;
  const S* Bm = (const S*)g.B + (long long)b * g.b_bstride;
  const S* B2 = DUAL ? (const S*)g.B2 + (long long)b * g.b_bstride : nullptr;
  const int tid = threadIdx.x, ty = tid >> 5, tx = tid & 31;
  float acc[4][4], acc2[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = acc2[i][j] = 0.f;

  for (int k0 = 0; k0 < g.K; k0 += BK) {
    for (int i = tid; i < BM * BK; i += NT) {
      const int mm = i / BK, kk = i % BK, gm = m0 + mm, gk = k0 + kk;
      As[kk][mm] = (gm < g.M && gk < g.K) ? to_f(A[(long long)gm * g.lda + gk]) : 0.f;
    }
    for (int i = tid; i < BN * BK; i += NT) {
      const int nn = i / BK, kk = i % BK, gn = n0 + nn, gk = k0 + kk;
      const bool ok = gn < g.N && gk < g.K;
      Bs[kk][nn] = ok ? to_f(Bm[(long long)gn * g.ldb + gk]) : 0.f;
      if (DUAL) B2s[kk][nn] = ok ? to_f(B2[(long long)gn * g.ldb + gk]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], bv[4], b2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        bv[j] = Bs[kk][tx + 32 * j];
        if (DUAL) b2[j] = B2s[kk][tx + 32 * j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(a[i], bv[j], acc[i][j]);
          if (DUAL) acc2[i][j] = fmaf(a[i], b2[j], acc2[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
      Cs[ty * 4 + i][tx + 32 * j] = DUAL ? silu_f(acc[i][j]) * acc2[i][j] : acc[i][j];
  __syncthreads();

  const Epi& e = g.epi;
  if (e.mode == EPI_STORE || e.mode == EPI_RESID || e.mode == EPI_SWIGLU) {
    for (int idx = tid; idx < BM * BN; idx += NT) {
      const int mm = idx / BN, nn = idx % BN, gm = m0 + mm, gn = n0 + nn;
      if (gm >= g.M || gn >= g.N) continue;
      float v = Cs[mm][nn];
      if (e.mode == EPI_RESID) v += to_f(((const S*)e.R)[(long long)gm * e.ldr + gn]);
      const long long row = e.rowmap ? e.rowmap[gm] : gm;
      const long long off = (long long)b * e.c_bstride + row * e.ldc + gn;
      if (e.out_f32)
        ((float*)e.C)[off] = v;
      else
        ((S*)e.C)[off] = from_f<S>(v);
    }
  } else {
    const int hpt = BN / e.d;
    for (int task = tid; task < BM * hpt; task += NT) {
      const int mm = task / hpt, hh = task % hpt, gm = m0 + mm, gn0 = n0 + hh * e.d;
      if (gm >= g.M || gn0 >= g.N) continue;
      float v[128];
      for (int t = 0; t < e.d; ++t) v[t] = Cs[mm][hh * e.d + t];
      epi_store_head<S>(e, b, gm, gn0, v);
    }
  }
}

void launch_gemm_simt(int dtype, const GemmDesc& g, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0 || g.batch <= 0) return;
  dim3 grid((g.M + BM - 1) / BM, (g.N + BN - 1) / BN, g.batch);
  if (g.B2) {
    WM_DISPATCH_S(dtype, launch_k(gemm_simt_kernel<S, true>, dim3(grid), dim3(NT), 0, st, g));
  } else {
    WM_DISPATCH_S(dtype, launch_k(gemm_simt_kernel<S, false>, dim3(grid), dim3(NT), 0, st, g));
  }
}

}  // namespace wm
