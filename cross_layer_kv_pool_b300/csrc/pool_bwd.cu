// Backward pass of the pool ("WhiteMatter: All-to-All Cross-Layer Connections
// via KV Mixing", 3 METHOD, "Cross-layer KV pool"; the gradients a truncated-
// backprop training schedule needs, 4 EXPERIMENTS). For N token rows and
// upstream gradients dK, dV of their cached channels, the forward pool is
// recomputed in fp32 and undone step by step:
//   RoPE^T (rotation by -pos) and K-norm backward      -> dY_K,   d kappa
//   dW_j += dY_j^T c_j,  dc_j = dY_j W_j                (batched over channels)
//   channel-norm backward                              -> dm,     d tau
//   da_{j,l} = <dm_j, n_l>,  dn_l = sum_j a_{j,l} dm_j  (per row)
//   dW_R += da^T x,  dn_R += da W_R                     (router)
//   per-source norm backward                           -> dh,     d sigma
// Everything is fp32 (weights converted once per call). The norm, RoPE and
// scatter steps are this file's kernels; the products, all plain GEMMs, run
// on the fp32 strided-batched GEMM of sgemm.cu (batched over channels or
// rows). Gains and weight gradients accumulate (+=); dstates is overwritten.
#include "kernels.h"

namespace wm {
namespace {

// ---------------------------------------------------------------------------
// Forward recompute
// ---------------------------------------------------------------------------

// n[r][l] = h * inv * sigma; x[r] = concat of n over the router sources; inv.
template <typename S>
__global__ void __launch_bounds__(256) bwd_src_norm_fwd(const S* __restrict__ states, int L, int D,
                                                        const S* __restrict__ sigma, float eps,
                                                        int p, int p_offset, int nR,
                                                        float* __restrict__ inv,
                                                        float* __restrict__ n,
                                                        float* __restrict__ x) {
  __shared__ float red[32];
  const long long rl = blockIdx.x;  // row * L + l
  const int l = (int)(rl % L);
  const long long r = rl / L;
  const S* h = states + rl * D;
  float ss = 0.f;
  for (int t = threadIdx.x; t < D; t += blockDim.x) {
    const float v = to_f(h[t]);
    ss += v * v;
  }
  ss = block_sum(ss, red);
  const float iv = rsqrtf(ss / (float)D + eps);
  if (threadIdx.x == 0) inv[rl] = iv;
  const bool src = (l % p) == p_offset;
  float* xr = x + (r * nR + l / p) * D;
  for (int t = threadIdx.x; t < D; t += blockDim.x) {
    const float v = to_f(h[t]) * iv * to_f(sigma[(size_t)l * D + t]);
    n[rl * D + t] = v;
    if (src) xr[t] = v;
  }
}

// m[j][r] = sum_l a[r][j][l] n[r][l]; rj[r][j] = rms(m); c[j][r] = m / rj * tau_j.
__global__ void __launch_bounds__(256) bwd_mix_fwd(const float* __restrict__ a,
                                                   const float* __restrict__ n, int N, int L, int D,
                                                   int k, const float* __restrict__ tau,
                                                   float eps, float* __restrict__ m,
                                                   float* __restrict__ rj, float* __restrict__ c) {
  __shared__ float red[32];
  __shared__ float coef[1024];
  const long long r = blockIdx.x;
  for (int i = threadIdx.x; i < k * L; i += blockDim.x) coef[i] = a[r * k * L + i];
  __syncthreads();
  const float* nr = n + r * L * D;
  for (int j = 0; j < k; ++j) {
    float ss = 0.f;
    for (int t = threadIdx.x; t < D; t += blockDim.x) {
      float acc = 0.f;
      for (int l = 0; l < L; ++l) acc = fmaf(coef[j * L + l], nr[(size_t)l * D + t], acc);
      m[((size_t)j * N + r) * D + t] = acc;
      ss += acc * acc;
    }
    ss = block_sum(ss, red);
    const float rr = sqrtf(ss / (float)D + eps);
    if (threadIdx.x == 0) rj[r * k + j] = rr;
    for (int t = threadIdx.x; t < D; t += blockDim.x)
      c[((size_t)j * N + r) * D + t] = m[((size_t)j * N + r) * D + t] / rr * tau[(size_t)j * D + t];
  }
}

// The same for k <= KMAX, one block per row reading each n element once: a
// thread holds the k mixed values of its column in registers.
template <int KMAX>
__global__ void __launch_bounds__(256) bwd_mix_fwd_k(const float* __restrict__ a,
                                                     const float* __restrict__ n, int N, int L,
                                                     int D, int k, const float* __restrict__ tau,
                                                     float eps, float* __restrict__ m,
                                                     float* __restrict__ rj, float* __restrict__ c) {
  __shared__ float coef[1024];
  __shared__ float red[KMAX][8];
  __shared__ float rr[KMAX];
  const long long r = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < k * L; i += blockDim.x) coef[i] = a[r * k * L + i];
  __syncthreads();
  const float* nr = n + r * L * D;
  float ss[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) ss[j] = 0.f;
  for (int t = threadIdx.x; t < D; t += blockDim.x) {
    float acc[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) acc[j] = 0.f;
    // eight source rows per step: their loads are in flight together
    int l = 0;
    for (; l + 8 <= L; l += 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = nr[(size_t)(l + u) * D + t];
#pragma unroll
      for (int u = 0; u < 8; ++u)
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (j < k) acc[j] = fmaf(coef[j * L + l + u], v[u], acc[j]);
    }
    for (; l < L; ++l) {
      const float v = nr[(size_t)l * D + t];
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < k) acc[j] = fmaf(coef[j * L + l], v, acc[j]);
    }
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < k) {
        m[((size_t)j * N + r) * D + t] = acc[j];
        ss[j] = fmaf(acc[j], acc[j], ss[j]);
      }
  }
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    const float v = warp_sum(ss[j]);
    if (lane == 0) red[j][warp] = v;
  }
  __syncthreads();
  if (threadIdx.x < k) {
    float t = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[threadIdx.x][w];
    rr[threadIdx.x] = sqrtf(t / (float)D + eps);
    rj[r * k + threadIdx.x] = rr[threadIdx.x];
  }
  __syncthreads();
  for (int j = 0; j < k; ++j) {
    const float inv = 1.f / rr[j];
    for (int t = threadIdx.x; t < D; t += blockDim.x) {
      const size_t i = ((size_t)j * N + r) * D + t;
      c[i] = m[i] * inv * tau[(size_t)j * D + t];
    }
  }
}

// ---------------------------------------------------------------------------
// Backward steps
// ---------------------------------------------------------------------------

// Keys: dk^ = RoPE^T(dK) (rotation by -pos), then the K-norm backward against
// kt = c W_K^T; writes dY[j][r][h*d + t] and accumulates d kappa_j. One block
// (d threads) per (channel, block of rows).
template <typename S>
__global__ void bwd_knorm(const S* __restrict__ dK, const float* __restrict__ kt,
                          const int* __restrict__ pos, int N, int k, int Hkv, int d,
                          const S* __restrict__ kappa, float eps, double rope_base, int rows,
                          float* __restrict__ dY, float* __restrict__ dkappa) {
  __shared__ float red[32];
  __shared__ float buf[256];
  const int j = blockIdx.y;
  const int t = threadIdx.x, half = d / 2;
  const float kap = to_f(kappa[(size_t)j * d + t]);
  const double theta = pow(rope_base, -2.0 * (double)(t % half) / (double)d);
  float dk_acc = 0.f;
  const long long r0 = (long long)blockIdx.x * rows;
  for (long long r = r0; r < r0 + rows && r < N; ++r) {
    double sn, cs;
    sincos((double)pos[r] * theta, &sn, &cs);
    for (int hh = 0; hh < Hkv; ++hh) {
      const float g = to_f(dK[(((size_t)r * k + j) * Hkv + hh) * d + t]);
      buf[t] = g;
      __syncthreads();
      // forward: y1 = x1 c - x2 s, y2 = x2 c + x1 s; transpose: x1 = y1 c + y2 s, x2 = y2 c - y1 s
      const float gp = buf[t < half ? t + half : t - half];
      const float dkh = t < half ? (float)(g * cs + gp * sn) : (float)(g * cs - gp * sn);
      __syncthreads();
      const float x = kt[(((size_t)j * N + r) * Hkv + hh) * d + t];
      const float ssx = block_sum(x * x, red);
      const float rho = sqrtf(ssx / (float)d + eps);
      const float gk = kap * dkh;
      const float sgx = block_sum(gk * x, red);
      dY[(((size_t)j * N + r) * Hkv + hh) * d + t] = gk / rho - x * sgx / ((float)d * rho * rho * rho);
      dk_acc += x / rho * dkh;
    }
  }
  atomicAdd(&dkappa[(size_t)j * d + t], dk_acc);
}

// Values: dY[j][r] = dV[r][j] as fp32.
template <typename S>
__global__ void bwd_copy_dv(const S* __restrict__ dV, int N, int k, int w, float* __restrict__ dY) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)N * k * w) return;
  const int t = (int)(i % w);
  const long long rj = i / w;
  const int j = (int)(rj % k);
  const long long r = rj / k;
  dY[((size_t)j * N + r) * w + t] = to_f(dV[i]);
}

// RMSNorm backward over rows of D (y = w * x / rr), in place on dx:
// dx = g / rr - x * sum(g * x) / (D rr^3) with g = w * dy; the w-gradient
// sum(x / rr * dy) over the rows is added to dw. One warp per row (8 rows in
// flight per block), the w-gradient gathered in shared memory (dynamic, D
// floats) and added once per block; block (chunk, gain gi) takes rows
// chunk * rows .. + rows, row q of gain gi at x + gi * xstride_gain + q *
// xstride_row.
__global__ void __launch_bounds__(256) bwd_rms_w(const float* __restrict__ x, long long xstride_gain,
                                                 long long xstride_row, const float* __restrict__ rr,
                                                 long long rr_stride_gain, long long rr_stride_row,
                                                 const float* __restrict__ w, int D, int rows_total,
                                                 int rows, float* __restrict__ dxy,
                                                 float* __restrict__ dw) {
  extern __shared__ float acc[];
  const int gi = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* wg = w + (size_t)gi * D;
  for (int t = threadIdx.x; t < D; t += blockDim.x) acc[t] = 0.f;
  __syncthreads();
  const int r0 = blockIdx.x * rows, r1 = min(r0 + rows, rows_total);
  for (int q = r0 + warp; q < r1; q += (int)(blockDim.x >> 5)) {
    const float* xr = x + gi * xstride_gain + q * xstride_row;
    float* dr = dxy + gi * xstride_gain + q * xstride_row;
    const float rv = rr[gi * rr_stride_gain + q * rr_stride_row];
    float s = 0.f;
    for (int t = lane; t < D; t += 32) s = fmaf(wg[t] * dr[t], xr[t], s);
    s = warp_sum(s);
    const float c3 = s / ((float)D * rv * rv * rv), iv = 1.f / rv;
    for (int t = lane; t < D; t += 32) {
      const float dy = dr[t], xv = xr[t];
      atomicAdd(&acc[t], xv * iv * dy);
      dr[t] = wg[t] * dy * iv - xv * c3;
    }
  }
  __syncthreads();
  for (int t = threadIdx.x; t < D; t += blockDim.x) atomicAdd(&dw[(size_t)gi * D + t], acc[t]);
}

// dn[r][R_i] += dx[r][i]
__global__ void bwd_scatter_dx(const float* __restrict__ dx, int N, int L, int D, int p,
                               int p_offset, int nR, float* __restrict__ dn) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)N * nR * D) return;
  const int t = (int)(i % D);
  const long long ri = i / D;
  const int s = (int)(ri % nR);
  const long long r = ri / nR;
  dn[(r * L + p_offset + (long long)s * p) * D + t] += dx[i];
}

// Source norm backward: dh = sigma*dn*inv - h*sum(sigma*dn*h)*inv^3/D, added to
// dstates (written on the first branch); d sigma_l accumulated. One warp per
// row (8 rows in flight per block), d sigma gathered in shared memory
// (dynamic, D floats) and added once per block; block (chunk, l) takes rows
// chunk * rows .. + rows of layer l.
template <typename S>
__global__ void __launch_bounds__(256) bwd_src_norm_w(const S* __restrict__ states, int N, int L,
                                                      int D, const float* __restrict__ inv,
                                                      const S* __restrict__ sigma,
                                                      const float* __restrict__ dn, int rows,
                                                      bool first, float* __restrict__ dstates,
                                                      float* __restrict__ dsigma) {
  extern __shared__ float acc[];
  const int l = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const S* sg = sigma + (size_t)l * D;
  for (int t = threadIdx.x; t < D; t += blockDim.x) acc[t] = 0.f;
  __syncthreads();
  const int r0 = blockIdx.x * rows, r1 = min(r0 + rows, N);
  for (int r = r0 + warp; r < r1; r += (int)(blockDim.x >> 5)) {
    const size_t base = ((size_t)r * L + l) * D;
    const float iv = inv[(size_t)r * L + l];
    float s = 0.f;
    for (int t = lane; t < D; t += 32) s = fmaf(to_f(sg[t]) * dn[base + t], to_f(states[base + t]), s);
    s = warp_sum(s);
    const float c3 = s * iv * iv * iv / (float)D;
    for (int t = lane; t < D; t += 32) {
      const float h = to_f(states[base + t]), g = dn[base + t];
      atomicAdd(&acc[t], h * iv * g);
      const float dh = to_f(sg[t]) * g * iv - h * c3;
      dstates[base + t] = first ? dh : dstates[base + t] + dh;
    }
  }
  __syncthreads();
  for (int t = threadIdx.x; t < D; t += blockDim.x) atomicAdd(&dsigma[(size_t)l * D + t], acc[t]);
}

template <typename S>
__global__ void to_f32(const S* __restrict__ src, long long n, float* __restrict__ dst) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) dst[i] = to_f(src[i]);
}

__global__ void broadcast_rows(const float* __restrict__ src, int n, int N, float* __restrict__ dst) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < (long long)N * n) dst[i] = src[i % n];
}

bool gemm_rm(bool ta, bool tb, int M, int N, int K, const float* A, long long lda, long long sa,
             const float* B, long long ldb, long long sb, float beta, float* C, long long ldc,
             long long sc, int batch, cudaStream_t st) {
  SgemmArgs g{ta, tb, M, N, K, A, lda, sa, B, ldb, sb, beta, C, ldc, sc, batch};
  return sgemm_rm(g, st) == cudaSuccess;
}

}  // namespace

// Workspace for N rows: fp32 buffers (see run_pool_backward), 256-byte aligned.
PoolBwdLayout pool_bwd_layout(const wm_config& c, long long N) {
  PoolBwdLayout lay;
  const long long L = c.L, D = c.D, k = c.k, w = (long long)c.Hkv * c.d;
  long long nR = 0;
  for (int l = 0; l < c.L; ++l) nR += (l % c.p) == c.p_offset;
  const long long sz[PoolBwdLayout::NB] = {
      N * L,          // inv
      N * L * D,      // n (one branch)
      N * nR * D,     // x (router input)
      N * k * L,      // a, then da
      k * N * D,      // m
      N * k,          // rms of m
      k * N * D,      // c
      k * N * w,      // kt = c W_K^T
      k * N * w,      // dY
      k * N * D,      // dc, then dm
      N * L * D,      // dn
      N * nR * D,     // dx
      k * L * nR * D, // W_R (fp32)
      k * w * D,      // W_K or W_V (fp32)
      2 * k * D,      // channel-norm gains (fp32)
      N * k * L,      // a (kept for the mix backward)
  };
  size_t o = 0;
  for (int i = 0; i < PoolBwdLayout::NB; ++i) {
    lay.off[i] = o;
    o += (size_t)((sz[i] * 4 + 255) / 256 * 256);
  }
  lay.total = o;
  return lay;
}

cudaError_t run_pool_backward(const PoolBwdArgs& q, cudaStream_t st) {
  const wm_config& c = *q.cfg;
  const int N = q.N, L = c.L, D = c.D, k = c.k, Hkv = c.Hkv, d = c.d, w = Hkv * d;
  int nR = 0;
  for (int l = 0; l < c.L; ++l) nR += (l % c.p) == c.p_offset;
  const PoolBwdLayout& lay = q.lay;
  auto buf = [&](int b) { return reinterpret_cast<float*>(static_cast<char*>(q.ws) + lay.off[b]); };
  float *inv = buf(PoolBwdLayout::INV), *n = buf(PoolBwdLayout::N_), *x = buf(PoolBwdLayout::X),
        *a = buf(PoolBwdLayout::A), *m = buf(PoolBwdLayout::M), *rj = buf(PoolBwdLayout::RJ),
        *cc = buf(PoolBwdLayout::C), *kt = buf(PoolBwdLayout::KT), *dY = buf(PoolBwdLayout::DY),
        *dc = buf(PoolBwdLayout::DC), *dn = buf(PoolBwdLayout::DN), *dx = buf(PoolBwdLayout::DX),
        *wr = buf(PoolBwdLayout::WR), *wp = buf(PoolBwdLayout::WP), *gains = buf(PoolBwdLayout::G),
        *a_keep = buf(PoolBwdLayout::AK);
  const wm_weights& W = *q.w;
  const long long WRn = (long long)k * L * nR * D, WPn = (long long)k * w * D;
  float* tau32 = gains;  // [2][k][D]
  WM_DISPATCH_S(c.dtype, {
    to_f32<S><<<(unsigned)((2LL * k * D + 255) / 256), 256, 0, st>>>((const S*)W.chan_norm, 2LL * k * D, tau32);
  });
  bool ok = true;
  for (int be = 0; be < 2 && ok; ++be) {
    const char* sig = static_cast<const char*>(W.src_norm) + (size_t)be * L * D * (c.dtype == WM_F32 ? 4 : 2);
    WM_DISPATCH_S(c.dtype, {
      bwd_src_norm_fwd<S><<<(unsigned)((long long)N * L), 256, 0, st>>>(
          (const S*)q.states, L, D, (const S*)sig, c.eps, c.p, c.p_offset, nR, inv, n, x);
    });
    // coefficients: the router (x W_R^T) or the constants
    if (W.static_coeff) {
      broadcast_rows<<<(unsigned)(((long long)N * k * L + 255) / 256), 256, 0, st>>>(
          W.static_coeff + (size_t)be * k * L, k * L, N, a_keep);
    } else {
      const char* wrs = static_cast<const char*>(W.Wr) + (size_t)be * WRn * (c.dtype == WM_F32 ? 4 : 2);
      WM_DISPATCH_S(c.dtype, {
        to_f32<S><<<(unsigned)((WRn + 255) / 256), 256, 0, st>>>((const S*)wrs, WRn, wr);
      });
      ok = ok && gemm_rm(false, true, N, k * L, nR * D, x, nR * D, 0, wr, nR * D, 0, 0.f, a_keep,
                         k * L, 0, 1, st);
    }
    if (k <= 16)
      bwd_mix_fwd_k<16><<<N, 256, 0, st>>>(a_keep, n, N, L, D, k, tau32 + (size_t)be * k * D, c.eps, m, rj, cc);
    else
      bwd_mix_fwd<<<N, 256, 0, st>>>(a_keep, n, N, L, D, k, tau32 + (size_t)be * k * D, c.eps, m, rj, cc);
    // projections: kt (keys only), dY, weight gradients and dc
    const char* wps = static_cast<const char*>(be == 0 ? W.Wk : W.Wv);
    WM_DISPATCH_S(c.dtype, {
      to_f32<S><<<(unsigned)((WPn + 255) / 256), 256, 0, st>>>((const S*)wps, WPn, wp);
    });
    if (be == 0) {
      ok = ok && gemm_rm(false, true, N, w, D, cc, D, (long long)N * D, wp, D, (long long)w * D,
                         0.f, kt, w, (long long)N * w, k, st);
      const int rows = 64;
      dim3 grid((N + rows - 1) / rows, k);
      WM_DISPATCH_S(c.dtype, {
        bwd_knorm<S><<<grid, d, 0, st>>>((const S*)q.dK, kt, q.pos, N, k, Hkv, d, (const S*)W.k_norm,
                                         c.eps, (double)c.rope_base, rows, dY, q.g.dk_norm);
      });
    } else {
      WM_DISPATCH_S(c.dtype, {
        bwd_copy_dv<S><<<(unsigned)(((long long)N * k * w + 255) / 256), 256, 0, st>>>(
            (const S*)q.dV, N, k, w, dY);
      });
    }
    float* dW = be == 0 ? q.g.dWk : q.g.dWv;
    // dW_j += dY_j^T c_j  ([w x N] [N x D]);  dc_j = dY_j W_j  ([N x w] [w x D])
    ok = ok && gemm_rm(true, false, w, D, N, dY, w, (long long)N * w, cc, D, (long long)N * D, 1.f,
                       dW, D, (long long)w * D, k, st);
    ok = ok && gemm_rm(false, false, N, D, w, dY, w, (long long)N * w, wp, D, (long long)w * D, 0.f,
                       dc, D, (long long)N * D, k, st);
    {  // channel norm backward, in place: dc -> dm
      const int rows = 64;
      dim3 grid((N + rows - 1) / rows, k);
      bwd_rms_w<<<grid, 256, (size_t)D * 4, st>>>(m, (long long)N * D, D, rj, 1, k,
                                                  tau32 + (size_t)be * k * D, D, N, rows, dc,
                                                  q.g.dchan_norm + (size_t)be * k * D);
    }
    // mix backward per row r: da_r [k x L] = dm_r [k x D] n_r^T; dn_r [L x D] = a_r^T dm_r
    ok = ok && gemm_rm(false, true, k, L, D, dc, (long long)N * D, D, n, D, (long long)L * D, 0.f, a,
                       L, (long long)k * L, N, st);
    ok = ok && gemm_rm(true, false, L, D, k, a_keep, L, (long long)k * L, dc, (long long)N * D, D,
                       0.f, dn, D, (long long)L * D, N, st);
    if (!W.static_coeff && q.g.dWr) {
      // router: dW_R += da^T x ([kL x N] [N x nR D]);  dx = da W_R ([N x kL] [kL x nR D])
      ok = ok && gemm_rm(true, false, k * L, nR * D, N, a, k * L, 0, x, nR * D, 0, 1.f,
                         q.g.dWr + (size_t)be * WRn, nR * D, 0, 1, st);
    }
    if (!W.static_coeff) {
      ok = ok && gemm_rm(false, false, N, nR * D, k * L, a, k * L, 0, wr, nR * D, 0, 0.f, dx, nR * D,
                         0, 1, st);
      bwd_scatter_dx<<<(unsigned)(((long long)N * nR * D + 255) / 256), 256, 0, st>>>(
          dx, N, L, D, c.p, c.p_offset, nR, dn);
    }
    {  // source norm backward into dstates
      const int rows = 64;
      dim3 grid((N + rows - 1) / rows, L);
      WM_DISPATCH_S(c.dtype, {
        bwd_src_norm_w<S><<<grid, 256, (size_t)D * 4, st>>>((const S*)q.states, N, L, D, inv,
                                                            (const S*)sig, dn, rows, be == 0,
                                                            q.dstates,
                                                            q.g.dsrc_norm + (size_t)be * L * D);
      });
    }
  }
  if (!ok) return cudaErrorUnknown;
  return cudaGetLastError();
}

}  // namespace wm
