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
// scatter steps are this file's kernels. The router's three products (a =
// x W_R^T, dx = da W_R, dW_R += da^T x; two thirds of the work) run on the
// tcgen05 GEMM engine with bf16 operands split exactly-to-16-bits: each fp32
// operand v = hi + lo (hi = bf16(v), lo = bf16(v - hi)), the left operand laid
// out along K as [hi | hi | lo] and the right one as [hi | lo | hi], so one
// product over 3K sums hi.hi + hi.lo + lo.hi in fp32 (the dropped lo.lo is
// below 2^-16 relative). The other products run on the fp32 GEMM of sgemm.cu
// (batched over channels or rows). Gains and weight gradients accumulate
// (+=); dstates is overwritten.
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

// The same, one warp per (row, layer) with the state held in registers: lane
// t loads 16-byte vectors t, t + 32, ... (NV of them, all in flight), sums
// their squares, and writes n (and x) as 16-byte stores from the registers.
template <typename S, int NV>
__global__ void __launch_bounds__(256) bwd_src_norm_fwd_w(const S* __restrict__ states, long long NL,
                                                          int L, int D, const S* __restrict__ sigma,
                                                          float eps, int p, int p_offset, int nR,
                                                          float* __restrict__ inv,
                                                          float* __restrict__ n,
                                                          float* __restrict__ x) {
  constexpr int VN = 16 / sizeof(S);
  const int lane = threadIdx.x & 31;
  const long long rl = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);  // row * L + l
  if (rl >= NL) return;  // warp-uniform
  const int l = (int)(rl % L);
  const long long r = rl / L;
  const S* h = states + rl * D;
  float v[NV][VN];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int c = (lane + 32 * k) * VN;
    if (c < D) {
      const uint4 u = *reinterpret_cast<const uint4*>(h + c);
      const S* e = reinterpret_cast<const S*>(&u);
#pragma unroll
      for (int i = 0; i < VN; ++i) v[k][i] = to_f(e[i]);
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k)
    if ((lane + 32 * k) * VN < D) {
#pragma unroll
      for (int i = 0; i < VN; ++i) ss += v[k][i] * v[k][i];
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float iv = rsqrtf(ss / (float)D + eps);
  if (lane == 0) inv[rl] = iv;
  const bool src = (l % p) == p_offset;
  float* xr = x + (r * nR + l / p) * D;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int c = (lane + 32 * k) * VN;
    if (c >= D) continue;
    const uint4 u = *reinterpret_cast<const uint4*>(sigma + (size_t)l * D + c);
    const S* g = reinterpret_cast<const S*>(&u);
#pragma unroll
    for (int i = 0; i < VN; i += 4) {
      const float4 o = make_float4(v[k][i] * iv * to_f(g[i]), v[k][i + 1] * iv * to_f(g[i + 1]),
                                   v[k][i + 2] * iv * to_f(g[i + 2]), v[k][i + 3] * iv * to_f(g[i + 3]));
      *reinterpret_cast<float4*>(n + rl * D + c + i) = o;
      if (src) *reinterpret_cast<float4*>(xr + c + i) = o;
    }
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
  // four consecutive columns per thread (D is a multiple of 64): 16-byte
  // loads of the row's L states, four states' loads in flight at a time
  for (int t = 4 * threadIdx.x; t < D; t += 4 * blockDim.x) {
    float4 acc[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    int l = 0;
    for (; l + 4 <= L; l += 4) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = *reinterpret_cast<const float4*>(nr + (size_t)(l + u) * D + t);
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (j < k) {
            const float a = coef[j * L + l + u];
            acc[j].x = fmaf(a, v[u].x, acc[j].x);
            acc[j].y = fmaf(a, v[u].y, acc[j].y);
            acc[j].z = fmaf(a, v[u].z, acc[j].z);
            acc[j].w = fmaf(a, v[u].w, acc[j].w);
          }
    }
    for (; l < L; ++l) {
      const float4 v = *reinterpret_cast<const float4*>(nr + (size_t)l * D + t);
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < k) {
          const float a = coef[j * L + l];
          acc[j].x = fmaf(a, v.x, acc[j].x);
          acc[j].y = fmaf(a, v.y, acc[j].y);
          acc[j].z = fmaf(a, v.z, acc[j].z);
          acc[j].w = fmaf(a, v.w, acc[j].w);
        }
    }
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < k) {
        *reinterpret_cast<float4*>(m + ((size_t)j * N + r) * D + t) = acc[j];
        ss[j] = fmaf(acc[j].x, acc[j].x, fmaf(acc[j].y, acc[j].y,
                fmaf(acc[j].z, acc[j].z, fmaf(acc[j].w, acc[j].w, ss[j]))));
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
    for (int t = 4 * threadIdx.x; t < D; t += 4 * blockDim.x) {
      const size_t i = ((size_t)j * N + r) * D + t;
      const float4 mv = *reinterpret_cast<const float4*>(m + i);
      const float4 tv = *reinterpret_cast<const float4*>(tau + (size_t)j * D + t);
      *reinterpret_cast<float4*>(c + i) =
          make_float4(mv.x * inv * tv.x, mv.y * inv * tv.y, mv.z * inv * tv.z, mv.w * inv * tv.w);
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
    // the angle and its reduction to [-pi, pi] in double, the sine and
    // cosine of the reduced angle in fp32 (double-precision sincos per row
    // and thread cost more than the rest of the kernel)
    const double ang = (double)pos[r] * theta;
    const double ared = ang - 6.283185307179586 * rint(ang * 0.15915494309189535);
    float sn, cs;
    sincosf((float)ared, &sn, &cs);
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
    // lane l takes columns 4l + 128i (D is a multiple of 64): 16-byte accesses
#pragma unroll 4
    for (int t = 4 * lane; t < D; t += 128) {
      const float4 w = *reinterpret_cast<const float4*>(wg + t);
      const float4 dy = *reinterpret_cast<const float4*>(dr + t);
      const float4 xv = *reinterpret_cast<const float4*>(xr + t);
      s = fmaf(w.x * dy.x, xv.x, fmaf(w.y * dy.y, xv.y, fmaf(w.z * dy.z, xv.z, fmaf(w.w * dy.w, xv.w, s))));
    }
    s = warp_sum(s);
    const float c3 = s / ((float)D * rv * rv * rv), iv = 1.f / rv;
#pragma unroll 4
    for (int t = 4 * lane; t < D; t += 128) {
      const float4 w = *reinterpret_cast<const float4*>(wg + t);
      const float4 dy = *reinterpret_cast<const float4*>(dr + t);
      const float4 xv = *reinterpret_cast<const float4*>(xr + t);
      atomicAdd(&acc[t], xv.x * iv * dy.x);
      atomicAdd(&acc[t + 1], xv.y * iv * dy.y);
      atomicAdd(&acc[t + 2], xv.z * iv * dy.z);
      atomicAdd(&acc[t + 3], xv.w * iv * dy.w);
      *reinterpret_cast<float4*>(dr + t) =
          make_float4(w.x * dy.x * iv - xv.x * c3, w.y * dy.y * iv - xv.y * c3,
                      w.z * dy.z * iv - xv.z * c3, w.w * dy.w * iv - xv.w * c3);
    }
  }
  __syncthreads();
  for (int t = threadIdx.x; t < D; t += blockDim.x) atomicAdd(&dw[(size_t)gi * D + t], acc[t]);
}

// bwd_rms_w with each row held in registers (NV float4 columns a lane, D =
// 128 NV; 16-byte aligned rows), the gains in shared memory and each warp's
// d w summed in a shared row of its own (as bwd_src_norm_wr). Dynamic shared
// memory: (1 + warps) D floats.
template <int NV>
__global__ void __launch_bounds__(256, 1) bwd_rms_wr(const float* __restrict__ x, long long xstride_gain,
                                                     long long xstride_row, const float* __restrict__ rr,
                                                     long long rr_stride_gain, long long rr_stride_row,
                                                     const float* __restrict__ w, int D, int rows_total,
                                                     int rows, float* __restrict__ dxy,
                                                     float* __restrict__ dw) {
  extern __shared__ float sm[];
  const int nw = (int)(blockDim.x >> 5);
  float* wgs = sm;        // [D] the gains
  float* wacc = sm + D;   // [warps][D] each warp's d w
  const int gi = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int t = threadIdx.x; t < D; t += blockDim.x) wgs[t] = w[(size_t)gi * D + t];
  for (int t = threadIdx.x; t < nw * D; t += blockDim.x) wacc[t] = 0.f;
  __syncthreads();
  float* acc = wacc + (size_t)warp * D + 4 * lane;
  const int r0 = blockIdx.x * rows, r1 = min(r0 + rows, rows_total);
  for (int q = r0 + warp; q < r1; q += nw) {
    const float* xr = x + gi * xstride_gain + q * xstride_row + 4 * lane;
    float* dr = dxy + gi * xstride_gain + q * xstride_row + 4 * lane;
    const float rv = rr[gi * rr_stride_gain + q * rr_stride_row];
    float4 dy[NV], xv[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      dy[k] = *reinterpret_cast<const float4*>(dr + 128 * k);
      xv[k] = *reinterpret_cast<const float4*>(xr + 128 * k);
    }
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const float4 wv = *reinterpret_cast<const float4*>(wgs + 4 * lane + 128 * k);
      s = fmaf(wv.x * dy[k].x, xv[k].x,
               fmaf(wv.y * dy[k].y, xv[k].y, fmaf(wv.z * dy[k].z, xv[k].z, fmaf(wv.w * dy[k].w, xv[k].w, s))));
    }
    s = warp_sum(s);
    const float c3 = s / ((float)D * rv * rv * rv), iv = 1.f / rv;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const float4 wv = *reinterpret_cast<const float4*>(wgs + 4 * lane + 128 * k);
      float4* ak = reinterpret_cast<float4*>(acc + 128 * k);
      float4 a4 = *ak;
      a4.x += xv[k].x * iv * dy[k].x;
      a4.y += xv[k].y * iv * dy[k].y;
      a4.z += xv[k].z * iv * dy[k].z;
      a4.w += xv[k].w * iv * dy[k].w;
      *ak = a4;
      *reinterpret_cast<float4*>(dr + 128 * k) =
          make_float4(wv.x * dy[k].x * iv - xv[k].x * c3, wv.y * dy[k].y * iv - xv[k].y * c3,
                      wv.z * dy[k].z * iv - xv[k].z * c3, wv.w * dy[k].w * iv - xv[k].w * c3);
    }
  }
  __syncthreads();
  for (int t = threadIdx.x; t < D; t += blockDim.x) {
    float v = 0.f;
    for (int i = 0; i < nw; ++i) v += wacc[(size_t)i * D + t];
    atomicAdd(&dw[(size_t)gi * D + t], v);
  }
}

// dn[r][R_i] += dx[r][i]
// The same four columns at a time (D % 4 == 0, 16-byte aligned rows).
__global__ void bwd_scatter_dx4(const float4* __restrict__ dx, int N, int L, int D4, int p,
                                int p_offset, int nR, float4* __restrict__ dn) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)N * nR * D4) return;
  const int t = (int)(i % D4);
  const long long ri = i / D4;
  const int s = (int)(ri % nR);
  const long long r = ri / nR;
  float4* d = dn + (r * L + p_offset + (long long)s * p) * D4 + t;
  const float4 a = dx[i], b = *d;
  *d = make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}
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
// Four consecutive storage-type values as fp32 (16- or 8-byte aligned).
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
// The same with scalar loads (operands whose alignment the caller does not fix).
template <typename S>
__device__ __forceinline__ float4 ld4s(const S* p) {
  return make_float4(to_f(p[0]), to_f(p[1]), to_f(p[2]), to_f(p[3]));
}

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
  // lane l takes columns 4l + 128i (D is a multiple of 64): 16-byte loads
  for (int r = r0 + warp; r < r1; r += (int)(blockDim.x >> 5)) {
    const size_t base = ((size_t)r * L + l) * D;
    const float iv = inv[(size_t)r * L + l];
    float s = 0.f;
#pragma unroll 4
    for (int t = 4 * lane; t < D; t += 128) {
      const float4 w = ld4s(sg + t), g = ld4(dn + base + t), h = ld4(states + base + t);
      s = fmaf(w.x * g.x, h.x, s);
      s = fmaf(w.y * g.y, h.y, s);
      s = fmaf(w.z * g.z, h.z, s);
      s = fmaf(w.w * g.w, h.w, s);
    }
    s = warp_sum(s);
    const float c3 = s * iv * iv * iv / (float)D;
#pragma unroll 4
    for (int t = 4 * lane; t < D; t += 128) {
      const float4 w = ld4s(sg + t), g = ld4(dn + base + t), h = ld4(states + base + t);
      atomicAdd(&acc[t], h.x * iv * g.x);
      atomicAdd(&acc[t + 1], h.y * iv * g.y);
      atomicAdd(&acc[t + 2], h.z * iv * g.z);
      atomicAdd(&acc[t + 3], h.w * iv * g.w);
      float4 dh = make_float4(w.x * g.x * iv - h.x * c3, w.y * g.y * iv - h.y * c3,
                              w.z * g.z * iv - h.z * c3, w.w * g.w * iv - h.w * c3);
      float4* o = reinterpret_cast<float4*>(dstates + base + t);
      if (!first) {
        const float4 prev = *o;
        dh.x += prev.x; dh.y += prev.y; dh.z += prev.z; dh.w += prev.w;
      }
      *o = dh;
    }
  }
  __syncthreads();
  for (int t = threadIdx.x; t < D; t += blockDim.x) atomicAdd(&dsigma[(size_t)l * D + t], acc[t]);
}

// Four consecutive storage-type values kept raw in registers (bf16: two
// registers), converted to fp32 where used.
template <typename S> struct Raw4;
template <> struct Raw4<float> {
  using T = float4;
  static __device__ __forceinline__ T load(const float* p) { return *reinterpret_cast<const float4*>(p); }
  static __device__ __forceinline__ float4 f(const T& v) { return v; }
};
template <> struct Raw4<__nv_bfloat16> {
  using T = uint2;
  static __device__ __forceinline__ T load(const __nv_bfloat16* p) { return *reinterpret_cast<const uint2*>(p); }
  static __device__ __forceinline__ float4 f(const T& u) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
};

// The same with each row held in registers (NV float4 columns a lane, D =
// 128 NV): every load of a row is in flight before its sum, the layer's gains
// sit in shared memory, and each warp sums d sigma over its rows in a shared
// row of its own (plain read-add-write, no atomics), the warps' rows added
// at the end. Dynamic shared memory: (2 + warps) D floats.
template <typename S, int NV>
__global__ void __launch_bounds__(256, 1) bwd_src_norm_wr(const S* __restrict__ states, int N, int L,
                                                          int D, const float* __restrict__ inv,
                                                          const S* __restrict__ sigma,
                                                          const float* __restrict__ dn, int rows,
                                                          bool first, float* __restrict__ dstates,
                                                          float* __restrict__ dsigma) {
  extern __shared__ float sm[];
  const int nw = (int)(blockDim.x >> 5);
  float* sgf = sm;                 // [D] the layer's gains in fp32
  float* wacc = sm + D;            // [warps][D] each warp's d sigma
  const int l = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int t = threadIdx.x; t < D; t += blockDim.x) sgf[t] = to_f(sigma[(size_t)l * D + t]);
  for (int t = threadIdx.x; t < nw * D; t += blockDim.x) wacc[t] = 0.f;
  __syncthreads();
  float* ds = wacc + (size_t)warp * D + 4 * lane;
  const int r0 = blockIdx.x * rows, r1 = min(r0 + rows, N);
  for (int r = r0 + warp; r < r1; r += (int)(blockDim.x >> 5)) {
    const size_t base = ((size_t)r * L + l) * D + 4 * lane;
    const float iv = inv[(size_t)r * L + l];
    float4 g[NV];
    typename Raw4<S>::T hr[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      g[k] = ld4(dn + base + 128 * k);
      hr[k] = Raw4<S>::load(states + base + 128 * k);
    }
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const float4 w = *reinterpret_cast<const float4*>(sgf + 4 * lane + 128 * k);
      const float4 h = Raw4<S>::f(hr[k]);
      s = fmaf(w.x * g[k].x, h.x, s);
      s = fmaf(w.y * g[k].y, h.y, s);
      s = fmaf(w.z * g[k].z, h.z, s);
      s = fmaf(w.w * g[k].w, h.w, s);
    }
    s = warp_sum(s);
    const float c3 = s * iv * iv * iv / (float)D;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const float4 w = *reinterpret_cast<const float4*>(sgf + 4 * lane + 128 * k);
      const float4 h = Raw4<S>::f(hr[k]);
      float4* dsk = reinterpret_cast<float4*>(ds + 128 * k);
      float4 a4 = *dsk;
      a4.x += h.x * iv * g[k].x;
      a4.y += h.y * iv * g[k].y;
      a4.z += h.z * iv * g[k].z;
      a4.w += h.w * iv * g[k].w;
      *dsk = a4;
      float4 dh = make_float4(w.x * g[k].x * iv - h.x * c3, w.y * g[k].y * iv - h.y * c3,
                              w.z * g[k].z * iv - h.z * c3, w.w * g[k].w * iv - h.w * c3);
      float4* o = reinterpret_cast<float4*>(dstates + base + 128 * k);
      if (!first) {
        const float4 prev = *o;
        dh.x += prev.x; dh.y += prev.y; dh.z += prev.z; dh.w += prev.w;
      }
      *o = dh;
    }
  }
  __syncthreads();
  for (int t = threadIdx.x; t < D; t += blockDim.x) {
    float v = 0.f;
    for (int w = 0; w < nw; ++w) v += wacc[(size_t)w * D + t];
    atomicAdd(&dsigma[(size_t)l * D + t], v);
  }
}

// Leading dimension (elements) of a split operand of K columns: 3K, rounded
// up to 8 so that rows start on 16-byte boundaries.
inline long long ld3(long long K) { return (3 * K + 7) / 8 * 8; }

__device__ __forceinline__ void split_hl(float v, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(v);
  lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}

// dst[r][j * C + c], j = 0, 1, 2: the split of src[r][c], left operand
// (right = false: hi, hi, lo) or right operand (right = true: hi, lo, hi).
__global__ void __launch_bounds__(256) split3_rows(const float* __restrict__ src, long long lds,
                                                   int R, int C, __nv_bfloat16* __restrict__ dst,
                                                   long long ldd, bool right) {
  const long long n = (long long)R * C;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / C;
    const int c = (int)(i - r * C);
    __nv_bfloat16 hi, lo;
    split_hl(src[r * lds + c], hi, lo);
    __nv_bfloat16* d = dst + r * ldd + c;
    d[0] = hi;
    d[C] = right ? lo : hi;
    d[2 * C] = right ? hi : lo;
  }
}

// The same four columns at a time: one 16-byte load, three 8-byte stores per
// thread (C, lds and ldd multiples of 4, src 16- and dst 8-byte aligned).
__global__ void __launch_bounds__(256) split3_rows4(const float* __restrict__ src, long long lds,
                                                    int R, int C4, __nv_bfloat16* __restrict__ dst,
                                                    long long ldd, bool right) {
  const long long n = (long long)R * C4;
  const int C = 4 * C4;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / C4;
    const int c = 4 * (int)(i - r * C4);
    const float4 v = *reinterpret_cast<const float4*>(src + r * lds + c);
    __nv_bfloat16 hi[4], lo[4];
    split_hl(v.x, hi[0], lo[0]);
    split_hl(v.y, hi[1], lo[1]);
    split_hl(v.z, hi[2], lo[2]);
    split_hl(v.w, hi[3], lo[3]);
    const uint2 h2 = *reinterpret_cast<const uint2*>(hi), l2 = *reinterpret_cast<const uint2*>(lo);
    uint2* d = reinterpret_cast<uint2*>(dst + r * ldd + c);
    d[0] = h2;
    *reinterpret_cast<uint2*>(dst + r * ldd + C + c) = right ? l2 : h2;
    *reinterpret_cast<uint2*>(dst + r * ldd + 2 * C + c) = right ? h2 : l2;
  }
}
// split3_rows, vectorised where the shapes allow
void launch_split3_rows(const float* src, long long lds, int R, int C, __nv_bfloat16* dst,
                        long long ldd, bool right, cudaStream_t st) {
  if (R <= 0 || C <= 0) return;
  const long long n = (long long)R * C;
  long long b = (n + 255) / 256;
  if (C % 4 == 0 && lds % 4 == 0 && ldd % 4 == 0 && (uintptr_t)src % 16 == 0 && (uintptr_t)dst % 8 == 0) {
    b = (n / 4 + 255) / 256;
    split3_rows4<<<(unsigned)(b < 65536LL * 16 ? b : 65536LL * 16), 256, 0, st>>>(src, lds, R, C / 4, dst,
                                                                             ldd, right);
  } else {
    split3_rows<<<(unsigned)(b < 65536LL * 16 ? b : 65536LL * 16), 256, 0, st>>>(src, lds, R, C, dst, ldd,
                                                                             right);
  }
}

// The same for the transpose: dst[c][j * R + r] from src[r][c] (32 x 32 tiles
// through shared memory, reads and writes coalesced).
// blockIdx.z selects a batch entry (src + z * sbs, dst + z * dbs).
__global__ void __launch_bounds__(256) split3_t(const float* __restrict__ src, long long lds, int R,
                                                int C, __nv_bfloat16* __restrict__ dst,
                                                long long ldd, bool right, long long sbs = 0,
                                                long long dbs = 0) {
  __shared__ float tile[32][33];
  src += blockIdx.z * sbs;
  dst += blockIdx.z * dbs;
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 8 rows of 32
  for (int y = ty; y < 32; y += 8) {
    const int r = r0 + y, c = c0 + tx;
    tile[y][tx] = (r < R && c < C) ? src[(long long)r * lds + c] : 0.f;
  }
  __syncthreads();
  for (int y = ty; y < 32; y += 8) {
    const int c = c0 + y, r = r0 + tx;
    if (c < C && r < R) {
      __nv_bfloat16 hi, lo;
      split_hl(tile[tx][y], hi, lo);
      __nv_bfloat16* d = dst + (long long)c * ldd + r;
      d[0] = hi;
      d[R] = right ? lo : hi;
      d[2 * R] = right ? hi : lo;
    }
  }
}

// split3_t with two source rows per lane (64 x CW tiles: CW source columns,
// read CW * 4 contiguous bytes a row), so each warp writes 128 contiguous
// bytes per destination row (R, ldd and dbs even, dst 4-byte aligned).
template <int CW>
__global__ void __launch_bounds__(256) split3_t2(const float* __restrict__ src, long long lds, int R,
                                                 int C, __nv_bfloat16* __restrict__ dst,
                                                 long long ldd, bool right, long long sbs,
                                                 long long dbs) {
  __shared__ float tile[64][CW + 1];
  src += blockIdx.z * sbs;
  dst += blockIdx.z * dbs;
  const int c0 = blockIdx.x * CW, r0 = blockIdx.y * 64;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int y = ty; y < 64; y += 8)
#pragma unroll
    for (int cx = tx; cx < CW; cx += 32) {
      const int r = r0 + y, c = c0 + cx;
      tile[y][cx] = (r < R && c < C) ? src[(long long)r * lds + c] : 0.f;
    }
  __syncthreads();
  const int r = r0 + 2 * tx;
  for (int y = ty; y < CW; y += 8) {
    const int c = c0 + y;
    if (c < C && r < R) {  // R even: r + 1 < R too
      __nv_bfloat162 hi, lo;
      split_hl(tile[2 * tx][y], hi.x, lo.x);
      split_hl(tile[2 * tx + 1][y], hi.y, lo.y);
      __nv_bfloat162* d = reinterpret_cast<__nv_bfloat162*>(dst + (long long)c * ldd + r);
      d[0] = hi;
      d[R / 2] = right ? lo : hi;
      d[R] = right ? hi : lo;
    }
  }
}
// da_r = dm_r n_r^T for every row r, on the tensor cores: dm_r [k x D] (row j
// of channel j at dm + j * ldj + r * D), n_r [L x D] (at n + r * L * D),
// da_r [k x L] (at da + r * k * L); k <= 16, L <= 32, D % 16 == 0. One warp
// per row: the m16n8k16 fragments are loaded straight from the fp32
// operands (8-byte pairs along D) and split exactly into bf16 hi + lo, the
// product taken as hi.hi + hi.lo + lo.hi with fp32 accumulation (lo.lo is
// below 2^-16 of the product); rows j >= k and columns l >= L are zero.
__device__ __forceinline__ void split_pair(float2 v, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(v.x - hf.x, v.y - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__global__ void __launch_bounds__(256) bwd_da_tc(const float* __restrict__ dm, long long ldj,
                                                 const float* __restrict__ n, int N, int L, int D,
                                                 int k, float* __restrict__ da) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long r = (long long)blockIdx.x * 8 + warp;
  if (r >= N) return;  // warp-uniform
  const int g = lane >> 2, t = lane & 3;
  // A rows g and g + 8 (channels), B columns nt * 8 + g (layers); absent
  // ones read row 0 and are zeroed
  const bool va0 = g < k, va1 = g + 8 < k;
  const float* A0 = dm + (long long)(va0 ? g : 0) * ldj + r * D + 2 * t;
  const float* A1 = dm + (long long)(va1 ? g + 8 : 0) * ldj + r * D + 2 * t;
  const float* Bp[4];
  bool vb[4];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    const int l = nt * 8 + g;
    vb[nt] = l < L;
    Bp[nt] = n + (r * L + (vb[nt] ? l : 0)) * D + 2 * t;
  }
  const float2 z = make_float2(0.f, 0.f);
  float acc[4][4] = {};
#pragma unroll 1
  for (int k0 = 0; k0 < D; k0 += 16) {
    const float2 a00 = va0 ? *reinterpret_cast<const float2*>(A0 + k0) : z;
    const float2 a10 = va1 ? *reinterpret_cast<const float2*>(A1 + k0) : z;
    const float2 a01 = va0 ? *reinterpret_cast<const float2*>(A0 + k0 + 8) : z;
    const float2 a11 = va1 ? *reinterpret_cast<const float2*>(A1 + k0 + 8) : z;
    float2 b0[4], b1[4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      b0[nt] = vb[nt] ? *reinterpret_cast<const float2*>(Bp[nt] + k0) : z;
      b1[nt] = vb[nt] ? *reinterpret_cast<const float2*>(Bp[nt] + k0 + 8) : z;
    }
    uint32_t ah[4], al[4];
    split_pair(a00, ah[0], al[0]);
    split_pair(a10, ah[1], al[1]);
    split_pair(a01, ah[2], al[2]);
    split_pair(a11, ah[3], al[3]);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      uint32_t bh0, bl0, bh1, bl1;
      split_pair(b0[nt], bh0, bl0);
      split_pair(b1[nt], bh1, bl1);
      mma_16816(acc[nt], ah, bh0, bh1);
      mma_16816(acc[nt], ah, bl0, bl1);
      mma_16816(acc[nt], al, bh0, bh1);
    }
  }
  float* out = da + r * k * L;
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = g + 8 * h;
      if (j >= k) continue;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int l = nt * 8 + 2 * t + e;
        if (l < L) out[j * L + l] = acc[nt][2 * h + e];
      }
    }
}

// dn_r = a_r^T dm_r for every row r, on the tensor cores: a_r [k x L] (at
// a + r * k * L), dm_r as in bwd_da_tc, dn_r [L x D] (at dn + r * L * D);
// k <= 16, L <= 32, D % 8 == 0. One warp per row: a_r^T's two 16-row
// fragments are split once; each 8-column step of D loads the four channel
// rows a lane's B fragment needs (8 lanes read 8 consecutive columns of one
// row), splits them and stores both 16-row output tiles with 8-byte stores.
__global__ void __launch_bounds__(256) bwd_dn_tc(const float* __restrict__ a,
                                                 const float* __restrict__ dm, long long ldj, int N,
                                                 int L, int D, int k, float* __restrict__ dn) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long r = (long long)blockIdx.x * 8 + warp;
  if (r >= N) return;  // warp-uniform
  const int g = lane >> 2, t = lane & 3;
  const float* ar = a + r * k * L;
  auto av = [&](int l, int j) { return (l < L && j < k) ? ar[j * L + l] : 0.f; };
  uint32_t ah[2][4], al[2][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const int l0 = mt * 16 + g, l1 = l0 + 8;
    split_pair(make_float2(av(l0, 2 * t), av(l0, 2 * t + 1)), ah[mt][0], al[mt][0]);
    split_pair(make_float2(av(l1, 2 * t), av(l1, 2 * t + 1)), ah[mt][1], al[mt][1]);
    split_pair(make_float2(av(l0, 2 * t + 8), av(l0, 2 * t + 9)), ah[mt][2], al[mt][2]);
    split_pair(make_float2(av(l1, 2 * t + 8), av(l1, 2 * t + 9)), ah[mt][3], al[mt][3]);
  }
  // the B rows (channels) 2t, 2t + 1, 2t + 8, 2t + 9 at column g of each step
  const float* Bj[4];
  bool vj[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int j = 2 * t + (i & 1) + (i >> 1) * 8;
    vj[i] = j < k;
    Bj[i] = dm + (long long)(vj[i] ? j : 0) * ldj + r * D + g;
  }
  float* out = dn + r * L * D + 2 * t;
  const bool w0 = g < L, w1 = g + 8 < L, w2 = g + 16 < L, w3 = g + 24 < L;
#pragma unroll 2
  for (int n0 = 0; n0 < D; n0 += 8) {
    float b[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) b[i] = vj[i] ? Bj[i][n0] : 0.f;
    uint32_t bh0, bl0, bh1, bl1;
    split_pair(make_float2(b[0], b[1]), bh0, bl0);
    split_pair(make_float2(b[2], b[3]), bh1, bl1);
    float c[2][4] = {};
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      mma_16816(c[mt], ah[mt], bh0, bh1);
      mma_16816(c[mt], ah[mt], bl0, bl1);
      mma_16816(c[mt], al[mt], bh0, bh1);
    }
    if (w0) *reinterpret_cast<float2*>(out + (long long)g * D + n0) = make_float2(c[0][0], c[0][1]);
    if (w1) *reinterpret_cast<float2*>(out + (long long)(g + 8) * D + n0) = make_float2(c[0][2], c[0][3]);
    if (w2) *reinterpret_cast<float2*>(out + (long long)(g + 16) * D + n0) = make_float2(c[1][0], c[1][1]);
    if (w3) *reinterpret_cast<float2*>(out + (long long)(g + 24) * D + n0) = make_float2(c[1][2], c[1][3]);
  }
}

// split3_t over a batch of blockIdx.z entries, vectorised where the shapes allow
void launch_split3_t(const float* src, long long lds, int R, int C, __nv_bfloat16* dst, long long ldd,
                     bool right, int batch, long long sbs, long long dbs, cudaStream_t st) {
  if (R <= 0 || C <= 0 || batch <= 0) return;
  if (R % 2 == 0 && ldd % 2 == 0 && dbs % 2 == 0 && (uintptr_t)dst % 4 == 0) {
    constexpr int CW = 128;  // 512 contiguous bytes read a source row (32: 20.3 ms a call, 128: 19.5)
    dim3 g((unsigned)((C + CW - 1) / CW), (unsigned)((R + 63) / 64), (unsigned)batch);
    split3_t2<CW><<<g, 256, 0, st>>>(src, lds, R, C, dst, ldd, right, sbs, dbs);
  } else {
    dim3 g((unsigned)((C + 31) / 32), (unsigned)((R + 31) / 32), (unsigned)batch);
    split3_t<<<g, 256, 0, st>>>(src, lds, R, C, dst, ldd, right, sbs, dbs);
  }
}

__global__ void add_f32(float* __restrict__ dst, const float* __restrict__ src, long long n) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    dst[i] += src[i];
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

// C[M][N] (fp32, ldc) = A B^T on the tensor cores for split operands A [M][3K]
// and B [N][3K] (bf16, leading dimensions lda, ldb). False if the engine
// does not take the shape (the caller then uses the fp32 GEMM).
bool gemm_split_tc(int M, int N, int K, const __nv_bfloat16* A, long long lda,
                   const __nv_bfloat16* B, long long ldb, float* C, long long ldc, uint32_t* flags,
                   cudaStream_t st, int batch = 1, long long abs = 0, long long bbs = 0,
                   long long cbs = 0) {
  GemmDesc g;
  g.M = M;
  g.N = N;
  g.K = 3 * K;
  g.batch = batch;
  g.A = A;
  g.lda = lda;
  g.a_bstride = abs;
  g.B = B;
  g.ldb = ldb;
  g.b_bstride = bbs;
  g.epi.mode = EPI_STORE;
  g.epi.out_f32 = 1;
  g.epi.C = C;
  g.epi.ldc = ldc;
  g.epi.c_bstride = cbs;
  g.epi.flags = flags;
  if (!gemm_tc_supported(g)) return false;
  return launch_gemm_tc(g, st, nullptr) == cudaSuccess;
}

inline unsigned blocks_for(long long n) {
  long long b = (n + 255) / 256;
  return (unsigned)(b > 148 * 32 ? 148 * 32 : (b < 1 ? 1 : b));
}

}  // namespace

// Workspace for N rows: fp32 buffers (see run_pool_backward), 256-byte aligned.
PoolBwdLayout pool_bwd_layout(const wm_config& c, long long N) {
  PoolBwdLayout lay;
  const long long L = c.L, D = c.D, k = c.k, w = (long long)c.Hkv * c.d;
  long long nR = 0;
  for (int l = 0; l < c.L; ++l) nR += (l % c.p) == c.p_offset;
  const long long kL = k * L, nRD = nR * D;
  auto bf = [](long long elems) { return (elems + 1) / 2; };  // bf16 elements in floats
  const long long sz[PoolBwdLayout::NB] = {
      64,             // flag word (256 bytes)
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
      bf(N * ld3(nRD)),    // x split (left operand of a = x W_R^T)
      bf(kL * ld3(nRD)),   // W_R split (right operand)
      bf(nRD * ld3(kL)),   // W_R^T split (right operand of dx = da W_R)
      bf(N * ld3(kL)),     // da split (left operand)
      bf(kL * ld3(N)),     // da^T split (left operand of dW_R = da^T x)
      bf(nRD * ld3(N)),    // x^T split (right operand)
      kL * nRD,            // dW_R of this call (fp32), then added
      bf(k * N * ld3(D)),  // c split, per channel (left operand of kt = c W^T)
      bf(k * w * ld3(D)),  // W split, per channel (right operand)
      bf(k * N * ld3(w)),  // dY split (left operand of dc = dY W)
      bf(k * D * ld3(w)),  // W^T split (right operand)
      bf(k * w * ld3(N)),  // dY^T split (left operand of dW = dY^T c)
      bf(k * D * ld3(N)),  // c^T split (right operand)
      k * w * D,           // dW of this call (fp32), then added
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
        *a_keep = buf(PoolBwdLayout::AK), *tmpw = buf(PoolBwdLayout::TMPW);
  auto bbuf = [&](int b) {
    return reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(q.ws) + lay.off[b]);
  };
  __nv_bfloat16 *sx = bbuf(PoolBwdLayout::SX), *sw = bbuf(PoolBwdLayout::SW),
                *swt = bbuf(PoolBwdLayout::SWT), *sda = bbuf(PoolBwdLayout::SDA),
                *sdat = bbuf(PoolBwdLayout::SDAT), *sxt = bbuf(PoolBwdLayout::SXT);
  uint32_t* flags = reinterpret_cast<uint32_t*>(q.ws);  // FLAGS is the first buffer
  const long long kL = (long long)k * L, nRD = (long long)nR * D;
  __nv_bfloat16 *sc = bbuf(PoolBwdLayout::SC), *swp = bbuf(PoolBwdLayout::SWP),
                *sdy = bbuf(PoolBwdLayout::SDY), *swpt = bbuf(PoolBwdLayout::SWPT),
                *sdyt = bbuf(PoolBwdLayout::SDYT), *sct = bbuf(PoolBwdLayout::SCT);
  float* tmpp = buf(PoolBwdLayout::TMPP);
  const long long kN = (long long)k * N;
  const wm_weights& W = *q.w;
  const long long WRn = (long long)k * L * nR * D, WPn = (long long)k * w * D;
  float* tau32 = gains;  // [2][k][D]
  WM_DISPATCH_S(c.dtype, {
    to_f32<S><<<(unsigned)((2LL * k * D + 255) / 256), 256, 0, st>>>((const S*)W.chan_norm, 2LL * k * D, tau32);
  });
  bool ok = true;
  for (int be = 0; be < 2 && ok; ++be) {
    const char* sig = static_cast<const char*>(W.src_norm) + (size_t)be * L * D * (c.dtype == WM_F32 ? 4 : 2);
// the warp source-norm recompute for NV vectors per lane (used inside the
// storage-type dispatch below, where S is defined)
#define WM_SNF(NV_)                                                                                    \
  bwd_src_norm_fwd_w<S, NV_><<<gw, 256, 0, st>>>((const S*)q.states, NL, L, D, (const S*)sig, c.eps, \
                                                 c.p, c.p_offset, nR, inv, n, x)
    WM_DISPATCH_S(c.dtype, {
      constexpr int VN = 16 / sizeof(S);
      const int nv = (D + 32 * VN - 1) / (32 * VN);
      const long long NL = (long long)N * L;
      const bool vec = D % VN == 0 && ((uintptr_t)q.states % 16 == 0) && ((uintptr_t)sig % 16 == 0) &&
                       D % 4 == 0 && nv <= 8;
      const unsigned gw = (unsigned)((NL + 7) / 8);
      if (vec) {
        switch (nv) {
          case 1: WM_SNF(1); break;
          case 2: WM_SNF(2); break;
          case 3: WM_SNF(3); break;
          case 4: WM_SNF(4); break;
          case 5: WM_SNF(5); break;
          case 6: WM_SNF(6); break;
          case 7: WM_SNF(7); break;
          default: WM_SNF(8); break;
        }
      } else {
        bwd_src_norm_fwd<S><<<(unsigned)NL, 256, 0, st>>>(
            (const S*)q.states, L, D, (const S*)sig, c.eps, c.p, c.p_offset, nR, inv, n, x);
      }

    });
#undef WM_SNF
    // coefficients: the router (x W_R^T) or the constants
    if (W.static_coeff) {
      broadcast_rows<<<(unsigned)(((long long)N * k * L + 255) / 256), 256, 0, st>>>(
          W.static_coeff + (size_t)be * k * L, k * L, N, a_keep);
    } else {
      const char* wrs = static_cast<const char*>(W.Wr) + (size_t)be * WRn * (c.dtype == WM_F32 ? 4 : 2);
      WM_DISPATCH_S(c.dtype, {
        to_f32<S><<<(unsigned)((WRn + 255) / 256), 256, 0, st>>>((const S*)wrs, WRn, wr);
      });
      // a = x W_R^T on the tensor cores (split operands), else in fp32
      launch_split3_rows(x, nRD, N, (int)nRD, sx, ld3(nRD), false, st);
      launch_split3_rows(wr, nRD, (int)kL, (int)nRD, sw, ld3(nRD), true, st);
      if (!gemm_split_tc(N, (int)kL, (int)nRD, sx, ld3(nRD), sw, ld3(nRD), a_keep, kL, flags, st))
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
      // kt = c W_K^T per channel on split operands (rows of all channels at once)
      launch_split3_rows(cc, D, (int)kN, D, sc, ld3(D), false, st);
      launch_split3_rows(wp, D, (int)(k * w), D, swp, ld3(D), true, st);
      if (!gemm_split_tc(N, w, D, sc, ld3(D), swp, ld3(D), kt, w, flags, st, k, N * ld3(D),
                         w * ld3(D), (long long)N * w))
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
    {
      launch_split3_rows(dY, w, (int)kN, w, sdy, ld3(w), false, st);
      launch_split3_t(wp, D, w, D, swpt, ld3(w), true, k, (long long)w * D, D * ld3(w), st);
      launch_split3_t(dY, w, N, w, sdyt, ld3(N), false, k, (long long)N * w, w * ld3(N), st);
      launch_split3_t(cc, D, N, D, sct, ld3(N), true, k, (long long)N * D, D * ld3(N), st);
    }
    if (gemm_split_tc(w, D, N, sdyt, ld3(N), sct, ld3(N), tmpp, D, flags, st, k, w * ld3(N),
                      D * ld3(N), (long long)w * D))
      add_f32<<<blocks_for((long long)k * w * D), 256, 0, st>>>(dW, tmpp, (long long)k * w * D);
    else
      ok = ok && gemm_rm(true, false, w, D, N, dY, w, (long long)N * w, cc, D, (long long)N * D, 1.f,
                         dW, D, (long long)w * D, k, st);
    if (!gemm_split_tc(N, D, w, sdy, ld3(w), swpt, ld3(w), dc, D, flags, st, k, N * ld3(w),
                       D * ld3(w), (long long)N * D))
      ok = ok && gemm_rm(false, false, N, D, w, dY, w, (long long)N * w, wp, D, (long long)w * D, 0.f,
                         dc, D, (long long)N * D, k, st);
    {  // channel norm backward, in place: dc -> dm
      const int rows = 64;
      dim3 grid((N + rows - 1) / rows, k);
      const int nvr = D % 128 == 0 ? D / 128 : 0;
      const float* tau_b = tau32 + (size_t)be * k * D;
      const bool al = (uintptr_t)m % 16 == 0 && (uintptr_t)dc % 16 == 0 && (uintptr_t)tau_b % 16 == 0;
#define WM_RMW(NV_)                                                                            \
  do {                                                                                         \
    const size_t smb = (size_t)D * 4 * (1 + 8);                                                \
    cudaFuncSetAttribute(bwd_rms_wr<NV_>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smb); \
    bwd_rms_wr<NV_><<<grid, 256, smb, st>>>(m, (long long)N * D, D, rj, 1, k, tau_b, D, N, rows, dc, \
                                            q.g.dchan_norm + (size_t)be * k * D);                 \
  } while (0)
      if (al && nvr == 14) WM_RMW(14);
      else if (al && nvr == 8) WM_RMW(8);
      else if (al && nvr == 4) WM_RMW(4);
      else if (al && nvr == 2) WM_RMW(2);
      else if (al && nvr == 1) WM_RMW(1);
      else
        bwd_rms_w<<<grid, 256, (size_t)D * 4, st>>>(m, (long long)N * D, D, rj, 1, k, tau_b, D, N,
                                                    rows, dc, q.g.dchan_norm + (size_t)be * k * D);
#undef WM_RMW
    }
    // mix backward per row r: da_r [k x L] = dm_r [k x D] n_r^T; dn_r [L x D] = a_r^T dm_r
    if (k <= 16 && L <= 32 && D % 16 == 0 && (uintptr_t)dc % 8 == 0 && (uintptr_t)n % 8 == 0)
      bwd_da_tc<<<(unsigned)((N + 7) / 8), 256, 0, st>>>(dc, (long long)N * D, n, N, L, D, k, a);
    else
      ok = ok && gemm_rm(false, true, k, L, D, dc, (long long)N * D, D, n, D, (long long)L * D, 0.f, a,
                         L, (long long)k * L, N, st);
    if (k <= 16 && L <= 32 && D % 8 == 0 && (uintptr_t)dn % 8 == 0)
      bwd_dn_tc<<<(unsigned)((N + 7) / 8), 256, 0, st>>>(a_keep, dc, (long long)N * D, N, L, D, k, dn);
    else
      ok = ok && gemm_rm(true, false, L, D, k, a_keep, L, (long long)k * L, dc, (long long)N * D, D,
                         0.f, dn, D, (long long)L * D, N, st);
    if (!W.static_coeff) {
      // router: dW_R += da^T x ([kL x N] [N x nR D]);  dx = da W_R ([N x kL] [kL x nR D]),
      // on the tensor cores with split operands (transposed where the
      // engine's K-major layout needs it), else in fp32
      launch_split3_rows(a, kL, N, (int)kL, sda, ld3(kL), false, st);
      launch_split3_t(wr, nRD, (int)kL, (int)nRD, swt, ld3(kL), true, 1, 0, 0, st);
      if (!gemm_split_tc(N, (int)nRD, (int)kL, sda, ld3(kL), swt, ld3(kL), dx, nRD, flags, st))
        ok = ok && gemm_rm(false, false, N, nR * D, k * L, a, k * L, 0, wr, nR * D, 0, 0.f, dx,
                           nR * D, 0, 1, st);
      if (q.g.dWr) {
        launch_split3_t(a, kL, N, (int)kL, sdat, ld3(N), false, 1, 0, 0, st);
        launch_split3_t(x, nRD, N, (int)nRD, sxt, ld3(N), true, 1, 0, 0, st);
        float* dwr = q.g.dWr + (size_t)be * WRn;
        if (gemm_split_tc((int)kL, (int)nRD, N, sdat, ld3(N), sxt, ld3(N), tmpw, nRD, flags, st))
          add_f32<<<blocks_for(kL * nRD), 256, 0, st>>>(dwr, tmpw, kL * nRD);
        else
          ok = ok && gemm_rm(true, false, k * L, nR * D, N, a, k * L, 0, x, nR * D, 0, 1.f, dwr,
                             nR * D, 0, 1, st);
      }
      if (D % 4 == 0 && (uintptr_t)dx % 16 == 0 && (uintptr_t)dn % 16 == 0)
        bwd_scatter_dx4<<<(unsigned)(((long long)N * nR * (D / 4) + 255) / 256), 256, 0, st>>>(
            reinterpret_cast<const float4*>(dx), N, L, D / 4, c.p, c.p_offset, nR,
            reinterpret_cast<float4*>(dn));
      else
        bwd_scatter_dx<<<(unsigned)(((long long)N * nR * D + 255) / 256), 256, 0, st>>>(
            dx, N, L, D, c.p, c.p_offset, nR, dn);
    }
    {  // source norm backward into dstates
      const int rows = 64;
      dim3 grid((N + rows - 1) / rows, L);
      const int nvr = D % 128 == 0 ? D / 128 : 0;
      const bool al = (uintptr_t)q.states % 16 == 0 && (uintptr_t)dn % 16 == 0 &&
                      (uintptr_t)q.dstates % 16 == 0;
#define WM_SNW(NV_)                                                                               \
  do {                                                                                            \
    const size_t smb = (size_t)D * 4 * (1 + 8);                                                   \
    cudaFuncSetAttribute(bwd_src_norm_wr<S, NV_>, cudaFuncAttributeMaxDynamicSharedMemorySize,    \
                         (int)smb);                                                               \
    bwd_src_norm_wr<S, NV_><<<grid, 256, smb, st>>>((const S*)q.states, N, L, D, inv,             \
                                                    (const S*)sig, dn, rows, be == 0, q.dstates, \
                                                    q.g.dsrc_norm + (size_t)be * L * D);          \
  } while (0)
      WM_DISPATCH_S(c.dtype, {
        if (al && nvr == 14) WM_SNW(14);
        else if (al && nvr == 8) WM_SNW(8);
        else if (al && nvr == 4) WM_SNW(4);
        else if (al && nvr == 2) WM_SNW(2);
        else if (al && nvr == 1) WM_SNW(1);
        else
          bwd_src_norm_w<S><<<grid, 256, (size_t)D * 4, st>>>((const S*)q.states, N, L, D, inv,
                                                              (const S*)sig, dn, rows, be == 0,
                                                              q.dstates,
                                                              q.g.dsrc_norm + (size_t)be * L * D);
      });
#undef WM_SNW
    }
  }
  if (!ok) return cudaErrorUnknown;
  return cudaGetLastError();
}

}  // namespace wm
