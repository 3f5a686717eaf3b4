// Element-wise and row-wise kernels: RoPE table, row metadata of a group,
// embedding gather, RMSNorm with the pool's per-source emissions.
#include "kernels.h"

namespace wm {

// 16-byte vector load/store of the storage type as floats.
template <typename S> struct VecT { static constexpr int N = 16 / sizeof(S); };

__device__ __forceinline__ void ld_vec(const float* p, float* v) {
  const float4 x = *reinterpret_cast<const float4*>(p);
  v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}
__device__ __forceinline__ void ld_vec(const __nv_bfloat16* p, float* v) {
  const uint4 x = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&x);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x; v[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void st_vec(float* p, const float* v) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void st_vec(__nv_bfloat16* p, const float* v) {
  uint4 x;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&x);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = x;
}

// ---------------------------------------------------------------------------
// RoPE table: tab[pos][t] = (cos, sin)(pos * base^(-2t/d)), angles in fp64.
// ---------------------------------------------------------------------------
__global__ void rope_table_kernel(float2* tab, int p0, int p1, int d, double base) {
  pdl_wait();
  pdl_trigger();
  const int half = d >> 1;
  const long long n = (long long)(p1 - p0) * half;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const int pos = p0 + (int)(idx / half), t = (int)(idx % half);
    const double theta = pow(base, -2.0 * (double)t / (double)d);
    double s, c;
    sincos((double)pos * theta, &s, &c);
    tab[(long long)pos * half + t] = make_float2((float)c, (float)s);
  }
}

void launch_rope_table(float2* tab, int p0, int p1, int d, float base, cudaStream_t st) {
  const long long n = (long long)(p1 - p0) * (d / 2);
  if (n <= 0) return;
  const int blocks = (int)((n + 255) / 256 < 1184 ? (n + 255) / 256 : 1184);
  launch_k(rope_table_kernel, dim3(blocks), dim3(256), 0, st, tab, p0, p1, d, (double)base);
}

// ---------------------------------------------------------------------------
// Rows of cyclic group q: row r = b * nq + u holds position i = q + u * g.
// ---------------------------------------------------------------------------
__global__ void group_rows_kernel(const int32_t* __restrict__ tokens, int B, int T, int g, int q,
                                  int nq, int pos0, int32_t* tok, int32_t* seq, int32_t* pos,
                                  int32_t* rowmap) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= B * nq) return;
  const int b = r / nq, u = r % nq, i = q + u * g;
  tok[r] = tokens[(long long)b * T + i];
  seq[r] = b;
  pos[r] = pos0 + i;
  if (rowmap) rowmap[r] = b * T + i;
}

void launch_group_rows(const int32_t* tokens, int B, int T, int g, int q, int nq, int32_t* tok,
                       int32_t* seq, int32_t* pos, int32_t* rowmap, cudaStream_t st, int pos0) {
  const int n = B * nq;
  launch_k(group_rows_kernel, dim3((n + 255) / 256), dim3(256), 0, st, tokens, B, T, g, q, nq, pos0, tok, seq, pos,
                                                     rowmap);
}

__global__ void decode_rows_kernel(const int32_t* __restrict__ tokens, int B, int t, int32_t* tok,
                                   int32_t* seq, int32_t* pos) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= B) return;
  tok[r] = tokens[r];
  seq[r] = r;
  pos[r] = t;
}

void launch_decode_rows(const int32_t* tokens, int B, int t, int32_t* tok, int32_t* seq,
                        int32_t* pos, cudaStream_t st) {
  launch_k(decode_rows_kernel, dim3((B + 255) / 256), dim3(256), 0, st, tokens, B, t, tok, seq, pos);
}

// Decode rows from device arrays: row b is sequence b at pos[b]; its RoPE
// table row is written here too (rows of equal positions get equal values).
__global__ void decode_rows_dev_kernel(const int32_t* __restrict__ tokens,
                                       const int32_t* __restrict__ pos_in, int B, int d,
                                       double base, int32_t* tok, int32_t* seq, int32_t* pos,
                                       float2* tab, int Tmax) {
  pdl_wait();
  pdl_trigger();
  const int half = d >> 1;
  const long long n = (long long)B * half;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(idx / half), t = (int)(idx % half);
    const int ps = pos_in[r];
    if (t == 0) {
      tok[r] = tokens[r];
      seq[r] = r;
      pos[r] = ps;
    }
    if (ps < 0 || ps >= Tmax) continue;  // the consumers flag the position
    const double theta = pow(base, -2.0 * (double)t / (double)d);
    double sn, cs;
    sincos((double)ps * theta, &sn, &cs);
    tab[(long long)ps * half + t] = make_float2((float)cs, (float)sn);
  }
}

void launch_decode_rows_dev(const int32_t* tokens, const int32_t* pos_in, int B, int d, float base,
                            int32_t* tok, int32_t* seq, int32_t* pos, float2* tab, int Tmax,
                            cudaStream_t st) {
  const long long n = (long long)B * (d / 2);
  const int blocks = (int)((n + 255) / 256 < 1184 ? (n + 255) / 256 : 1184);
  launch_k(decode_rows_dev_kernel, dim3(blocks), dim3(256), 0, st, tokens, pos_in, B, d,
           (double)base, tok, seq, pos, tab, Tmax);
}

// ---------------------------------------------------------------------------
// h^0 = embed[token]; an out-of-range id writes zeros and sets a flag.
// ---------------------------------------------------------------------------
template <typename S>
__global__ void embed_kernel(const int32_t* __restrict__ tok, const S* __restrict__ embed, int V,
                             int D, S* __restrict__ out, long long ld_out, uint32_t* flags) {
  pdl_wait();
  pdl_trigger();
  constexpr int VN = VecT<S>::N;
  const int r = blockIdx.x;
  const int id = tok[r];
  const bool ok = id >= 0 && id < V;
  if (!ok && threadIdx.x == 0) atomicOr(flags, FLAG_BAD_TOKEN);
  S* o = out + (long long)r * ld_out;
  const S* e = embed + (long long)(ok ? id : 0) * D;
  for (int c = threadIdx.x * VN; c < D; c += blockDim.x * VN) {
    if (ok) {
      *reinterpret_cast<uint4*>(o + c) = *reinterpret_cast<const uint4*>(e + c);
    } else {
      *reinterpret_cast<uint4*>(o + c) = make_uint4(0, 0, 0, 0);
    }
  }
}

void launch_embed(int dtype, const int32_t* tok, int N, const void* embed, int V, int D, void* out,
                  long long ld_out, uint32_t* flags, cudaStream_t st) {
  if (N <= 0) return;
  WM_DISPATCH_S(dtype, launch_k(embed_kernel<S>, dim3(N), dim3(128), 0, st, tok, (const S*)embed, V, D, (S*)out,
                                                         ld_out, flags));
}

// ---------------------------------------------------------------------------
// Layer-input RMSNorm with the pool's emissions: one warp per (row, layer),
// eight rows per block. The row is read twice (the second time from L1).
// ---------------------------------------------------------------------------
constexpr int NORM_ROWS = 8;             // rows per 256-thread block
constexpr int NORM_WARP_MIN_ROWS = 1024;  // fewer rows: a block per row

template <typename S>
__global__ void __launch_bounds__(32 * NORM_ROWS) norm_emit_kernel(
    const S* __restrict__ X, long long ldx_row, long long ldx_l, int l0, int D, int L,
    const S* __restrict__ gain_in, S* __restrict__ xn, float* __restrict__ inv_out,
    const S* __restrict__ src_norm, S* __restrict__ rin, int N, int nR, int p, int p_off,
    float eps) {
  pdl_wait();
  pdl_trigger();
  constexpr int VN = VecT<S>::N;
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * NORM_ROWS + (threadIdx.x >> 5), l = l0 + blockIdx.y;
  if (r >= N) return;  // warp-uniform
  const S* x = X + (long long)r * ldx_row + (long long)l * ldx_l;
  float ss = 0.f;
#pragma unroll 4
  for (int c = lane * VN; c < D; c += 32 * VN) {
    float v[VN];
    ld_vec(x + c, v);
#pragma unroll
    for (int i = 0; i < VN; ++i) ss += v[i] * v[i];
  }
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / (float)D + eps);
  if (lane == 0) inv_out[(long long)r * L + l] = inv;
  const bool in_R = rin != nullptr && (l % p) == p_off;
  const int ridx = (l - p_off) / p;
  if (xn == nullptr && !in_R) return;
  const long long rin_b = (long long)N * nR * D;
  for (int c = lane * VN; c < D; c += 32 * VN) {
    float v[VN], o[VN], gv[VN];
    ld_vec(x + c, v);
    if (xn) {
      ld_vec(gain_in + (long long)l * D + c, gv);
#pragma unroll
      for (int i = 0; i < VN; ++i) o[i] = v[i] * inv * gv[i];
      st_vec(xn + (long long)r * D + c, o);
    }
    if (in_R) {
#pragma unroll
      for (int beta = 0; beta < 2; ++beta) {
        ld_vec(src_norm + ((long long)beta * L + l) * D + c, gv);
#pragma unroll
        for (int i = 0; i < VN; ++i) o[i] = v[i] * inv * gv[i];
        st_vec(rin + beta * rin_b + (long long)r * nR * D + (long long)ridx * D + c, o);
      }
    }
  }
}

// The same with the row held in registers: lane t loads vectors t, t + 32, ...
// (NV of them, all issued before the first is used) and writes the outputs
// from them, so the row is read once with every load in flight. The sums run
// in the same order as the loop above (bit-identical results).
template <typename S, int NV>
__global__ void __launch_bounds__(32 * NORM_ROWS) norm_emit_regs_kernel(
    const S* __restrict__ X, long long ldx_row, long long ldx_l, int l0, int D, int L,
    const S* __restrict__ gain_in, S* __restrict__ xn, float* __restrict__ inv_out,
    const S* __restrict__ src_norm, S* __restrict__ rin, int N, int nR, int p, int p_off,
    float eps) {
  pdl_wait();
  pdl_trigger();
  constexpr int VN = VecT<S>::N;
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * NORM_ROWS + (threadIdx.x >> 5), l = l0 + blockIdx.y;
  if (r >= N) return;  // warp-uniform
  const S* x = X + (long long)r * ldx_row + (long long)l * ldx_l;
  float v[NV][VN];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int c = (lane + 32 * k) * VN;
    if (c < D) ld_vec(x + c, v[k]);
  }
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k)
    if ((lane + 32 * k) * VN < D) {
#pragma unroll
      for (int i = 0; i < VN; ++i) ss += v[k][i] * v[k][i];
    }
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / (float)D + eps);
  if (lane == 0) inv_out[(long long)r * L + l] = inv;
  const bool in_R = rin != nullptr && (l % p) == p_off;
  const int ridx = (l - p_off) / p;
  const long long rin_b = (long long)N * nR * D;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int c = (lane + 32 * k) * VN;
    if (c >= D) continue;
    float o[VN], gv[VN];
    if (xn) {
      ld_vec(gain_in + (long long)l * D + c, gv);
#pragma unroll
      for (int i = 0; i < VN; ++i) o[i] = v[k][i] * inv * gv[i];
      st_vec(xn + (long long)r * D + c, o);
    }
    if (in_R) {
#pragma unroll
      for (int beta = 0; beta < 2; ++beta) {
        ld_vec(src_norm + ((long long)beta * L + l) * D + c, gv);
#pragma unroll
        for (int i = 0; i < VN; ++i) o[i] = v[k][i] * inv * gv[i];
        st_vec(rin + beta * rin_b + (long long)r * nR * D + (long long)ridx * D + c, o);
      }
    }
  }
}

// Few rows (a decode step): one 256-thread block per (row, layer), more loads
// in flight per row than a warp has.
template <typename S>
__global__ void norm_emit_block_kernel(const S* __restrict__ X, long long ldx_row, long long ldx_l,
                                 int l0, int D, int L, const S* __restrict__ gain_in,
                                 S* __restrict__ xn, float* __restrict__ inv_out,
                                 const S* __restrict__ src_norm, S* __restrict__ rin, int N,
                                 int nR, int p, int p_off, float eps) {
  pdl_wait();
  pdl_trigger();
  constexpr int VN = VecT<S>::N;
  __shared__ float red[32];
  const int r = blockIdx.x, l = l0 + blockIdx.y;
  const S* x = X + (long long)r * ldx_row + (long long)l * ldx_l;
  float ss = 0.f;
  for (int c = threadIdx.x * VN; c < D; c += blockDim.x * VN) {
    float v[VN];
    ld_vec(x + c, v);
#pragma unroll
    for (int i = 0; i < VN; ++i) ss += v[i] * v[i];
  }
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / (float)D + eps);
  if (threadIdx.x == 0) inv_out[(long long)r * L + l] = inv;
  const bool in_R = rin != nullptr && (l % p) == p_off;
  const int ridx = (l - p_off) / p;
  if (xn == nullptr && !in_R) return;
  const long long rin_b = (long long)N * nR * D;
  for (int c = threadIdx.x * VN; c < D; c += blockDim.x * VN) {
    float v[VN], o[VN], gv[VN];
    ld_vec(x + c, v);
    if (xn) {
      ld_vec(gain_in + (long long)l * D + c, gv);
#pragma unroll
      for (int i = 0; i < VN; ++i) o[i] = v[i] * inv * gv[i];
      st_vec(xn + (long long)r * D + c, o);
    }
    if (in_R) {
#pragma unroll
      for (int beta = 0; beta < 2; ++beta) {
        ld_vec(src_norm + ((long long)beta * L + l) * D + c, gv);
#pragma unroll
        for (int i = 0; i < VN; ++i) o[i] = v[i] * inv * gv[i];
        st_vec(rin + beta * rin_b + (long long)r * nR * D + (long long)ridx * D + c, o);
      }
    }
  }
}

void launch_norm_emit(int dtype, const void* X, long long ldx_row, long long ldx_l, int N, int l0,
                      int nl, int D, int L, const void* gain_in, void* xn, float* inv,
                      const void* src_norm, void* rin, int nR, int p, int p_off, float eps,
                      cudaStream_t st) {
  if (N <= 0 || nl <= 0) return;
  if (N < NORM_WARP_MIN_ROWS) {
    WM_DISPATCH_S(dtype, launch_k(norm_emit_block_kernel<S>, dim3(N, nl), dim3(256), 0, st,
                                  (const S*)X, ldx_row, ldx_l, l0, D, L, (const S*)gain_in,
                                  (S*)xn, inv, (const S*)src_norm, (S*)rin, N, nR, p, p_off, eps));
    return;
  }
  dim3 grid((N + NORM_ROWS - 1) / NORM_ROWS, nl);
  // rows of up to 8 vectors per lane stay in registers
  const int nv = (D + 32 * (dtype == WM_BF16 ? 8 : 4) - 1) / (32 * (dtype == WM_BF16 ? 8 : 4));
#define WM_EMIT_REGS(NV_)                                                                           \
  WM_DISPATCH_S(dtype, launch_k(norm_emit_regs_kernel<S, NV_>, dim3(grid), dim3(32 * NORM_ROWS), 0, \
                                st, (const S*)X, ldx_row, ldx_l, l0, D, L, (const S*)gain_in,      \
                                (S*)xn, inv, (const S*)src_norm, (S*)rin, N, nR, p, p_off, eps))
  switch (nv) {
    case 1: WM_EMIT_REGS(1); return;
    case 2: WM_EMIT_REGS(2); return;
    case 3: WM_EMIT_REGS(3); return;
    case 4: WM_EMIT_REGS(4); return;
    case 5: WM_EMIT_REGS(5); return;
    case 6: WM_EMIT_REGS(6); return;
    case 7: WM_EMIT_REGS(7); return;
    case 8: WM_EMIT_REGS(8); return;
    default: break;
  }
#undef WM_EMIT_REGS
  WM_DISPATCH_S(dtype, launch_k(norm_emit_kernel<S>, dim3(grid), dim3(32 * NORM_ROWS), 0, st,
                                (const S*)X, ldx_row, ldx_l, l0, D, L, (const S*)gain_in, (S*)xn,
                                inv, (const S*)src_norm, (S*)rin, N, nR, p, p_off, eps));
}

// y = RMSNorm(x; gain): one warp per row, eight rows per block.
template <typename S>
__global__ void __launch_bounds__(32 * NORM_ROWS) rmsnorm_kernel(
    const S* __restrict__ X, long long ldx, int row0, int rstride, int D,
    const S* __restrict__ gain, S* __restrict__ y, float eps, int N) {
  pdl_wait();
  pdl_trigger();
  constexpr int VN = VecT<S>::N;
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * NORM_ROWS + (threadIdx.x >> 5);
  if (r >= N) return;  // warp-uniform
  const S* x = X + (long long)(row0 + (long long)r * rstride) * ldx;
  float ss = 0.f;
#pragma unroll 4
  for (int c = lane * VN; c < D; c += 32 * VN) {
    float v[VN];
    ld_vec(x + c, v);
#pragma unroll
    for (int i = 0; i < VN; ++i) ss += v[i] * v[i];
  }
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / (float)D + eps);
  for (int c = lane * VN; c < D; c += 32 * VN) {
    float v[VN], gv[VN];
    ld_vec(x + c, v);
    ld_vec(gain + c, gv);
#pragma unroll
    for (int i = 0; i < VN; ++i) v[i] = v[i] * inv * gv[i];
    st_vec(y + (long long)r * D + c, v);
  }
}

// The same with the row held in registers (as norm_emit_regs_kernel).
template <typename S, int NV>
__global__ void __launch_bounds__(32 * NORM_ROWS) rmsnorm_regs_kernel(
    const S* __restrict__ X, long long ldx, int row0, int rstride, int D,
    const S* __restrict__ gain, S* __restrict__ y, float eps, int N) {
  pdl_wait();
  pdl_trigger();
  constexpr int VN = VecT<S>::N;
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * NORM_ROWS + (threadIdx.x >> 5);
  if (r >= N) return;  // warp-uniform
  const S* x = X + (long long)(row0 + (long long)r * rstride) * ldx;
  float v[NV][VN];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int c = (lane + 32 * k) * VN;
    if (c < D) ld_vec(x + c, v[k]);
  }
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k)
    if ((lane + 32 * k) * VN < D) {
#pragma unroll
      for (int i = 0; i < VN; ++i) ss += v[k][i] * v[k][i];
    }
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / (float)D + eps);
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int c = (lane + 32 * k) * VN;
    if (c >= D) continue;
    float gv[VN], o[VN];
    ld_vec(gain + c, gv);
#pragma unroll
    for (int i = 0; i < VN; ++i) o[i] = v[k][i] * inv * gv[i];
    st_vec(y + (long long)r * D + c, o);
  }
}

template <typename S>
__global__ void rmsnorm_block_kernel(const S* __restrict__ X, long long ldx, int row0, int rstride,
                               int D, const S* __restrict__ gain, S* __restrict__ y, float eps) {
  pdl_wait();
  pdl_trigger();
  constexpr int VN = VecT<S>::N;
  __shared__ float red[32];
  const int r = blockIdx.x;
  const S* x = X + (long long)(row0 + (long long)r * rstride) * ldx;
  float ss = 0.f;
  for (int c = threadIdx.x * VN; c < D; c += blockDim.x * VN) {
    float v[VN];
    ld_vec(x + c, v);
#pragma unroll
    for (int i = 0; i < VN; ++i) ss += v[i] * v[i];
  }
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / (float)D + eps);
  for (int c = threadIdx.x * VN; c < D; c += blockDim.x * VN) {
    float v[VN], gv[VN];
    ld_vec(x + c, v);
    ld_vec(gain + c, gv);
#pragma unroll
    for (int i = 0; i < VN; ++i) v[i] = v[i] * inv * gv[i];
    st_vec(y + (long long)r * D + c, v);
  }
}

void launch_rmsnorm(int dtype, const void* X, long long ldx, int row0, int rstride, int N, int D,
                    const void* gain, void* y, float eps, cudaStream_t st) {
  if (N <= 0) return;
  if (N < NORM_WARP_MIN_ROWS) {
    WM_DISPATCH_S(dtype, launch_k(rmsnorm_block_kernel<S>, dim3(N), dim3(256), 0, st,
                                  (const S*)X, ldx, row0, rstride, D, (const S*)gain, (S*)y, eps));
    return;
  }
  const dim3 grid((N + NORM_ROWS - 1) / NORM_ROWS);
  const int nv = (D + 32 * (dtype == WM_BF16 ? 8 : 4) - 1) / (32 * (dtype == WM_BF16 ? 8 : 4));
#define WM_RMS_REGS(NV_)                                                                         \
  WM_DISPATCH_S(dtype, launch_k(rmsnorm_regs_kernel<S, NV_>, grid, dim3(32 * NORM_ROWS), 0, st, \
                                (const S*)X, ldx, row0, rstride, D, (const S*)gain, (S*)y, eps, N))
  switch (nv) {
    case 1: WM_RMS_REGS(1); return;
    case 2: WM_RMS_REGS(2); return;
    case 3: WM_RMS_REGS(3); return;
    case 4: WM_RMS_REGS(4); return;
    case 5: WM_RMS_REGS(5); return;
    case 6: WM_RMS_REGS(6); return;
    case 7: WM_RMS_REGS(7); return;
    case 8: WM_RMS_REGS(8); return;
    default: break;
  }
#undef WM_RMS_REGS
  WM_DISPATCH_S(dtype, launch_k(rmsnorm_kernel<S>, grid, dim3(32 * NORM_ROWS), 0, st, (const S*)X, ldx,
                                row0, rstride, D, (const S*)gain, (S*)y, eps, N));
}

__global__ void broadcast_coeff_kernel(const float* __restrict__ stat, long long total, int n_per_row,
                                       float* __restrict__ coeff) {
  pdl_wait();
  pdl_trigger();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x)
    coeff[i] = stat[i % n_per_row];
}

void launch_broadcast_coeff(const float* stat, int N, int n_per_row, float* coeff, cudaStream_t st) {
  const long long total = (long long)N * n_per_row;
  if (total <= 0) return;
  const long long b = (total + 255) / 256;
  launch_k(broadcast_coeff_kernel, dim3((int)(b < 4096 ? b : 4096)), dim3(256), 0, st, stat, total, n_per_row, coeff);
}

}  // namespace wm
