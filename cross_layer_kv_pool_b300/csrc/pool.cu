// The pool's mix and channel norm for N token rows:
//   m^b_j = sum_l a^b_{j,l} * inv_l * src_norm[b][l] (.) h_l,
//   c^b_j = RMSNorm(m^b_j; chan_norm[b][j]),
// written channel-major: mixed[b][j][row][:], the operand layout of the
// per-channel projections.
#include "kernels.h"

namespace wm {

// CUDA-core engine, one block per row.
template <typename S>
__global__ void __launch_bounds__(256) mix_simt_kernel(const MixArgs a) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float mbuf[];  // [D]
  __shared__ float red[32];
  const int r = blockIdx.x;
  const S* hs = (const S*)a.stash + (long long)r * a.ld_row;
  const float* inv = a.inv + (long long)r * a.inv_ld;
  const S* sn = (const S*)a.src_norm;
  const S* cn = (const S*)a.chan_norm;
  S* out = (S*)a.mixed;
  for (int beta = 0; beta < 2; ++beta) {
    for (int j = 0; j < a.k; ++j) {
      const float* cf = a.coeff + (((long long)r * 2 + beta) * a.k + j) * a.L;
      float ss = 0.f;
      for (int t = threadIdx.x; t < a.D; t += blockDim.x) {
        float acc = 0.f;
        for (int l = 0; l < a.L; ++l)
          acc += cf[l] * (inv[l] * to_f(sn[((long long)beta * a.sn_layers + l) * a.D + t]) *
                          to_f(hs[(long long)l * a.D + t]));
        mbuf[t] = acc;
        ss += acc * acc;
      }
      ss = block_sum(ss, red);
      const float im = rsqrtf(ss / (float)a.D + a.eps);
      for (int t = threadIdx.x; t < a.D; t += blockDim.x)
        out[(((long long)beta * a.k + j) * a.N + r) * a.D + t] =
            from_f<S>(mbuf[t] * im * to_f(cn[((long long)beta * a.cn_channels + j) * a.D + t]));
    }
  }
}

// ---------------------------------------------------------------------------
// Streaming engine (bf16 storage): one persistent CTA per SM walks token rows.
// Each row's contiguous L x D stack streams through shared memory in chunks of
// MIX_LC layers, each chunk together with both branches' source-norm gains of
// those layers, by bulk TMA copies into a ring of MIX_STAGES stages (so the
// next chunks, also of the next row, load while this one is mixed). inv_rms
// folds into the coefficients. The block's two halves take one branch each;
// every thread owns 4 adjacent columns and all k channel accumulators of its
// branch (packed f32x2 FMAs), so each staged element is read once per branch
// for all k outputs. The channel RMSNorm is a block reduction; the output is
// written channel-major with 8-byte stores.
// ---------------------------------------------------------------------------
namespace {
constexpr int MIX_C = 4;  // columns per thread

__device__ __forceinline__ uint32_t sa32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ bool mix_mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t addr = sa32(bar);
  unsigned long long t0 = 0;
  for (uint32_t it = 0;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    if (ok) return true;
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (it == 0) t0 = t;
    else if (t - t0 > 4000000000ull) return false;
  }
}
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %2};\n\tmov.b64 rb, {%3, %4};\n\tmov.b64 rd, {%0, %1};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rd;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void ld4_bf16(const __nv_bfloat16* p, float* v) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}
}  // namespace

constexpr int MIX_LC = 4;      // source layers per staged chunk
constexpr int MIX_STAGES = 4;  // chunks in flight

template <int K, int NT>
__global__ void __launch_bounds__(NT, 1) mix_stream_kernel(const MixArgs a, uint32_t* flags) {
  extern __shared__ __align__(128) uint8_t msm[];
  constexpr int HALF = NT / 2;  // threads per branch
  const int L = a.L, D = a.D;
  const int nc = (L + MIX_LC - 1) / MIX_LC;
  // stage s: [MIX_LC][D] states, then [2][MIX_LC][D] source-norm gains
  const size_t stage_elems = (size_t)3 * MIX_LC * D;
  __nv_bfloat16* stages = reinterpret_cast<__nv_bfloat16*>(msm);
  float* coef = reinterpret_cast<float*>(msm + MIX_STAGES * stage_elems * 2);  // [2][L][K]
  float* red = coef + (size_t)2 * L * K;                                        // [2K][32]
  float* scale = red + 2 * K * 32;                                              // [2K]
  uint64_t* bar = reinterpret_cast<uint64_t*>(scale + 2 * K + (2 * K & 1));     // [MIX_STAGES]
  const int tid = threadIdx.x, lane = tid & 31;
  const int beta = tid / HALF, bt = tid % HALF, wb = bt >> 5;  // branch, thread and warp in branch
  const int t0 = bt * MIX_C;
  const __nv_bfloat16* src = (const __nv_bfloat16*)a.stash;
  const __nv_bfloat16* sn = (const __nv_bfloat16*)a.src_norm;
  const __nv_bfloat16* cn = (const __nv_bfloat16*)a.chan_norm + (size_t)beta * a.cn_channels * D;
  __nv_bfloat16* out = (__nv_bfloat16*)a.mixed + (size_t)beta * K * a.N * D;

  if (tid == 0) {
    for (int i = 0; i < MIX_STAGES; ++i)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sa32(&bar[i])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  {  // an earlier kernel of this call timed out: leave before issuing anything
    __shared__ int stop;
    if (tid == 0) stop = (*(volatile const uint32_t*)flags & FLAG_TIMEOUT) != 0;
    __syncthreads();
    if (stop) return;
  }
  // Chunk q of this block: row blockIdx.x + (q / nc) * gridDim.x, layers of chunk q % nc.
  auto issue = [&](int q) {
    const long long r = blockIdx.x + (long long)(q / nc) * gridDim.x;
    if (r >= a.N) return;
    const int c = (int)(q % nc), l0 = c * MIX_LC, lc = min(MIX_LC, L - l0);
    const int st = (int)(q % MIX_STAGES);
    const uint32_t bytes = (uint32_t)lc * D * 2;
    __nv_bfloat16* dst = stages + st * stage_elems;
    const uint32_t b = sa32(&bar[st]);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(3 * bytes)
                 : "memory");
    const __nv_bfloat16* srcs[3] = {src + r * a.ld_row + (long long)l0 * D,
                                    sn + (long long)l0 * D, sn + ((long long)a.sn_layers + l0) * D};
    for (int i = 0; i < 3; ++i)
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
              sa32(dst + (size_t)i * MIX_LC * D)),
          "l"(srcs[i]), "r"(bytes), "r"(b)
          : "memory");
  };
  if (tid == 0)
    for (int q = 0; q < MIX_STAGES; ++q) issue(q);
  bool ok = true;
  float acc[K][MIX_C];
  int q = 0;
  for (int r = blockIdx.x; r < a.N; r += gridDim.x) {
    // coefficients of this row, scaled by the inverse RMS of each source
    for (int i = tid; i < 2 * L * K; i += NT) {
      const int be = i / (L * K), l = (i / K) % L, j = i % K;
      coef[i] = a.coeff[(((long long)r * 2 + be) * K + j) * L + l] * a.inv[(long long)r * a.inv_ld + l];
    }
#pragma unroll
    for (int j = 0; j < K; ++j)
#pragma unroll
      for (int c = 0; c < MIX_C; ++c) acc[j][c] = 0.f;
    for (int c = 0; c < nc; ++c, ++q) {
      const int st = q % MIX_STAGES;
      if (!mix_mbar_wait(&bar[st], (uint32_t)((q / MIX_STAGES) & 1))) ok = false;
      __syncthreads();
      if (t0 < D) {
        const int l0 = c * MIX_LC, lc = min(MIX_LC, L - l0);
        const __nv_bfloat16* hs = stages + st * stage_elems + t0;
        const __nv_bfloat16* gs = hs + (size_t)(1 + beta) * MIX_LC * D;
        const float* cf = coef + ((size_t)beta * L + l0) * K;
#pragma unroll 1
        for (int ll = 0; ll < lc; ++ll, hs += D, gs += D, cf += K) {
          float h[MIX_C], sg[MIX_C];
          ld4_bf16(hs, h);
          ld4_bf16(gs, sg);
#pragma unroll
          for (int e = 0; e < MIX_C; ++e) h[e] *= sg[e];
#pragma unroll
          for (int j = 0; j < K; ++j) {
            const float cj = cf[j];
            ffma2(acc[j][0], acc[j][1], cj, h[0], h[1]);
            ffma2(acc[j][2], acc[j][3], cj, h[2], h[3]);
          }
        }
      }
      __syncthreads();  // stage st is free: refill it
      if (tid == 0) issue(q + MIX_STAGES);
    }
    // channel norms: sum of squares over D for each (beta, j)
#pragma unroll
    for (int j = 0; j < K; ++j) {
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < MIX_C; ++e) ss += acc[j][e] * acc[j][e];
      ss = warp_sum(ss);
      if (lane == 0) red[(beta * K + j) * 32 + wb] = ss;
    }
    __syncthreads();
    if (tid < 2 * K) {
      float ss = 0.f;
      for (int w = 0; w < HALF / 32; ++w) ss += red[tid * 32 + w];
      scale[tid] = rsqrtf(ss / (float)D + a.eps);
    }
    __syncthreads();
    if (t0 < D) {
#pragma unroll
      for (int j = 0; j < K; ++j) {
        float g[MIX_C];
        ld4_bf16(cn + (size_t)j * D + t0, g);
        const float sc = scale[beta * K + j];
        __nv_bfloat162 o0 = __floats2bfloat162_rn(acc[j][0] * sc * g[0], acc[j][1] * sc * g[1]);
        __nv_bfloat162 o1 = __floats2bfloat162_rn(acc[j][2] * sc * g[2], acc[j][3] * sc * g[3]);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&o0);
        u.y = *reinterpret_cast<uint32_t*>(&o1);
        *reinterpret_cast<uint2*>(out + ((size_t)j * a.N + r) * D + t0) = u;
      }
    }
    __syncthreads();  // coef, red and scale are free for the next row
  }
  if (!ok && tid == 0) atomicOr(flags, FLAG_TIMEOUT);
}

template <int K, int NT>
bool launch_mix_stream_nt(const MixArgs& a, uint32_t* flags, cudaStream_t st) {
  const size_t smem = (size_t)MIX_STAGES * 3 * MIX_LC * a.D * 2 + (size_t)2 * a.L * K * 4 +
                      2 * K * 32 * 4 + (2 * K + 2) * 4 + 8 * MIX_STAGES + 128;
  if (smem > 227 * 1024) return false;
  if (cudaFuncSetAttribute(mix_stream_kernel<K, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return false;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = a.N < sms ? a.N : sms;
  launch_k(mix_stream_kernel<K, NT>, dim3(grid), dim3(NT), smem, st, a, flags);
  return true;
}

// Smallest block whose halves (one per branch) cover D/4 columns each and
// still leave registers for 4k accumulators per thread (one block per SM).
template <int K>
bool launch_mix_stream(const MixArgs& a, uint32_t* flags, cudaStream_t st) {
  const int need = 2 * (a.D / MIX_C);
  if (need <= 256) return launch_mix_stream_nt<K, 256>(a, flags, st);
  if (need <= 512) return launch_mix_stream_nt<K, 512>(a, flags, st);
  if (need <= 896 && K <= 14) return launch_mix_stream_nt<K, 896>(a, flags, st);
  if (need <= 1024 && K <= 8) return launch_mix_stream_nt<K, 1024>(a, flags, st);
  return false;
}

// ---------------------------------------------------------------------------
// One channel (k = 1, the feedback-free variant's per-layer pool): a weighted
// sum of the row's L states, about 1 FMA per byte, so CUDA cores keep pace
// with HBM. One block per row, 8 columns per thread (16-byte loads of the
// state and both gains), fp32 sums of the exact state x gain products. Like
// the tensor-core mixer it writes u = tau (.) m and the row's sum of squares
// (one part) for the projection epilogue.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void unpack8(const uint4& u, float* v) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

__global__ void __launch_bounds__(1024) mix1_kernel(const MixArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ float coef[2][64];
  __shared__ float red[2][32];
  const long long r = blockIdx.x;
  const int L = a.L, D = a.D;
  const int t0 = threadIdx.x * 8;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  for (int i = threadIdx.x; i < 2 * L; i += blockDim.x) {
    const int be = i / L, l = i % L;
    coef[be][l] = a.coeff[(r * 2 + be) * L + l] * a.inv[r * a.inv_ld + l];
  }
  __syncthreads();
  const __nv_bfloat16* hs = (const __nv_bfloat16*)a.stash + r * a.ld_row + t0;
  const __nv_bfloat16* gk = (const __nv_bfloat16*)a.src_norm + t0;
  const __nv_bfloat16* gv = gk + (size_t)a.sn_layers * D;
  float mk[8], mv[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) mk[e] = mv[e] = 0.f;
  if (t0 < D) {
#pragma unroll 4
    for (int l = 0; l < L; ++l) {
      float h[8], sk[8], sv[8];
      unpack8(*reinterpret_cast<const uint4*>(hs + (size_t)l * D), h);
      unpack8(*reinterpret_cast<const uint4*>(gk + (size_t)l * D), sk);
      unpack8(*reinterpret_cast<const uint4*>(gv + (size_t)l * D), sv);
      const float ck = coef[0][l], cv = coef[1][l];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        mk[e] = fmaf(ck, sk[e] * h[e], mk[e]);
        mv[e] = fmaf(cv, sv[e] * h[e], mv[e]);
      }
    }
  }
  float ssk = 0.f, ssv = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    ssk += mk[e] * mk[e];
    ssv += mv[e] * mv[e];
  }
  ssk = warp_sum(ssk);
  ssv = warp_sum(ssv);
  if (lane == 0) {
    red[0][warp] = ssk;
    red[1][warp] = ssv;
  }
  __syncthreads();
  if (threadIdx.x < 2) {
    float s2 = 0.f;
    for (int w = 0; w < nw; ++w) s2 += red[threadIdx.x][w];
    a.chan_ss[r * 2 + threadIdx.x] = s2;  // [N][2][1][1]
  }
  if (t0 < D) {
#pragma unroll
    for (int be = 0; be < 2; ++be) {
      float g[8];
      unpack8(*reinterpret_cast<const uint4*>((const __nv_bfloat16*)a.chan_norm +
                                              (size_t)be * a.cn_channels * D + t0),
              g);
      const float* m = be ? mv : mk;
      uint4 o;
      __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int i = 0; i < 4; ++i) ob[i] = __floats2bfloat162_rn(m[2 * i] * g[2 * i], m[2 * i + 1] * g[2 * i + 1]);
      *reinterpret_cast<uint4*>((__nv_bfloat16*)a.mixed + ((size_t)be * a.N + r) * D + t0) = o;
    }
  }
}

int launch_mix(int dtype, const MixArgs& a, bool simt, cudaStream_t st, uint32_t* flags) {
  if (a.N <= 0) return 0;
  if (dtype == WM_BF16 && !simt && a.k == 1 && a.chan_ss && a.L <= 64 && a.D % 8 == 0 &&
      a.D <= 8 * 1024 && (uintptr_t)a.stash % 16 == 0 && a.ld_row % 8 == 0 &&
      (uintptr_t)a.src_norm % 16 == 0 && (uintptr_t)a.chan_norm % 16 == 0 &&
      (uintptr_t)a.mixed % 16 == 0) {
    const int threads = ((a.D / 8 + 31) / 32) * 32;
    launch_k(mix1_kernel, dim3(a.N), dim3(threads), 0, st, a);
    return 1;
  }
  const bool stream_ok = dtype == WM_BF16 && !simt && a.D % (8 * MIX_C) == 0 &&
                         ((uintptr_t)a.stash % 16 == 0) && (a.ld_row % 8 == 0);
  if (dtype == WM_BF16 && !simt) {
    const int parts = launch_mix_tc(a, st, flags);
    if (parts) return parts;  // P > 0, or -1: its launch failed
  }
  if (stream_ok) {
    bool done = false;
    switch (a.k) {
      case 1: done = launch_mix_stream<1>(a, flags, st); break;
      case 2: done = launch_mix_stream<2>(a, flags, st); break;
      case 4: done = launch_mix_stream<4>(a, flags, st); break;
      case 8: done = launch_mix_stream<8>(a, flags, st); break;
      case 12: done = launch_mix_stream<12>(a, flags, st); break;
      case 14: done = launch_mix_stream<14>(a, flags, st); break;
      case 16: done = launch_mix_stream<16>(a, flags, st); break;
      default: break;
    }
    if (done) return 0;
  }
  WM_DISPATCH_S(dtype, launch_k(mix_simt_kernel<S>, dim3(a.N), dim3(256), a.D * sizeof(float), st, a));
  return 0;
}

}  // namespace wm
