// Shared device/host definitions for libwm (B300, sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/wm.h"

namespace wm {

// ---------------------------------------------------------------------------
// Programmatic dependent launch. Kernels go out through launch_k, which lets
// a kernel's CTAs start while its predecessor in the stream drains. Every
// such kernel calls pdl_wait() in each thread before it reads or writes any
// global memory that another kernel writes or reads (only shared-memory,
// TMEM and barrier set-up, tensor-map prefetch and loads of constant weights
// may come first), so that it sees the predecessor's results and its grid
// cannot complete before the predecessor's. pdl_trigger() lets the
// successor's CTAs be scheduled.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t st, Args... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kern, static_cast<KArgs>(args)...);
}

// Device-side check bits, OR-ed into the workspace flag word.
enum : uint32_t {
  FLAG_BAD_TOKEN = 1u,     // token id outside [0, V)
  FLAG_BAD_SEQ = 2u,       // sequence index outside [0, B)
  FLAG_BAD_POS = 4u,       // position outside [0, Tmax)
  FLAG_TIMEOUT = 8u,       // a bounded wait gave up
};

// ---------------------------------------------------------------------------
// Storage-type conversions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename S> __device__ __forceinline__ S from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide sum for blockDim.x <= 1024; ``red`` holds >= 32 floats.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float t = (lane < nw) ? red[lane] : 0.f;
  return warp_sum(t);
}

__device__ __forceinline__ float silu_f(float x) { return x / (1.f + expf(-x)); }

// ---------------------------------------------------------------------------
// GEMM description shared by the tensor-core and CUDA-core engines.
//   C[b][m][n] = epilogue( sum_k A[b][m][k] * B[b][n][k] )
// A and B are K-contiguous (row-major [rows][K]) in the storage type.
// ---------------------------------------------------------------------------
enum EpiMode : int {
  EPI_STORE = 0,       // C = acc                         (C in storage type or fp32)
  EPI_RESID = 1,       // C = acc + R                     (storage type)
  EPI_SWIGLU = 2,      // C = silu(acc_B) * acc_B2        (storage type)
  EPI_QNORM_ROPE = 3,  // per head: RoPE_pos(RMSNorm_d(acc; gain))      -> C
  EPI_KV = 4,          // batch index = channel j; keys: RoPE(RMSNorm_d(acc; gain_j)),
                       // values: acc; scattered to cache[seq][j][h][pos][:]
};

struct Epi {
  int mode = EPI_STORE;
  int out_f32 = 0;               // EPI_STORE: C is fp32
  void* C = nullptr;
  long long ldc = 0, c_bstride = 0;
  const void* R = nullptr;       // EPI_RESID residual [M][ldr]
  long long ldr = 0;
  const int* rowmap = nullptr;   // EPI_STORE: C row index of tile row m (nullable)
  const void* gain = nullptr;    // norm gains [d] (+ gain_bstride per batch)
  long long gain_bstride = 0;
  const int* pos = nullptr;      // [M] absolute positions (RoPE, cache slot)
  const int* seq = nullptr;      // [M] sequence of each row (EPI_KV)
  const float2* rope = nullptr;  // [Tmax][d/2] (cos, sin)
  int d = 0;
  float eps = 1e-6f;
  void* cache_k = nullptr;
  void* cache_v = nullptr;
  int k = 0, Hkv = 0, Tmax = 0, B = 0;
  int kv_branch = 0;             // EPI_KV: 0 = keys (norm + RoPE), 1 = values (raw)
  // EPI_KV with a deferred channel norm (nullable): the input rows are
  // u = tau (.) m and output row ``row`` of channel b is scaled by
  // rsqrt(sum_c chan_ss[row][kv_branch][b][c] / chan_D + eps), the channel
  // RMSNorm's factor (the projection is linear in its input).
  const float* chan_ss = nullptr;
  int chan_parts = 0;
  int chan_ss_k = 0;             // channels per branch in the chan_ss layout
  float chan_D = 1.f;
  int chan0 = 0;                 // EPI_KV: cache channel of batch 0 (channel = chan0 + batch)
  uint32_t* flags = nullptr;
};

__device__ __forceinline__ float chan_scale(const Epi& e, long long row, int channel) {
  const float* p = e.chan_ss + ((row * 2 + e.kv_branch) * e.chan_ss_k + channel) * e.chan_parts;
  float s = 0.f;
  for (int c = 0; c < e.chan_parts; ++c) s += p[c];
  return rsqrtf(s / e.chan_D + e.eps);
}

struct GemmDesc {
  int M = 0, N = 0, K = 0, batch = 1;
  const void* A = nullptr;
  long long lda = 0, a_bstride = 0;
  const void* B = nullptr;
  long long ldb = 0, b_bstride = 0;
  const void* B2 = nullptr;      // EPI_SWIGLU second operand (same strides as B)
  // B (and B2) are weights that no kernel writes: the tensor-core engine may
  // request them before its predecessor in the stream has finished.
  bool b_const = false;
  bool no_cluster = false;       // split K through global atomics, never a cluster
  bool wait_probe = false;       // test aid (WM_FLAG_WAIT_PROBE): see gemm_tc.cu
  Epi epi;
  // Zero-filled fp32 scratch for split-K (nullable): when a GEMM has too few
  // output tiles to occupy the GPU, K is split across CTAs that add their
  // partial tiles here; a finalize kernel applies the epilogue and re-zeroes.
  float* partial = nullptr;
  long long partial_elems = 0;
  // Optional L2 prefetch (tensor-core engine): byte ranges that a later
  // product reads. Each CTA fetches its share into L2 once its own loads are
  // issued, so the transfer overlaps this product's reduction and epilogue
  // instead of opening the next product. Ranges must be 16-byte aligned with
  // sizes multiples of 16; unused entries are null.
  const void* pf[2] = {nullptr, nullptr};
  long long pf_bytes[2] = {0, 0};
};

// Per-head epilogue on one row's d values (EPI_QNORM_ROPE and the key branch
// of EPI_KV): RMSNorm over the head with ``gain`` then rotate-half RoPE at
// ``pos`` using the (cos, sin) table row ``rt``.
template <typename S>
__device__ __forceinline__ void head_norm_rope(float* v, int d, const S* gain, float eps,
                                               const float2* rt) {
  float ss = 0.f;
  for (int t = 0; t < d; ++t) ss += v[t] * v[t];
  const float inv = rsqrtf(ss / (float)d + eps);
  for (int t = 0; t < d; ++t) v[t] = v[t] * inv * to_f(gain[t]);
  const int half = d >> 1;
  for (int t = 0; t < half; ++t) {
    const float2 cs = rt[t];
    const float x1 = v[t], x2 = v[t + half];
    v[t] = x1 * cs.x - x2 * cs.y;
    v[t + half] = x2 * cs.x + x1 * cs.y;
  }
}

}  // namespace wm
