// Strictly causal channel attention: row n (sequence seq[n], position pos[n])
// attends to keys s < pos[n] of one cache channel; query head h reads KV head
// h*Hkv/Hq; a row with no visible key gets 0.
#include "kernels.h"

namespace wm {

// CUDA-core engine: one warp per (row, query head), online softmax over the
// visible keys, each lane owning d/32 of the head's dimensions.
template <typename S>
__global__ void __launch_bounds__(128) attn_simt_kernel(const AttnArgs a) {
  const int lane = threadIdx.x & 31;
  const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (wid >= (long long)a.N * a.Hq) return;
  const int r = (int)(wid / a.Hq), h = (int)(wid % a.Hq);
  const int hk = h * a.Hkv / a.Hq;
  const int per = a.d >> 5;  // 2 or 4
  S* out = (S*)a.out + (long long)r * a.Hq * a.d + (long long)h * a.d;
  const int sq = a.seq[r], i = a.pos[r];
  if (sq < 0 || sq >= a.B || i < 0 || i >= a.Tmax) {
    if (lane == 0) atomicOr(a.flags, sq < 0 || sq >= a.B ? FLAG_BAD_SEQ : FLAG_BAD_POS);
    for (int e = 0; e < per; ++e) out[lane * per + e] = from_f<S>(0.f);
    return;
  }
  const long long base = (((long long)sq * a.k + a.channel) * a.Hkv + hk) * a.Tmax * a.d;
  const S* Kp = (const S*)a.cache_k + base;
  const S* Vp = (const S*)a.cache_v + base;
  const S* qp = (const S*)a.q + (long long)r * a.Hq * a.d + (long long)h * a.d;
  float qv[4], o[4];
  const float scale = 1.0f / sqrtf((float)a.d);
  for (int e = 0; e < per; ++e) {
    qv[e] = to_f(qp[lane * per + e]) * scale;
    o[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int s = 0; s < i; ++s) {
    float part = 0.f;
    for (int e = 0; e < per; ++e) part += qv[e] * to_f(Kp[(long long)s * a.d + lane * per + e]);
    const float z = warp_sum(part);
    const float mn = fmaxf(m, z);
    const float corr = expf(m - mn);
    const float pz = expf(z - mn);
    l = l * corr + pz;
    for (int e = 0; e < per; ++e)
      o[e] = o[e] * corr + pz * to_f(Vp[(long long)s * a.d + lane * per + e]);
    m = mn;
  }
  for (int e = 0; e < per; ++e) out[lane * per + e] = from_f<S>(i > 0 ? o[e] / l : 0.f);
}

void launch_attention(int dtype, const AttnArgs& a, bool simt, cudaStream_t st) {
  if (a.N <= 0) return;
  (void)simt;
  const long long warps = (long long)a.N * a.Hq;
  const int blocks = (int)((warps + 3) / 4);
  WM_DISPATCH_S(dtype, attn_simt_kernel<S><<<blocks, 128, 0, st>>>(a));
}

}  // namespace wm
