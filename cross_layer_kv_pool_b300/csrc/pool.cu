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
  extern __shared__ float mbuf[];  // [D]
  __shared__ float red[32];
  const int r = blockIdx.x;
  const S* hs = (const S*)a.stash + (long long)r * a.ld_row;
  const float* inv = a.inv + (long long)r * a.L;
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
          acc += cf[l] * (inv[l] * to_f(sn[((long long)beta * a.L + l) * a.D + t]) *
                          to_f(hs[(long long)l * a.D + t]));
        mbuf[t] = acc;
        ss += acc * acc;
      }
      ss = block_sum(ss, red);
      const float im = rsqrtf(ss / (float)a.D + a.eps);
      for (int t = threadIdx.x; t < a.D; t += blockDim.x)
        out[(((long long)beta * a.k + j) * a.N + r) * a.D + t] =
            from_f<S>(mbuf[t] * im * to_f(cn[((long long)beta * a.k + j) * a.D + t]));
    }
  }
}

void launch_mix(int dtype, const MixArgs& a, bool simt, cudaStream_t st) {
  if (a.N <= 0) return;
  (void)simt;
  WM_DISPATCH_S(dtype, mix_simt_kernel<S><<<a.N, 256, a.D * sizeof(float), st>>>(a));
}

}  // namespace wm
