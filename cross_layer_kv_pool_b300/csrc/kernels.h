// Host-side launch functions of libwm's kernels (internal interface).
#pragma once

#include "common.cuh"

namespace wm {

// Storage-type dispatch helper: dtype is WM_F32 or WM_BF16.
#define WM_DISPATCH_S(dtype, ...)                          \
  do {                                                     \
    if ((dtype) == WM_F32) {                               \
      using S = float;                                     \
      __VA_ARGS__;                                         \
    } else {                                               \
      using S = __nv_bfloat16;                             \
      __VA_ARGS__;                                         \
    }                                                      \
  } while (0)

inline size_t elem_size(int dtype) { return dtype == WM_F32 ? 4 : 2; }

// ---- elem.cu ---------------------------------------------------------------
void launch_rope_table(float2* tab, int p0, int p1, int d, float base, cudaStream_t st);
// Rows of group q (positions pos0 + q + g*u) of B sequences of T tokens.
void launch_group_rows(const int32_t* tokens, int B, int T, int g, int q, int nq,
                       int32_t* tok, int32_t* seq, int32_t* pos, int32_t* rowmap, cudaStream_t st,
                       int pos0 = 0);
void launch_decode_rows_dev(const int32_t* tokens, const int32_t* pos_in, int B, int d, float base,
                            int32_t* tok, int32_t* seq, int32_t* pos, float2* tab, int Tmax,
                            cudaStream_t st);
void launch_decode_rows(const int32_t* tokens, int B, int t, int32_t* tok, int32_t* seq,
                        int32_t* pos, cudaStream_t st);
void launch_embed(int dtype, const int32_t* tok, int N, const void* embed, int V, int D,
                  void* out, long long ld_out, uint32_t* flags, cudaStream_t st);
// Per (row, layer l = l0 + y): inv_rms of X[row][l] -> inv[row*L + l];
// optional xn = X*inv*gain_in[l]; for l in the router set, rin[beta][row][ridx*D..]
// = X*inv*src_norm[beta][l].
void launch_norm_emit(int dtype, const void* X, long long ldx_row, long long ldx_l, int N,
                      int l0, int nl, int D, int L, const void* gain_in, void* xn,
                      float* inv, const void* src_norm, void* rin, int nR, int p, int p_off,
                      float eps, cudaStream_t st);
// y[r] = RMSNorm(X[row0 + r*rstride]; gain) for r < N.
void launch_rmsnorm(int dtype, const void* X, long long ldx, int row0, int rstride, int N, int D,
                    const void* gain, void* y, float eps, cudaStream_t st);
void launch_broadcast_coeff(const float* stat, int N, int n_per_row, float* coeff,
                            cudaStream_t st);

// ---- gemm_simt.cu / gemm_tc.cu --------------------------------------------
void launch_gemm_simt(int dtype, const GemmDesc& g, cudaStream_t st);
bool gemm_tc_supported(const GemmDesc& g);
cudaError_t launch_gemm_tc(const GemmDesc& g, cudaStream_t st, int* launches);

// ---- attn.cu ---------------------------------------------------------------
struct AttnArgs {
  const void* q;          // [N][Hq][d]
  int N;
  const int32_t* seq;
  const int32_t* pos;
  int channel;
  const void* cache_k;    // [B][k][Hkv][Tmax][d]
  const void* cache_v;
  int B, k, Hq, Hkv, d, Tmax;
  void* out;              // [N][Hq*d]
  uint32_t* flags;
  // Optional arrival counters (zero on entry, left zero): the decode
  // engine's last key split of each (row, KV head) merges the splits itself.
  int* counters = nullptr;
  long long counter_elems = 0;
};
// Returns the number of kernels launched. kv_len: the largest visible key
// count when the host knows it (decode), else 0. part: fp32 scratch for the
// decode engine's key splits (part_elems floats), nullable.
int launch_attention(int dtype, const AttnArgs& a, bool simt, cudaStream_t st, int nq, int kv_len,
                     float* part, long long part_elems);
// Prefill attention on tcgen05 (attn_pair.cu): two query tiles of one
// sequence and KV head per CTA, sharing every K and V block.
bool attention_tc_supported(const AttnArgs& a, int nq);
cudaError_t launch_attention_pair(const AttnArgs& a, int nq, cudaStream_t st);

// ---- sgemm.cu --------------------------------------------------------------
// C[b] = op(A[b]) op(B[b]) + beta C[b] for b < batch, fp32, row-major: op(A)
// is M x K (A stored K x M when ta), op(B) K x N (B stored N x K when tb);
// sa, sb, sc are the strides between batch entries (0 broadcasts).
struct SgemmArgs {
  bool ta, tb;
  int M, N, K;
  const float* A;
  long long lda, sa;
  const float* B;
  long long ldb, sb;
  float beta;
  float* C;
  long long ldc, sc;
  int batch;
};
cudaError_t sgemm_rm(const SgemmArgs& g, cudaStream_t st);

// ---- pool.cu ---------------------------------------------------------------
// Bytes per row of the tensor-core mixer's coefficient tiles: [2 branches]
// [hi, lo][16 channels][40] bf16 (32 layers + 8 of padding per row).
constexpr long long MIX_ATILE_BYTES = 2 * 2 * 16 * 40 * 2;

struct MixArgs {
  const void* stash;      // [N][L][D] source states
  long long ld_row;       // elements between rows (L*D for a stash)
  const float* inv;       // [N][L] inverse RMS of each source state
  const float* coeff;     // [N][2][k][L]
  const void* src_norm;   // [2][L][D]
  const void* chan_norm;  // [2][k][D]
  void* mixed;            // [2][k][N][D]
  float* chan_ss;         // [N][2][k][8] slice sums of squares (deferred-norm output)
  // scratch of the tensor-core mixer (nullable: that mixer is then not used):
  // per row the hi/lo bf16 coefficient tile, MIX_ATILE_BYTES bytes
  void* atile;
  int N, L, D, k;         // rows, source layers mixed (the first L of each row), width, channels
  int inv_ld;             // floats between rows of inv (>= L)
  int sn_layers;          // layers per branch in src_norm (>= L)
  int cn_channels;        // channels per branch in chan_norm (>= k)
  float eps;
};
// Runs the mixer. Returns 0 if ``mixed`` holds the channel-normed c, or P > 0
// if it holds u = tau (.) m with the norm deferred: chan_ss then holds P
// partial sums of squares per (row, branch, channel) and the norm factor is
// rsqrt(sum / D + eps) (applied by the projection epilogue, or in place by
// launch_mix_normalize); -1 if a launch failed.
int launch_mix(int dtype, const MixArgs& a, bool simt, cudaStream_t st, uint32_t* flags);
// Tensor-core mixer (bf16 mma.sync, deferred norm); returns P, 0 if the
// shape is outside its envelope (k > 16, L > 32, no slicing of D into at
// most 8 slices of at most 448 columns, misaligned operands), or -1 if a
// launch failed.
int launch_mix_tc(const MixArgs& a, cudaStream_t st, uint32_t* flags);

// ---------------------------------------------------------------------------
// Backward pass of the pool (pool_bwd.cu)
// ---------------------------------------------------------------------------
struct PoolBwdLayout {
  // FLAGS first: the flag word sits where wm_check_flags reads it. SX .. TMPW
  // hold the router products' bf16 hi/lo operands, SC .. TMPP the channel
  // projections' (see pool_bwd.cu).
  enum { FLAGS, INV, N_, X, A, M, RJ, C, KT, DY, DC, DN, DX, WR, WP, G, AK,
         SX, SW, SWT, SDA, SDAT, SXT, TMPW, SC, SWP, SDY, SWPT, SDYT, SCT, TMPP, NB };
  size_t off[NB];
  size_t total;
};
PoolBwdLayout pool_bwd_layout(const wm_config& c, long long N);
struct PoolBwdArgs {
  const wm_config* cfg;
  const wm_weights* w;
  const void* states;  // [N][L][D] storage type
  int N;
  const int* pos;      // [N]
  const void* dK;      // [N][k][Hkv][d] storage type
  const void* dV;
  float* dstates;      // [N][L][D] fp32, overwritten
  wm_pool_grads g;     // fp32 accumulators
  void* ws;
  PoolBwdLayout lay;
};
cudaError_t run_pool_backward(const PoolBwdArgs& q, cudaStream_t st);
void launch_mix_normalize(const MixArgs& a, int parts, cudaStream_t st);

}  // namespace wm
