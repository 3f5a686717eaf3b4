// Contraction engine for few rows (M <= 64, the decode step): bf16 mma.sync.
//
// One CTA computes 16 output columns (16 weight rows) for all M <= 64 rows,
// streaming its weight rows and the activation block through a 3-stage
// cp.async pipeline over K in chunks of 64. Four warps each own 16 activation
// rows. Weight traffic, the whole cost of these products, is spread over
// N / 16 CTAs (112 for N = 1792) instead of one 128-row tile per column block.
// Residual and SwiGLU epilogues are fused; per-head epilogues (q-norm, K/V
// projection) write fp32 sums for the shared finalize kernel.
#include "kernels.h"

namespace wm {
namespace sk {

constexpr int BN = 16, BKC = 64, STAGES = 3, NT = 128, LDS = BKC + 8;

__device__ __forceinline__ uint32_t sa(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void cp16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sa(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                      uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// DUAL: B and B2 (SwiGLU gate and up) share the activation loads.
template <bool DUAL>
__global__ void __launch_bounds__(NT) skinny_kernel(const GemmDesc g, float* fp32_out) {
  pdl_wait();
  pdl_trigger();
  __shared__ __align__(16) __nv_bfloat16 sA[STAGES][64][LDS];
  __shared__ __align__(16) __nv_bfloat16 sB[STAGES][(DUAL ? 2 : 1) * BN][LDS];
  const int b = blockIdx.y;
  const int n0 = blockIdx.x * BN;
  const __nv_bfloat16* A = (const __nv_bfloat16*)g.A + (long long)b * g.a_bstride;
  const __nv_bfloat16* Bm = (const __nv_bfloat16*)g.B + (long long)b * g.b_bstride;
  const __nv_bfloat16* B2 = DUAL ? (const __nv_bfloat16*)g.B2 + (long long)b * g.b_bstride : nullptr;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkc = (g.K + BKC - 1) / BKC;
  auto load = [&](int kc, int st) {
    const int k0 = kc * BKC;
    for (int c = threadIdx.x; c < 64 * (BKC / 8); c += NT) {
      const int m = c / (BKC / 8), part = c % (BKC / 8), k = k0 + part * 8;
      const bool v = m < g.M && k < g.K;
      cp16(&sA[st][m][part * 8], A + (long long)(v ? m : 0) * g.lda + (v ? k : 0), v);
    }
    for (int c = threadIdx.x; c < (DUAL ? 2 : 1) * BN * (BKC / 8); c += NT) {
      const int rr = c / (BKC / 8), part = c % (BKC / 8), k = k0 + part * 8;
      const int which = rr / BN, n = n0 + rr % BN;
      const bool v = n < g.N && k < g.K;
      const __nv_bfloat16* src = (which ? B2 : Bm) + (long long)(v ? n : 0) * g.ldb + (v ? k : 0);
      cp16(&sB[st][rr][part * 8], src, v);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  float acc[DUAL ? 4 : 2][4];
#pragma unroll
  for (int i = 0; i < (DUAL ? 4 : 2); ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < nkc) load(s, s);
    else asm volatile("cp.async.commit_group;" ::: "memory");
  }
  for (int kc = 0; kc < nkc; ++kc) {
    const int st = kc % STAGES;
    asm volatile("cp.async.wait_group %0;" ::"n"(STAGES - 2) : "memory");
    __syncthreads();
    if (kc + STAGES - 1 < nkc) load(kc + STAGES - 1, (kc + STAGES - 1) % STAGES);
    else asm volatile("cp.async.commit_group;" ::: "memory");
#pragma unroll
    for (int ks = 0; ks < BKC / 16; ++ks) {
      uint32_t a[4];
      ldsm4(sa(&sA[st][warp * 16 + (lane & 15)][ks * 16 + (lane >> 4) * 8]), a[0], a[1], a[2], a[3]);
#pragma unroll
      for (int half = 0; half < (DUAL ? 2 : 1); ++half) {
        // two 8-column n-tiles, k = ks*16 .. ks*16+15: rows (lane & 7) + 8 * (lane >> 4)
        uint32_t b0, b1, b2, b3;
        ldsm4(sa(&sB[st][half * BN + (lane & 7) + ((lane >> 4) << 3)][ks * 16 + ((lane >> 3) & 1) * 8]),
              b0, b1, b2, b3);
        mma(acc[half * 2 + 0], a, b0, b1);
        mma(acc[half * 2 + 1], a, b2, b3);
      }
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  // epilogue: thread holds rows (warp*16 + lane/4, +8), columns 2*(lane%4) (+1) of each n-tile
  const Epi& e = g.epi;
  const int r0 = warp * 16 + (lane >> 2);
#pragma unroll
  for (int half_row = 0; half_row < 2; ++half_row) {
    const int row = r0 + half_row * 8;
    if (row >= g.M) continue;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int col = n0 + nt * 8 + 2 * (lane & 3) + e2;
        if (col >= g.N) continue;
        float v = acc[nt][half_row * 2 + e2];
        if (DUAL) {
          const float u = acc[2 + nt][half_row * 2 + e2];
          v = v / (1.f + __expf(-v)) * u;
        }
        if (fp32_out) {
          fp32_out[((long long)b * g.M + row) * g.N + col] = v;
          continue;
        }
        if (e.mode == EPI_RESID) v += __bfloat162float(((const __nv_bfloat16*)e.R)[(long long)row * e.ldr + col]);
        const long long orow = (e.mode == EPI_STORE && e.rowmap) ? e.rowmap[row] : row;
        const long long off = (long long)b * e.c_bstride + orow * e.ldc + col;
        if (e.out_f32)
          ((float*)e.C)[off] = v;
        else
          ((__nv_bfloat16*)e.C)[off] = __float2bfloat16_rn(v);
      }
    }
  }
}

}  // namespace sk

bool gemm_skinny_supported(const GemmDesc& g) {
  auto a16 = [](const void* p) { return ((uintptr_t)p & 15u) == 0; };
  if (g.M < 1 || g.M > 64 || g.N < 1 || g.K < 1 || g.K % 8 || g.batch < 1) return false;
  if (!a16(g.A) || !a16(g.B) || (g.B2 && !a16(g.B2))) return false;
  if (g.lda % 8 || g.ldb % 8 || (g.batch > 1 && (g.a_bstride % 8 || g.b_bstride % 8))) return false;
  if ((g.epi.mode == EPI_QNORM_ROPE || g.epi.mode == EPI_KV) &&
      (!g.partial || (long long)g.batch * g.M * g.N > g.partial_elems))
    return false;
  return true;
}

// Runs the product; per-head epilogues go through the fp32 sums in g.partial
// and the finalize kernel. Returns the number of kernels launched.
int launch_gemm_skinny(const GemmDesc& g, cudaStream_t st) {
  const bool head = g.epi.mode == EPI_QNORM_ROPE || g.epi.mode == EPI_KV;
  dim3 grid((g.N + sk::BN - 1) / sk::BN, g.batch);
  float* f32 = head ? g.partial : nullptr;
  if (g.B2)
    launch_k(sk::skinny_kernel<true>, dim3(grid), dim3(sk::NT), 0, st, g, f32);
  else
    launch_k(sk::skinny_kernel<false>, dim3(grid), dim3(sk::NT), 0, st, g, f32);
  if (!head) return 1;
  return 1 + launch_finalize_head(g, st);
}

}  // namespace wm
