// Pool mixer on tcgen05 with the layer operand in tensor memory (bf16).
//
// Per token and branch b the mix is the small contraction
//   M^b [D x k] = X^b [D x L] . A^b^T [L x k],
//   X^b_{t,l} = src_norm[b][l][t] h_l[t],     A^b_{j,l} = a^b_{j,l} inv_l,
// followed by the channel RMSNorm of each column of M^b ("WhiteMatter:
// All-to-All Cross-Layer Connections via KV Mixing", 3 METHOD, "Cross-layer
// KV pool"). Its operands are what the step must stream (the L x D states of
// every token) and it is bound by HBM; the work here is arranged so that the
// SM spends as few instructions per byte as possible:
//
//   - the states of one row and one 128- or 256-column slice arrive by one
//     TMA box {W columns, L layers} (producer warp);
//   - converter warps (one thread per column: TMEM lane) multiply the states
//     by the resident source-norm gains and split the exact product into a
//     bf16 hi + lo pair (both branches), and store them straight into tensor
//     memory as the MMA's A operand (M = 128 columns, K = layers);
//   - a coefficient warp builds the row's B operand in shared memory: the
//     k x L coefficients times inv_l, split hi | lo along K (128-byte rows,
//     128-byte swizzle);
//   - one thread issues tcgen05.mma (M 128, N 16, K 16) for X_hi.A_hi +
//     X_lo.A_hi + X_hi.A_lo into an fp32 accumulator in tensor memory (the
//     missing X_lo.A_lo term is below 2^-16 relative);
//   - epilogue warps read the accumulator (16x256b, the m16n8 fragment), form
//     u = tau (.) m, reduce the slice's sums of squares of m per channel, and
//     write u transposed (stmatrix) into a staging tile that a storer warp
//     sends out with one bulk copy per (branch, channel) row segment.
// Everything is double-buffered per row (tensor-memory operands and
// accumulators, coefficient tiles, staging tiles) and the states run through
// a ring of NS stages, so the six roles work on different rows at once.
//
// As in the mma.sync mixer, the channel norm needs sums over all D columns,
// which no CTA sees: the kernel writes u = tau (.) m and the slice's sums of
// squares of m; the K/V projection (linear in its input) applies
// rsqrt(sum / D + eps) to its output rows.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kernels.h"

namespace wm {
namespace mt {

constexpr unsigned long long WAIT_NS = 4000000000ull;  // 4 s bound on any wait
constexpr int MAX_NS = 6;                               // state ring stages

struct Geo {
  int CT;     // 128-column tiles per CTA (1 or 2)
  int W;      // columns per CTA
  int CS;     // column slices (CTAs per row)
  int LP;     // layers rounded up to 16 or 32 (MMA K)
  int NS;     // state ring stages
  int NCV;    // converter warps (4 * CT), also the epilogue warp count
  int OSTR;   // staging row stride (elements), W + 8: conflict-free stmatrix
  int tmem_cols, buf_cols, a_cols;  // allocation, columns per buffer, A columns per (tile, branch, half)
  unsigned off_stage, off_b, off_out, off_red, off_bar, smem;
};

__device__ __forceinline__ uint32_t su32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait; false on timeout or when another role already gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try(b, parity)) return true;
  const unsigned long long t0 = gtimer();
  while (true) {
    if (mbar_try(b, parity)) return true;
    if (*abort_flag) return false;
    if (gtimer() - t0 > WAIT_NS) return false;
  }
}
// One lane waits, the warp learns the outcome.
__device__ __forceinline__ bool warp_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                                          int lane) {
  int ok = 1;
  if (lane == 0) ok = mbar_wait(b, parity, abort_flag) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}
__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// A from tensor memory, B from shared memory, D in tensor memory.
__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                        uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
      : "memory");
}
// K-major operand tile with 128-byte swizzle: rows of 128 B, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;            // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset
  d |= (uint64_t)1 << 46;            // descriptor version
  d |= (uint64_t)2 << 61;            // 128-byte swizzle
  return d;
}
// kind::f16: bf16 A and B, fp32 D, K-major, M = 128, N = 16.
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}
// 16 lanes x 16 columns: the m16n8 accumulator fragment, twice along columns.
__device__ __forceinline__ void tmem_ld16x256x2(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr));
}
__device__ __forceinline__ void stsm4t(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2,
                                       uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr),
               "r"(r0), "r"(r1), "r"(r2), "r"(r3)
               : "memory");
}
// x*y of two bf16 pairs as an exact hi + lo pair of bf16 pairs: the product
// of two 8-bit significands has at most 16 bits; hi holds it rounded to 8
// bits and the residual (at most 8 bits) is exact in lo.
__device__ __forceinline__ void bmul2_split(uint32_t x, uint32_t y, uint32_t& hi, uint32_t& lo) {
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(hi) : "r"(x), "r"(y));
  const uint32_t nhi = hi ^ 0x80008000u;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(lo) : "r"(x), "r"(y), "r"(nhi));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ void tma_load3(const CUtensorMap* map, uint64_t* bar, void* dst, int c0,
                                          int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(su32(dst)),
      "l"(map), "r"(su32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Byte offset of K element e (0..63) in row j of a 128-byte-swizzled K-major tile.
__device__ __forceinline__ uint32_t swz(int j, int e) {
  return (uint32_t)(j * 128 + ((((e >> 3) ^ (j & 7)) << 4) | ((e & 7) << 1)));
}

__global__ void __launch_bounds__(20 * 32, 1)
    mix_tmem_kernel(const __grid_constant__ CUtensorMap tmS, const MixArgs a, const Geo g,
                    uint32_t* flags) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NCV = g.NCV;
  const int W_PROD = 2 * NCV, W_MMA = 2 * NCV + 1, W_COEF = 2 * NCV + 2, W_STORE = 2 * NCV + 3;
  const int slice = (int)(blockIdx.x % g.CS);
  const long long rg = blockIdx.x / g.CS, nrg = gridDim.x / g.CS;
  const int c0 = slice * g.W;
  const int L = a.L, K = a.k, D = a.D;
  const long long nrows = rg < a.N ? (a.N - 1 - rg) / nrg + 1 : 0;  // rows of this CTA

  uint8_t* stage = sm + g.off_stage;                         // [NS][L][W] bf16
  uint8_t* btile = sm + g.off_b;                             // [2 buf][2 branch][16][128 B]
  __nv_bfloat16* otile = (__nv_bfloat16*)(sm + g.off_out);   // [2 buf][2][16][OSTR]
  float* red = (float*)(sm + g.off_red);                     // [2 buf][NCV][32]
  uint64_t* full = (uint64_t*)(sm + g.off_bar);              // [NS]
  uint64_t* empty = full + MAX_NS;                           // [NS]
  uint64_t* a_full = empty + MAX_NS;                         // [2]
  uint64_t* b_full = a_full + 2;                             // [2]
  uint64_t* mma_done = b_full + 2;                           // [2]
  uint64_t* d_empty = mma_done + 2;                          // [2]
  uint64_t* o_full = d_empty + 2;                            // [2]
  uint64_t* o_empty = o_full + 2;                            // [2]
  uint64_t* mma_final = o_empty + 2;
  uint32_t* tmem_holder = (uint32_t*)(mma_final + 1);
  volatile int* abort_flag = (volatile int*)(tmem_holder + 1);
  volatile int* stop = abort_flag + 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < g.NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], NCV);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&a_full[i], NCV);
      mbar_init(&b_full[i], 1);
      mbar_init(&mma_done[i], 1);
      mbar_init(&d_empty[i], NCV);
      mbar_init(&o_full[i], NCV);
      mbar_init(&o_empty[i], 1);
    }
    mbar_init(mma_final, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmS) : "memory");
  }
  // coefficient tiles start at zero: rows j >= k and layers l >= L stay zero
  for (int i = threadIdx.x; i < 2 * 2 * 16 * 128 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(btile)[i] = make_uint4(0u, 0u, 0u, 0u);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  // every access above touched shared memory only; the predecessor's outputs next
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) *stop = (*(volatile const uint32_t*)flags & FLAG_TIMEOUT) != 0;
  __syncthreads();
  // An earlier kernel of this call timed out: leave before allocating or
  // issuing anything (one wait limit per call).
  if (*stop) return;
  if (warp == W_MMA) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     su32(tmem_holder)),
                 "r"((uint32_t)g.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_holder;
  // tensor-memory columns: buffer b at b * buf_cols; in it the A operands
  // (tile c, branch be, half p) at ((c * 2 + be) * 2 + p) * a_cols, then the
  // accumulators (tile c, branch be) at 4 * CT * a_cols + (c * 2 + be) * 16
  auto a_col = [&](int b, int c, int be, int p) {
    return (uint32_t)(b * g.buf_cols + ((c * 2 + be) * 2 + p) * g.a_cols);
  };
  auto d_col = [&](int b, int c, int be) {
    return (uint32_t)(b * g.buf_cols + 4 * g.CT * g.a_cols + (c * 2 + be) * 16);
  };

  bool ok = true;
  if (warp < NCV) {
    // ---------------- converters: one thread per column (TMEM lane) ----------------
    const int ct = warp >> 2, q = warp & 3;
    const int t = ct * 128 + q * 32 + lane;  // column within the slice
    const __nv_bfloat16* sn = (const __nv_bfloat16*)a.src_norm;
    const int npair = (L + 1) / 2;
    uint32_t gk[16], gv[16];  // source-norm gains of this column, layer pairs
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      uint32_t x = 0u, y = 0u;
      if (i < npair) {
        const int l0 = 2 * i, l1 = 2 * i + 1;
        const size_t col = (size_t)c0 + t;
        const uint16_t k0 = __bfloat16_as_ushort(sn[(size_t)l0 * D + col]);
        const uint16_t v0 = __bfloat16_as_ushort(sn[((size_t)a.sn_layers + l0) * D + col]);
        const uint16_t k1 = l1 < L ? __bfloat16_as_ushort(sn[(size_t)l1 * D + col]) : 0;
        const uint16_t v1 = l1 < L ? __bfloat16_as_ushort(sn[((size_t)a.sn_layers + l1) * D + col]) : 0;
        x = (uint32_t)k0 | ((uint32_t)k1 << 16);
        y = (uint32_t)v0 | ((uint32_t)v1 << 16);
      }
      gk[i] = x;
      gv[i] = y;
    }
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    for (long long r = 0; r < nrows && ok; ++r) {
      const int s = (int)(r % g.NS), b = (int)(r & 1);
      if (!warp_wait(&full[s], (uint32_t)((r / g.NS) & 1), abort_flag, lane)) { ok = false; break; }
      if (r >= 2 && !warp_wait(&mma_done[b], (uint32_t)(((r >> 1) - 1) & 1), abort_flag, lane)) {
        ok = false;
        break;
      }
      fence_after();
      const __nv_bfloat16* hs = (const __nv_bfloat16*)(stage + (size_t)s * L * g.W * 2) + t;
      uint32_t hp[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        uint32_t x = 0u;
        if (i < npair) {
          const uint32_t h0 = __bfloat16_as_ushort(hs[(size_t)(2 * i) * g.W]);
          const uint32_t h1 = 2 * i + 1 < L ? __bfloat16_as_ushort(hs[(size_t)(2 * i + 1) * g.W]) : 0u;
          x = h0 | (h1 << 16);
        }
        hp[i] = x;
      }
      // the stage's states are in registers: the producer may refill it
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
      for (int be = 0; be < 2; ++be) {
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) bmul2_split(hp[i], be ? gv[i] : gk[i], hi[i], lo[i]);
        const uint32_t th = tmem + lane_off + a_col(b, ct, be, 0);
        const uint32_t tl = tmem + lane_off + a_col(b, ct, be, 1);
        if (g.LP == 32) {
          tmem_st16(th, hi);
          tmem_st16(tl, lo);
        } else {
          tmem_st8(th, hi);
          tmem_st8(tl, lo);
        }
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[b]);
    }
  } else if (warp < 2 * NCV) {
    // ---------------- epilogue: accumulators -> u = tau (.) m, sums of squares ----------------
    const int e = warp - NCV, ct = e >> 2, q = e & 3;
    const int gq = lane >> 2, tq = lane & 3;
    const __nv_bfloat16* cn = (const __nv_bfloat16*)a.chan_norm;
    // tau of this thread's outputs: [branch][lane half h][row 0/8][j 2tq, 2tq+1, 8+2tq, 9+2tq]
    float tau[2][2][2][4];
#pragma unroll
    for (int be = 0; be < 2; ++be)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int j = (jj >> 1) * 8 + 2 * tq + (jj & 1);
            const int t = ct * 128 + q * 32 + h * 16 + rr * 8 + gq;
            tau[be][h][rr][jj] =
                j < K ? __bfloat162float(cn[((size_t)be * a.cn_channels + j) * D + c0 + t]) : 0.f;
          }
    for (long long r = 0; r < nrows && ok; ++r) {
      const int b = (int)(r & 1);
      if (!warp_wait(&mma_done[b], (uint32_t)((r >> 1) & 1), abort_flag, lane)) { ok = false; break; }
      fence_after();
      uint32_t acc[2][2][8];
#pragma unroll
      for (int be = 0; be < 2; ++be)
#pragma unroll
        for (int h = 0; h < 2; ++h)
          tmem_ld16x256x2(tmem + ((uint32_t)(q * 32 + h * 16) << 16) + d_col(b, ct, be), acc[be][h]);
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&d_empty[b]);
      // staging tile of this row: free once the storer has read row r - 2's
      if (r >= 2 && !warp_wait(&o_empty[b], (uint32_t)(((r >> 1) - 1) & 1), abort_flag, lane)) {
        ok = false;
        break;
      }
      float ss[2][4];
#pragma unroll
      for (int be = 0; be < 2; ++be) {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) ss[be][jj] = 0.f;
        uint32_t pk[2][4];  // [lane half][matrix]: bf16 pairs of u
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // acc[be][h]: {rows gq, cols 2tq, 2tq+1}, {rows gq+8, same}, then cols + 8
          float m[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) m[i] = __uint_as_float(acc[be][h][i]);
          // fragment index i -> (row rr, column jj): i = (jj >> 1) * 4 + rr * 2 + (jj & 1)
#pragma unroll
          for (int rr = 0; rr < 2; ++rr)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const float v = m[(jj >> 1) * 4 + rr * 2 + (jj & 1)];
              ss[be][jj] = fmaf(v, v, ss[be][jj]);
            }
#pragma unroll
          for (int mi = 0; mi < 4; ++mi) {  // matrix mi: rows rr = mi & 1, columns 8 * (mi >> 1)
            const int rr = mi & 1, jh = mi >> 1;
            const float u0 = m[jh * 4 + rr * 2] * tau[be][h][rr][jh * 2];
            const float u1 = m[jh * 4 + rr * 2 + 1] * tau[be][h][rr][jh * 2 + 1];
            pk[h][mi] = pack_bf16(u0, u1);
          }
        }
        // transposed 8 x 8 blocks into staging rows (branch, channel): lane
        // 8i + x gives the address of row x of matrix i
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int mi = lane >> 3, x = lane & 7;
          const int j = (mi >> 1) * 8 + x;
          const int tcol = ct * 128 + q * 32 + h * 16 + (mi & 1) * 8;
          const __nv_bfloat16* dst = otile + ((size_t)(b * 2 + be) * 16 + j) * g.OSTR + tcol;
          stsm4t(su32(dst), pk[h][0], pk[h][1], pk[h][2], pk[h][3]);
        }
      }
      // sums of squares over this warp's 32 columns: reduce over the eight
      // lanes that share tq
#pragma unroll
      for (int be = 0; be < 2; ++be)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          float v = ss[be][jj];
          v += __shfl_xor_sync(0xffffffffu, v, 4);
          v += __shfl_xor_sync(0xffffffffu, v, 8);
          v += __shfl_xor_sync(0xffffffffu, v, 16);
          ss[be][jj] = v;
        }
      if (gq == 0) {
        float* rw = red + ((size_t)b * NCV + e) * 32;
#pragma unroll
        for (int be = 0; be < 2; ++be)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) rw[be * 16 + (jj >> 1) * 8 + 2 * tq + (jj & 1)] = ss[be][jj];
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_full[b]);
    }
  } else if (warp == W_PROD) {
    // ---------------- producer: one TMA box {W, L} per row ----------------
    long long issued = 0;
    if (lane == 0) {
      const uint32_t bytes = (uint32_t)(L * g.W * 2);
      for (long long r = 0; r < nrows; ++r) {
        const int s = (int)(r % g.NS);
        if (r >= g.NS && !mbar_wait(&empty[s], (uint32_t)(((r / g.NS) - 1) & 1), abort_flag)) {
          ok = false;
          break;
        }
        const long long row = rg + r * nrg;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(&full[s])),
                     "r"(bytes)
                     : "memory");
        tma_load3(&tmS, &full[s], stage + (size_t)s * L * g.W * 2, c0, 0, (int)row);
        issued = r + 1;
      }
      // Drain: every issued box has landed before the CTA may exit.
      volatile int no_abort = 0;
      for (long long r = issued - g.NS > 0 ? issued - g.NS : 0; r < issued; ++r)
        mbar_wait(&full[r % g.NS], (uint32_t)((r / g.NS) & 1), &no_abort);
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  } else if (warp == W_MMA) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const int nks = g.LP / 16;
      for (long long r = 0; r < nrows && ok; ++r) {
        const int b = (int)(r & 1);
        const uint32_t ph = (uint32_t)((r >> 1) & 1);
        if (!mbar_wait(&a_full[b], ph, abort_flag) || !mbar_wait(&b_full[b], ph, abort_flag) ||
            (r >= 2 && !mbar_wait(&d_empty[b], ph ^ 1, abort_flag))) {
          ok = false;
          break;
        }
        fence_after();
#pragma unroll 1
        for (int c = 0; c < g.CT; ++c)
#pragma unroll 1
          for (int be = 0; be < 2; ++be) {
            const uint32_t d = tmem + d_col(b, c, be);
            const uint32_t bt = su32(btile + (size_t)(b * 2 + be) * 2048);
            for (int s = 0; s < nks; ++s) {
              const uint32_t ah = tmem + a_col(b, c, be, 0) + 8 * s;
              const uint32_t al = tmem + a_col(b, c, be, 1) + 8 * s;
              const uint64_t bh = sdesc(bt + 32 * s), bl = sdesc(bt + 64 + 32 * s);
              umma_ts(d, ah, bh, IDESC, s > 0 ? 1u : 0u);
              umma_ts(d, al, bh, IDESC, 1u);
              umma_ts(d, ah, bl, IDESC, 1u);
            }
          }
        umma_commit(&mma_done[b]);
      }
      // every issued MMA has completed before tensor memory is released
      umma_commit(mma_final);
      volatile int no_abort = 0;
      mbar_wait(mma_final, 0, &no_abort);
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  } else if (warp == W_COEF) {
    // ---------------- coefficient tiles: A = a * inv, hi | lo along K ----------------
    // lane = source layer l; entry i = be * k + j of the row's 2k x L values
    const int ncoef = 2 * K * L;
    float cf[32];
    float inv = 0.f;
    auto fetch = [&](long long r) {
      const long long row = rg + r * nrg;
      const bool v = r < nrows && lane < L;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        cf[i] = (v && i < 2 * K) ? a.coeff[row * ncoef + (long long)i * L + lane] : 0.f;
      inv = v ? a.inv[row * a.inv_ld + lane] : 0.f;
    };
    fetch(0);
    for (long long r = 0; r < nrows && ok; ++r) {
      const int b = (int)(r & 1);
      if (r >= 2 && !warp_wait(&mma_done[b], (uint32_t)(((r >> 1) - 1) & 1), abort_flag, lane)) {
        ok = false;
        break;
      }
      if (lane < L) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (i < 2 * K) {
            const int be = i >= K ? 1 : 0, j = i - be * K;
            const float v = cf[i] * inv;
            const __nv_bfloat16 hi = __float2bfloat16_rn(v);
            const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
            uint8_t* t = btile + (size_t)(b * 2 + be) * 2048;
            *reinterpret_cast<__nv_bfloat16*>(t + swz(j, lane)) = hi;
            *reinterpret_cast<__nv_bfloat16*>(t + swz(j, 32 + lane)) = lo;
          }
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&b_full[b]);
      fetch(r + 1);
    }
  } else if (warp == W_STORE) {
    // ---------------- storer: staging rows -> u, sums of squares -> chan_ss ----------------
    __nv_bfloat16* out = (__nv_bfloat16*)a.mixed;
    for (long long r = 0; r < nrows && ok; ++r) {
      const int b = (int)(r & 1);
      const long long row = rg + r * nrg;
      if (!warp_wait(&o_full[b], (uint32_t)((r >> 1) & 1), abort_flag, lane)) { ok = false; break; }
      if (lane < 2 * K) {
        const int be = lane / K, j = lane - be * K;
        const __nv_bfloat16* src = otile + ((size_t)(b * 2 + be) * 16 + j) * g.OSTR;
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                         out + ((size_t)lane * a.N + row) * D + c0),
                     "r"(su32(src)), "r"((uint32_t)(g.W * 2))
                     : "memory");
        float v = 0.f;
        const float* rs = red + (size_t)b * NCV * 32 + be * 16 + j;
        for (int w = 0; w < NCV; ++w) v += rs[w * 32];
        a.chan_ss[(((size_t)row * 2 + be) * K + j) * g.CS + slice] = v;
      }
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_empty[b]);
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
  if (!ok && lane == 0) {
    *abort_flag = 1;
    atomicOr(flags, FLAG_TIMEOUT);
  }
  fence_before();
  __syncthreads();
  if (warp == W_MMA) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"((uint32_t)g.tmem_cols)
                 : "memory");
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

bool make_geo(const MixArgs& a, Geo& g) {
  if (a.D % 128) return false;
  g.CT = (a.D % 256 == 0) ? 2 : 1;
  g.W = 128 * g.CT;
  g.CS = a.D / g.W;
  if (g.CS > 8) return false;  // chan_ss holds at most 8 parts per (row, branch, channel)
  g.LP = a.L <= 16 ? 16 : 32;
  g.NCV = 4 * g.CT;
  g.OSTR = g.W + 8;
  g.a_cols = g.LP / 2;
  g.buf_cols = 4 * g.CT * g.a_cols + 2 * g.CT * 16;
  int cols = 32;
  while (cols < 2 * g.buf_cols) cols *= 2;
  g.tmem_cols = cols;
  const unsigned stage = (unsigned)a.L * g.W * 2;
  const unsigned btile = 2u * 2 * 2048;
  const unsigned otile = 2u * 2 * 16 * g.OSTR * 2;
  const unsigned redb = 2u * g.NCV * 32 * 4;
  const unsigned bars = (2 * MAX_NS + 13) * 8 + 16;
  g.off_b = 0;
  g.off_stage = btile;
  const unsigned budget = 227u * 1024 - 1024;  // 1 KB for aligning the base
  const unsigned fixed = btile + otile + redb + bars + 64;
  int ns = MAX_NS;
  while (ns > 2 && fixed + ns * ((stage + 127) / 128 * 128) > budget) --ns;
  if (fixed + ns * ((stage + 127) / 128 * 128) > budget) return false;
  g.NS = ns;
  g.off_out = g.off_stage + ns * ((stage + 127) / 128 * 128);
  g.off_out = (g.off_out + 127) / 128 * 128;
  g.off_red = g.off_out + otile;
  g.off_bar = (g.off_red + redb + 7) / 8 * 8;
  g.smem = g.off_bar + bars + 1024;
  return true;
}

}  // namespace mt

// Returns the number of column slices (the deferred norm's part count), or 0
// if the shape is outside this kernel's envelope (the caller then takes the
// mma.sync mixer).
int launch_mix_tmem(const MixArgs& a, cudaStream_t st, uint32_t* flags) {
  if (a.N <= 0 || a.k < 1 || a.k > 16 || a.L < 1 || a.L > 32 || !a.chan_ss) return 0;
  if ((uintptr_t)a.stash % 16 || a.ld_row % 8 || a.D % 8 || (uintptr_t)a.mixed % 16) return 0;
  mt::Geo g{};
  if (!mt::make_geo(a, g)) return 0;
  auto enc = mt::encode_fn();
  if (!enc) return 0;
  CUtensorMap map;
  cuuint64_t dims[3] = {(cuuint64_t)a.D, (cuuint64_t)a.L, (cuuint64_t)a.N};
  cuuint64_t strides[2] = {(cuuint64_t)a.D * 2, (cuuint64_t)a.ld_row * 2};
  cuuint32_t box[3] = {(cuuint32_t)g.W, (cuuint32_t)a.L, 1};
  cuuint32_t es[3] = {1, 1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.stash), dims, strides, box,
          es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return 0;
  if (cudaFuncSetAttribute(mt::mix_tmem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)g.smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long nrg = sms / g.CS;
  if (nrg < 1) nrg = 1;
  if (nrg > a.N) nrg = a.N;
  const int threads = (2 * g.NCV + 4) * 32;
  if (launch_k(mt::mix_tmem_kernel, dim3((unsigned)(nrg * g.CS)), dim3(threads), g.smem, st, map, a,
               g, flags) != cudaSuccess)
    return 0;
  return g.CS;
}

}  // namespace wm
