// Pool mixer on the tensor cores (bf16 storage), mma.sync.
//
// Per token and branch b the mix is a small dense contraction
//   M^b [k x D] = A^b [k x L] . X^b [L x D],
//   A^b_{j,l} = a^b_{j,l} inv_l,     X^b_{l,t} = src_norm[b][l][t] h_l[t],
// followed by the channel RMSNorm of each row of M^b ("WhiteMatter: All-to-All
// Cross-Layer Connections via KV Mixing", 3 METHOD, "Cross-layer KV pool").
// At 1.3B widths it is 2kL*D = 1.4M MAC per token against 204 kB of HBM
// traffic. The fp32 FMA pipes (35 TFMA/s measured) would need more time than
// HBM does; bf16 mma.sync (287 TMAC/s measured) needs about 60% of it even
// with three products per tile: A is split into hi + lo bf16 halves (~16
// significant bits) and X, the product of a stored bf16 state and its bf16
// gain, is split exactly into hi + lo; X_hi.A_hi + X_lo.A_hi + X_hi.A_lo keep
// the mix near fp32 accuracy. (The contraction is too narrow for tcgen05:
// with N = k <= 16 channels one M128 N16 K16 instruction costs ~100 cycles.)
//
// Work layout. D is cut into CS column slices of W = 32 * nwc columns; a CTA
// owns one slice for the rows rg, rg + nrg, ... Warp roles:
//   compute warps (nwc): each owns 32 columns (four n8 tiles) of both
//     branches; its source-norm gains live in registers in the B-fragment
//     layout for the whole kernel. Per row: ldmatrix the coefficient tile
//     (A, hi and lo) and the states (B, transposed), split gain x state into
//     hi + lo, 24 mma.sync per K16 step; then the epilogue: u = tau (.) m
//     (bf16) into a staging tile by stmatrix, and the sums of squares of m,
//     both with packed fp32x2 multiplies. The channel-norm gains tau sit in
//     a per-warp table in shared memory, read once per row: held in
//     registers they pushed the warp past 128 registers into spills
//     (0.465 ms against 0.431 ms per 8,192 rows);
//   feeder warp: lane 0 brings each row into a ring of NS stages: the
//     states with ONE four-dimensional TMA box {64 columns, LP layers, W/64
//     column blocks, 1 row} under the 128-byte swizzle (consecutive layers in
//     consecutive 128-byte rows: conflict-free for ldmatrix.trans; the layers
//     past L of the K padding arrive zero-filled), and the row's hi/lo
//     coefficient tile with one bulk copy. The tiles are built beforehand by
//     mix_atile_kernel: a feeder that computed them itself, sharing its
//     sub-partition's issue slots with busy compute warps, took ~2.3 us per
//     row for ~300 instructions;
//   storer warp: sends each row's staging tile out with ONE four-dimensional
//     TMA store {64 columns, 2k channel planes, W/64 blocks, 1 row} and sums
//     the compute warps' partial sums of squares into the slice's value.
// (Per-layer and per-channel bulk copies cost ~0.1 us each to issue: 28 of
// each per row limited an earlier version to ~3.5 us per row.)
// The channel RMSNorm factor needs sums over all D columns, which no CTA sees:
// the kernel writes u = tau (.) m and, per row, branch, channel and slice, the
// slice's sum of squares of m; the consumer of the channels (the K/V
// projection, linear in its input) applies rsqrt(sum / D + eps) to its output
// rows. launch_mix_normalize produces c itself where a caller asks for it.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kernels.h"

namespace wm {
namespace {

constexpr int NTW = 4;      // n8 tiles per compute warp (32 columns)
constexpr int MAX_CW = 14;  // compute warps (+ feeder + storer = 16 warps: 128 registers)
constexpr int NS = 4;       // stages (rows in flight): the row's states and coefficient tile
constexpr int NOB = 2;      // output staging tiles (rows being stored)

struct MixGeo {
  int CS;    // column slices
  int W;     // columns per CTA
  int nwc;   // compute warps (W / 32)
  int LP;    // L rounded up to 16 or 32 (MMA K)
  int AST;   // padded row stride (elements) of the coefficient tiles
  int NB;    // 64-column blocks per CTA (W / 64)
  unsigned state_bytes, stage_bytes, out_bytes;
  unsigned off_stage, off_out, off_red, off_tau, off_bar, smem;
};

constexpr unsigned long long WAIT_NS = 4000000000ull;  // 4 s bound on any wait
// Time limit of one suspended try_wait before it checks again: 100 ns was
// ~2.5% faster per launch than the hardware's default limit.
constexpr uint32_t SUSPEND_NS = 100;

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
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity), "r"(SUSPEND_NS)
      : "memory");
  return ok != 0;
}
// Spin wait of the storer (one lane, waiting on the compute warps): non-
// blocking tests, the clock read every 256 of them; false on timeout or when
// another warp already gave up. A suspended try_wait there resumed well after
// the phase had completed (~1,600 cycles late in shared-memory clock stamps).
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __noinline__ bool mbar_spin(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
  unsigned long long t0 = 0;
  for (uint32_t i = 0;; ++i) {
    if (mbar_test(b, parity)) return true;
    if ((i & 255u) == 255u) {
      if (*abort_flag) return false;
      const unsigned long long t = gtimer();
      if (t0 == 0) t0 = t;
      else if (t - t0 > WAIT_NS) return false;
    }
  }
}
// Bounded wait; false on timeout or when another warp already gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
  if (mbar_test(b, parity)) return true;  // the usual case: already complete, cheaper than try_wait
  if (mbar_try(b, parity)) return true;
  const unsigned long long t0 = gtimer();
  while (true) {
    if (mbar_try(b, parity)) return true;
    if (*abort_flag) return false;
    if (gtimer() - t0 > WAIT_NS) return false;
  }
}
// One lane waits (acquiring the completed phase), the warp learns the
// outcome; __syncwarp then orders the other lanes' reads after that acquire.
__device__ __forceinline__ bool warp_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                                          int lane) {
  int ok = 1;
  if (lane == 0) ok = mbar_wait(b, parity, abort_flag) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm4t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void stsm4(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2,
                                      uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr),
               "r"(r0), "r"(r1), "r"(r2), "r"(r3)
               : "memory");
}
// x*y of two bf16 pairs as an exact hi + lo pair of bf16 pairs: the product
// of two 8-bit significands has at most 16 bits, hi holds it rounded to 8
// bits and the rounding residual (at most 8 bits) is exact in lo.
__device__ __forceinline__ void bmul2_split(uint32_t x, uint32_t y, uint32_t& hi, uint32_t& lo) {
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(hi) : "r"(x), "r"(y));
  const uint32_t nhi = hi ^ 0x80008000u;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(lo) : "r"(x), "r"(y), "r"(nhi));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// The first product of an accumulator: D = A.B (no zeroing pass).
__device__ __forceinline__ void mma16816_first(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  const float z = 0.f;
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
}
// (x0, x1) * (y0, y1) with one packed fp32 multiply
__device__ __forceinline__ void fmul2(float x0, float x1, float y0, float y1, float& d0, float& d1) {
  asm("{\n\t.reg .b64 a, b, c;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mul.rn.f32x2 c, a, b;\n\tmov.b64 {%0, %1}, c;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(x0), "f"(x1), "f"(y0), "f"(y1));
}
// (s0, s1) += (x0, x1) * (x0, x1) with one packed fp32 fma
__device__ __forceinline__ void fsq2(float x0, float x1, float& s0, float& s1) {
  asm("{\n\t.reg .b64 a, c;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 c, {%0, %1};\n\t"
      "fma.rn.f32x2 c, a, a, c;\n\tmov.b64 {%0, %1}, c;\n\t}"
      : "+f"(s0), "+f"(s1)
      : "f"(x0), "f"(x1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Address of 16-byte chunk ``c16`` of 128-byte row ``row`` of a tile stored
// with the 128-byte swizzle (the layout TMA writes and reads).
__device__ __forceinline__ uint32_t swz128(uint32_t base, int row, int c16) {
  return base + (uint32_t)row * 128u + (uint32_t)((c16 ^ (row & 7)) << 4);
}
__device__ __forceinline__ void tma_load4(const CUtensorMap* map, uint64_t* bar, uint32_t dst, int c0,
                                          int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(map), "r"(su32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void tma_store4(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                           int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(map),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(su32(bar))
      : "memory");
}

// The mixer's per-row coefficient tiles: A^b_{j,l} = a^b_{j,l} inv_l split
// into bf16 hi + lo (hi = bf16(A), lo = bf16(A - hi)), laid out as the
// mixer's ldmatrix reads them, [2 b][2 hi/lo][16 j][40] (j >= k, l >= L and
// the 8 padding columns zero). One block of 128 threads per row; each thread
// writes pairs of entries.
__global__ void __launch_bounds__(128) mix_atile_kernel(const MixArgs a) {
  pdl_wait();
  pdl_trigger();
  const long long row = blockIdx.x;
  const int L = a.L, K = a.k;
  const float* cf = a.coeff + row * 2 * K * L;
  const float* iv = a.inv + row * a.inv_ld;
  uint32_t* out = reinterpret_cast<uint32_t*>((uint8_t*)a.atile + row * MIX_ATILE_BYTES);
  // 2 * 2 * 16 rows of 20 pairs
  for (int p = threadIdx.x; p < 2 * 2 * 16 * 20; p += blockDim.x) {
    const int rr = p / 20, l0 = (p - rr * 20) * 2;
    const int be = rr >> 5, hl = (rr >> 4) & 1, j = rr & 15;
    float v[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int l = l0 + e;
      float x = 0.f;
      if (j < K && l < L) {
        const float A = cf[(be * K + j) * L + l] * iv[l];
        const float hi = __bfloat162float(__float2bfloat16_rn(A));
        x = hl ? A - hi : hi;
      }
      v[e] = x;
    }
    out[p] = pack_bf16(v[0], v[1]);
  }
}

__global__ void __launch_bounds__((MAX_CW + 2) * 32, 1)
    mix_tc_kernel(const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmU,
                  const MixArgs a, const MixGeo g, uint32_t* flags) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwc = g.nwc, W_FEED = nwc, W_STORE = nwc + 1;
  const int slice = (int)(blockIdx.x % g.CS);
  const long long rg = blockIdx.x / g.CS, nrg = gridDim.x / g.CS;
  const int L = a.L, D = a.D, K = a.k, AST = g.AST, LP = g.LP, NB = g.NB;
  const int c0 = slice * g.W;
  const int nks = LP / 16;
  const long long nrows = rg < a.N ? (a.N - 1 - rg) / nrg + 1 : 0;  // rows of this CTA
  // stage s: the states, [NB blocks][LP layers] rows of 128 B (64 columns),
  // swizzled, then the row's coefficient tile [2 be][2 hi/lo][16 j][AST]
  const uint32_t stage0 = su32(sm + g.off_stage);
  // staging tile ob: [NB blocks][2k channel planes] rows of 128 B, swizzled,
  // then one spare 128-byte row that takes the padding channels k..15
  const uint32_t out0 = su32(sm + g.off_out);
  float* red = reinterpret_cast<float*>(sm + g.off_red);                      // [NOB][nwc][32]
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + g.off_bar);               // [NS]
  uint64_t* empty = full + NS;                                                // [NS]
  uint64_t* ofull = empty + NS;                                               // [NOB]
  uint64_t* oempty = ofull + NOB;                                             // [NOB]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(oempty + NOB);
  volatile int* stop = abort_flag + 1;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], nwc);
    }
    for (int i = 0; i < NOB; ++i) {
      mbar_init(&ofull[i], nwc);
      mbar_init(&oempty[i], 1);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmS) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmU) : "memory");
  }
  // everything above touched only shared memory
  pdl_wait();
  pdl_trigger();
  if (tid == 0) *stop = (*(volatile const uint32_t*)flags & FLAG_TIMEOUT) != 0;
  __syncthreads();
  // an earlier kernel of this call timed out: leave before issuing anything
  if (*stop) return;

  bool ok = true;
  if (warp < nwc) {
    // ---------------- compute warps ----------------
    const int gq = lane >> 2, tq = lane & 3;
    const int wcol = warp * NTW * 8;  // first column of this warp within the slice
    const __nv_bfloat16* sn = (const __nv_bfloat16*)a.src_norm;
    const __nv_bfloat16* cn = (const __nv_bfloat16*)a.chan_norm;
    // Source-norm gains in the B-fragment layout of ldmatrix.trans below:
    // gf[be][ks][np][i]: i = 0, 1 -> n-tile 2np (layers 2tq.., 2tq+8..),
    // i = 2, 3 -> n-tile 2np + 1; layers >= L are zero.
    uint32_t gf[2][2][2][4];
#pragma unroll
    for (int be = 0; be < 2; ++be)
#pragma unroll
      for (int ks = 0; ks < 2; ++ks)
#pragma unroll
        for (int np = 0; np < 2; ++np)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int nt = 2 * np + (i >> 1);
            const int l0 = ks * 16 + 2 * tq + (i & 1) * 8;
            const size_t col = (size_t)c0 + wcol + nt * 8 + gq;
            const size_t rowb = (size_t)be * a.sn_layers;
            const uint32_t x0 = l0 < L ? __bfloat16_as_ushort(sn[(rowb + l0) * D + col]) : 0u;
            const uint32_t x1 = l0 + 1 < L ? __bfloat16_as_ushort(sn[(rowb + l0 + 1) * D + col]) : 0u;
            gf[be][ks][np][i] = x0 | (x1 << 16);
          }
    // channel-norm gains of this thread's outputs, [branch][n-tile][row half]
    // as entry (be * 4 + nt) * 2 + h, kept in shared memory: [4][32 lanes] uint4
    uint32_t* taus = reinterpret_cast<uint32_t*>(sm + g.off_tau) + (size_t)warp * 512;
#pragma unroll
    for (int be = 0; be < 2; ++be)
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int j = gq + 8 * h, p = (be * 4 + nt) * 2 + h;
          taus[((p >> 2) * 32 + lane) * 4 + (p & 3)] =
              j < K ? *reinterpret_cast<const uint32_t*>(cn + ((size_t)be * a.cn_channels + j) * D + c0 +
                                                         wcol + nt * 8 + 2 * tq)
                    : 0u;
        }
    __syncwarp();
    // ldmatrix.trans rows: lane -> layer lr of the K16 step, 8-column chunk
    const int lr = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int blk = wcol >> 6;                       // 64-column block of this warp
    const int cchunk = ((wcol & 63) >> 3) + (lane >> 4);  // chunk of n-tile pair 0
    for (long long r = 0; r < nrows && ok; ++r) {
      const int s = (int)(r % NS), ob = (int)(r % NOB);
      if (!warp_wait(&full[s], (uint32_t)((r / NS) & 1), abort_flag, lane)) {
        ok = false;
        break;
      }
      const uint32_t st = stage0 + (uint32_t)s * g.stage_bytes;
      const __nv_bfloat16* at =
          reinterpret_cast<const __nv_bfloat16*>(sm + g.off_stage + (size_t)s * g.stage_bytes + g.state_bytes);
      float acc[2][NTW][4];
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        if (ks < nks) {
          uint32_t A[2][2][4];
#pragma unroll
          for (int be = 0; be < 2; ++be)
#pragma unroll
            for (int hl = 0; hl < 2; ++hl)
              ldsm4(su32(at + ((size_t)(be * 2 + hl) * 16 + (lane & 15)) * AST + ks * 16 + (lane >> 4) * 8),
                    A[be][hl]);
          const int row = blk * LP + ks * 16 + lr;  // 128-byte row of (block, layer)
#pragma unroll
          for (int np = 0; np < NTW / 2; ++np) {
            uint32_t h[4];
            ldsm4t(swz128(st, row, cchunk + 2 * np), h);
            uint32_t xk[2][4], xv[2][4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              bmul2_split(h[i], gf[0][ks][np][i], xk[0][i], xk[1][i]);
              bmul2_split(h[i], gf[1][ks][np][i], xv[0][i], xv[1][i]);
            }
            // A_hi X_hi (+) A_hi X_lo (+) A_lo X_hi; A_lo X_lo is below 2^-16 relative
            if (ks == 0) {
              mma16816_first(acc[0][2 * np], A[0][0], xk[0][0], xk[0][1]);
              mma16816_first(acc[0][2 * np + 1], A[0][0], xk[0][2], xk[0][3]);
              mma16816_first(acc[1][2 * np], A[1][0], xv[0][0], xv[0][1]);
              mma16816_first(acc[1][2 * np + 1], A[1][0], xv[0][2], xv[0][3]);
            } else {
              mma16816(acc[0][2 * np], A[0][0], xk[0][0], xk[0][1]);
              mma16816(acc[0][2 * np + 1], A[0][0], xk[0][2], xk[0][3]);
              mma16816(acc[1][2 * np], A[1][0], xv[0][0], xv[0][1]);
              mma16816(acc[1][2 * np + 1], A[1][0], xv[0][2], xv[0][3]);
            }
            mma16816(acc[0][2 * np], A[0][0], xk[1][0], xk[1][1]);
            mma16816(acc[0][2 * np + 1], A[0][0], xk[1][2], xk[1][3]);
            mma16816(acc[1][2 * np], A[1][0], xv[1][0], xv[1][1]);
            mma16816(acc[1][2 * np + 1], A[1][0], xv[1][2], xv[1][3]);
            mma16816(acc[0][2 * np], A[0][1], xk[0][0], xk[0][1]);
            mma16816(acc[0][2 * np + 1], A[0][1], xk[0][2], xk[0][3]);
            mma16816(acc[1][2 * np], A[1][1], xv[0][0], xv[0][1]);
            mma16816(acc[1][2 * np + 1], A[1][1], xv[0][2], xv[0][3]);
          }
        }
      }
      // the row's states and coefficient tile are consumed
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      // sums of squares of m per (branch, channel) over this warp's columns
      float ss[2][2];
#pragma unroll
      for (int be = 0; be < 2; ++be)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // even and odd columns summed apart (one packed fma per n-tile)
          float v0 = 0.f, v1 = 0.f;
#pragma unroll
          for (int nt = 0; nt < NTW; ++nt) fsq2(acc[be][nt][2 * h], acc[be][nt][2 * h + 1], v0, v1);
          float v = v0 + v1;
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          v += __shfl_xor_sync(0xffffffffu, v, 2);
          ss[be][h] = v;
        }
      // u = tau (.) m as bf16 pairs, the m16n8 fragments being stmatrix's
      uint32_t pk[2][NTW][2];
      uint32_t tau[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = *reinterpret_cast<const uint4*>(taus + (q * 32 + lane) * 4);
        tau[4 * q] = v.x; tau[4 * q + 1] = v.y; tau[4 * q + 2] = v.z; tau[4 * q + 3] = v.w;
      }
#pragma unroll
      for (int be = 0; be < 2; ++be)
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // bf16 -> fp32 is a 16-bit shift of the pair's halves
            const uint32_t tp = tau[(be * 4 + nt) * 2 + h];
            float ux, uy;
            fmul2(acc[be][nt][2 * h], acc[be][nt][2 * h + 1], __uint_as_float(tp << 16),
                  __uint_as_float(tp & 0xffff0000u), ux, uy);
            pk[be][nt][h] = pack_bf16(ux, uy);
          }
      // staging tile ob is free once the storer has read row r - NOB's
      if (r >= NOB && !warp_wait(&oempty[ob], (uint32_t)(((r / NOB) - 1) & 1), abort_flag, lane)) {
        ok = false;
        break;
      }
      {
        // matrix i of an x4 store: n-tile 2q + (i >> 1), channel rows 8 * (i & 1)..;
        // lane 8i + x gives the address of row x of matrix i: channel plane
        // be * k + j, block blk, chunk of the n-tile (channels >= k go to the
        // spare row)
        const uint32_t ot = out0 + (uint32_t)ob * g.out_bytes;
        const int i = lane >> 3, x = lane & 7;
        const int j = (i & 1) * 8 + x;
#pragma unroll
        for (int be = 0; be < 2; ++be)
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int nt = 2 * q + (i >> 1);
            const int c16 = ((wcol & 63) >> 3) + nt;
            const uint32_t addr = j < K ? swz128(ot, blk * 2 * K + be * K + j, c16)
                                        : ot + (uint32_t)(2 * K * NB) * 128u + (uint32_t)(c16 << 4);
            stsm4(addr, pk[be][2 * q][0], pk[be][2 * q][1], pk[be][2 * q + 1][0], pk[be][2 * q + 1][1]);
          }
      }
      if (tq == 0) {
        float* rw = red + ((size_t)ob * nwc + warp) * 32;
#pragma unroll
        for (int be = 0; be < 2; ++be)
#pragma unroll
          for (int h = 0; h < 2; ++h) rw[be * 16 + gq + 8 * h] = ss[be][h];
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&ofull[ob]);
    }
  } else if (warp == W_FEED) {
    // ---------------- feeder: lane 0 issues each row's two copies ----------------
    const uint8_t* tiles = (const uint8_t*)a.atile;
    long long issued = 0;
    if (lane == 0) {
      for (long long r = 0; r < nrows; ++r) {
        const int s = (int)(r % NS);
        const long long row = rg + r * nrg;
        if (r >= NS && !mbar_wait(&empty[s], (uint32_t)(((r / NS) - 1) & 1), abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t st = stage0 + (uint32_t)s * g.stage_bytes;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(&full[s])),
                     "r"(g.state_bytes + (uint32_t)MIX_ATILE_BYTES)
                     : "memory");
        // states: one box {64, LP, NB, 1}; layers >= L arrive as zeros
        tma_load4(&tmS, &full[s], st, 0, 0, c0 / 64, (int)row);
        bulk_load(st + g.state_bytes, tiles + row * MIX_ATILE_BYTES, (uint32_t)MIX_ATILE_BYTES, &full[s]);
        issued = r + 1;
      }
      // copies still in flight land before the CTA may exit
      volatile int no_abort = 0;
      for (long long r = issued - NS > 0 ? issued - NS : 0; r < issued; ++r)
        mbar_wait(&full[r % NS], (uint32_t)((r / NS) & 1), &no_abort);
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  } else if (warp == W_STORE) {
    // ---------------- storer: staging tile -> u, sums of squares -> chan_ss ----------------
    for (long long r = 0; r < nrows && ok; ++r) {
      const int ob = (int)(r % NOB);
      const long long row = rg + r * nrg;
      int okw = 1;
      if (lane == 0) okw = mbar_spin(&ofull[ob], (uint32_t)((r / NOB) & 1), abort_flag) ? 1 : 0;
      okw = __shfl_sync(0xffffffffu, okw, 0);
      __syncwarp();
      if (!okw) {
        ok = false;
        break;
      }
      if (lane == 0) tma_store4(&tmU, out0 + (uint32_t)ob * g.out_bytes, 0, 0, c0 / 64, (int)row);
      if (lane < 2 * K) {
        const int be = lane >= K ? 1 : 0, j = lane - be * K;
        float v = 0.f;
        const float* rs = red + (size_t)ob * nwc * 32 + be * 16 + j;
        for (int w = 0; w < nwc; ++w) v += rs[w * 32];
        a.chan_ss[(((size_t)row * 2 + be) * K + j) * g.CS + slice] = v;
      }
      if (lane == 0) {
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&oempty[ob]);
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
  if (!ok && lane == 0) {
    *abort_flag = 1;
    atomicOr(flags, FLAG_TIMEOUT);
  }
}

// c = s * u in place: one block per (branch, channel, row) of the deferred-norm output.
__global__ void __launch_bounds__(256) mix_normalize_kernel(void* mixed, const float* chan_ss,
                                                            int parts, int N, int k, int D,
                                                            float eps) {
  pdl_wait();
  pdl_trigger();
  const long long r = blockIdx.x;  // (b * k + j) * N + row
  const int row = (int)(r % N);
  const long long bj = r / N;
  const int j = (int)(bj % k), be = (int)(bj / k);
  const float* p = chan_ss + (((long long)row * 2 + be) * k + j) * parts;
  float s = 0.f;
  for (int c = 0; c < parts; ++c) s += p[c];
  const float sc = rsqrtf(s / (float)D + eps);
  __nv_bfloat16* x = (__nv_bfloat16*)mixed + r * D;
  for (int t = threadIdx.x; t < D; t += blockDim.x)
    x[t] = __float2bfloat16_rn(__bfloat162float(x[t]) * sc);
}

// Geometry for a slice count CS, or false if it does not fit.
bool mix_geo(const MixArgs& a, int CS, MixGeo& g) {
  if (a.D % (64 * CS)) return false;
  g.CS = CS;
  g.W = a.D / CS;
  if (g.W > 32 * MAX_CW) return false;
  g.nwc = g.W / 32;
  g.NB = g.W / 64;
  g.LP = a.L <= 16 ? 16 : 32;
  g.AST = 40;
  g.state_bytes = (unsigned)g.LP * g.W * 2;                                // multiple of 1024
  g.stage_bytes = (g.state_bytes + (unsigned)MIX_ATILE_BYTES + 1023u) / 1024u * 1024u;
  g.out_bytes = ((unsigned)(2 * a.k * g.NB + 1) * 128u + 1023u) / 1024u * 1024u;
  const unsigned redb = (unsigned)NOB * g.nwc * 32 * 4;
  const unsigned bars = (2 * NS + 2 * NOB) * 8 + 16;
  g.off_stage = 0;
  g.off_out = g.off_stage + NS * g.stage_bytes;
  g.off_red = g.off_out + NOB * g.out_bytes;
  g.off_tau = (g.off_red + redb + 15) / 16 * 16;
  g.off_bar = g.off_tau + (unsigned)g.nwc * 2048u;
  g.smem = g.off_bar + bars + 1024;  // + alignment of the base to 1024 bytes
  return g.smem <= 227u * 1024;
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

}  // namespace

int launch_mix_tc(const MixArgs& a, cudaStream_t st, uint32_t* flags) {
  if (a.N <= 0 || a.k < 1 || a.k > 16 || a.L < 1 || a.L > 32 || !a.atile) return 0;
  if ((uintptr_t)a.atile % 16) return 0;
  if (!a.chan_ss || (uintptr_t)a.stash % 16 || a.ld_row % 8 || (uintptr_t)a.src_norm % 4 ||
      (uintptr_t)a.chan_norm % 4 || (uintptr_t)a.mixed % 16 || a.D % 64)
    return 0;
  MixGeo g{};
  bool found = false;
  for (int cs = 1; cs <= 8 && !found; ++cs) found = mix_geo(a, cs, g);
  if (!found) return 0;
  auto enc = encode_fn();
  if (!enc) return 0;
  // states [N][L][D] (row stride ld_row) as {64 columns, L, D/64 blocks, N}
  CUtensorMap ms, mu;
  {
    cuuint64_t dims[4] = {64, (cuuint64_t)a.L, (cuuint64_t)(a.D / 64), (cuuint64_t)a.N};
    cuuint64_t strides[3] = {(cuuint64_t)a.D * 2, 128, (cuuint64_t)a.ld_row * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)g.LP, (cuuint32_t)g.NB, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (enc(&ms, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(a.stash), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return 0;
  }
  // u [2k][N][D] as {64 columns, 2k planes, D/64 blocks, N}
  {
    cuuint64_t dims[4] = {64, (cuuint64_t)(2 * a.k), (cuuint64_t)(a.D / 64), (cuuint64_t)a.N};
    cuuint64_t strides[3] = {(cuuint64_t)a.N * a.D * 2, 128, (cuuint64_t)a.D * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)(2 * a.k), (cuuint32_t)g.NB, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (enc(&mu, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.mixed, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return 0;
  }
  if (cudaFuncSetAttribute(mix_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)g.smem) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long nrg = sms / g.CS;
  if (nrg < 1) nrg = 1;
  if (nrg > a.N) nrg = a.N;
  // a failed launch is an error of the call, not a shape to hand to another mixer
  if (launch_k(mix_atile_kernel, dim3((unsigned)a.N), dim3(128), 0, st, a) != cudaSuccess) return -1;
  if (launch_k(mix_tc_kernel, dim3((unsigned)(nrg * g.CS)), dim3((g.nwc + 2) * 32), g.smem, st, ms, mu, a,
               g, flags) != cudaSuccess)
    return -1;
  return g.CS;
}

void launch_mix_normalize(const MixArgs& a, int parts, cudaStream_t st) {
  if (a.N <= 0 || parts <= 0) return;
  launch_k(mix_normalize_kernel, dim3((unsigned)(2LL * a.k * a.N)), dim3(256), 0, st, a.mixed, a.chan_ss, parts, a.N,
                                                                    a.k, a.D, a.eps);
}

}  // namespace wm
