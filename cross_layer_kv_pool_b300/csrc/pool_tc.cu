// Pool mixer on the tensor cores (bf16 storage).
//
// Per token and branch b the mix is a small dense contraction
//   M^b [k x D] = A^b [k x L] . X^b [L x D],
//   A^b_{j,l} = a^b_{j,l} inv_l,     X^b_{l,t} = src_norm[b][l][t] h_l[t],
// followed by the channel RMSNorm of each row of M^b ("WhiteMatter: All-to-All
// Cross-Layer Connections via KV Mixing", 3 METHOD, "Cross-layer KV pool").
// At 1.3B widths it is 2kL*D = 1.4M MAC per token against 204 kB of HBM
// traffic, 13.8 flop/B: streaming at the HBM rate needs ~90 TFLOP/s, more than
// the fp32 FMA pipes deliver, so the contraction runs on bf16 mma.sync.
// A is split into hi + lo bf16 halves (~16 significant bits); X, the product
// of a stored bf16 state and its bf16 gain, is split exactly into hi + lo;
// three MMAs (hi.hi, hi.lo, lo.hi) keep the mix near fp32 accuracy.
//
// Layout of the work: D is cut into CS column slices of W <= 448 columns; a
// CTA owns one slice for a subset of the rows (rows rg, rg + nrg, ...). Its
// slice of both branches' source-norm gains stays resident in shared memory.
// One producer warp streams the states through a ring of 16-layer chunks
// (bulk TMA copies, one per layer, into padded rows so ldmatrix.trans is
// conflict-free). Each compute warp owns 32 columns (four n8 tiles) of both
// branches; the 16 x 8 accumulator tiles hold all k <= 16 channels. The
// compute warps also build each row's hi/lo bf16 A tile together, one row
// ahead (each its share, from coefficients prefetched a row earlier). Warps
// synchronise only through mbarriers, so they drift by up to a row and one
// warp's epilogue overlaps another's MMAs. Outputs go through a
// double-buffered shared tile that a storer warp writes out with one bulk copy
// per (branch, channel) row segment (full-line writes instead of 16-byte
// pieces of eight rows per warp store).
//
// The channel RMSNorm's factor needs sums of squares over all D columns, which
// no single CTA sees. The kernel therefore writes u = tau (.) m (the gained,
// not yet normalised channel) and, per row, branch, channel and slice, the
// slice's sum of squares of m; the consumer of the channels (the K/V
// projection, which is linear in its input) applies rsqrt(sum / D + eps) to
// its output rows. launch_mix_normalize produces c itself where a caller
// asks for it.
#include <mutex>

#include "kernels.h"

namespace wm {
namespace {

constexpr int NTW = 4;        // n8 tiles per compute warp (32 columns)
constexpr int MAXV = 4;       // tile entries per compute thread per row (2kL <= 4 * 32 * warps)
constexpr int MAX_WARPS = 14; // + producer + storer = 16 warps, 4 per SM sub-partition (128 registers)
constexpr int RS = 4;         // rows in the coefficient-tile ring (>= 4, see the row loop)

struct MixGeo {
  int CS;    // column slices
  int W;     // columns per CTA
  int LP;    // L rounded up to a multiple of 16 (MMA K)
  int SROW;  // padded row stride (elements) of staged states and gains
  int AST;   // padded row stride (elements) of the coefficient tiles
  int nstg;  // 16-layer chunks in the state ring
  int nwc;   // compute warps (W / 32)
  int OST;   // padded row stride (elements) of the output tiles
  unsigned off_stage, off_atile, off_ss, off_out, off_bar, smem;
};

__device__ __forceinline__ uint32_t su32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Bounded phase wait: false after ~4 s (the caller records a timeout flag).
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity) {
  unsigned long long t0 = 0;
  for (uint32_t it = 0;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (it == 0) t0 = t;
    else if (t - t0 > 4000000000ull) return false;
  }
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
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

__global__ void __launch_bounds__((MAX_WARPS + 2) * 32, 1)
    mix_tc_kernel(const MixArgs a, const MixGeo g, uint32_t* flags) {
  extern __shared__ __align__(128) uint8_t sm[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = blockIdx.x % g.CS;            // column slice
  const long long rg = blockIdx.x / g.CS;        // first row
  const long long nrg = gridDim.x / g.CS;        // row stride
  const int L = a.L, D = a.D, K = a.k, W = g.W, SROW = g.SROW, AST = g.AST, LP = g.LP;
  const int c0 = rank * W;
  const int nks = LP / 16;
  const int atile_elems = 2 * 2 * 16 * AST;
  __nv_bfloat16* gains = reinterpret_cast<__nv_bfloat16*>(sm);                // [2][LP][SROW]
  __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(sm + g.off_stage);  // [nstg][16][SROW]
  __nv_bfloat16* atile = reinterpret_cast<__nv_bfloat16*>(sm + g.off_atile);  // [RS][2][2][16][AST]
  float* red = reinterpret_cast<float*>(sm + g.off_ss);                       // [RS][nwc][32]
  uint32_t* sscnt = reinterpret_cast<uint32_t*>(red + RS * g.nwc * 32);       // [RS]
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + g.off_bar);               // [nstg]
  uint64_t* empty = full + g.nstg;                                            // [nstg]
  uint64_t* afull = empty + g.nstg;                                           // [RS]
  uint64_t* ofull = afull + RS;                                               // [2]
  uint64_t* oempty = ofull + 2;                                               // [2]
  __nv_bfloat16* otile = reinterpret_cast<__nv_bfloat16*>(sm + g.off_out);    // [2][2][k][OST]
  const int otile_elems = 2 * K * g.OST;
  const __nv_bfloat16* sn = (const __nv_bfloat16*)a.src_norm;

  // Resident gains of this slice (rows l >= L zero); zeroed ring, tiles and sums.
  {
    const int w8 = W / 8, per_b = LP * w8;
    for (int i = tid; i < 2 * per_b; i += blockDim.x) {
      const int be = i / per_b, rem = i - be * per_b, l = rem / w8, c8 = (rem - l * w8) * 8;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (l < L) v = *reinterpret_cast<const uint4*>(sn + ((size_t)be * a.sn_layers + l) * D + c0 + c8);
      *reinterpret_cast<uint4*>(gains + ((size_t)be * LP + l) * SROW + c8) = v;
    }
    for (unsigned o = g.off_stage + 16u * tid; o < g.off_bar; o += 16u * blockDim.x)
      *reinterpret_cast<uint4*>(sm + o) = make_uint4(0u, 0u, 0u, 0u);
  }
  if (tid == 0) {
    for (int i = 0; i < g.nstg; ++i) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&full[i])) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(&empty[i])), "r"(g.nwc)
                   : "memory");
    }
    for (int i = 0; i < RS; ++i)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(&afull[i])), "r"(g.nwc)
                   : "memory");
    for (int i = 0; i < 2; ++i) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(&ofull[i])), "r"(g.nwc)
                   : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&oempty[i])) : "memory");
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  // everything above touched only weights and shared memory
  pdl_wait();
  pdl_trigger();
  // A bounded wait of an earlier kernel of this call gave up: nothing has
  // been issued yet, so the CTA leaves at once (one wait limit per call).
  if (*(volatile const uint32_t*)flags & FLAG_TIMEOUT) return;

  bool ok = true;
  if (warp == g.nwc) {
    // ------------- producer: lane 0 streams the state chunks
    if (lane == 0) {
      const __nv_bfloat16* src = (const __nv_bfloat16*)a.stash;
      int q = 0;
      for (;; ++q) {
        const long long row = rg + (long long)(q / nks) * nrg;
        if (row >= a.N) break;
        const int ks = q % nks, st = q % g.nstg;
        if (q >= g.nstg) ok = tc_wait(su32(&empty[st]), (uint32_t)((q / g.nstg - 1) & 1));
        if (!ok) break;
        const int l0 = ks * 16, lc = min(16, L - l0);
        const uint32_t b = su32(&full[st]);
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b),
                     "r"((uint32_t)(lc * W * 2))
                     : "memory");
        const __nv_bfloat16* s0 = src + row * a.ld_row + (long long)l0 * D + c0;
        __nv_bfloat16* d0 = stage + (size_t)st * 16 * SROW;
        for (int l = 0; l < lc; ++l)
          asm volatile(
              "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
              "[%3];" ::"r"(su32(d0 + (size_t)l * SROW)),
              "l"(s0 + (long long)l * D), "r"((uint32_t)(W * 2)), "r"(b)
              : "memory");
      }
      // copies still in flight land before the CTA may exit
      for (int p = max(0, q - g.nstg); p < q; ++p)
        tc_wait(su32(&full[p % g.nstg]), (uint32_t)((p / g.nstg) & 1));
    }
    __syncwarp();
  } else if (warp == g.nwc + 1) {
    // ------------- storer: the row's output tile leaves by bulk copies, one per
    // (branch, channel) row segment of W columns
    __nv_bfloat16* out = (__nv_bfloat16*)a.mixed;
    long long it = 0;
    for (long long row = rg; row < a.N; row += nrg, ++it) {
      const int os = (int)(it & 1);
      if (ok) ok = tc_wait(su32(&ofull[os]), (uint32_t)((it >> 1) & 1));
      const __nv_bfloat16* ot = otile + (size_t)os * otile_elems;
      for (int idx = lane; idx < 2 * K; idx += 32)
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                         out + ((size_t)idx * a.N + row) * D + c0),
                     "r"(su32(ot + (size_t)idx * g.OST)), "r"((uint32_t)(W * 2))
                     : "memory");
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(su32(&oempty[os]));
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  } else {
    // ------------- compute warps
    const int gq = lane >> 2, tq = lane & 3;
    const __nv_bfloat16* cn = (const __nv_bfloat16*)a.chan_norm;
    const int wcol = warp * NTW * 8;  // first column of this warp within the slice
    // This warp's share of each row's coefficient tile: entries idx = tid + NC * i
    // (i < MAXV) of the row's 2kL values; tile offset (hi half) and source layer fixed.
    const int NC = g.nwc * 32, ncoef = 2 * K * L;
    uint32_t pk[MAXV];
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
      const int idx = tid + NC * i;
      const int be = idx / (K * L), j = (idx / L) % K, l = idx % L;
      pk[i] = idx < ncoef ? ((uint32_t)(((be * 2) * 16 + j) * AST + l) | ((uint32_t)l << 16))
                          : 0xffffffffu;
    }
    float pc[MAXV], pi[MAXV];
    auto fetch = [&](long long row) {
#pragma unroll
      for (int i = 0; i < MAXV; ++i) {
        const bool v = row < a.N && pk[i] != 0xffffffffu;
        pc[i] = v ? a.coeff[row * ncoef + tid + NC * i] : 0.f;
        pi[i] = v ? a.inv[row * a.inv_ld + (pk[i] >> 16)] : 0.f;
      }
    };
    auto convert = [&](long long it_dst) {  // prefetched values -> tile of iteration it_dst
      __nv_bfloat16* at = atile + (size_t)(it_dst % RS) * atile_elems;
#pragma unroll
      for (int i = 0; i < MAXV; ++i) {
        if (pk[i] != 0xffffffffu) {
          const float v = pc[i] * pi[i];
          const __nv_bfloat16 hi = __float2bfloat16_rn(v);
          const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
          const uint32_t o = pk[i] & 0xffffu;
          at[o] = hi;
          at[o + 16 * AST] = lo;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(su32(&afull[it_dst % RS]));
    };
    // channel-norm gains of this thread's outputs: [branch][n-tile][row half]
    uint32_t tau[2][NTW][2];
#pragma unroll
    for (int be = 0; be < 2; ++be)
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int j = gq + 8 * h;
          tau[be][nt][h] =
              j < K ? *reinterpret_cast<const uint32_t*>(cn + ((size_t)be * a.cn_channels + j) * D + c0 + wcol +
                                                         nt * 8 + 2 * tq)
                    : 0u;
        }
    float acc[2][NTW][4];
#pragma unroll
    for (int be = 0; be < 2; ++be)
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt) acc[be][nt][0] = acc[be][nt][1] = acc[be][nt][2] = acc[be][nt][3] = 0.f;
    const int lr = (lane & 7) + ((lane >> 3) & 1) * 8;  // ldmatrix.trans source row (layer)
    const int lc8 = (lane >> 4) * 8;                     // and column offset
    // Tiles run one row ahead of use: a warp converts row it + 1's share at the
    // start of row it, then waits for row it's tile (all warps' shares). A warp
    // at row it has seen row it - 1's tile complete, so every warp has started
    // row it - 2 and finished row it - 3: the slot written at row it (last used
    // by row it + 1 - RS) is free for RS >= 4.
    fetch(rg);
    convert(0);
    fetch(rg + nrg);
    int q = 0;
    long long it = 0;
    for (long long row = rg; row < a.N; row += nrg, ++it) {
      const int slot = (int)(it % RS);
      if (row + nrg < a.N) {
        convert(it + 1);
        fetch(row + 2 * nrg);
      }
      if (ok) ok = tc_wait(su32(&afull[slot]), (uint32_t)((it / RS) & 1));
      const __nv_bfloat16* at = atile + (size_t)slot * atile_elems;
      for (int ks = 0; ks < nks; ++ks, ++q) {
        const int st = q % g.nstg;
        if (ok) ok = tc_wait(su32(&full[st]), (uint32_t)((q / g.nstg) & 1));
        uint32_t A[2][2][4];
#pragma unroll
        for (int be = 0; be < 2; ++be)
#pragma unroll
          for (int hl = 0; hl < 2; ++hl)
            ldsm4(su32(at + ((size_t)(be * 2 + hl) * 16 + (lane & 15)) * AST + ks * 16 + (lane >> 4) * 8),
                  A[be][hl]);
        const __nv_bfloat16* sb = stage + (size_t)st * 16 * SROW + (size_t)lr * SROW + wcol + lc8;
        const __nv_bfloat16* gk0 = gains + (size_t)(ks * 16 + lr) * SROW + wcol + lc8;
        const __nv_bfloat16* gv0 = gk0 + (size_t)LP * SROW;
#pragma unroll
        for (int np = 0; np < NTW / 2; ++np) {
          uint32_t h[4], gk[4], gv[4], xk[2][4], xv[2][4];
          ldsm4t(su32(sb + np * 16), h);
          ldsm4t(su32(gk0 + np * 16), gk);
          ldsm4t(su32(gv0 + np * 16), gv);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            bmul2_split(h[i], gk[i], xk[0][i], xk[1][i]);
            bmul2_split(h[i], gv[i], xv[0][i], xv[1][i]);
          }
          // A_hi X_hi + A_hi X_lo + A_lo X_hi (A_lo X_lo is below 2^-16 relative)
#pragma unroll
          for (int t = 0; t < 3; ++t) {
            const int ha = t == 2 ? 1 : 0, hx = t == 1 ? 1 : 0;
            mma16816(acc[0][2 * np], A[0][ha], xk[hx][0], xk[hx][1]);
            mma16816(acc[0][2 * np + 1], A[0][ha], xk[hx][2], xk[hx][3]);
            mma16816(acc[1][2 * np], A[1][ha], xv[hx][0], xv[hx][1]);
            mma16816(acc[1][2 * np + 1], A[1][ha], xv[hx][2], xv[hx][3]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(su32(&empty[st]));
      }
      // this warp's sums of squares per (branch, channel) into its entry of the row's slot
      float* rw = red + ((size_t)slot * g.nwc + warp) * 32;
#pragma unroll
      for (int be = 0; be < 2; ++be)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float s = 0.f;
#pragma unroll
          for (int nt = 0; nt < NTW; ++nt)
            s += acc[be][nt][2 * h] * acc[be][nt][2 * h] + acc[be][nt][2 * h + 1] * acc[be][nt][2 * h + 1];
          s += __shfl_xor_sync(0xffffffffu, s, 1);
          s += __shfl_xor_sync(0xffffffffu, s, 2);
          if (tq == 0) rw[be * 16 + gq + 8 * h] = s;
        }
      // u = tau (.) m into the row's output tile (free once the storer has read
      // the tile of row it - 2)
      const int os = (int)(it & 1);
      if (it >= 2 && ok) ok = tc_wait(su32(&oempty[os]), (uint32_t)(((it >> 1) - 1) & 1));
      __nv_bfloat16* ot = otile + (size_t)os * otile_elems + wcol + 2 * tq;
#pragma unroll
      for (int be = 0; be < 2; ++be)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int j = gq + 8 * h;
          if (j < K) {
            __nv_bfloat16* orow = ot + (size_t)(be * K + j) * g.OST;
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt) {
              // bf16 -> fp32 is a 16-bit shift of the pair's halves
              const float tx = __uint_as_float(tau[be][nt][h] << 16);
              const float ty = __uint_as_float(tau[be][nt][h] & 0xffff0000u);
              const __nv_bfloat162 o =
                  __floats2bfloat162_rn(acc[be][nt][2 * h] * tx, acc[be][nt][2 * h + 1] * ty);
              *reinterpret_cast<__nv_bfloat162*>(orow + nt * 8) = o;
            }
          }
        }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(su32(&ofull[os]));
      // The last warp of the row adds the warps' sums and publishes the slice's
      // (the slot is reused at row it + RS, which no warp reaches before all
      // have left row it).
      __syncwarp();
      uint32_t last = 0;
      if (lane == 0) {
        __threadfence_block();
        last = atomicAdd(&sscnt[slot], 1u) == (uint32_t)(g.nwc - 1);
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        __threadfence_block();
        const float* rs = red + (size_t)slot * g.nwc * 32 + lane;
        float v = 0.f;
        for (int w = 0; w < g.nwc; ++w) v += rs[w * 32];
        const int be = lane >> 4, j = lane & 15;
        if (j < K) a.chan_ss[(((size_t)row * 2 + be) * K + j) * g.CS + rank] = v;
        if (lane == 0) atomicExch(&sscnt[slot], 0u);
      }
#pragma unroll
      for (int be = 0; be < 2; ++be)
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt)
          acc[be][nt][0] = acc[be][nt][1] = acc[be][nt][2] = acc[be][nt][3] = 0.f;
    }
  }
  if (!ok) atomicOr(flags, FLAG_TIMEOUT);
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
  if (a.D % (32 * CS)) return false;
  g.CS = CS;
  g.W = a.D / CS;
  if (g.W > 32 * MAX_WARPS) return false;
  g.nwc = g.W / 32;
  if (2 * a.k * a.L > MAXV * 32 * g.nwc) return false;
  g.LP = (a.L + 15) / 16 * 16;
  g.SROW = g.W % 64 == 0 ? g.W + 8 : g.W + 40;  // row stride = 16 B mod 128 B
  g.AST = g.LP + 8;
  g.OST = g.SROW;
  const unsigned gains = 2u * g.LP * g.SROW * 2, stage = 16u * g.SROW * 2;
  const unsigned atile = (unsigned)RS * 2 * 2 * 16 * g.AST * 2, ss = RS * (g.nwc * 32 + 1) * 4 + 12;
  const unsigned otile = 2u * 2 * a.k * g.OST * 2;
  const unsigned fixed = gains + atile + ss + otile + (RS + 4) * 8 + 160;
  const unsigned budget = 227u * 1024;
  if (fixed >= budget) return false;
  int nstg = (int)((budget - fixed) / (stage + 16));
  if (nstg > 8) nstg = 8;
  const int nks = g.LP / 16;
  if (nstg < 2 * nks && nstg < 4) return false;
  g.nstg = nstg;
  g.off_stage = gains;
  g.off_atile = g.off_stage + (unsigned)nstg * stage;
  g.off_ss = g.off_atile + atile;
  g.off_out = g.off_ss + (ss + 15) / 16 * 16;
  g.off_bar = g.off_out + otile;
  g.smem = g.off_bar + (2u * nstg + RS + 4) * 8;
  return g.smem <= budget;
}

}  // namespace

int launch_mix_tc(const MixArgs& a, cudaStream_t st, uint32_t* flags) {
  if (a.N <= 0 || a.k < 1 || a.k > 16 || a.L < 1 || a.L > 64) return 0;
  if (!a.chan_ss || (uintptr_t)a.stash % 16 || a.ld_row % 8 || (uintptr_t)a.src_norm % 16 ||
      (uintptr_t)a.chan_norm % 4 || (uintptr_t)a.mixed % 16)
    return 0;
  MixGeo g{};
  bool found = false;
  for (int cs = 1; cs <= 8 && !found; ++cs) found = mix_geo(a, cs, g);
  if (!found) return 0;
  if (cudaFuncSetAttribute(mix_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)g.smem) !=
      cudaSuccess)
    return 0;
  // persistent grid: every resident CTA (cached per shared-memory size and device)
  static std::mutex mu;
  static int cached_smem = -1, cached_dev = -1, cached_nwc = -1, cached_blocks = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  int blocks = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (cached_smem != (int)g.smem || cached_dev != dev || cached_nwc != g.nwc) {
      int per_sm = 0, sms = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mix_tc_kernel,
                                                        (g.nwc + 2) * 32, g.smem) != cudaSuccess ||
          cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          per_sm < 1) {
        cudaGetLastError();
        return 0;
      }
      cached_blocks = per_sm * sms;
      cached_smem = (int)g.smem;
      cached_dev = dev;
      cached_nwc = g.nwc;
    }
    blocks = cached_blocks;
  }
  long long nrg = blocks / g.CS;
  if (nrg < 1) nrg = 1;
  if (nrg > a.N) nrg = a.N;
  launch_k(mix_tc_kernel, dim3((unsigned)(nrg * g.CS)), dim3((g.nwc + 2) * 32), g.smem, st, a, g, flags);
  return cudaGetLastError() == cudaSuccess ? g.CS : 0;
}

void launch_mix_normalize(const MixArgs& a, int parts, cudaStream_t st) {
  if (a.N <= 0 || parts <= 0) return;
  launch_k(mix_normalize_kernel, dim3((unsigned)(2LL * a.k * a.N)), dim3(256), 0, st, a.mixed, a.chan_ss, parts, a.N,
                                                                    a.k, a.D, a.eps);
}

}  // namespace wm
