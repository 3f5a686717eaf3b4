// Strictly causal channel attention on tcgen05 tensor cores (bf16, prefill).
//
// A CTA owns one KV head and one tile of up to 128 query rows (M): R
// consecutive token rows of one sequence times the G = Hq/Hkv query heads
// that read this KV head, packed in (row, head) order. The Q tile is one 3-D
// TMA box {64 dims, G heads, R rows} per 64-dim chunk, which lands exactly in
// that order. Keys and values stream in blocks of 128 positions of the channel.
//
//   warps 0, 3   TMA: the Q tile and K blocks (three-stage ring), V blocks
//                (two-stage ring), from separate threads so K runs ahead;
//   warp 1       tcgen05.mma, per key block j:
//                  S(j) = Q K_j^T   (K-major smem operands, fp32 into one of
//                                    two TMEM buffers),
//                  O += P(j) V_j    (P from TMEM, V an MN-major smem operand);
//                issued as O(j), S(j + 2), so that S(j + 1) is ready while
//                the softmax still works on block j;
//   warps 4-11   two softmax warpgroups, both one thread per query row (TMEM
//                lane): warpgroup w takes keys 64w .. 64w + 63 of every block.
//                The two threads of a row swap their maxima through shared
//                memory (a 64-thread named barrier per lane quarter), then
//                each writes P = 2^(s*scale - base) for its keys back into
//                TMEM as bf16 pairs over the S buffer's first 64 columns and
//                keeps its own part of the row sum. The base is raised lazily,
//                only when a row maximum exceeds it by more than 8 (P stays
//                below 2^8); then each thread rescales its half of the row's O
//                in TMEM. O is read once, at the end, each thread its half.
//                The control warpgroup gives registers to the softmax
//                warpgroups (setmaxnreg).
// Every wait is bounded: on timeout the CTA raises FLAG_TIMEOUT, stops issuing,
// drains its copies and MMAs, frees TMEM and returns. The two warps that share
// a lane quarter decide together whether to stop, so neither is left at a
// named barrier.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kernels.h"

namespace wm {
namespace atc {

constexpr int BQ = 128, BKEY = 128, NTHREADS = 384;  // 3 warpgroups: control, softmax x2
constexpr int NSK = 3, NSV = 2;                       // K and V ring stages
// Register split: 384 threads x 168 at launch = 64512; the control warpgroup
// keeps 88, each softmax warpgroup takes 208: 128 x 88 + 256 x 208 = 64512
// (per SM sub-partition, one control and two softmax warps: 32 x 504 <= 16384).
constexpr int REG_CTRL = 88, REG_SOFTMAX = 208;
constexpr unsigned long long WAIT_NS = 4000000000ull;

struct Params {
  const int* seq;
  const int* pos;
  void* out;          // [N][Hq][HD] bf16
  uint32_t* flags;
  int N, Hq, Hkv, G, rpt, nq, Tmax, k, channel, B;
  int nseq, tps, tiles;  // sequences of the call, tiles per sequence, all tiles (x KV heads)
  float scale_log2;   // log2(e) / sqrt(d)
};

// Tile ``idx`` of the persistent schedule. The tiles of one (sequence, KV
// head) are consecutive, so the CTAs working at the same time share that
// sequence's K/V blocks through L2 (a position-major order re-read the whole
// channel from DRAM once per tile row). Within a sequence the order is
// t = tps-1, tps-2, ... for the first half and 0, 1, ... for the second, so a
// CTA whose tiles lie half a sequence apart (148 CTAs, 8 tiles per sequence)
// alternates heavy and light tiles.
struct Tile {
  int b, hk, r0, nrows, sq, nkb;
  bool seq_ok;
};
// Warp-collective (every lane gets the same result).
__device__ __forceinline__ Tile tile_of(const Params& p, int idx, int lane) {
  Tile tl;
  const int pr = idx / p.tps, i = idx % p.tps, half = (p.tps + 1) / 2;
  const int t = i < half ? p.tps - 1 - i : i - half;
  tl.b = pr / p.Hkv;
  tl.hk = pr % p.Hkv;
  tl.r0 = tl.b * p.nq + t * p.rpt;
  tl.nrows = max(0, min(p.rpt, (tl.b + 1) * p.nq - tl.r0));
  int maxp = 0;
  for (int r = tl.r0 + lane; r < tl.r0 + tl.nrows; r += 32) maxp = max(maxp, p.pos[r]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) maxp = max(maxp, __shfl_xor_sync(0xffffffffu, maxp, o));
  maxp = min(maxp, p.Tmax);
  tl.sq = p.seq[tl.r0];
  tl.seq_ok = tl.sq >= 0 && tl.sq < p.B;
  tl.nkb = tl.seq_ok ? (maxp + BKEY - 1) / BKEY : 0;  // an invalid sequence reads no keys
  return tl;
}

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
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes)
               : "memory");
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
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try(b, parity)) return true;
  const unsigned long long t0 = gtimer();
  while (true) {
    if (mbar_try(b, parity)) return true;
    if (*abort_flag) return false;
    if (gtimer() - t0 > WAIT_NS) return false;
  }
}
__device__ __forceinline__ void tma3(const CUtensorMap* m, uint64_t* bar, void* dst, int c0, int c1,
                                     int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(su32(dst)),
      "l"(m), "r"(su32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void umma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                     uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          su32(bar))
      : "memory");
}
// 128-byte swizzled operand tile: rows of 128 B, 8-row groups 1024 B apart
// (SBO); for the MN-major value operand, LBO is the distance between its
// 64-column chunks.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(lbo >> 4) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// kind::f16, bf16 A/B, fp32 D, M = 128; b_mn: B is MN-major.
__host__ __device__ constexpr uint32_t idesc(int n, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn ? (1u << 16) : 0u) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(BQ >> 4) << 24);
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld32_nw(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// 64 consecutive columns of this thread's TMEM lane, one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* v) {
  uint32_t r[64];
  tmem_ld32_nw(taddr, r);
  tmem_ld32_nw(taddr + 32, r + 32);
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]),
      "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]),
      "r"(r[30]), "r"(r[31])
      : "memory");
}

// max(a, b, c) in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// 2^x on the special-function unit (inputs here are <= 8; results below the
// smallest normal flush to zero, far below bf16 resolution of the row sum)
__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// packed pairs of fp32 (one instruction for two lanes of arithmetic)
__device__ __forceinline__ unsigned long long f2pack(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2unpack(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b,
                                                    unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long fadd2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

template <int HD>
struct Smem {
  static constexpr int QB = BQ * HD * 2;     // one Q tile
  static constexpr int KB = BKEY * HD * 2;   // one K (or V) block
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + QB;          // NSK stages
  static constexpr int OFF_V = OFF_K + NSK * KB;    // NSV stages
  static constexpr int OFF_X = OFF_V + NSV * KB;    // max exchange [2][2][128], sums [2][128]
  static constexpr int OFF_BAR = OFF_X + 6 * 128 * 4;
  static constexpr int BYTES = 1024 + OFF_BAR + 256;
  // S buffers b = 0, 1 (128 fp32 columns each; P, bf16 pairs, overwrites the
  // first 64 after S is read) at b * 128, O (HD columns) at 256
  static constexpr int TMEM_COLS = 512;
};

// A from tensor memory (P), B from shared memory (V), D in tensor memory.
__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                        uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}

// Named barrier ``id`` over the 64 threads of two warps; the AND of ``v``.
__device__ __forceinline__ void bar_pair(int id) {
  asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
}
__device__ __forceinline__ bool bar_pair_and(int id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, 64, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id)
      : "memory");
  return r != 0;
}

// Persistent: CTA c takes tiles c, c + gridDim.x, ... The key blocks of all
// its tiles form one sequence (counter gb) that drives the K/V ring and the
// S/P buffers, so the next tile's Q, first K/V blocks and first two S
// products proceed while the softmax warps finish the current tile.
template <int HD>
__global__ void __launch_bounds__(NTHREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const Params p) {
  pdl_wait();
  pdl_trigger();
  using SM = Smem<HD>;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  float* xmax = (float*)(sm + SM::OFF_X);   // [block parity][warpgroup][row]
  float* xsum = xmax + 4 * 128;             // [warpgroup][row]
  uint64_t* bar = (uint64_t*)(sm + SM::OFF_BAR);
  uint64_t* q_full = bar + 0;
  uint64_t* q_empty = bar + 1;         // the tile's S products are done
  uint64_t* k_full = bar + 2;          // [NSK]
  uint64_t* k_empty = k_full + NSK;    // [NSK]
  uint64_t* v_full = k_empty + NSK;    // [NSV]
  uint64_t* v_empty = v_full + NSV;    // [NSV]
  uint64_t* s_full = v_empty + NSV;    // [buffer]: S of block gb is in TMEM
  uint64_t* p_full = s_full + 2;       // [buffer]: P of block gb written (8 warps arrive)
  uint64_t* pv_done = p_full + 2;      // O += P V of block gb complete
  uint64_t* o_free = pv_done + 1;      // the softmax warps have read the tile's O (8 arrive)
  uint64_t* mma_done = o_free + 1;
  uint32_t* tmem_holder = (uint32_t*)(mma_done + 1);
  volatile int* abort_flag = (volatile int*)(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 8);
    }
    for (int i = 0; i < NSK; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < NSV; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(pv_done, 1);
    mbar_init(o_free, 8);
    mbar_init(mma_done, 1);
    // A bounded wait of an earlier kernel of this call gave up: every role
    // stops before issuing anything, so one timeout costs one wait limit per
    // call rather than one per launch.
    *abort_flag = (*(volatile const uint32_t*)p.flags & FLAG_TIMEOUT) ? 1 : 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     su32(tmem_holder)),
                 "r"((uint32_t)SM::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_holder;
  // read by every thread here, before any role can have timed out, so that
  // the two warps of a lane quarter agree
  const bool entry_ok = *abort_flag == 0;
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REG_CTRL));
  if (warp == 0 || warp == 3) {
    // ---------------- TMA producers (lane 0; the warp computes tile metadata):
    // warp 0 the Q tiles and K blocks, warp 3 the V blocks, so that K runs
    // ahead of V by its deeper ring
    const bool kq = warp == 0;
    const int ns = kq ? NSK : NSV;
    uint64_t* full = kq ? k_full : v_full;
    uint64_t* empty = kq ? k_empty : v_empty;
    const CUtensorMap* map = kq ? &tmK : &tmV;
    uint8_t* ring = sm + (kq ? SM::OFF_K : SM::OFF_V);
    bool ok = entry_ok;
    int gb = 0, nqi = 0;  // K or V blocks issued, Q tiles issued
    uint32_t used = 0, lastk = 0;
    for (int idx = blockIdx.x; idx < p.tiles && ok; idx += gridDim.x) {
      const Tile tl = tile_of(p, idx, lane);
      if (lane == 0) {
        if (kq) {
          if (!tl.seq_ok) atomicOr(p.flags, FLAG_BAD_SEQ);
          // one Q buffer: the previous tile's S products have read it
          if (!mbar_wait(q_empty, (nqi & 1) ^ 1, abort_flag)) ok = false;
          if (ok) {
            // the box fills R*G rows of each 128-row operand chunk; rows past
            // them feed only accumulator rows that are never read back
            mbar_expect_tx(q_full, (uint32_t)((HD / 64) * p.G * p.rpt * 128));
            for (int c = 0; c < HD / 64; ++c)
              tma3(&tmQ, q_full, sm + SM::OFF_Q + c * BQ * 128, c * 64, tl.hk * p.G, tl.r0);
            ++nqi;
          }
        }
        const int zc = ((tl.sq * p.k) + p.channel) * p.Hkv + tl.hk;
        for (int j = 0; j < tl.nkb && ok; ++j, ++gb) {
          const int s = gb % ns;
          const uint32_t ph = (gb / ns) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, abort_flag)) { ok = false; break; }
          mbar_expect_tx(&full[s], (uint32_t)SM::KB);
          for (int c = 0; c < HD / 64; ++c)
            tma3(map, &full[s], ring + s * SM::KB + c * BKEY * 128, c * 64, j * BKEY, zc);
          used |= 1u << s;
          lastk = (lastk & ~(1u << s)) | (ph << s);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    if (lane == 0) {
      if (!ok) {
        *abort_flag = 1;
        atomicOr(p.flags, FLAG_TIMEOUT);
      }
      // Drain: every issued copy has landed before the CTA may exit.
      volatile int no_abort = 0;
      if (kq && nqi > 0) mbar_wait(q_full, (nqi - 1) & 1, &no_abort);
      for (int s = 0; s < ns; ++s)
        if (used & (1u << s)) mbar_wait(&full[s], (lastk >> s) & 1, &no_abort);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (lane 0) ----------------
    // tcgen05.mma operations of this thread execute in issue order, so
    // S(gb + 2) (issued after O += P(gb) V, into the same buffer) cannot
    // overwrite P(gb) before the product has read it.
    bool ok = entry_ok;
    int gb = 0, it = 0, o_waited = 0;
    constexpr uint32_t id_qk = idesc(BKEY, false);
    constexpr uint32_t id_pv = idesc(HD, true);
    for (int idx = blockIdx.x; idx < p.tiles && ok; idx += gridDim.x, ++it) {
      const Tile tl = tile_of(p, idx, lane);
      if (lane == 0) {
        const uint32_t sQ = su32(sm + SM::OFF_Q);
        if (!mbar_wait(q_full, it & 1, abort_flag)) ok = false;
        fence_after();
        const int g0 = gb;  // first block of this tile
        auto qk = [&](int j) -> bool {
          const int g = g0 + j;
          if (!mbar_wait(&k_full[g % NSK], (g / NSK) & 1, abort_flag)) return false;
          fence_after();
          const uint32_t sK = su32(sm + SM::OFF_K + (g % NSK) * SM::KB);
#pragma unroll
          for (int k16 = 0; k16 < HD / 16; ++k16) {
            const uint32_t off = (k16 >> 2) * BQ * 128 + (k16 & 3) * 32;
            const uint32_t offk = (k16 >> 2) * BKEY * 128 + (k16 & 3) * 32;
            umma(tmem + (g & 1) * 128, sdesc(sQ + off, 16), sdesc(sK + offk, 16), id_qk, k16 > 0);
          }
          commit(&s_full[g & 1]);
          commit(&k_empty[g % NSK]);
          return true;
        };
        auto pv = [&](int j) -> bool {
          const int g = g0 + j;
          if (!mbar_wait(&p_full[g & 1], (g >> 1) & 1, abort_flag)) return false;
          fence_after();
          const uint32_t sV = su32(sm + SM::OFF_V + (g % NSV) * SM::KB);
#pragma unroll
          for (int k16 = 0; k16 < BKEY / 16; ++k16)
            umma_ts(tmem + 256, tmem + (g & 1) * 128 + k16 * 8,
                    sdesc(sV + k16 * 16 * 128, BKEY * 128), id_pv, (j > 0 || k16 > 0) ? 1u : 0u);
          commit(pv_done);
          return true;
        };
        for (int j = 0; j < 2 && j < tl.nkb && ok; ++j) ok = qk(j);
        if (ok && tl.nkb > 0) {
          // the first product of this tile overwrites O: every earlier tile's O
          // must have been read back
          while (o_waited < it && ok) {
            if (!mbar_wait(o_free, o_waited & 1, abort_flag)) ok = false;
            ++o_waited;
          }
          fence_after();
        }
        for (int j = 0; j < tl.nkb && ok; ++j) {
          const int g = g0 + j;
          if (!mbar_wait(&v_full[g % NSV], (g / NSV) & 1, abort_flag)) { ok = false; break; }
          if (!pv(j)) { ok = false; break; }
          commit(&v_empty[g % NSV]);
          if (j + 2 < tl.nkb && !qk(j + 2)) { ok = false; break; }
        }
        if (ok) commit(q_empty);  // this tile's S products are issued and in order before
        gb = g0 + tl.nkb;
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    if (lane == 0) {
      if (!ok) {
        *abort_flag = 1;
        atomicOr(p.flags, FLAG_TIMEOUT);
      }
      commit(mma_done);
      volatile int no_abort = 0;
      mbar_wait(mma_done, 0, &no_abort);
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REG_SOFTMAX));
    // ------------- softmax warps: keys 64wg .. 64wg + 63 of each block, one
    // thread per query row
    constexpr int HK = BKEY / 2;         // keys per thread and block
    const int wg = (warp - 4) >> 2;
    const int quarter = warp & 3;        // TMEM lane quarter this warp may access
    const int pair = 1 + quarter;        // named barrier of the two warps of this quarter
    const int m = quarter * 32 + lane;   // query row of the tile = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const float sl2 = p.scale_log2;
    bool ok = entry_ok;
    int gb = 0;
    auto warp_wait = [&](uint64_t* bb, uint32_t parity) -> bool {
      int w = 1;
      if (lane == 0) w = mbar_wait(bb, parity, abort_flag) ? 1 : 0;
      return __shfl_sync(0xffffffffu, w, 0) != 0;
    };
    for (int idx = blockIdx.x; idx < p.tiles && ok; idx += gridDim.x) {
      const Tile tl = tile_of(p, idx, lane);
      const int mrows = tl.nrows * p.G;
      const bool valid = m < mrows;
      const int r = tl.r0 + (valid ? m / p.G : 0);
      const int h = tl.hk * p.G + (valid ? m % p.G : 0);
      int ps = valid ? p.pos[r] : 0;
      if (valid && (ps < 0 || ps >= p.Tmax)) {
        if (wg == 0) atomicOr(p.flags, FLAG_BAD_POS);
        ps = 0;
      }
      float mrun = -INFINITY, l = 0.f;  // exponent base (log2 units) and this half's row sum
      for (int j = 0; j < tl.nkb && ok; ++j, ++gb) {
        if (!bar_pair_and(pair, warp_wait(&s_full[gb & 1], (gb >> 1) & 1))) { ok = false; break; }
        fence_after();
        const uint32_t s_base = lane_base + (gb & 1) * 128;
        // This thread's HK scores, one TMEM load wait.
        const int nvis = min(max(ps - j * BKEY - HK * wg, 0), HK);
        float sv[HK];
        {
          uint32_t* ru = reinterpret_cast<uint32_t*>(sv);
#pragma unroll
          for (int c = 0; c < HK / 32; ++c) tmem_ld32_nw(s_base + HK * wg + c * 32, ru + 32 * c);
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        }
        if (!__all_sync(0xffffffffu, nvis == HK)) {
#pragma unroll
          for (int i = 0; i < HK; ++i)
            if (i >= nvis) sv[i] = -INFINITY;
        }
        float mx;
        {
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int i = 0; i < HK; i += 8)
#pragma unroll
            for (int q = 0; q < 4; ++q) m4[q] = fmax3(m4[q], sv[i + 2 * q], sv[i + 2 * q + 1]);
          mx = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3])) * sl2;  // scaled log2 units
        }
        // the row maximum over both halves (both threads then take the same
        // decisions below); the slot alternates with the block parity
        float* xm = xmax + (gb & 1) * 256;
        xm[wg * 128 + m] = mx;
        bar_pair(pair);
        mx = fmaxf(mx, xm[(wg ^ 1) * 128 + m]);
        float corr = 1.f;
        bool resc = false;
        if (mx > mrun + 8.f) {
          // O and l hold blocks < j taken against the old base (nothing if the
          // row had no visible key yet)
          if (j > 0 && mrun != -INFINITY) {
            resc = true;
            corr = ex2(mrun - mx);
          }
          mrun = mx;
        }
        const float base = mrun == -INFINITY ? 0.f : mrun;
        if (__any_sync(0xffffffffu, resc)) {  // the partner warp holds the same rows
          // O holds the products of blocks < j once the previous one landed
          if (!bar_pair_and(pair, warp_wait(pv_done, (gb - 1) & 1))) { ok = false; break; }
          fence_after();
          l *= corr;
#pragma unroll
          for (int c = 0; c < HD / 64; ++c) {
            uint32_t ro[32];
            const uint32_t oa = lane_base + 256 + (HD / 2) * wg + c * 32;
            tmem_ld32_nw(oa, ro);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
            for (int i = 0; i < 32; ++i) ro[i] = __float_as_uint(__uint_as_float(ro[i]) * corr);
            tmem_st32(oa, ro);
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        }
        // P = 2^(s * scale - base) as bf16 pairs over the buffer's columns
        // 32wg .. 32wg + 31 (16 at a time; the partner read its scores there
        // before the barrier above); this half's row sum in two packed sums.
        const unsigned long long sc2 = f2pack(sl2, sl2), nb2 = f2pack(-base, -base);
        unsigned long long rs2[2] = {0ull, 0ull};
#pragma unroll
        for (int c = 0; c < HK / 32; ++c) {
          uint32_t pw[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int i = 32 * c + 2 * e;
            float x0, x1;
            f2unpack(ffma2(f2pack(sv[i], sv[i + 1]), sc2, nb2), x0, x1);
            const float e0 = ex2(x0), e1 = ex2(x1);
            rs2[e & 1] = fadd2(rs2[e & 1], f2pack(e0, e1));
            __nv_bfloat162 hh = __floats2bfloat162_rn(e0, e1);
            pw[e] = *reinterpret_cast<uint32_t*>(&hh);
          }
          tmem_st16(s_base + (HK / 2) * wg + 16 * c, pw);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        {
          float a0, a1, b0, b1;
          f2unpack(rs2[0], a0, a1);
          f2unpack(rs2[1], b0, b1);
          l += (a0 + a1) + (b0 + b1);
        }
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[gb & 1]);
      }
      if (!ok) break;
      const bool have_o = tl.nkb > 0;
      if (have_o) {
        if (!bar_pair_and(pair, warp_wait(pv_done, (gb - 1) & 1))) { ok = false; break; }
        fence_after();
      }
      // the row sum over both halves, then O / l, this thread's HD/2 dims
      xsum[wg * 128 + m] = l;
      bar_pair(pair);
      l += xsum[(wg ^ 1) * 128 + m];
      const float inv = (valid && ps > 0 && l > 0.f) ? 1.f / l : 0.f;
      __nv_bfloat16* dst = (__nv_bfloat16*)p.out + ((long long)r * p.Hq + h) * HD + (HD / 2) * wg;
#pragma unroll
      for (int c = 0; c < HD / 64; ++c) {
        float o[32];
        if (have_o) tmem_ld32(lane_base + 256 + (HD / 2) * wg + c * 32, o);
        else
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0.f;
        if (valid) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 u;
            __nv_bfloat162* hh = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              hh[e] = __floats2bfloat162_rn(o[i + 2 * e] * inv, o[i + 2 * e + 1] * inv);
            *reinterpret_cast<uint4*>(dst + 32 * c + i) = u;
          }
        }
      }
      // O (and the sums slot) may be reused by the next tile
      fence_before();
      bar_pair(pair);
      if (lane == 0) mbar_arrive(o_free);
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      atomicOr(p.flags, FLAG_TIMEOUT);
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"((uint32_t)SM::TMEM_COLS)
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

bool map3(CUtensorMap* m, const void* ptr, cuuint64_t d0, cuuint64_t d1, cuuint64_t d2,
          cuuint64_t s1, cuuint64_t s2, cuuint32_t b0, cuuint32_t b1, cuuint32_t b2) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int HD>
cudaError_t run(const AttnArgs& a, int nq, cudaStream_t st) {
  using SM = Smem<HD>;
  const int G = a.Hq / a.Hkv;
  // rows per tile: a full 128-row tile, or a short sequence's rows
  int rpt = BQ / G;
  if (rpt > nq) rpt = nq;
  CUtensorMap mq, mk, mv;
  // q as [N][Hq][HD]: box {64 dims, G heads, rpt rows}
  if (!map3(&mq, a.q, HD, a.Hq, a.N, (cuuint64_t)HD * 2, (cuuint64_t)a.Hq * HD * 2, 64, G, rpt))
    return cudaErrorInvalidValue;
  // cache as [B*k*Hkv][Tmax][HD]: box {64 dims, 128 positions, 1}
  const cuuint64_t planes = (cuuint64_t)a.B * a.k * a.Hkv;
  if (!map3(&mk, a.cache_k, HD, a.Tmax, planes, (cuuint64_t)HD * 2, (cuuint64_t)a.Tmax * HD * 2, 64,
            BKEY, 1))
    return cudaErrorInvalidValue;
  if (!map3(&mv, a.cache_v, HD, a.Tmax, planes, (cuuint64_t)HD * 2, (cuuint64_t)a.Tmax * HD * 2, 64,
            BKEY, 1))
    return cudaErrorInvalidValue;
  Params p;
  p.seq = a.seq; p.pos = a.pos; p.out = a.out; p.flags = a.flags;
  p.N = a.N; p.Hq = a.Hq; p.Hkv = a.Hkv; p.G = G; p.rpt = rpt; p.nq = nq; p.Tmax = a.Tmax;
  p.k = a.k; p.channel = a.channel; p.B = a.B;
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
  p.nseq = a.N / nq;
  p.tps = (nq + rpt - 1) / rpt;
  p.tiles = p.nseq * p.tps * a.Hkv;
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<HD>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SM::BYTES);
  if (e != cudaSuccess) return e;
  int sms = 148, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  dim3 grid((unsigned)(p.tiles < sms ? p.tiles : sms));
  launch_k(attn_tc_kernel<HD>, dim3(grid), dim3(NTHREADS), SM::BYTES, st, mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace atc

// The tensor-core path takes structured calls (rows = B sequences of nq
// consecutive rows, one sequence per tile) whose G heads fit a 128-row tile.
bool attention_tc_supported(const AttnArgs& a, int nq) {
  if (nq <= 0 || a.N % nq) return false;
  const int G = a.Hq / a.Hkv;
  if (G > atc::BQ || (a.d != 64 && a.d != 128)) return false;
  if (((uintptr_t)a.q | (uintptr_t)a.cache_k | (uintptr_t)a.cache_v | (uintptr_t)a.out) & 15u)
    return false;
  return atc::encode_fn() != nullptr;
}

cudaError_t launch_attention_tc(const AttnArgs& a, int nq, cudaStream_t st) {
  return a.d == 128 ? atc::run<128>(a, nq, st) : atc::run<64>(a, nq, st);
}

}  // namespace wm
