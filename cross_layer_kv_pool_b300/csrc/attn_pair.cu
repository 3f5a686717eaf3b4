// Strictly causal channel attention on tcgen05 tensor cores (bf16, prefill):
// two query tiles per CTA that share every key and value block.
//
// A tile is up to 128 query rows (M): R consecutive token rows of one
// sequence times the G = Hq/Hkv query heads that read one KV head, packed in
// (row, head) order. A CTA takes a pair of adjacent tiles A, B of the same
// sequence and KV head (token rows r0 .. r0 + 2R), so that one K block and one
// V block (128 positions of the channel) feed both tiles. Tensor memory holds
// S_A, S_B (128 fp32 columns each; P, bf16 pairs, overwrites the first 64 of
// its tile's S after the softmax has read it) and the output accumulators
// O_A, O_B.
//
//   warp 0       takes the pairs (a global counter, longest first) and
//                publishes them to the other roles; TMA of the pair's two Q
//                tiles and of the K blocks through a three-stage ring;
//   warp 3       TMA of the V blocks through a two-stage ring;
//   warp 1       allocates tensor memory;
//   warps 4-7    tile A, warps 8-11 tile B: one thread per query row (TMEM
//                lane), all 128 keys of a block: row maximum, P = 2^(s*scale
//                - base) written back into TMEM as bf16 pairs, the row sum;
//                the base is raised lazily (only when a row maximum exceeds it
//                by more than 8, so P stays below 2^8), and then the thread
//                rescales its row of O in TMEM. The warpgroup meets at a named
//                barrier once P is written, and its leading lane issues the
//                tile's products itself: O_X += P_X(j) V_j, then S_X(j + 1).
//                The products of one thread execute in issue order, so
//                S_X(j + 1) cannot overwrite P_X(j) before it is read, and
//                when S_X(j + 1) is complete, O_X += P_X(j) V_j is too. The
//                two tiles run out of step: the tensor pipe computes one
//                tile's products while the other tile's softmax runs.
// Each tile waits on and releases every K and V block of the pair, read or
// not, so the rings' phases advance in step for both tiles.
// ("WhiteMatter: All-to-All Cross-Layer Connections via KV Mixing", 3 METHOD,
// "Per-layer channel selection": layer l reads channel l mod k; token i sees
// positions s < i.) Every wait is bounded: on timeout the CTA raises
// FLAG_TIMEOUT, stops issuing, drains its copies and products, frees tensor
// memory and returns; it also returns before issuing anything when an
// earlier kernel of the call has raised that flag.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kernels.h"

namespace wm {
namespace apr {

constexpr int BQ = 128, BKEY = 128, NTHREADS = 384;  // control, softmax A, softmax B warpgroups
constexpr int NSK = 3, NSV = 2;                       // K and V ring stages
// Register split: 384 threads x 168 at launch = 64512; the control warpgroup
// keeps 88, each softmax warpgroup takes 208: 128 x 88 + 256 x 208 = 64512.
constexpr int REG_CTRL = 88, REG_SOFTMAX = 208;
constexpr unsigned long long WAIT_NS = 4000000000ull;
// Roles that read the pair numbers warp 0 publishes: the V producer and the
// two softmax warpgroups' leading warps (one lane each).
constexpr int SCHED_READERS = 3;

struct Params {
  const int* seq;
  const int* pos;
  void* out;            // [N][Hq][HD] bf16
  uint32_t* flags;
  int N, Hq, Hkv, G, rpt, nq, Tmax, k, channel, B;
  int nseq, ppt, pairs;  // sequences, pairs per (sequence, KV head), all pairs
  int chunk_groups;      // (sequence, KV head) groups per chunk of the pair list
  // nullable: [0] the next pair of the dynamic schedule, [1] CTAs finished;
  // zero on entry, left zero (the last CTA to finish resets them)
  int* sched;
  float scale_log2;      // log2(e) / sqrt(d)
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
// One lane waits (acquiring the phase), the warp learns the outcome.
__device__ __forceinline__ bool warp_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                                          int lane) {
  int ok = 1;
  if (lane == 0) ok = mbar_wait(b, parity, abort_flag) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}
// This CTA's pair number for its iteration ``it``, published by warp 0 in a
// two-slot ring (warp-collective; false if the wait gave up).
__device__ __forceinline__ bool next_pair(uint64_t* full, uint64_t* empty, volatile int* slot, int it,
                                          volatile int* abort_flag, int lane, int& n) {
  int ok = 1, v = 0;
  if (lane == 0) {
    ok = mbar_wait(&full[it & 1], (it >> 1) & 1, abort_flag) ? 1 : 0;
    if (ok) {
      v = slot[it & 1];
      mbar_arrive(&empty[it & 1]);
    }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  n = __shfl_sync(0xffffffffu, v, 0);
  return ok != 0;
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
// A and B from shared memory.
__device__ __forceinline__ void umma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
// A from tensor memory (P), B from shared memory (V).
__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                        uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
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
// 32 consecutive fp32 columns of this thread's TMEM lane (no wait).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
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
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

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
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The persistent schedule. The (sequence, KV head) groups of pairs are cut
// into chunks of chunk_groups consecutive groups; list entry n lies in chunk
// n / (chunk_groups * ppt) and, within it, the heaviest pair (the last tiles,
// most keys) of every group comes first, then the next heaviest, and so on.
// With a pair counter (dynamic schedule) the list is one chunk and each CTA
// takes the next entry when it starts a pair: greedy longest-first list
// scheduling, whose last pairs are the shortest, so the CTAs finish close
// together (at 1.3B, group 15 of 64 sequences, this reads ~310 MB of K/V
// from DRAM per launch where L2-sized chunks read ~165 MB, yet it is the
// faster: the tail, not DRAM, sets the time). Without a counter the chunks
// hold about one pair per CTA (the CTAs working at one time share the
// chunk's K/V blocks through L2) and CTA c
// takes entry it * G + c in even rounds ``it`` and it * G + (G - 1 - c) in odd
// ones (G CTAs), so that a CTA that drew a heavy pair in one round draws a
// light one in the next.
__device__ __forceinline__ int pair_index(int it) {
  const int g = (int)gridDim.x, c = (int)blockIdx.x;
  return it * g + ((it & 1) ? g - 1 - c : c);
}
struct Pair {
  int hk, sq, r0[2], nrows[2], nkb[2];
  bool seq_ok;
};
// Warp-collective (every lane gets the same result).
__device__ __forceinline__ Pair pair_of(const Params& p, int n, int lane) {
  Pair pr;
  const int per_chunk = p.chunk_groups * p.ppt;
  const int g0 = (n / per_chunk) * p.chunk_groups, m = n % per_chunk;
  const int gsz = min(p.chunk_groups, p.nseq * p.Hkv - g0);  // groups in this chunk
  const int sh = g0 + m % gsz, t = p.ppt - 1 - m / gsz;
  const int b = sh / p.Hkv;
  pr.hk = sh % p.Hkv;
  pr.sq = p.seq[b * p.nq];
  pr.seq_ok = pr.sq >= 0 && pr.sq < p.B;
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    const int u0 = (2 * t + x) * p.rpt;                // first token row of the tile
    pr.r0[x] = b * p.nq + u0;
    pr.nrows[x] = max(0, min(p.rpt, p.nq - u0));
    int maxp = 0;
    for (int r = lane; r < pr.nrows[x]; r += 32) maxp = max(maxp, p.pos[pr.r0[x] + r]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) maxp = max(maxp, __shfl_xor_sync(0xffffffffu, maxp, o));
    maxp = min(maxp, p.Tmax);
    pr.nkb[x] = pr.seq_ok ? (maxp + BKEY - 1) / BKEY : 0;  // an invalid sequence reads no keys
  }
  return pr;
}

template <int HD>
struct Smem {
  static constexpr int QB = BQ * HD * 2;     // one Q tile
  static constexpr int KB = BKEY * HD * 2;   // one K (or V) block
  static constexpr int OFF_Q = 0;            // tiles A, B
  static constexpr int OFF_K = OFF_Q + 2 * QB;       // NSK stages
  static constexpr int OFF_V = OFF_K + NSK * KB;     // NSV stages
  static constexpr int OFF_BAR = OFF_V + NSV * KB;
  static constexpr int BYTES = 1024 + OFF_BAR + 512;
  static_assert(BYTES <= 232448, "dynamic shared memory above the per-block limit");
  // q_full, q_empty[2], k_full[NSK], k_empty[2][NSK], v_full[NSV],
  // v_empty[2][NSV], s_full[2], o_done[2], mma_done[2], sched_full[2],
  // sched_empty[2]; then the TMEM address, the abort flag, the two schedule
  // slots and the two tiles' pair numbers
  static constexpr int NBAR = 1 + 2 + 3 * NSK + 3 * NSV + 2 + 2 + 2 + 4;
  static_assert(NBAR * 8 + 24 <= 512, "barrier area");
  // TMEM columns: S_A at 0, S_B at 128 (P over the first 64 of each), O_A at
  // 256, O_B at 256 + HD
  static constexpr int TMEM_COLS = 512;
};

// Named barrier ``id`` over the 128 threads of one softmax warpgroup. The
// warp reconverges first (its leading lane may come from issuing products),
// so that all 32 lanes arrive together.
__device__ __forceinline__ void wg_sync(int id) {
  __syncwarp();
  asm volatile("barrier.sync.aligned %0, 128;" ::"r"(id) : "memory");
}
// The same barrier, returning the OR of ``v`` over the 128 threads, so that
// every thread of the warpgroup takes the same decision.
__device__ __forceinline__ bool wg_any(int id, bool v) {
  uint32_t r;
  __syncwarp();
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\t"
      "barrier.red.or.aligned.pred q, %2, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id)
      : "memory");
  return r != 0;
}

template <int HD>
__global__ void __launch_bounds__(NTHREADS, 1)
    attn_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const Params p) {
  pdl_wait();
  pdl_trigger();
  using SM = Smem<HD>;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  uint64_t* q_full = (uint64_t*)(sm + SM::OFF_BAR);
  uint64_t* q_empty = q_full + 1;          // [tile]: the tile's S products have read its Q
  uint64_t* k_full = q_empty + 2;          // [NSK]
  uint64_t* k_empty = k_full + NSK;        // [tile][NSK]: the tile is done with the stage's block
  uint64_t* v_full = k_empty + 2 * NSK;    // [NSV]
  uint64_t* v_empty = v_full + NSV;        // [tile][NSV]: the tile is done with the stage's block
  uint64_t* s_full = v_empty + 2 * NSV;    // [tile]: S_X of the next block is in TMEM
  uint64_t* o_done = s_full + 2;           // [tile]: the pair's products into O_X are complete
  uint64_t* mma_done = o_done + 2;         // [tile]: drain before exit
  uint64_t* sched_full = mma_done + 2;     // [2]: the slot holds this CTA's next pair number
  uint64_t* sched_empty = sched_full + 2;  // [2]: every reader has read the slot
  uint32_t* tmem_holder = (uint32_t*)(sched_empty + 2);
  volatile int* abort_flag = (volatile int*)(tmem_holder + 1);
  volatile int* sched_slot = abort_flag + 1;  // [2]
  volatile int* tile_pair = sched_slot + 2;   // [tile]: pair number, leader to warpgroup

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&q_empty[x], 1);
      mbar_init(&s_full[x], 1);
      mbar_init(&o_done[x], 1);
      mbar_init(&mma_done[x], 1);
      for (int i = 0; i < NSK; ++i) mbar_init(&k_empty[x * NSK + i], 1);
      for (int i = 0; i < NSV; ++i) mbar_init(&v_empty[x * NSV + i], 1);
    }
    for (int i = 0; i < NSK; ++i) mbar_init(&k_full[i], 1);
    for (int i = 0; i < NSV; ++i) mbar_init(&v_full[i], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sched_full[i], 1);
      mbar_init(&sched_empty[i], SCHED_READERS);
    }
    // A bounded wait of an earlier kernel of this call gave up: every role
    // stops before issuing anything (one wait limit per call).
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
  const bool entry_ok = *abort_flag == 0;
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REG_CTRL));
  if (warp == 0 || warp == 3) {
    // ---------------- TMA producers (lane 0): warp 0 takes the pairs, loads
    // the Q tiles and K blocks, warp 3 the V blocks
    const bool kq = warp == 0;
    const int ns = kq ? NSK : NSV;
    uint64_t* full = kq ? k_full : v_full;
    uint64_t* empty = kq ? k_empty : v_empty;  // [tile][ns]
    const CUtensorMap* map = kq ? &tmK : &tmV;
    uint8_t* ring = sm + (kq ? SM::OFF_K : SM::OFF_V);
    bool ok = entry_ok;
    int gb = 0, nqi = 0;  // K or V blocks issued, Q pairs issued
    uint32_t used = 0, lastph = 0;
    for (int it = 0; ok; ++it) {
      int idx = 0;
      if (kq) {
        // take the next pair and publish it to the other roles
        int okp = 1;
        if (lane == 0) {
          idx = p.sched ? atomicAdd(p.sched, 1) : pair_index(it);
          if (mbar_wait(&sched_empty[it & 1], ((it >> 1) & 1) ^ 1, abort_flag)) {
            sched_slot[it & 1] = idx;
            mbar_arrive(&sched_full[it & 1]);
          } else {
            okp = 0;
          }
        }
        idx = __shfl_sync(0xffffffffu, idx, 0);
        if (!__shfl_sync(0xffffffffu, okp, 0)) { ok = false; break; }
      } else if (!next_pair(sched_full, sched_empty, sched_slot, it, abort_flag, lane, idx)) {
        ok = false;
        break;
      }
      if (idx >= p.pairs) break;
      const Pair pr = pair_of(p, idx, lane);
      const int nkb = max(pr.nkb[0], pr.nkb[1]);
      if (lane == 0) {
        if (kq) {
          if (!pr.seq_ok) atomicOr(p.flags, FLAG_BAD_SEQ);
          // the Q buffers: both tiles' S products of the previous pair have read them
          for (int x = 0; x < 2 && ok; ++x)
            if (!mbar_wait(&q_empty[x], (nqi & 1) ^ 1, abort_flag)) ok = false;
          if (ok) {
            // each box fills R*G rows of a 128-row operand chunk; rows past
            // them feed only accumulator rows that are never read back
            mbar_expect_tx(q_full, (uint32_t)(2 * (HD / 64) * p.G * p.rpt * 128));
#pragma unroll
            for (int x = 0; x < 2; ++x)
              for (int c = 0; c < HD / 64; ++c)
                tma3(&tmQ, q_full, sm + SM::OFF_Q + x * SM::QB + c * BQ * 128, c * 64, pr.hk * p.G,
                     pr.r0[x]);
            ++nqi;
          }
        }
        const int zc = ((pr.sq * p.k) + p.channel) * p.Hkv + pr.hk;
        for (int j = 0; j < nkb && ok; ++j, ++gb) {
          const int s = gb % ns;
          const uint32_t ph = (gb / ns) & 1;
          // both tiles have released the block now in this stage (each
          // releases every block, read or not)
          for (int x = 0; x < 2 && ok; ++x)
            if (!mbar_wait(&empty[x * ns + s], ph ^ 1, abort_flag)) ok = false;
          if (!ok) break;
          mbar_expect_tx(&full[s], (uint32_t)SM::KB);
          for (int c = 0; c < HD / 64; ++c)
            tma3(map, &full[s], ring + s * SM::KB + c * BKEY * 128, c * 64, j * BKEY, zc);
          used |= 1u << s;
          lastph = (lastph & ~(1u << s)) | (ph << s);
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
        if (used & (1u << s)) mbar_wait(&full[s], (lastph >> s) & 1, &no_abort);
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REG_SOFTMAX));
    // ------------- softmax warpgroups: warpgroup x owns tile x, one thread
    // per query row (TMEM lane), all 128 keys of each block. Its leader (lane
    // 0 of its first warp) takes the pair numbers and issues the tile's
    // products: S_X(0), then per block O_X += P_X(j) V_j and S_X(j + 1).
    const int x = (warp - 4) >> 2;
    const int quarter = warp & 3;        // TMEM lane quarter this warp may access
    const bool lead_warp = quarter == 0;
    const bool leader = lead_warp && lane == 0;
    const int bar_id = 1 + x;            // the warpgroup's named barrier
    const int m = quarter * 32 + lane;   // query row of the tile = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t s_base = lane_base + x * 128;
    const uint32_t o_base = lane_base + 256 + x * HD;
    const float sl2 = p.scale_log2;
    constexpr uint32_t id_qk = idesc(BKEY, false);
    constexpr uint32_t id_pv = idesc(HD, true);
    const uint32_t sQ = su32(sm + SM::OFF_Q + x * SM::QB);
    bool lead_ok = entry_ok;  // the leader's waits have all succeeded
    bool issued = false;      // the leader has issued products (drain at exit)
    int cs = 0, gk = 0;       // S_X phases consumed; the pair's first block in the CTA's sequence
    // S_X = Q_X K^T of the block in K stage ``ks`` (leader only)
    auto issue_qk = [&](int ks) {
      const uint32_t sK = su32(sm + SM::OFF_K + ks * SM::KB);
#pragma unroll
      for (int k16 = 0; k16 < HD / 16; ++k16) {
        const uint32_t off = (k16 >> 2) * BQ * 128 + (k16 & 3) * 32;
        const uint32_t offk = (k16 >> 2) * BKEY * 128 + (k16 & 3) * 32;
        umma_ss(tmem + x * 128, sdesc(sQ + off, 16), sdesc(sK + offk, 16), id_qk, k16 > 0);
      }
      commit(&s_full[x]);
      commit(&k_empty[x * NSK + ks]);
    };
    for (int it = 0;; ++it) {
      // ---- the pair: the leader's warp takes its number and issues S_X(0)
      int idx = 0;
      Pair pr;
      if (lead_warp) {
        if (lead_ok && !next_pair(sched_full, sched_empty, sched_slot, it, abort_flag, lane, idx))
          lead_ok = false;
        if (lead_ok && idx < p.pairs) {
          pr = pair_of(p, idx, lane);
          if (lane == 0) {
            tile_pair[x] = idx;
            const int nkb = max(pr.nkb[0], pr.nkb[1]);
            const int nkbx = x ? pr.nkb[1] : pr.nkb[0];
            if (!mbar_wait(q_full, it & 1, abort_flag)) lead_ok = false;
            // every block of the pair is waited on and released by both
            // tiles, read or not: the stages' phases advance in step
            if (lead_ok && nkb > 0 && !mbar_wait(&k_full[gk % NSK], (gk / NSK) & 1, abort_flag))
              lead_ok = false;
            if (lead_ok) {
              fence_after();
              if (nkbx > 0) issue_qk(gk % NSK);
              else if (nkb > 0) mbar_arrive(&k_empty[x * NSK + gk % NSK]);
              if (nkbx <= 1) commit(&q_empty[x]);
              issued = true;
            }
          }
          lead_ok = __shfl_sync(0xffffffffu, lead_ok ? 1 : 0, 0) != 0;
        }
      }
      const bool end = lead_warp && lane == 0 && lead_ok && idx >= p.pairs;
      if (wg_any(bar_id, (leader && !lead_ok) || end || *abort_flag)) break;
      if (!lead_warp) pr = pair_of(p, tile_pair[x], lane);
      const int nkb = max(pr.nkb[0], pr.nkb[1]);
      const int nkbx = x ? pr.nkb[1] : pr.nkb[0];
      const int mrows = (x ? pr.nrows[1] : pr.nrows[0]) * p.G;
      const bool valid = m < mrows;
      const int r = (x ? pr.r0[1] : pr.r0[0]) + (valid ? m / p.G : 0);
      const int h = pr.hk * p.G + (valid ? m % p.G : 0);
      int ps = valid ? p.pos[r] : 0;
      if (valid && (ps < 0 || ps >= p.Tmax)) {
        atomicOr(p.flags, FLAG_BAD_POS);
        ps = 0;
      }
      float mrun = -INFINITY, l = 0.f;  // exponent base (log2 units) and the row sum
      bool stop = false;
      for (int j = 0; j < nkbx; ++j, ++cs) {
        // S_X(j) is in TMEM: the leader waits, the warpgroup follows
        if (leader && lead_ok && !mbar_wait(&s_full[x], cs & 1, abort_flag)) lead_ok = false;
        if (wg_any(bar_id, (leader && !lead_ok) || *abort_flag)) { stop = true; break; }
        fence_after();
        float sv[BKEY];
        {
          uint32_t* ru = reinterpret_cast<uint32_t*>(sv);
#pragma unroll
          for (int c = 0; c < BKEY / 32; ++c) tmem_ld32(s_base + c * 32, ru + 32 * c);
          tmem_wait_ld();
        }
        // keys visible to this row in the block; rows past the tile's last
        // query row are never stored, so they skip the mask
        const int nvis = valid ? min(max(ps - j * BKEY, 0), BKEY) : BKEY;
        if (!__all_sync(0xffffffffu, nvis == BKEY)) {
#pragma unroll
          for (int i = 0; i < BKEY; ++i)
            if (i >= nvis) sv[i] = -INFINITY;
        }
        float mx;
        {
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int i = 0; i < BKEY; i += 8)
#pragma unroll
            for (int q = 0; q < 4; ++q) m4[q] = fmax3(m4[q], sv[i + 2 * q], sv[i + 2 * q + 1]);
          mx = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3])) * sl2;  // scaled log2 units
        }
        float corr = 1.f;
        bool resc = false;
        if (mx > mrun + 8.f) {
          // O and l hold blocks < j taken against the old base (nothing if the
          // row had no visible key yet); O_X += P_X(j - 1) V is complete
          // because S_X(j), issued after it by the same thread, is
          if (j > 0 && mrun != -INFINITY) {
            resc = true;
            corr = ex2(mrun - mx);
          }
          mrun = mx;
        }
        const float base = mrun == -INFINITY ? 0.f : mrun;
        if (__any_sync(0xffffffffu, resc)) {
          l *= corr;
#pragma unroll 1
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t ro[32];
            tmem_ld32(o_base + c * 32, ro);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) ro[i] = __float_as_uint(__uint_as_float(ro[i]) * corr);
            tmem_st32(o_base + c * 32, ro);
          }
        }
        // P = 2^(s * scale - base) as bf16 pairs over the buffer's first 64
        // columns, 32 at a time; the row sum in two packed sums
        const unsigned long long sc2 = f2pack(sl2, sl2), nb2 = f2pack(-base, -base);
        unsigned long long rs2[2] = {0ull, 0ull};
#pragma unroll
        for (int c = 0; c < BKEY / 64; ++c) {
          uint32_t pw[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int i = 64 * c + 2 * e;
            float x0, x1;
            f2unpack(ffma2(f2pack(sv[i], sv[i + 1]), sc2, nb2), x0, x1);
            const float e0 = ex2(x0), e1 = ex2(x1);
            rs2[e & 1] = fadd2(rs2[e & 1], f2pack(e0, e1));
            pw[e] = pack_bf16(e0, e1);
          }
          tmem_st32(s_base + 32 * c, pw);
        }
        tmem_wait_st();
        {
          float a0, a1, b0, b1;
          f2unpack(rs2[0], a0, a1);
          f2unpack(rs2[1], b0, b1);
          l += (a0 + a1) + (b0 + b1);
        }
        // P_X(j) and any rescaled O_X are in TMEM
        fence_before();
        wg_sync(bar_id);
        if (leader && lead_ok) {
          fence_after();
          const int g = gk + j;
          if (!mbar_wait(&v_full[g % NSV], (g / NSV) & 1, abort_flag)) {
            lead_ok = false;
          } else {
            const uint32_t sV = su32(sm + SM::OFF_V + (g % NSV) * SM::KB);
#pragma unroll
            for (int k16 = 0; k16 < BKEY / 16; ++k16)
              umma_ts(tmem + 256 + x * HD, tmem + x * 128 + k16 * 8,
                      sdesc(sV + k16 * 16 * 128, BKEY * 128), id_pv, (j > 0 || k16 > 0) ? 1u : 0u);
            commit(&v_empty[x * NSV + g % NSV]);
            if (j == nkbx - 1) commit(&o_done[x]);
            if (j + 1 < nkb) {
              // S_X(j + 1) (after the product that reads P_X(j): one thread's
              // products execute in issue order)
              if (!mbar_wait(&k_full[(g + 1) % NSK], ((g + 1) / NSK) & 1, abort_flag)) {
                lead_ok = false;
              } else if (j + 1 < nkbx) {
                fence_after();
                issue_qk((g + 1) % NSK);
              } else {
                mbar_arrive(&k_empty[x * NSK + (g + 1) % NSK]);  // a block this tile skips
              }
            }
            if (j + 2 == nkbx) commit(&q_empty[x]);  // those were the pair's last S products
          }
        }
      }
      if (stop) break;
      if (leader && lead_ok) {
        if (nkbx == 0) commit(&o_done[x]);  // nothing issued: keeps one phase per pair
        // the blocks this tile skips (past its last visible key), waited on
        // and released in the order the other tile reads them (V_j, then
        // K_(j+1); K_nkbx was taken above or in the prologue), so that
        // neither tile holds back a block the other needs first
        for (int j = nkbx; j < nkb && lead_ok; ++j) {
          const int g = gk + j;
          if (!mbar_wait(&v_full[g % NSV], (g / NSV) & 1, abort_flag)) {
            lead_ok = false;
            break;
          }
          mbar_arrive(&v_empty[x * NSV + g % NSV]);
          if (j + 1 < nkb) {
            if (!mbar_wait(&k_full[(g + 1) % NSK], ((g + 1) / NSK) & 1, abort_flag)) {
              lead_ok = false;
              break;
            }
            mbar_arrive(&k_empty[x * NSK + (g + 1) % NSK]);
          }
        }
        if (lead_ok && !mbar_wait(&o_done[x], it & 1, abort_flag)) lead_ok = false;
      }
      // the pair's products into O_X are complete
      if (wg_any(bar_id, (leader && !lead_ok) || *abort_flag)) break;
      fence_after();
      gk += nkb;
      const float inv = (valid && ps > 0 && l > 0.f) ? 1.f / l : 0.f;
      __nv_bfloat16* dst = (__nv_bfloat16*)p.out + ((long long)r * p.Hq + h) * HD;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t o[32];
        if (nkbx > 0) {
          tmem_ld32(o_base + c * 32, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        if (valid) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 u;
            u.x = pack_bf16(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv);
            u.y = pack_bf16(__uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv);
            u.z = pack_bf16(__uint_as_float(o[i + 4]) * inv, __uint_as_float(o[i + 5]) * inv);
            u.w = pack_bf16(__uint_as_float(o[i + 6]) * inv, __uint_as_float(o[i + 7]) * inv);
            *reinterpret_cast<uint4*>(dst + 32 * c + i) = u;
          }
        }
      }
      // the next pair's first product into O_X is issued after the next
      // block barrier, which every thread reaches after these reads
      fence_before();
    }
    if (leader) {
      if (!lead_ok) {
        *abort_flag = 1;
        atomicOr(p.flags, FLAG_TIMEOUT);
      }
      // Drain: no product of this tile is in flight when the CTA exits.
      if (issued) {
        commit(&mma_done[x]);
        volatile int no_abort = 0;
        mbar_wait(&mma_done[x], 0, &no_abort);
      }
    }
  }
  fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && p.sched) {
    // every pair number this CTA will take is taken; the last CTA to get
    // here leaves the counters zero for the next launch
    __threadfence();
    if (atomicAdd(p.sched + 1, 1) == (int)gridDim.x - 1) {
      p.sched[0] = 0;
      p.sched[1] = 0;
    }
  }
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
  // tiles per sequence: as few as hold its nq rows at <= 128/G rows each,
  // made even so that they pair up; rows spread evenly over them
  const int cap = BQ / G;
  int tiles = (nq + cap - 1) / cap;
  tiles += tiles & 1;
  const int rpt = (nq + tiles - 1) / tiles;
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
  p.ppt = tiles / 2;
  p.pairs = p.nseq * p.ppt * a.Hkv;
  p.sched = (a.counters && a.counter_elems >= 2) ? a.counters : nullptr;
  cudaError_t e = cudaFuncSetAttribute(attn_pair_kernel<HD>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SM::BYTES);
  if (e != cudaSuccess) return e;
  int sms = 148, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  dim3 grid((unsigned)(p.pairs < sms ? p.pairs : sms));
  // dynamic: one chunk, longest first over all groups (the last pairs handed
  // out are the shortest); static: about one pair per CTA per chunk
  const int per_cta = (int)grid.x / p.ppt > 1 ? (int)grid.x / p.ppt : 1;
  p.chunk_groups = p.sched ? p.nseq * a.Hkv : per_cta;
  launch_k(attn_pair_kernel<HD>, dim3(grid), dim3(NTHREADS), SM::BYTES, st, mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace apr

// The tensor-core path takes structured calls (rows = sequences of nq
// consecutive rows) whose G heads fit a 128-row tile.
bool attention_tc_supported(const AttnArgs& a, int nq) {
  if (nq <= 0 || a.N % nq) return false;
  const int G = a.Hq / a.Hkv;
  if (G > apr::BQ || (a.d != 64 && a.d != 128)) return false;
  if (((uintptr_t)a.q | (uintptr_t)a.cache_k | (uintptr_t)a.cache_v | (uintptr_t)a.out) & 15u)
    return false;
  return apr::encode_fn() != nullptr;
}

cudaError_t launch_attention_pair(const AttnArgs& a, int nq, cudaStream_t st) {
  return a.d == 128 ? apr::run<128>(a, nq, st) : apr::run<64>(a, nq, st);
}

}  // namespace wm
