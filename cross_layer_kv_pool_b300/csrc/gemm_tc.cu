// Tensor-core GEMM engine for bf16 operands on sm_103a (tcgen05 + TMA + TMEM).
//
//   C[b][m][n] = epilogue( sum_k A[b][m][k] * B[b][n][k] ),  fp32 accumulation
//
// Persistent kernel, one CTA per SM, 192 threads in three roles:
//   warp 0      one lane issues TMA loads of 128x64 A and BNx64 B tiles (128-byte
//               swizzle) into a ring of shared-memory stages;
//   warp 1      one lane issues tcgen05.mma (M=128, N=BN, K=16) into one of two
//               TMEM accumulators, committing stage releases and tile completion
//               to mbarriers; the warp also owns the TMEM allocation;
//   warps 2-5   read the accumulator rows back with tcgen05.ld (each warp owns
//               the 32 TMEM lanes of its quarter), apply the fused epilogue and
//               store to global memory, then hand the accumulator back.
// Every mbarrier wait is bounded: on timeout the kernel raises FLAG_TIMEOUT,
// stops issuing work, drains its copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kernels.h"

namespace wm {
namespace tc {

constexpr int BM = 128, BK = 64, NTHREADS = 192;
constexpr unsigned long long WAIT_NS = 4000000000ull;  // 4 s bound on any wait
constexpr unsigned long long PROBE_NS = 2000000ull;    // 2 ms: the wait_probe barrier

struct Params {
  int M, N, K, batch;
  int m_tiles, n_tiles, num_kb;
  int ksplit, kb_per;     // split-K: K slices per output tile, k-blocks per slice
  long long total_tiles;  // output tiles x ksplit
  int vec_out, vec_res, vec_fin;
  float* partial;         // split-K accumulation target [batch][M][N] (x2 when DUAL)
  int cluster_red;        // split-K over a thread-block cluster, reduced in shared memory
  int b_const;            // B tiles may be requested before the predecessor grid ends
  int wait_probe;         // test aid: the MMA issuer first waits on a barrier nothing completes
  const char* pf[2];      // L2 prefetch ranges for a later product (GemmDesc::pf)
  long long pf_bytes[2];
  Epi epi;
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
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
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait; false on timeout or when another role already gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long limit_ns = WAIT_NS) {
  if (mbar_try(b, parity)) return true;
  const unsigned long long t0 = gtimer();
  while (true) {
    if (mbar_try(b, parity)) return true;
    if (*abort_flag) return false;
    if (gtimer() - t0 > limit_ns) return false;
  }
}
__device__ __forceinline__ void tma_load3(const CUtensorMap* map, uint64_t* bar, void* dst, int c0,
                                          int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(su32(dst)),
      "l"(map), "r"(su32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                     uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          su32(bar))
      : "memory");
}
// K-major operand tile, 128-byte swizzle: rows of 128 B, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;              // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;    // stride byte offset
  d |= (uint64_t)1 << 46;              // descriptor version
  d |= (uint64_t)2 << 61;              // 128-byte swizzle
  return d;
}
// kind::f16 instruction descriptor: bf16 A/B, fp32 D, both K-major, M = 128.
__host__ __device__ constexpr uint32_t idesc_bf16(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
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
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Thread-block cluster: full barrier (release/acquire) and loads from the
// shared memory of CTA ``rank`` of this cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}
__device__ __forceinline__ uint32_t peer_addr(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_peer(uint32_t a) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float4 ld_peer4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a));
  return v;
}

__device__ __forceinline__ void st_bf16x32(__nv_bfloat16* p, const float* v) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[8 * q + 2 * i], v[8 * q + 2 * i + 1]);
    reinterpret_cast<uint4*>(p)[q] = u;
  }
}
__device__ __forceinline__ void ld_bf16x32(const __nv_bfloat16* p, float* v) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 u = reinterpret_cast<const uint4*>(p)[q];
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      v[8 * q + 2 * i] = f.x;
      v[8 * q + 2 * i + 1] = f.y;
    }
  }
}

// RMSNorm over one head held in registers, gain, then rotate-half RoPE.
// Gains are read 8 at a time and the (cos, sin) table 2 pairs at a time.
template <int HD>
__device__ __forceinline__ void norm_rope(float (&v)[HD], const __nv_bfloat16* gain, float eps,
                                          const float2* rt) {
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < HD; ++i) ss += v[i] * v[i];
  const float inv = rsqrtf(ss / (float)HD + eps);
#pragma unroll
  for (int i = 0; i < HD; i += 8) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(gain + i));
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 g = __bfloat1622float2(g2[e]);
      v[i + 2 * e] *= inv * g.x;
      v[i + 2 * e + 1] *= inv * g.y;
    }
  }
  const float4* rt4 = reinterpret_cast<const float4*>(rt);
#pragma unroll
  for (int t = 0; t < HD / 2; t += 2) {
    const float4 cs = __ldg(rt4 + t / 2);
    float x1 = v[t], x2 = v[t + HD / 2];
    v[t] = x1 * cs.x - x2 * cs.y;
    v[t + HD / 2] = x2 * cs.x + x1 * cs.y;
    x1 = v[t + 1];
    x2 = v[t + 1 + HD / 2];
    v[t + 1] = x1 * cs.z - x2 * cs.w;
    v[t + 1 + HD / 2] = x2 * cs.z + x1 * cs.w;
  }
}

// ---------------------------------------------------------------------------
// Epilogue of one 128 x BN tile: this thread owns accumulator row ``lane_row``.
// ---------------------------------------------------------------------------
template <int BN, bool DUAL, int MODE, int HD>
__device__ __forceinline__ void epilogue_tile(const Params& p, uint32_t taddr, int row, int bidx,
                                              int n0) {
  const Epi& e = p.epi;
  const bool row_ok = row < p.M;
  if constexpr (MODE == EPI_QNORM_ROPE || MODE == EPI_KV) {
#pragma unroll 1
    for (int h0 = 0; h0 < BN; h0 += HD) {
      float v[HD];
      __syncwarp();
      {
        uint32_t r[32];
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          tmem_ld32(taddr + h0 + 32 * c, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[32 * c + i] = __uint_as_float(r[i]);
        }
      }
      const int col0 = n0 + h0;
      if (!row_ok || col0 >= p.N) continue;
      const int ps = e.pos[row];
      if (ps < 0 || ps >= e.Tmax) {
        atomicOr(e.flags, FLAG_BAD_POS);
        continue;
      }
      const float2* rt = e.rope + (long long)ps * (HD / 2);
      __nv_bfloat16* dst;
      if constexpr (MODE == EPI_QNORM_ROPE) {
        norm_rope<HD>(v, (const __nv_bfloat16*)e.gain, e.eps, rt);
        dst = (__nv_bfloat16*)e.C + (long long)row * e.ldc + col0;
      } else {
        const int sq = e.seq[row];
        if (sq < 0 || sq >= e.B) {
          atomicOr(e.flags, FLAG_BAD_SEQ);
          continue;
        }
        if (e.chan_ss) {
          const float cs = chan_scale(e, row, bidx);
#pragma unroll
          for (int t = 0; t < HD; ++t) v[t] *= cs;
        }
        if (e.kv_branch == 0)
          norm_rope<HD>(v, (const __nv_bfloat16*)e.gain + (long long)bidx * e.gain_bstride, e.eps,
                        rt);
        dst = (__nv_bfloat16*)(e.kv_branch == 0 ? e.cache_k : e.cache_v) +
              ((((long long)sq * e.k + e.chan0 + bidx) * e.Hkv + col0 / HD) * e.Tmax + ps) * HD;
      }
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) st_bf16x32(dst + 32 * c, v + 32 * c);
    }
  } else {
    constexpr int CW = (BN % 32 == 0) ? 32 : 16;  // columns per TMEM load
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += CW) {
      uint32_t r[CW];
      float v[CW];
      __syncwarp();
      if constexpr (CW == 32) tmem_ld32(taddr + c0, *reinterpret_cast<uint32_t(*)[32]>(r));
      else tmem_ld16(taddr + c0, r);
      if constexpr (DUAL) {
        uint32_t r2[CW];
        if constexpr (CW == 32) tmem_ld32(taddr + BN + c0, *reinterpret_cast<uint32_t(*)[32]>(r2));
        else tmem_ld16(taddr + BN + c0, r2);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < CW; ++i) {
          const float gt = __uint_as_float(r[i]);
          v[i] = gt / (1.f + __expf(-gt)) * __uint_as_float(r2[i]);
        }
      } else {
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < CW; ++i) v[i] = __uint_as_float(r[i]);
      }
      const int col = n0 + c0;
      if (!row_ok || col >= p.N) continue;
      const bool full = col + CW <= p.N;
      if constexpr (MODE == EPI_RESID) {
        const __nv_bfloat16* rp = (const __nv_bfloat16*)e.R + (long long)row * e.ldr + col;
        if (full && p.vec_res) {
#pragma unroll
          for (int q = 0; q < CW / 8; ++q) {
            const uint4 u = reinterpret_cast<const uint4*>(rp)[q];
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 f = __bfloat1622float2(h[i]);
              v[8 * q + 2 * i] += f.x;
              v[8 * q + 2 * i + 1] += f.y;
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < CW; ++i)
            if (col + i < p.N) v[i] += __bfloat162float(rp[i]);
        }
      }
      const long long orow = (MODE == EPI_STORE && e.rowmap) ? e.rowmap[row] : row;
      const long long off = (long long)bidx * e.c_bstride + orow * e.ldc + col;
      if (e.out_f32) {
        float* cp = (float*)e.C + off;
        if (full && p.vec_out) {
#pragma unroll
          for (int i = 0; i < CW; i += 4)
            *reinterpret_cast<float4*>(cp + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        } else {
#pragma unroll
          for (int i = 0; i < CW; ++i)
            if (col + i < p.N) cp[i] = v[i];
        }
      } else {
        __nv_bfloat16* cp = (__nv_bfloat16*)e.C + off;
        if (full && p.vec_out) {
#pragma unroll
          for (int q = 0; q < CW / 8; ++q) {
            uint4 u;
            __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              h[i] = __floats2bfloat162_rn(v[8 * q + 2 * i], v[8 * q + 2 * i + 1]);
            reinterpret_cast<uint4*>(cp)[q] = u;
          }
        } else {
#pragma unroll
          for (int i = 0; i < CW; ++i)
            if (col + i < p.N) cp[i] = __float2bfloat16_rn(v[i]);
        }
      }
    }
  }
}

// Split-K: add this slice's accumulator row into the fp32 partial sums.
template <int BN, bool DUAL>
__device__ __forceinline__ void partial_tile(const Params& p, uint32_t taddr, int row, int bidx,
                                             int n0) {
  constexpr int CW = (BN % 32 == 0) ? 32 : 16;
  const bool row_ok = row < p.M;
  const long long plane = (long long)p.batch * p.M * p.N;
#pragma unroll 1
  for (int half = 0; half < (DUAL ? 2 : 1); ++half) {
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += CW) {
      uint32_t r[CW];
      __syncwarp();
      if constexpr (CW == 32) tmem_ld32(taddr + half * BN + c0, *reinterpret_cast<uint32_t(*)[32]>(r));
      else tmem_ld16(taddr + half * BN + c0, r);
      tmem_wait_ld();
      const int col = n0 + c0;
      if (!row_ok || col >= p.N) continue;
      float* dst = p.partial + half * plane + ((long long)bidx * p.M + row) * p.N + col;
      if (col + CW <= p.N && (p.N % 4) == 0) {
#pragma unroll
        for (int i = 0; i < CW; i += 4)
          atomicAdd(reinterpret_cast<float4*>(dst + i),
                    make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]),
                                __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3])));
      } else {
        for (int i = 0; i < CW && col + i < p.N; ++i) atomicAdd(dst + i, __uint_as_float(r[i]));
      }
    }
  }
}

// Per-head epilogue of one (row, head) whose HD sums sit in one warp, lane l
// holding dims l + 32c (so every RoPE pair (t, t + HD/2) is in one lane).
template <int MODE, int HD>
__device__ __forceinline__ void head_out(const Params& p, int bidx, int row, int hh, int lane,
                                         float (&v)[HD / 32]) {
  constexpr int VPL = HD / 32;
  const Epi& e = p.epi;
  const int ps = e.pos[row];
  if (ps < 0 || ps >= e.Tmax) {
    if (lane == 0) atomicOr(e.flags, FLAG_BAD_POS);
    return;
  }
  const __nv_bfloat16* gain;
  __nv_bfloat16* dst;
  bool rotate = true;
  if constexpr (MODE == EPI_QNORM_ROPE) {
    gain = (const __nv_bfloat16*)e.gain;
    dst = (__nv_bfloat16*)e.C + (long long)row * e.ldc + hh * HD;
  } else {
    const int sq = e.seq[row];
    if (sq < 0 || sq >= e.B) {
      if (lane == 0) atomicOr(e.flags, FLAG_BAD_SEQ);
      return;
    }
    if (e.chan_ss) {
      const float cs = chan_scale(e, row, bidx);
#pragma unroll
      for (int c = 0; c < VPL; ++c) v[c] *= cs;
    }
    rotate = e.kv_branch == 0;
    gain = (const __nv_bfloat16*)e.gain + (long long)bidx * e.gain_bstride;
    dst = (__nv_bfloat16*)(e.kv_branch == 0 ? e.cache_k : e.cache_v) +
          ((((long long)sq * e.k + e.chan0 + bidx) * e.Hkv + hh) * e.Tmax + ps) * HD;
  }
  if (rotate) {
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < VPL; ++c) ss += v[c] * v[c];
    ss = warp_sum(ss);
    const float inv = rsqrtf(ss / (float)HD + e.eps);
#pragma unroll
    for (int c = 0; c < VPL; ++c) v[c] *= inv * __bfloat162float(gain[lane + 32 * c]);
    const float2* rt = e.rope + (long long)ps * (HD / 2);
#pragma unroll
    for (int c = 0; c < VPL / 2; ++c) {  // pair (lane + 32c, lane + 32c + HD/2)
      const float2 cs = rt[lane + 32 * c];
      const float x1 = v[c], x2 = v[c + VPL / 2];
      v[c] = x1 * cs.x - x2 * cs.y;
      v[c + VPL / 2] = x2 * cs.x + x1 * cs.y;
    }
  }
#pragma unroll
  for (int c = 0; c < VPL; ++c) dst[lane + 32 * c] = __float2bfloat16_rn(v[c]);
}

// Plain-mode epilogue of outputs (row, col .. col + 3) (SwiGLU already
// applied): residual, then store. ``vec``: one 4-wide access each (widths and
// alignments allow it, no row map); else element by element up to N.
template <int MODE>
__device__ __forceinline__ void plain_out4(const Params& p, int bidx, int row, int col,
                                           float (&o)[4], bool vec) {
  const Epi& e = p.epi;
  if (vec) {
    if constexpr (MODE == EPI_RESID) {
      const uint2 rr = *reinterpret_cast<const uint2*>((const __nv_bfloat16*)e.R +
                                                       (long long)row * e.ldr + col);
      const float2 r0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&rr.x));
      const float2 r1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&rr.y));
      o[0] += r0.x; o[1] += r0.y; o[2] += r1.x; o[3] += r1.y;
    }
    const long long off = (long long)bidx * e.c_bstride + (long long)row * e.ldc + col;
    if (e.out_f32) {
      *reinterpret_cast<float4*>((float*)e.C + off) = make_float4(o[0], o[1], o[2], o[3]);
    } else {
      uint2 w;
      __nv_bfloat162 a = __floats2bfloat162_rn(o[0], o[1]), b = __floats2bfloat162_rn(o[2], o[3]);
      w.x = *reinterpret_cast<uint32_t*>(&a);
      w.y = *reinterpret_cast<uint32_t*>(&b);
      *reinterpret_cast<uint2*>((__nv_bfloat16*)e.C + off) = w;
    }
    return;
  }
  const long long orow = (MODE == EPI_STORE && e.rowmap) ? e.rowmap[row] : row;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (col + i >= p.N) break;
    float v = o[i];
    if constexpr (MODE == EPI_RESID) v += __bfloat162float(((const __nv_bfloat16*)e.R)[(long long)row * e.ldr + col + i]);
    const long long off = (long long)bidx * e.c_bstride + orow * e.ldc + col + i;
    if (e.out_f32)
      ((float*)e.C)[off] = v;
    else
      ((__nv_bfloat16*)e.C)[off] = __float2bfloat16_rn(v);
  }
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + __expf(-g)) * u; }

// Epilogue applied to summed split-K partials; re-zeroes what it read. Norm
// modes: one warp per (row, head). Plain modes: four outputs per thread.
template <int MODE, int HD>
__global__ void __launch_bounds__(256) finalize_kernel(const Params p) {
  pdl_wait();
  pdl_trigger();
  const long long plane = (long long)p.batch * p.M * p.N;
  if constexpr (MODE == EPI_QNORM_ROPE || MODE == EPI_KV) {
    constexpr int VPL = HD / 32;
    const int lane = threadIdx.x & 31;
    const int heads = p.N / HD;
    const long long task = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
    if (task >= (long long)p.batch * p.M * heads) return;  // warp-uniform
    const int hh = (int)(task % heads);
    const int row = (int)((task / heads) % p.M);
    const int bidx = (int)(task / ((long long)heads * p.M));
    float* src = p.partial + ((long long)bidx * p.M + row) * p.N + hh * HD;
    float v[VPL];
#pragma unroll
    for (int c = 0; c < VPL; ++c) {
      v[c] = src[lane + 32 * c];
      src[lane + 32 * c] = 0.f;
    }
    head_out<MODE, HD>(p, bidx, row, hh, lane, v);
  } else {
    const Epi& e = p.epi;
    const bool vec = (p.N % 4) == 0 && (e.ldc % 4) == 0 && (e.c_bstride % 4) == 0 &&
                     ((uintptr_t)e.C % 16) == 0 &&
                     (MODE != EPI_RESID || ((e.ldr % 4) == 0 && ((uintptr_t)e.R % 8) == 0)) &&
                     !(MODE == EPI_STORE && e.rowmap);
    const int quads = (p.N + 3) / 4;  // four columns per thread, per row
    const long long step = (long long)gridDim.x * blockDim.x;
    for (long long tq = blockIdx.x * (long long)blockDim.x + threadIdx.x;
         tq < (long long)p.batch * p.M * quads; tq += step) {
      const int col = (int)(tq % quads) * 4;
      const int row = (int)((tq / quads) % p.M);
      const int bidx = (int)(tq / ((long long)quads * p.M));
      const long long i = ((long long)bidx * p.M + row) * p.N + col;
      float o[4];
      if (vec) {
        const float4 v = *reinterpret_cast<float4*>(p.partial + i);
        *reinterpret_cast<float4*>(p.partial + i) = make_float4(0.f, 0.f, 0.f, 0.f);
        o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
        if constexpr (MODE == EPI_SWIGLU) {
          const float4 u = *reinterpret_cast<float4*>(p.partial + plane + i);
          *reinterpret_cast<float4*>(p.partial + plane + i) = make_float4(0.f, 0.f, 0.f, 0.f);
          o[0] = silu_mul(o[0], u.x); o[1] = silu_mul(o[1], u.y);
          o[2] = silu_mul(o[2], u.z); o[3] = silu_mul(o[3], u.w);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          o[q] = 0.f;
          if (col + q < p.N) {
            o[q] = p.partial[i + q];
            p.partial[i + q] = 0.f;
            if constexpr (MODE == EPI_SWIGLU) {
              o[q] = silu_mul(o[q], p.partial[plane + i + q]);
              p.partial[plane + i + q] = 0.f;
            }
          }
        }
      }
      plain_out4<MODE>(p, bidx, row, col, o, vec);
    }
  }
}

// This CTA's share of the L2 prefetch ranges: one contiguous, 4 KB-aligned
// piece of each range, issued as bulk prefetches whose lines L2 keeps in
// preference to normal and evict-first ones. Nothing waits for them.
__device__ __forceinline__ void prefetch_share(const Params& p) {
  if (!p.pf[0] && !p.pf[1]) return;
  uint64_t keep;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep));
  const long long nb = gridDim.x;
#pragma unroll 1
  for (int r = 0; r < 2; ++r) {
    const long long bytes = p.pf_bytes[r];
    if (!p.pf[r]) continue;
    const long long chunk = ((bytes + nb - 1) / nb + 4095) & ~4095LL;
    const long long lo = (long long)blockIdx.x * chunk, hi = min(bytes, lo + chunk);
    for (long long off = lo; off < hi; off += 65536) {
      const uint32_t sz = (uint32_t)min(65536LL, hi - off);
      asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(p.pf[r] + off),
                   "r"(sz), "l"(keep)
                   : "memory");
    }
  }
}

// Split-K over a cluster: the CTAs of one output tile each hold their K
// slice's accumulator rows in shared memory (``red``, RS floats per row);
// CTA ``rank`` sums rows rank, rank + ks, ... over the cluster in a fixed
// order and applies the epilogue. Warp ``we`` of ``nw`` takes every nw-th of
// those rows; each lane issues all its loads of a row before adding them.
template <int BN, bool DUAL, int MODE, int HD, int RS>
__device__ __forceinline__ void cluster_reduce(const Params& p, const float* red, int we, int nw,
                                               int lane) {
  constexpr int KS_MAX = 8;
  const int ks = p.ksplit, rank = (int)(blockIdx.x % ks);
  const long long ot = blockIdx.x / ks;
  const int tiles_per_batch = p.m_tiles * p.n_tiles;
  const int bidx = (int)(ot / tiles_per_batch), rem = (int)(ot % tiles_per_batch);
  const int nt = rem % p.n_tiles, mt = rem / p.n_tiles;
  const int n0 = nt * BN, rows = min(BM, p.M - mt * BM);
  uint32_t peer[KS_MAX];
#pragma unroll
  for (int q = 0; q < KS_MAX; ++q) peer[q] = q < ks ? peer_addr(su32(red), q) : 0u;
  for (int j = rank + we * ks; j < rows; j += nw * ks) {
    const int row = mt * BM + j;
    if constexpr (MODE == EPI_QNORM_ROPE || MODE == EPI_KV) {
      constexpr int VPL = HD / 32;
#pragma unroll 1
      for (int h0 = 0; h0 < BN && n0 + h0 < p.N; h0 += HD) {
        float a[KS_MAX][VPL];
        const uint32_t off = (uint32_t)(j * RS + h0 + lane) * 4u;
#pragma unroll
        for (int q = 0; q < KS_MAX; ++q)
#pragma unroll
          for (int c = 0; c < VPL; ++c) a[q][c] = q < ks ? ld_peer(peer[q] + off + 128u * c) : 0.f;
        float v[VPL];
#pragma unroll
        for (int c = 0; c < VPL; ++c) {
          v[c] = a[0][c];
#pragma unroll
          for (int q = 1; q < KS_MAX; ++q) v[c] += a[q][c];
        }
        head_out<MODE, HD>(p, bidx, row, (n0 + h0) / HD, lane, v);
      }
    } else {
      for (int c = 4 * lane; c < BN && n0 + c < p.N; c += 128) {
        const uint32_t off = (uint32_t)(j * RS + c) * 4u;
        const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
        float4 a[KS_MAX], b[KS_MAX];
#pragma unroll
        for (int q = 0; q < KS_MAX; ++q) {
          a[q] = q < ks ? ld_peer4(peer[q] + off) : z4;
          b[q] = (DUAL && q < ks) ? ld_peer4(peer[q] + off + BN * 4u) : z4;
        }
        float4 g = a[0], u = b[0];
#pragma unroll
        for (int q = 1; q < KS_MAX; ++q) {
          g.x += a[q].x; g.y += a[q].y; g.z += a[q].z; g.w += a[q].w;
          if constexpr (DUAL) { u.x += b[q].x; u.y += b[q].y; u.z += b[q].z; u.w += b[q].w; }
        }
        float o[4] = {g.x, g.y, g.z, g.w};
        if constexpr (DUAL) {
          o[0] = silu_mul(g.x, u.x); o[1] = silu_mul(g.y, u.y);
          o[2] = silu_mul(g.z, u.z); o[3] = silu_mul(g.w, u.w);
        }
        plain_out4<MODE>(p, bidx, row, n0 + c, o, p.vec_fin != 0 && n0 + c + 4 <= p.N);
      }
    }
  }
}

constexpr int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p *= 2;
  return p;
}

template <int BN, bool DUAL>
struct Cfg {
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M = 128");
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES * (DUAL ? 2 : 1);
  static_assert(STAGE_BYTES % 1024 == 0, "operand tiles stay 1024-byte aligned");
  static constexpr int STAGES_RAW = (220 * 1024) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  static constexpr int ACC_COLS = BN * (DUAL ? 2 : 1);
  static constexpr int ACC_STRIDE = pow2_at_least(ACC_COLS);  // accumulator 1 column offset
  static constexpr int TMEM_COLS = 2 * ACC_STRIDE;
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + 256;
  // cluster split-K: accumulator rows staged over the (then idle) stage ring
  static constexpr int RED_STRIDE = ACC_COLS + 4;
  static_assert(BM * RED_STRIDE * 4 <= STAGES * STAGE_BYTES, "staged rows fit the ring");
};

// Cluster split-K: copy this thread's accumulator row (tile row ``j``) into
// the staging rows ``red`` (RS floats per row) of this CTA's shared memory.
template <int BN, bool DUAL, int RS>
__device__ __forceinline__ void stage_row(const Params& p, uint32_t taddr, int j, bool row_ok,
                                          float* red) {
  constexpr int CW = (BN % 32 == 0) ? 32 : 16;
#pragma unroll 1
  for (int c0 = 0; c0 < BN * (DUAL ? 2 : 1); c0 += CW) {
    uint32_t r[CW];
    __syncwarp();
    if constexpr (CW == 32) tmem_ld32(taddr + c0, *reinterpret_cast<uint32_t(*)[32]>(r));
    else tmem_ld16(taddr + c0, r);
    tmem_wait_ld();
    if (!row_ok) continue;
    float4* dst = reinterpret_cast<float4*>(red + (long long)j * RS + c0);
#pragma unroll
    for (int i = 0; i < CW; i += 4)
      dst[i / 4] = make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]),
                               __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
  }
}

template <int BN, bool DUAL, int MODE, int HD>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmB2, const Params p) {
  using C = Cfg<BN, DUAL>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full = (uint64_t*)(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint64_t* probe = mma_done + 1;  // wait_probe: a barrier that nothing completes
  uint32_t* tmem_holder = (uint32_t*)(probe + 1);
  volatile int* abort_flag = (volatile int*)(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(mma_done, 1);
    mbar_init(probe, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmB) : "memory");
    if (DUAL) asm volatile("prefetch.tensormap [%0];" ::"l"(&tmB2) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     su32(tmem_holder)),
                 "r"((uint32_t)C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int tiles_per_batch = p.m_tiles * p.n_tiles;
  if (!(warp == 0 && lane == 0)) pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      // Weight tiles of the first two ring stages go out before the wait for
      // the predecessor grid (its results are only read through A). More
      // measured slower on decode steps: A tiles issued after the wait queue
      // behind the weight tiles still in flight.
      constexpr int PRE_MAX = C::STAGES < 2 ? C::STAGES : 2;
      int pre = 0;
      if (p.b_const && blockIdx.x < p.total_tiles) {
        const long long ot = blockIdx.x / p.ksplit;
        const int bidx = (int)(ot / tiles_per_batch);
        const int nt = (int)(ot % tiles_per_batch) % p.n_tiles;
        const int kb0 = (int)(blockIdx.x % p.ksplit) * p.kb_per;
        const int kb1 = min(p.num_kb, kb0 + p.kb_per);
        for (int kb = kb0; kb < kb1 && pre < PRE_MAX; ++kb, ++pre) {
          uint8_t* sa = smem + pre * C::STAGE_BYTES;
          mbar_expect_tx(&full[pre], C::STAGE_BYTES);
          tma_load3(&tmB, &full[pre], sa + C::A_BYTES, kb * BK, nt * BN, bidx);
          if (DUAL) tma_load3(&tmB2, &full[pre], sa + C::A_BYTES + C::B_BYTES, kb * BK, nt * BN, bidx);
        }
      }
      pdl_wait();
      int stage = 0, issued = 0;
      uint32_t phase = 0, used = 0, last_phase = 0;
      bool ok = true;
      for (long long t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
        const long long ot = t / p.ksplit;
        const int ks = (int)(t % p.ksplit);
        const int bidx = (int)(ot / tiles_per_batch);
        const int rem = (int)(ot % tiles_per_batch);
        const int nt = rem % p.n_tiles, mt = rem / p.n_tiles;  // column tiles fastest
        const int kb0 = ks * p.kb_per, kb1 = min(p.num_kb, kb0 + p.kb_per);
        for (int kb = kb0; kb < kb1; ++kb, ++issued) {
          // Another role gave up (or the call had already timed out): stop,
          // once the stages whose B tiles went out early have their A tiles
          // too (their byte counts are posted in full).
          if (issued >= pre && *abort_flag) {
            ok = false;
            break;
          }
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * C::STAGE_BYTES;
          if (issued >= pre) {  // else its B tiles and byte count are already posted
            mbar_expect_tx(&full[stage], C::STAGE_BYTES);
            tma_load3(&tmB, &full[stage], sa + C::A_BYTES, kb * BK, nt * BN, bidx);
            if (DUAL) tma_load3(&tmB2, &full[stage], sa + C::A_BYTES + C::B_BYTES, kb * BK, nt * BN, bidx);
          }
          tma_load3(&tmA, &full[stage], sa, kb * BK, mt * BM, bidx);
          used |= 1u << stage;
          last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(p.epi.flags, FLAG_TIMEOUT);
      } else {
        prefetch_share(p);
      }
      // Drain: every issued copy has landed before the CTA may exit.
      volatile int no_abort = 0;
      for (int s = 0; s < C::STAGES; ++s)
        if (used & (1u << s)) mbar_wait(&full[s], (last_phase >> s) & 1, &no_abort);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t idesc = idesc_bf16(BN);
      int stage = 0, it = 0;
      uint32_t phase = 0;
      bool ok = true;
      // A bounded wait of an earlier kernel of this call gave up: issue
      // nothing, so that one timeout costs one wait limit per call rather
      // than one per launch.
      if (*(volatile uint32_t*)p.epi.flags & FLAG_TIMEOUT) {
        ok = false;
        *abort_flag = 1;
      } else if (p.wait_probe) {
        // test aid: a wait that runs out (nothing arrives at ``probe``)
        if (!mbar_wait(probe, 0, abort_flag, PROBE_NS)) ok = false;
      }
      for (long long t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        fence_after();
        const uint32_t d_tmem = tmem_base + acc * C::ACC_STRIDE;
        const int kb0 = (int)(t % p.ksplit) * p.kb_per, kb1 = min(p.num_kb, kb0 + p.kb_per);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          fence_after();
          const uint32_t sa = su32(smem + stage * C::STAGE_BYTES);
          const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
          for (int k16 = 0; k16 < BK / 16; ++k16) {
            const uint32_t accum = (kb != kb0) || (k16 != 0);
            if constexpr (DUAL && 2 * BN <= 256) {
              // The second operand's tile follows the first in the stage and
              // its accumulator follows the first's in tensor memory: one
              // M128 N(2 BN) product covers both, reading the A tile from
              // shared memory once instead of twice (with two N = 128
              // products per K step the operand reads, 16 KB per 128 cycles,
              // held the gate/up products at 229 us per 8,192-row launch;
              // 197 us this way).
              umma(d_tmem, sdesc(sa + 32 * k16), sdesc(sb + 32 * k16), idesc_bf16(2 * BN), accum);
            } else {
              umma(d_tmem, sdesc(sa + 32 * k16), sdesc(sb + 32 * k16), idesc, accum);
              if (DUAL) umma(d_tmem + BN, sdesc(sa + 32 * k16), sdesc(sb + C::B_BYTES + 32 * k16), idesc, accum);
            }
          }
          umma_commit(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok) umma_commit(&tfull[acc]);
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(p.epi.flags, FLAG_TIMEOUT);
      }
      // Every issued MMA has completed before TMEM is released.
      umma_commit(mma_done);
      volatile int no_abort = 0;
      mbar_wait(mma_done, 0, &no_abort);
    }
  } else {
    // ---------------- epilogue warps ----------------
    const int quarter = warp & 3;
    int it = 0;
    for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull[acc], acc_phase, abort_flag) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) {
          *abort_flag = 1;
          atomicOr(p.epi.flags, FLAG_TIMEOUT);
        }
        break;
      }
      fence_after();
      const long long ot = t / p.ksplit;
      const int bidx = (int)(ot / tiles_per_batch);
      const int rem = (int)(ot % tiles_per_batch);
      const int nt = rem % p.n_tiles, mt = rem / p.n_tiles;  // column tiles fastest
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * C::ACC_STRIDE;
      if (p.cluster_red) {
        // this CTA holds exactly one tile; the stage ring is idle from here on
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        stage_row<BN, DUAL, C::RED_STRIDE>(p, taddr, quarter * 32 + lane,
                                           mt * BM + quarter * 32 + lane < p.M,
                                           reinterpret_cast<float*>(smem));
      } else if (p.partial)
        partial_tile<BN, DUAL>(p, taddr, mt * BM + quarter * 32 + lane, bidx, nt * BN);
      else
        epilogue_tile<BN, DUAL, MODE, HD>(p, taddr, mt * BM + quarter * 32 + lane, bidx, nt * BN);
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"((uint32_t)C::TMEM_COLS)
                 : "memory");
  }
  if (p.cluster_red) {
    cluster_sync();  // every CTA of the cluster has staged its rows
    cluster_reduce<BN, DUAL, MODE, HD, C::RED_STRIDE>(p, reinterpret_cast<const float*>(smem),
                                                      warp, NTHREADS / 32, lane);
    cluster_sync();  // no CTA leaves while a peer may still read its rows
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
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

bool make_map(CUtensorMap* m, const void* ptr, long long K, long long rows, long long batch,
              long long ld, long long bstride, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)batch};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2,
                           (cuuint64_t)(batch > 1 ? bstride : rows * ld) * 2};
  cuuint32_t box[3] = {(cuuint32_t)BK, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Plain-mode outputs may be moved four at a time (see plain_out4).
bool fin_vectorisable(const GemmDesc& g) {
  const Epi& e = g.epi;
  return (g.N % 4) == 0 && (e.ldc % 4) == 0 && (e.c_bstride % 4) == 0 &&
         ((uintptr_t)e.C % 16) == 0 &&
         (e.mode != EPI_RESID || ((e.ldr % 4) == 0 && ((uintptr_t)e.R % 8) == 0)) &&
         !(e.mode == EPI_STORE && e.rowmap);
}

// How many clusters of ``ks`` CTAs of this kernel can be resident at once
// (asked once per kernel and size; the dynamic shared memory size is set).
template <int BN, bool DUAL, int MODE, int HD>
int max_clusters(int ks) {
  static int known[9] = {-1, -1, -1, -1, -1, -1, -1, -1, -1};
  if (ks < 2 || ks > 8) return 0;
  if (known[ks] < 0) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)ks);
    lc.blockDim = dim3(NTHREADS);
    lc.dynamicSmemBytes = (size_t)Cfg<BN, DUAL>::SMEM;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)ks;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    lc.attrs = at;
    lc.numAttrs = 1;
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<BN, DUAL, MODE, HD>, &lc);
    known[ks] = e == cudaSuccess ? n : 0;
    if (e != cudaSuccess) cudaGetLastError();  // clear the query's error
  }
  return known[ks];
}

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

template <int BN, bool DUAL, int MODE, int HD>
cudaError_t run(const GemmDesc& g, cudaStream_t st, int* launches) {
  using C = Cfg<BN, DUAL>;
  CUtensorMap ta, tb, tb2;
  if (!make_map(&ta, g.A, g.K, g.M, g.batch, g.lda, g.a_bstride, BM)) return cudaErrorInvalidValue;
  if (!make_map(&tb, g.B, g.K, g.N, g.batch, g.ldb, g.b_bstride, BN)) return cudaErrorInvalidValue;
  if (DUAL) {
    if (!make_map(&tb2, g.B2, g.K, g.N, g.batch, g.ldb, g.b_bstride, BN))
      return cudaErrorInvalidValue;
  } else {
    tb2 = tb;
  }
  Params p;
  p.M = g.M; p.N = g.N; p.K = g.K; p.batch = g.batch;
  p.m_tiles = (g.M + BM - 1) / BM;
  p.n_tiles = (g.N + BN - 1) / BN;
  p.num_kb = (g.K + BK - 1) / BK;
  const long long out_tiles = (long long)p.m_tiles * p.n_tiles * g.batch;
  p.ksplit = 1;
  p.kb_per = p.num_kb;
  p.partial = nullptr;
  p.cluster_red = 0;
  const int sms = num_sms();
  auto kern = gemm_tc_kernel<BN, DUAL, MODE, HD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  // Few output tiles (decode-sized M): split K over a cluster of up to 8
  // CTAs that sum their slices through distributed shared memory; the
  // largest split whose clusters are all resident at once (one wave).
  if (!g.no_cluster && g.M <= BM && out_tiles * 2 <= sms && p.num_kb >= 4) {
    long long ks0 = sms / out_tiles;
    if (ks0 > 8) ks0 = 8;
    if (ks0 > p.num_kb / 2) ks0 = p.num_kb / 2;
    for (int ks = (int)ks0; ks >= 2; --ks) {
      const int kb_per = (p.num_kb + ks - 1) / ks;
      const int kse = (p.num_kb + kb_per - 1) / kb_per;
      if (kse != ks) continue;
      if (max_clusters<BN, DUAL, MODE, HD>(ks) >= out_tiles) {
        p.ksplit = ks;
        p.kb_per = kb_per;
        p.cluster_red = 1;
        break;
      }
    }
  }
  const long long need = (long long)g.batch * g.M * g.N * (DUAL ? 2 : 1);
  // split-K only for one row tile (decode-sized M): for more rows the fp32
  // atomics of the partial tiles cost more than the idle SMs it recovers
  if (!p.cluster_red && g.partial && g.M <= BM && need <= g.partial_elems && out_tiles * 2 <= sms &&
      p.num_kb >= 4 &&
      (MODE != EPI_QNORM_ROPE && MODE != EPI_KV ? true : (g.N % HD == 0))) {
    int ks = (int)((sms + out_tiles - 1) / out_tiles);
    ks = min(ks, p.num_kb / 2);
    p.kb_per = (p.num_kb + ks - 1) / ks;
    p.ksplit = (p.num_kb + p.kb_per - 1) / p.kb_per;
    if (p.ksplit > 1) p.partial = g.partial;
    else p.kb_per = p.num_kb;
  }
  p.total_tiles = out_tiles * p.ksplit;
  p.epi = g.epi;
  const size_t osz = g.epi.out_f32 ? 4 : 2;
  p.vec_out = ((uintptr_t)g.epi.C % 16 == 0) && ((g.epi.ldc * osz) % 16 == 0) &&
              ((g.epi.c_bstride * osz) % 16 == 0);
  p.vec_res = ((uintptr_t)g.epi.R % 16 == 0) && ((g.epi.ldr * 2) % 16 == 0);
  p.vec_fin = fin_vectorisable(g);
  p.b_const = g.b_const ? 1 : 0;
  p.wait_probe = g.wait_probe ? 1 : 0;
  for (int r = 0; r < 2; ++r) {
    const bool use = g.pf[r] && g.pf_bytes[r] > 0 && (uintptr_t)g.pf[r] % 16 == 0 && g.pf_bytes[r] % 16 == 0;
    p.pf[r] = use ? static_cast<const char*>(g.pf[r]) : nullptr;
    p.pf_bytes[r] = use ? g.pf_bytes[r] : 0;
  }
  if (p.cluster_red) {
    // one CTA per (output tile, K slice); a cluster holds one tile's slices
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)p.total_tiles);
    lc.blockDim = dim3(NTHREADS);
    lc.dynamicSmemBytes = C::SMEM;
    lc.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)p.ksplit;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = 2;
    e = cudaLaunchKernelEx(&lc, kern, ta, tb, tb2, p);
    if (launches) ++*launches;
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  const long long grid = p.total_tiles < sms ? p.total_tiles : sms;
  launch_k(kern, dim3((unsigned)grid), dim3(NTHREADS), C::SMEM, st, ta, tb, tb2, p);
  if (launches) ++*launches;
  if (p.partial) {
    long long work = (MODE == EPI_QNORM_ROPE || MODE == EPI_KV)
                         ? 32LL * g.batch * g.M * (g.N / (HD > 0 ? HD : 1))
                         : ((long long)g.batch * g.M * g.N + 3) / 4;
    long long blocks = (work + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    launch_k(finalize_kernel<MODE, (HD > 0 ? HD : 64)>, dim3((unsigned)blocks), dim3(256), 0, st, p);
    if (launches) ++*launches;
  }
  return cudaGetLastError();
}

}  // namespace tc

bool gemm_tc_supported(const GemmDesc& g) {
  auto a16 = [](const void* p) { return ((uintptr_t)p & 15u) == 0; };
  if (g.M <= 0 || g.N <= 0 || g.K <= 0 || g.batch <= 0) return false;
  if (!a16(g.A) || !a16(g.B) || (g.B2 && !a16(g.B2))) return false;
  if (g.lda % 8 || g.ldb % 8) return false;
  if (g.batch > 1 && (g.a_bstride % 8 || g.b_bstride % 8)) return false;
  if (g.epi.mode == EPI_QNORM_ROPE || g.epi.mode == EPI_KV) {
    if ((g.epi.d != 64 && g.epi.d != 128) || g.N % g.epi.d) return false;
  }
  if ((g.epi.mode == EPI_SWIGLU) != (g.B2 != nullptr)) return false;
  return tc::encode_fn() != nullptr;
}

namespace {
// Tile width with the fewest waves of tiles over the SMs, weighing each wave
// by the tile width plus a fixed per-tile cost (tiles of one GEMM run
// concurrently, one per SM, so the last partial wave sets the time).
int pick_bn(const GemmDesc& g, const int* cands, int n) {
  const long long m_tiles = (g.M + tc::BM - 1) / tc::BM;
  const long long sms = tc::num_sms();
  int best = cands[0];
  long long best_cost = -1;
  for (int i = 0; i < n; ++i) {
    const long long bn = cands[i];
    const long long tiles = m_tiles * ((g.N + bn - 1) / bn) * g.batch;
    const long long waves = (tiles + sms - 1) / sms;
    const long long cost = waves * (bn + 48);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = (int)bn;
    }
  }
  return best;
}
}  // namespace

cudaError_t launch_gemm_tc(const GemmDesc& g, cudaStream_t st, int* launches) {
  static const int kPlain[] = {256, 224, 128};
  switch (g.epi.mode) {
    case EPI_SWIGLU:
      return tc::run<128, true, EPI_SWIGLU, 0>(g, st, launches);
    case EPI_STORE:
    case EPI_RESID: {
      const int bn = pick_bn(g, kPlain, 3);
      if (g.epi.mode == EPI_STORE) {
        switch (bn) {
          case 256: return tc::run<256, false, EPI_STORE, 0>(g, st, launches);
          case 224: return tc::run<224, false, EPI_STORE, 0>(g, st, launches);
          case 128: return tc::run<128, false, EPI_STORE, 0>(g, st, launches);
          default: return tc::run<112, false, EPI_STORE, 0>(g, st, launches);
        }
      }
      switch (bn) {
        case 256: return tc::run<256, false, EPI_RESID, 0>(g, st, launches);
        case 224: return tc::run<224, false, EPI_RESID, 0>(g, st, launches);
        case 128: return tc::run<128, false, EPI_RESID, 0>(g, st, launches);
        default: return tc::run<112, false, EPI_RESID, 0>(g, st, launches);
      }
    }
    case EPI_QNORM_ROPE:
    case EPI_KV: {
      static const int kHeads[] = {256, 128};
      const bool wide = g.N % 256 == 0 && pick_bn(g, kHeads, 2) == 256;
      if (g.epi.mode == EPI_QNORM_ROPE) {
        if (g.epi.d == 128)
          return wide ? tc::run<256, false, EPI_QNORM_ROPE, 128>(g, st, launches)
                      : tc::run<128, false, EPI_QNORM_ROPE, 128>(g, st, launches);
        return wide ? tc::run<256, false, EPI_QNORM_ROPE, 64>(g, st, launches)
                    : tc::run<128, false, EPI_QNORM_ROPE, 64>(g, st, launches);
      }
      if (g.epi.d == 128)
        return wide ? tc::run<256, false, EPI_KV, 128>(g, st, launches)
                    : tc::run<128, false, EPI_KV, 128>(g, st, launches);
      return wide ? tc::run<256, false, EPI_KV, 64>(g, st, launches) : tc::run<128, false, EPI_KV, 64>(g, st, launches);
    }
  }
  return cudaErrorNotSupported;
}

}  // namespace wm
