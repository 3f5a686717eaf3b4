// Strictly causal channel attention: row n (sequence seq[n], position pos[n])
// attends to keys s < pos[n] of one cache channel; query head h reads KV head
// h*Hkv/Hq; a row with no visible key gets 0.
#include <cuda_fp16.h>

#include "kernels.h"

namespace wm {

// CUDA-core engine: one warp per (row, query head), online softmax over the
// visible keys, each lane owning d/32 of the head's dimensions.
template <typename S>
__global__ void __launch_bounds__(128) attn_simt_kernel(const AttnArgs a) {
  pdl_wait();
  pdl_trigger();
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

// ---------------------------------------------------------------------------
// Tensor-core engine (bf16): flash attention on mma.sync m16n8k16.
// A CTA owns one KV head and a tile of consecutive rows; the G = Hq/Hkv query
// heads of each row are packed into the 64-row M dimension (row-major: M-row
// m = row (m / G), head hk*G + m % G). The tile is processed as maximal runs of
// rows sharing a sequence, so any row list is handled; rows of one sequence
// that are contiguous (every prefill group) form a single run. Keys stream
// through shared memory in blocks of 64 with cp.async double buffering; the
// softmax is online in fp32 (exp2 with the 1/sqrt(d) scale folded in).
// ---------------------------------------------------------------------------
namespace {
constexpr int AWARPS = 8, AQ = 16 * AWARPS, AKV = 32, ATHREADS = 32 * AWARPS;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// Transpose of an 8 x 8 bf16 matrix held one row pair per lane (the layout of
// an m16n8 accumulator quarter packed to bf16x2).
__device__ __forceinline__ uint32_t movm_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
}  // namespace

template <int HD>
__global__ void __launch_bounds__(ATHREADS, 2) attn_mma_kernel(const AttnArgs a, int rpt, int nq) {
  pdl_wait();
  pdl_trigger();
  constexpr int LDS = HD + 8;  // padded smem row (elements): conflict-free ldmatrix
  extern __shared__ __align__(16) uint8_t sm[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(sm);
  __nv_bfloat16* sK = sQ + AQ * LDS;           // [2][AKV][LDS]
  __nv_bfloat16* sV = sK + 2 * AKV * LDS;      // [2][AKV][LDS]
  __shared__ int s_pos[AQ];
  __shared__ int s_maxp;

  const int G = a.Hq / a.Hkv;
  const int hk = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int t0, t1;  // rows of this tile
  if (nq > 0) {
    const int tps = (nq + rpt - 1) / rpt;
    const int b = blockIdx.x / tps, t = tps - 1 - blockIdx.x % tps;  // late positions first
    t0 = b * nq + t * rpt;
    t1 = min(t0 + rpt, (b + 1) * nq);
  } else {
    t0 = blockIdx.x * rpt;
    t1 = min(t0 + rpt, a.N);
  }
  const float sl2 = 1.4426950408889634f / sqrtf((float)HD);
  const __nv_bfloat16* qg = (const __nv_bfloat16*)a.q;
  __nv_bfloat16* og = (__nv_bfloat16*)a.out;

  for (int ra = t0; ra < t1;) {
    // ---- the run [ra, rb) of rows sharing sequence seq[ra] ----
    const int sq = a.seq[ra];
    int rb = ra + 1;
    while (rb < t1 && a.seq[rb] == sq) ++rb;
    const int mrows = (rb - ra) * G;
    const bool seq_ok = sq >= 0 && sq < a.B;
    __syncthreads();  // previous run finished with shared memory
    if (threadIdx.x == 0) s_maxp = 0;
    __syncthreads();
    if (threadIdx.x < AQ) {
      int p = -1;
      if (threadIdx.x < mrows) {
        p = a.pos[ra + threadIdx.x / G];
        if (!seq_ok || p < 0 || p >= a.Tmax) {
          if (threadIdx.x % G == 0) atomicOr(a.flags, seq_ok ? FLAG_BAD_POS : FLAG_BAD_SEQ);
          p = -2;  // invalid row: output zeros
        }
      }
      s_pos[threadIdx.x] = p;
      if (p > 0) atomicMax(&s_maxp, p);
    }
    // Q tile: M-row m -> q[row][head]
    for (int c = threadIdx.x; c < AQ * (HD / 8); c += ATHREADS) {
      const int m = c / (HD / 8), part = c % (HD / 8);
      const bool v = m < mrows;
      const int r = ra + (v ? m / G : 0), h = hk * G + (v ? m % G : 0);
      cp_async16(sQ + m * LDS + part * 8, qg + ((long long)r * a.Hq + h) * HD + part * 8, v);
    }
    cp_async_commit();
    __syncthreads();
    const int maxp = s_maxp;
    const int nkb = (maxp + AKV - 1) / AKV;
    const long long kvbase = seq_ok ? (((long long)sq * a.k + a.channel) * a.Hkv + hk) * a.Tmax * HD : 0;
    const __nv_bfloat16* Kg = (const __nv_bfloat16*)a.cache_k + kvbase;
    const __nv_bfloat16* Vg = (const __nv_bfloat16*)a.cache_v + kvbase;

    auto load_kv = [&](int kb, int buf) {
      for (int c = threadIdx.x; c < AKV * (HD / 8); c += ATHREADS) {
        const int rr = c / (HD / 8), part = c % (HD / 8);
        const int s = kb * AKV + rr;
        const bool v = s < maxp;
        const long long off = (long long)(v ? s : 0) * HD + part * 8;
        cp_async16(sK + (buf * AKV + rr) * LDS + part * 8, Kg + off, v);
        cp_async16(sV + (buf * AKV + rr) * LDS + part * 8, Vg + off, v);
      }
      cp_async_commit();
    };
    if (nkb > 0) load_kv(0, 0);

    // per-thread rows: g and g + 8 of this warp's 16
    const int mr0 = warp * 16 + (lane >> 2), mr1 = mr0 + 8;
    const int p0 = s_pos[mr0], p1 = s_pos[mr1];
    float o[HD / 8][4];
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    cp_async_wait<0>();  // Q (and the first K/V block) landed
    __syncthreads();
    const uint32_t qaddr = smem_addr(sQ + (warp * 16 + (lane & 15)) * LDS + (lane >> 4) * 8);

    for (int kb = 0; kb < nkb; ++kb) {
      const int buf = kb & 1;
      if (kb + 1 < nkb) {
        load_kv(kb + 1, buf ^ 1);
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncthreads();
      // values to fp16 in place (exact for bf16 inputs of normal range), so
      // that P V runs with P in fp16 instead of bf16
      {
        __nv_bfloat162* vb2 = reinterpret_cast<__nv_bfloat162*>(sV + buf * AKV * LDS);
        for (int c = threadIdx.x; c < AKV * (LDS / 2); c += ATHREADS) {
          const float2 f = __bfloat1622float2(vb2[c]);
          reinterpret_cast<__half2*>(vb2)[c] = __floats2half2_rn(f.x, f.y);
        }
      }
      __syncthreads();
      const __nv_bfloat16* Kb = sK + buf * AKV * LDS;
      const __nv_bfloat16* Vb = sV + buf * AKV * LDS;
      // S = Q K^T for 16 rows x 64 keys
      float sc[AKV / 8][4];
#pragma unroll
      for (int nt = 0; nt < AKV / 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < HD / 16; ks += 2) {
        uint32_t qa[4], qb[4];
        ldsm_x4(qaddr + ks * 32, qa[0], qa[1], qa[2], qa[3]);
        ldsm_x4(qaddr + ks * 32 + 32, qb[0], qb[1], qb[2], qb[3]);
#pragma unroll
        for (int nt = 0; nt < AKV / 8; ++nt) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(smem_addr(Kb + (nt * 8 + (lane & 7)) * LDS + ks * 16 + (lane >> 3) * 8), b0, b1,
                  b2, b3);
          mma_bf16(sc[nt], qa, b0, b1);
          mma_bf16(sc[nt], qb, b2, b3);
        }
      }
      // mask keys s >= pos of the row, online softmax
      float mx0 = m0, mx1 = m1;
#pragma unroll
      for (int nt = 0; nt < AKV / 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int s = kb * AKV + nt * 8 + 2 * (lane & 3) + e;
          sc[nt][e] = s < p0 ? sc[nt][e] * sl2 : -INFINITY;
          sc[nt][2 + e] = s < p1 ? sc[nt][2 + e] * sl2 : -INFINITY;
          mx0 = fmaxf(mx0, sc[nt][e]);
          mx1 = fmaxf(mx1, sc[nt][2 + e]);
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float base0 = mx0 == -INFINITY ? 0.f : mx0;
      const float base1 = mx1 == -INFINITY ? 0.f : mx1;
      const float corr0 = exp2f(m0 - base0), corr1 = exp2f(m1 - base1);
      m0 = mx0;
      m1 = mx1;
      float rs0 = 0.f, rs1 = 0.f;
      uint32_t pf[AKV / 16][4];
#pragma unroll
      for (int nt = 0; nt < AKV / 8; ++nt) {
        const float e0 = exp2f(sc[nt][0] - base0), e1 = exp2f(sc[nt][1] - base0);
        const float e2 = exp2f(sc[nt][2] - base1), e3 = exp2f(sc[nt][3] - base1);
        rs0 += e0 + e1;
        rs1 += e2 + e3;
        pf[nt >> 1][(nt & 1) * 2 + 0] = pack_f16(e0, e1);
        pf[nt >> 1][(nt & 1) * 2 + 1] = pack_f16(e2, e3);
      }
      l0 = l0 * corr0 + rs0;
      l1 = l1 * corr1 + rs1;
#pragma unroll
      for (int i = 0; i < HD / 8; ++i) {
        o[i][0] *= corr0; o[i][1] *= corr0;
        o[i][2] *= corr1; o[i][3] *= corr1;
      }
      // O += P V
#pragma unroll
      for (int j = 0; j < AKV / 16; ++j) {
        const uint32_t pa[4] = {pf[j][0], pf[j][1], pf[j][2], pf[j][3]};
#pragma unroll
        for (int dn = 0; dn < HD / 8; dn += 2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(smem_addr(Vb + (j * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LDS + dn * 8 +
                              (lane >> 4) * 8),
                    b0, b1, b2, b3);
          mma_f16(o[dn], pa, b0, b1);
          mma_f16(o[dn + 1], pa, b2, b3);
        }
      }
      __syncthreads();  // this buffer may be overwritten by the next prefetch
    }
    // quad-reduce the row sums, normalise, store
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float i0 = p0 > 0 ? 1.f / l0 : 0.f, i1 = p1 > 0 ? 1.f / l1 : 0.f;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int m = half ? mr1 : mr0;
      const float inv = half ? i1 : i0;
      if (m >= mrows) continue;
      const int r = ra + m / G, h = hk * G + m % G;
      __nv_bfloat16* dst = og + ((long long)r * a.Hq + h) * HD + 2 * (lane & 3);
#pragma unroll
      for (int dn = 0; dn < HD / 8; ++dn) {
        const float x = o[dn][half * 2] * inv, y = o[dn][half * 2 + 1] * inv;
        *reinterpret_cast<__nv_bfloat162*>(dst + dn * 8) = __floats2bfloat162_rn(x, y);
      }
    }
    ra = rb;
  }
}

template <int HD>
void launch_attn_mma(const AttnArgs& a, int nq, cudaStream_t st) {
  const int G = a.Hq / a.Hkv;
  const int rpt = AQ / G;
  int tiles;
  if (nq > 0) {
    const int B = a.N / nq;
    tiles = B * ((nq + rpt - 1) / rpt);
  } else {
    tiles = (a.N + rpt - 1) / rpt;
  }
  const size_t smem = (size_t)(AQ + 4 * AKV) * (HD + 8) * 2;
  cudaFuncSetAttribute(attn_mma_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  dim3 grid(tiles, a.Hkv);
  launch_k(attn_mma_kernel<HD>, dim3(grid), dim3(ATHREADS), smem, st, a, rpt, nq);
}

// ---------------------------------------------------------------------------
// Decode engine (bf16, one query row per sequence): flash-decoding. A CTA owns
// (row, KV head, key split); its G query heads form one 16-row MMA tile. Four
// warps take every 4th block of 32 keys of the split with warp-private,
// double-buffered cp.async tiles (no block-wide barrier in the loop), keep
// their own online-softmax state, and merge through shared memory at the end.
// With several splits, each writes (max, sum, unnormalised output) and
// attn_combine_kernel merges them.
// ---------------------------------------------------------------------------
namespace {
constexpr int DWARPS = 4, DKEYS = 32, DBUF = 3;
}

// Merge of nsplit (max, sum, unnormalised output) partials of one (row, head).
template <int HD>
__device__ __forceinline__ float merge_splits(const float* src, int nsplit, int d) {
  float M = -INFINITY;
  for (int z = 0; z < nsplit; ++z) M = fmaxf(M, __ldcg(src + z * (HD + 2) + HD));
  const float base = M == -INFINITY ? 0.f : M;
  float L = 0.f, acc = 0.f;
  for (int z = 0; z < nsplit; ++z) {
    const float f = exp2f(__ldcg(src + z * (HD + 2) + HD) - base);
    L += f * __ldcg(src + z * (HD + 2) + HD + 1);
    acc += f * __ldcg(src + z * (HD + 2) + d);
  }
  return L > 0.f ? acc / L : 0.f;
}

// 16-byte cp.async whose line is the first candidate for eviction from L2.
__device__ __forceinline__ void cp_async16_ef(void* dst, const void* src, bool valid, uint64_t pol) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(smem_addr(dst)),
               "l"(src), "r"(n), "l"(pol)
               : "memory");
}

// HT (G <= 8 query heads per KV head): the products are taken transposed,
// S^T = K Q^T and O^T = V^T P^T, so keys and dimensions fill the 16 rows of
// each MMA and the G heads its 8 columns; P^T reaches the second product's
// operand layout through movmatrix. Without HT, the G heads are the rows of a
// 16-row tile (rows >= G wasted).
template <int HD, bool HT>
__global__ void __launch_bounds__(32 * DWARPS) attn_decode_kernel(const AttnArgs a, int nsplit,
                                                                  float* part) {
  pdl_wait();
  pdl_trigger();
  // The keys and values are read once per step: their lines go first when L2
  // needs room (the weights that the next products prefetch stay).
  uint64_t stream_pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(stream_pol));
  constexpr int LDS = HD + 8;
  extern __shared__ __align__(16) uint8_t sm[];
  __shared__ int last_split;
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(sm);          // [16][LDS]
  __nv_bfloat16* sKV = sQ + 16 * LDS;                                 // [warp][DBUF][K,V][DKEYS][LDS]
  float* sO = reinterpret_cast<float*>(sm);                           // [warp][16][HD + 2], reused
  const int G = a.Hq / a.Hkv;
  const int n = blockIdx.x / a.Hkv, hk = blockIdx.x % a.Hkv, z = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sq = a.seq[n], ps = a.pos[n];
  const bool ok = sq >= 0 && sq < a.B && ps >= 0 && ps < a.Tmax;
  if (!ok && threadIdx.x == 0) atomicOr(a.flags, (sq < 0 || sq >= a.B) ? FLAG_BAD_SEQ : FLAG_BAD_POS);
  const int visible = ok ? ps : 0;
  int span = (visible + nsplit - 1) / nsplit;
  span = (span + DKEYS - 1) / DKEYS * DKEYS;
  const int k0 = min(visible, z * span), k1 = min(visible, k0 + span);
  const int nblk = (k1 - k0 + DKEYS - 1) / DKEYS;
  const long long kvbase = ok ? (((long long)sq * a.k + a.channel) * a.Hkv + hk) * a.Tmax * HD : 0;
  const __nv_bfloat16* Kg = (const __nv_bfloat16*)a.cache_k + kvbase;
  const __nv_bfloat16* Vg = (const __nv_bfloat16*)a.cache_v + kvbase;
  const __nv_bfloat16* qg = (const __nv_bfloat16*)a.q;
  // Q rows: the G heads of this KV head (rows >= G are zero)
  for (int c = threadIdx.x; c < 16 * (HD / 8); c += 32 * DWARPS) {
    const int m = c / (HD / 8), part8 = c % (HD / 8);
    const bool v = m < G;
    cp_async16(sQ + m * LDS + part8 * 8,
               qg + ((long long)n * a.Hq + hk * G + (v ? m : 0)) * HD + part8 * 8, v);
  }
  cp_async_commit();
  __nv_bfloat16* myKV = sKV + warp * DBUF * 2 * DKEYS * LDS;
  auto load_blk = [&](int blk, int buf) {
    __nv_bfloat16* dK = myKV + (buf * 2 + 0) * DKEYS * LDS;
    __nv_bfloat16* dV = myKV + (buf * 2 + 1) * DKEYS * LDS;
    for (int c = lane; c < DKEYS * (HD / 8); c += 32) {
      const int rr = c / (HD / 8), part8 = c % (HD / 8);
      const int s = k0 + blk * DKEYS + rr;
      const bool v = s < k1;
      const long long off = (long long)(v ? s : 0) * HD + part8 * 8;
      cp_async16_ef(dK + rr * LDS + part8 * 8, Kg + off, v, stream_pol);
      cp_async16_ef(dV + rr * LDS + part8 * 8, Vg + off, v, stream_pol);
    }
    cp_async_commit();
  };
  const float sl2 = 1.4426950408889634f / sqrtf((float)HD);
  // HT: o[mt] holds O^T rows (dims) mt * 16 + lane / 4 (+ 8), heads 2 (lane % 4)
  // (+ 1); m0, l0 / m1, l1 are those two heads' running max and sum.
  // Otherwise o[dn] holds heads lane / 4 (+ 8), dims dn * 8 + 2 (lane % 4) (+ 1).
  float o[HT ? HD / 16 : HD / 8][4];
#pragma unroll
  for (int i = 0; i < (HT ? HD / 16 : HD / 8); ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  if constexpr (HT) {
    // this warp's first blocks, then Q^T as B operands (head lane / 4), kept in registers
    int blk = warp, buf = 0;
#pragma unroll
    for (int i = 0; i < DBUF - 1; ++i) {
      if (blk + i * DWARPS < nblk) load_blk(blk + i * DWARPS, i);
      else cp_async_commit();
    }
    cp_async_wait<DBUF - 2>();
    __syncthreads();  // Q visible to every warp
    uint32_t qf[HD / 16][2];
#pragma unroll
    for (int ks = 0; ks < HD / 16; ks += 2)
      ldsm_x4(smem_addr(sQ + (lane & 7) * LDS + ks * 16 + (lane >> 3) * 8), qf[ks][0], qf[ks][1],
              qf[ks + 1][0], qf[ks + 1][1]);

  for (; blk < nblk; blk += DWARPS, buf = (buf + 1 == DBUF ? 0 : buf + 1)) {
    const int ahead = blk + (DBUF - 1) * DWARPS;
    if (ahead < nblk) load_blk(ahead, buf == 0 ? DBUF - 1 : buf - 1);
    else cp_async_commit();
    cp_async_wait<DBUF - 1>();
    __syncwarp();
    const __nv_bfloat16* Kb = myKV + (buf * 2 + 0) * DKEYS * LDS;
    const __nv_bfloat16* Vb = myKV + (buf * 2 + 1) * DKEYS * LDS;
    // S^T: keys mt * 16 + lane / 4 (+ 8), heads hA = 2 (lane % 4), hA + 1.
    // Written in this order (the volatile asm statements keep it in the
    // emitted code; the final schedule is the assembler's): every K
    // fragment first, then the products over four independent accumulators
    // (even and odd k steps of both key tiles).
    float st[DKEYS / 16][4], st2[DKEYS / 16][4];
    {
      uint32_t ka[DKEYS / 16][HD / 16][4];
#pragma unroll
      for (int mt = 0; mt < DKEYS / 16; ++mt)
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks)
          ldsm_x4(smem_addr(Kb + (mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LDS + ks * 16 +
                            (lane >> 4) * 8),
                  ka[mt][ks][0], ka[mt][ks][1], ka[mt][ks][2], ka[mt][ks][3]);
#pragma unroll
      for (int mt = 0; mt < DKEYS / 16; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) st[mt][i] = st2[mt][i] = 0.f;
#pragma unroll
      for (int ks = 0; ks < HD / 16; ++ks)
#pragma unroll
        for (int mt = 0; mt < DKEYS / 16; ++mt)
          mma_bf16((ks & 1) ? st2[mt] : st[mt], ka[mt][ks], qf[ks][0], qf[ks][1]);
    }
    // V^T fragments for O^T += V^T P^T, loaded before the softmax needs them
    uint32_t va[HD / 16][DKEYS / 16][4];
#pragma unroll
    for (int j = 0; j < DKEYS / 16; ++j)
#pragma unroll
      for (int mt = 0; mt < HD / 16; ++mt)
        ldsm_x4_t(smem_addr(Vb + (j * 16 + (lane & 7) + (lane >> 4) * 8) * LDS + mt * 16 +
                            ((lane >> 3) & 1) * 8),
                  va[mt][j][0], va[mt][j][1], va[mt][j][2], va[mt][j][3]);
#pragma unroll
    for (int mt = 0; mt < DKEYS / 16; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) st[mt][i] += st2[mt][i];
    float mx0 = m0, mx1 = m1;
#pragma unroll
    for (int mt = 0; mt < DKEYS / 16; ++mt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int key = k0 + blk * DKEYS + mt * 16 + (lane >> 2) + hh * 8;
        const bool vis = key < k1;
        st[mt][2 * hh] = vis ? st[mt][2 * hh] * sl2 : -INFINITY;
        st[mt][2 * hh + 1] = vis ? st[mt][2 * hh + 1] * sl2 : -INFINITY;
        mx0 = fmaxf(mx0, st[mt][2 * hh]);
        mx1 = fmaxf(mx1, st[mt][2 * hh + 1]);
      }
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, x));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, x));
    }
    const float base0 = mx0 == -INFINITY ? 0.f : mx0, base1 = mx1 == -INFINITY ? 0.f : mx1;
    const float corr0 = exp2f(m0 - base0), corr1 = exp2f(m1 - base1);
    m0 = mx0;
    m1 = mx1;
    // P^T quarters (keys x heads) -> B operands (heads x keys) of O^T += V^T P^T
    uint32_t pb[DKEYS / 16][2];
#pragma unroll
    for (int mt = 0; mt < DKEYS / 16; ++mt) {
      const float e0 = exp2f(st[mt][0] - base0), e1 = exp2f(st[mt][1] - base1);
      const float e2 = exp2f(st[mt][2] - base0), e3 = exp2f(st[mt][3] - base1);
      l0 = l0 * (mt == 0 ? corr0 : 1.f) + e0 + e2;
      l1 = l1 * (mt == 0 ? corr1 : 1.f) + e1 + e3;
      __nv_bfloat162 p01 = __floats2bfloat162_rn(e0, e1), p23 = __floats2bfloat162_rn(e2, e3);
      pb[mt][0] = movm_t(*reinterpret_cast<uint32_t*>(&p01));
      pb[mt][1] = movm_t(*reinterpret_cast<uint32_t*>(&p23));
    }
#pragma unroll
    for (int i = 0; i < HD / 16; ++i) {
      o[i][0] *= corr0; o[i][1] *= corr1;
      o[i][2] *= corr0; o[i][3] *= corr1;
    }
#pragma unroll
    for (int j = 0; j < DKEYS / 16; ++j)
#pragma unroll
      for (int mt = 0; mt < HD / 16; ++mt) mma_bf16(o[mt], va[mt][j], pb[j][0], pb[j][1]);
    __syncwarp();  // this buffer is refilled DBUF - 1 blocks later
  }
  } else {

  // this warp's blocks: warp, warp + DWARPS, ...; DBUF - 1 of them in flight
  int blk = warp, buf = 0;
#pragma unroll
  for (int i = 0; i < DBUF - 1; ++i) {
    if (blk + i * DWARPS < nblk) load_blk(blk + i * DWARPS, i);
    else cp_async_commit();
  }
  cp_async_wait<DBUF - 2>();
  __syncthreads();  // Q visible to every warp
  const uint32_t qaddr = smem_addr(sQ + (lane & 15) * LDS + (lane >> 4) * 8);
  for (; blk < nblk; blk += DWARPS, buf = (buf + 1 == DBUF ? 0 : buf + 1)) {
    const int ahead = blk + (DBUF - 1) * DWARPS;
    if (ahead < nblk) load_blk(ahead, buf == 0 ? DBUF - 1 : buf - 1);
    else cp_async_commit();
    cp_async_wait<DBUF - 1>();
    __syncwarp();
    const __nv_bfloat16* Kb = myKV + (buf * 2 + 0) * DKEYS * LDS;
    const __nv_bfloat16* Vb = myKV + (buf * 2 + 1) * DKEYS * LDS;
    float sc[DKEYS / 8][4];
#pragma unroll
    for (int nt = 0; nt < DKEYS / 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < HD / 16; ks += 2) {
      uint32_t qa[4], qb[4];
      ldsm_x4(qaddr + ks * 32, qa[0], qa[1], qa[2], qa[3]);
      ldsm_x4(qaddr + ks * 32 + 32, qb[0], qb[1], qb[2], qb[3]);
#pragma unroll
      for (int nt = 0; nt < DKEYS / 8; ++nt) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_addr(Kb + (nt * 8 + (lane & 7)) * LDS + ks * 16 + (lane >> 3) * 8), b0, b1, b2, b3);
        mma_bf16(sc[nt], qa, b0, b1);
        mma_bf16(sc[nt], qb, b2, b3);
      }
    }
    float mx0 = m0, mx1 = m1;
#pragma unroll
    for (int nt = 0; nt < DKEYS / 8; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const bool vis = k0 + blk * DKEYS + nt * 8 + 2 * (lane & 3) + e < k1;
        sc[nt][e] = vis ? sc[nt][e] * sl2 : -INFINITY;
        sc[nt][2 + e] = vis ? sc[nt][2 + e] * sl2 : -INFINITY;
        mx0 = fmaxf(mx0, sc[nt][e]);
        mx1 = fmaxf(mx1, sc[nt][2 + e]);
      }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float base0 = mx0 == -INFINITY ? 0.f : mx0, base1 = mx1 == -INFINITY ? 0.f : mx1;
    const float corr0 = exp2f(m0 - base0), corr1 = exp2f(m1 - base1);
    m0 = mx0;
    m1 = mx1;
    float rs0 = 0.f, rs1 = 0.f;
    uint32_t pf[DKEYS / 16][4];
#pragma unroll
    for (int nt = 0; nt < DKEYS / 8; ++nt) {
      const float e0 = exp2f(sc[nt][0] - base0), e1 = exp2f(sc[nt][1] - base0);
      const float e2 = exp2f(sc[nt][2] - base1), e3 = exp2f(sc[nt][3] - base1);
      rs0 += e0 + e1;
      rs1 += e2 + e3;
      __nv_bfloat162 p01 = __floats2bfloat162_rn(e0, e1), p23 = __floats2bfloat162_rn(e2, e3);
      pf[nt >> 1][(nt & 1) * 2 + 0] = *reinterpret_cast<uint32_t*>(&p01);
      pf[nt >> 1][(nt & 1) * 2 + 1] = *reinterpret_cast<uint32_t*>(&p23);
    }
    l0 = l0 * corr0 + rs0;
    l1 = l1 * corr1 + rs1;
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) {
      o[i][0] *= corr0; o[i][1] *= corr0;
      o[i][2] *= corr1; o[i][3] *= corr1;
    }
#pragma unroll
    for (int j = 0; j < DKEYS / 16; ++j) {
      const uint32_t pa[4] = {pf[j][0], pf[j][1], pf[j][2], pf[j][3]};
#pragma unroll
      for (int dn = 0; dn < HD / 8; dn += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_addr(Vb + (j * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LDS + dn * 8 +
                            (lane >> 4) * 8), b0, b1, b2, b3);
        mma_bf16(o[dn], pa, b0, b1);
        mma_bf16(o[dn + 1], pa, b2, b3);
      }
    }
    __syncwarp();  // this buffer is refilled DBUF - 1 blocks later
  }
  }
  if constexpr (HT) {
  cp_async_wait<0>();
#pragma unroll
  for (int x = 4; x < 32; x <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, x);
    l1 += __shfl_xor_sync(0xffffffffu, l1, x);
  }
  __syncthreads();  // all warps are done with their tiles: reuse shared memory
  float* mine = sO + (size_t)warp * 16 * (HD + 2);
  {
    const int hA = 2 * (lane & 3), hB = hA + 1, dr = lane >> 2;
#pragma unroll
    for (int mt = 0; mt < HD / 16; ++mt) {
      mine[hA * (HD + 2) + mt * 16 + dr] = o[mt][0];
      mine[hB * (HD + 2) + mt * 16 + dr] = o[mt][1];
      mine[hA * (HD + 2) + mt * 16 + dr + 8] = o[mt][2];
      mine[hB * (HD + 2) + mt * 16 + dr + 8] = o[mt][3];
    }
    if (lane < 4) {
      mine[hA * (HD + 2) + HD] = m0;
      mine[hA * (HD + 2) + HD + 1] = l0;
      mine[hB * (HD + 2) + HD] = m1;
      mine[hB * (HD + 2) + HD + 1] = l1;
    }
  }
  } else {
  cp_async_wait<0>();
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  __syncthreads();  // all warps are done with their tiles: reuse shared memory
  // per-warp state: sO[w][row][0..HD) = o, [HD] = m, [HD + 1] = l
  float* mine = sO + (size_t)warp * 16 * (HD + 2);
  const int g0 = lane >> 2, g1 = g0 + 8;
#pragma unroll
  for (int dn = 0; dn < HD / 8; ++dn) {
    const int d0 = dn * 8 + 2 * (lane & 3);
    mine[g0 * (HD + 2) + d0] = o[dn][0];
    mine[g0 * (HD + 2) + d0 + 1] = o[dn][1];
    mine[g1 * (HD + 2) + d0] = o[dn][2];
    mine[g1 * (HD + 2) + d0 + 1] = o[dn][3];
  }
  if ((lane & 3) == 0) {
    mine[g0 * (HD + 2) + HD] = m0;
    mine[g0 * (HD + 2) + HD + 1] = l0;
    mine[g1 * (HD + 2) + HD] = m1;
    mine[g1 * (HD + 2) + HD + 1] = l1;
  }
  }
  __syncthreads();
  // merge the warps: thread (head h, dims) for h < G
  for (int idx = threadIdx.x; idx < G * HD; idx += 32 * DWARPS) {
    const int h = idx / HD, d = idx % HD;
    float M = -INFINITY;
    for (int w = 0; w < DWARPS; ++w) M = fmaxf(M, sO[((size_t)w * 16 + h) * (HD + 2) + HD]);
    const float base = M == -INFINITY ? 0.f : M;
    float L = 0.f, acc = 0.f;
    for (int w = 0; w < DWARPS; ++w) {
      const float* st = sO + ((size_t)w * 16 + h) * (HD + 2);
      const float f = exp2f(st[HD] - base);
      L += f * st[HD + 1];
      acc += f * st[d];
    }
    const int head = hk * G + h;
    if (nsplit == 1) {
      const float v = (visible > 0 && L > 0.f) ? acc / L : 0.f;
      ((__nv_bfloat16*)a.out)[((long long)n * a.Hq + head) * HD + d] = __float2bfloat16_rn(v);
    } else {
      float* dst = part + (((long long)n * a.Hq + head) * nsplit + z) * (HD + 2);
      dst[d] = acc;
      if (d == 0) {
        dst[HD] = M;
        dst[HD + 1] = L;
      }
    }
  }
  if (nsplit == 1 || !a.counters) return;
  // The last split of this (row, KV head) to arrive merges all of them.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(a.counters + blockIdx.x, 1);
    last_split = prev == nsplit - 1;
    if (last_split) a.counters[blockIdx.x] = 0;  // ready for the next launch
  }
  __syncthreads();
  if (!last_split) return;
  __threadfence();
  for (int idx = threadIdx.x; idx < G * HD; idx += 32 * DWARPS) {
    const int head = hk * G + idx / HD, d = idx % HD;
    const float* src = part + ((long long)n * a.Hq + head) * nsplit * (HD + 2);
    ((__nv_bfloat16*)a.out)[((long long)n * a.Hq + head) * HD + d] =
        __float2bfloat16_rn(merge_splits<HD>(src, nsplit, d));
  }
}

template <int HD>
__global__ void attn_combine_kernel(const AttnArgs a, int nsplit, const float* part) {
  pdl_wait();
  pdl_trigger();
  const long long nh = blockIdx.x;  // (row, head)
  const int d = threadIdx.x;
  if (d >= HD) return;
  ((__nv_bfloat16*)a.out)[nh * HD + d] =
      __float2bfloat16_rn(merge_splits<HD>(part + nh * nsplit * (HD + 2), nsplit, d));
}

// One CTA per (row, KV head, key split), one CTA per SM (shared memory). The
// split count keeps the grid within one wave: a second wave costs a full
// CTA start-up and drain, more than the idle SMs of a short first wave.
template <int HD>
int launch_attn_decode(const AttnArgs& a, int kv_len, float* part, long long part_elems,
                       cudaStream_t st) {
  int sms = 148, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long ctas = (long long)a.N * a.Hkv;
  int nsplit = (int)(sms / ctas);
  nsplit = max(1, min(nsplit, min(16, (kv_len + 4 * DKEYS - 1) / (4 * DKEYS))));
  if (nsplit > 1 && (long long)a.N * a.Hq * nsplit * (HD + 2) > part_elems) nsplit = 1;
  const bool fused = nsplit > 1 && a.counters && ctas <= a.counter_elems;
  AttnArgs aa = a;
  if (!fused) aa.counters = nullptr;
  const size_t smem_loop = (size_t)(16 + DWARPS * DBUF * 2 * DKEYS) * (HD + 8) * 2;
  const size_t smem_merge = (size_t)DWARPS * 16 * (HD + 2) * 4;
  const size_t smem = smem_loop > smem_merge ? smem_loop : smem_merge;
  dim3 grid((unsigned)ctas, nsplit);
  if (a.Hq / a.Hkv <= 8) {
    cudaFuncSetAttribute(attn_decode_kernel<HD, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    launch_k(attn_decode_kernel<HD, true>, dim3(grid), dim3(32 * DWARPS), smem, st, aa, nsplit, part);
  } else {
    cudaFuncSetAttribute(attn_decode_kernel<HD, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    launch_k(attn_decode_kernel<HD, false>, dim3(grid), dim3(32 * DWARPS), smem, st, aa, nsplit, part);
  }
  if (nsplit > 1 && !fused) {
    launch_k(attn_combine_kernel<HD>, dim3((unsigned)((long long)a.N * a.Hq)), dim3(HD), 0, st, a, nsplit, part);
    return 2;
  }
  return 1;
}

// nq > 0 declares the rows as B = N / nq sequences of nq consecutive rows
// (cyclic groups and decode steps); 0 = no structure assumed.
int launch_attention(int dtype, const AttnArgs& a, bool simt, cudaStream_t st, int nq, int kv_len,
                     float* part, long long part_elems) {
  if (a.N <= 0) return 0;
  const int G = a.Hq / a.Hkv;
  // one row per sequence (decode steps): split the keys across CTAs
  if (dtype == WM_BF16 && !simt && nq == 1 && G <= 16 && kv_len > 0) {
    return a.d == 128 ? launch_attn_decode<128>(a, kv_len, part, part_elems, st)
                      : launch_attn_decode<64>(a, kv_len, part, part_elems, st);
  }
  // prefill groups (several rows per sequence) run on tcgen05; single-row
  // sequences (decode) and unstructured row lists run on mma.sync
  if (dtype == WM_BF16 && !simt && nq >= 8 && attention_tc_supported(a, nq)) {
    launch_attention_pair(a, nq, st);
    return 1;
  }
  if (dtype == WM_BF16 && !simt && G <= AQ) {
    if (nq > 0 && a.N % nq) nq = 0;
    if (a.d == 128) launch_attn_mma<128>(a, nq, st);
    else launch_attn_mma<64>(a, nq, st);
    return 1;
  }
  const long long warps = (long long)a.N * a.Hq;
  const int blocks = (int)((warps + 3) / 4);
  WM_DISPATCH_S(dtype, launch_k(attn_simt_kernel<S>, dim3(blocks), dim3(128), 0, st, a));
  return 1;
}

}  // namespace wm
