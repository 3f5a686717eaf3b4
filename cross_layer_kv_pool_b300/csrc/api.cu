// libwm C ABI: argument validation, workspace layout and the host-side
// drivers of the pool, the cyclic Gauss-Seidel pass and the decode step.
// Every arithmetic step runs in the kernels launched from here.
#include <cstring>
#include <mutex>

#include "kernels.h"

using namespace wm;

namespace {

enum Buf {
  B_FLAGS, B_ROPE, B_TOK, B_SEQ, B_POS, B_ROWMAP, B_STASH, B_HMID, B_HL, B_XN, B_Q, B_O,
  B_ACT, B_RIN, B_INV, B_COEFF, B_MIXED, B_CHSS, B_ATILE, B_LASTX, B_PARTIAL, B_CNT, B_ATTNP, B_END,
  NBUF
};

struct Layout {
  size_t off[NBUF];
  size_t total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }


int count_nR(const wm_config& c) {
  int n = 0;
  for (int l = 0; l < c.L; ++l) n += (l % c.p) == c.p_offset;
  return n;
}

Layout make_layout(const wm_config& c, long long N, long long Tmax) {
  const size_t es = elem_size(c.dtype);
  const long long nR = count_nR(c);
  size_t sz[NBUF];
  sz[B_FLAGS] = 256;
  sz[B_ROPE] = (size_t)Tmax * (c.d / 2) * sizeof(float2);
  sz[B_TOK] = sz[B_SEQ] = sz[B_POS] = sz[B_ROWMAP] = (size_t)N * 4;
  sz[B_STASH] = (size_t)N * c.L * c.D * es;
  sz[B_HMID] = sz[B_HL] = sz[B_XN] = sz[B_LASTX] = (size_t)N * c.D * es;
  sz[B_Q] = sz[B_O] = (size_t)N * c.Hq * c.d * es;
  sz[B_ACT] = (size_t)N * c.F * es;
  sz[B_RIN] = (size_t)2 * N * nR * c.D * es;
  sz[B_INV] = (size_t)N * c.L * 4;
  sz[B_COEFF] = (size_t)N * 2 * c.k * c.L * 4;
  sz[B_MIXED] = (size_t)N * 2 * c.k * c.D * es;
  sz[B_CHSS] = (size_t)N * 2 * c.k * 8 * 4;  // deferred channel-norm partial sums
  sz[B_ATILE] = c.dtype == WM_BF16 ? (size_t)N * MIX_ATILE_BYTES : 0;  // mixer coefficient tiles
  {  // split-K partial sums for GEMMs of at most 128 rows
    const long long rows = N < 128 ? N : 128;
    long long w = 2LL * c.F;
    const long long cand[] = {(long long)c.Hq * c.d, c.D, 2LL * c.k * c.L,
                              (long long)c.k * c.Hkv * c.d};
    for (long long v : cand) w = v > w ? v : w;
    sz[B_PARTIAL] = (size_t)rows * w * 4;
  }
  // arrival counters of the decode attention's key splits, per (row, KV head)
  sz[B_CNT] = (size_t)(N < 1024 ? N : 1024) * c.Hkv * 4;
  // decode attention key-split partials (at most 16 splits, rows <= 1024)
  sz[B_ATTNP] = (size_t)(N < 1024 ? N : 1024) * c.Hq * 16 * (c.d + 2) * 4;
  sz[B_END] = 0;
  Layout lay;
  size_t o = 0;
  for (int i = 0; i < NBUF; ++i) {
    lay.off[i] = o;
    o += align256(sz[i]);
  }
  lay.total = o;
  return lay;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

wm_status check_config(const wm_config* c) {
  if (!c) return WM_ERR_INVALID_ARG;
  if (c->L < 1 || c->L > 256 || c->D < 64 || c->D % 64 || c->D > 8192) return WM_ERR_INVALID_ARG;
  if (c->k < 1 || c->k > c->L || c->p < 1 || c->p_offset < 0 || c->p_offset >= c->p)
    return WM_ERR_INVALID_ARG;
  if (c->Hq < 1 || c->Hkv < 1 || c->Hq % c->Hkv) return WM_ERR_INVALID_ARG;
  if (c->F < 64 || c->F % 64 || c->V < 1 || !(c->eps >= 0.f) || !(c->rope_base > 0.f))
    return WM_ERR_INVALID_ARG;
  if (c->dtype != WM_F32 && c->dtype != WM_BF16) return WM_ERR_INVALID_ARG;
  if (c->d != 64 && c->d != 128) return WM_ERR_UNSUPPORTED;
  if (count_nR(*c) < 1) return WM_ERR_INVALID_ARG;
  if (c->flags & ~(uint32_t)(WM_FLAG_SIMT_GEMM | WM_FLAG_NO_CLUSTER | WM_FLAG_WAIT_PROBE))
    return WM_ERR_INVALID_ARG;
  return WM_OK;
}

wm_status check_weights(const wm_weights* w) {
  if (!w) return WM_ERR_INVALID_ARG;
  const void* ps[] = {w->embed, w->lm_head, w->final_norm, w->in_norm, w->post_norm,
                      w->q_norm, w->Wq, w->Wo, w->Wgate, w->Wup, w->Wdown, w->src_norm,
                      w->Wr, w->chan_norm, w->Wk, w->Wv, w->k_norm};
  for (const void* p : ps)
    if (!p || !aligned16(p)) return WM_ERR_INVALID_ARG;
  if (w->static_coeff && !aligned16(w->static_coeff)) return WM_ERR_INVALID_ARG;
  return WM_OK;
}

wm_status check_ws(const wm_config& c, void* ws, size_t ws_bytes, long long N, long long Tmax) {
  if (!ws || ((uintptr_t)ws & 255u)) return WM_ERR_WORKSPACE;
  if (ws_bytes < make_layout(c, N, Tmax).total) return WM_ERR_WORKSPACE;
  return WM_OK;
}

struct Ctx {
  mutable cudaError_t err = cudaSuccess;   // first failed launch of this call
  mutable long long launches = 0;          // kernels launched by this call
  const wm_config* c;
  const wm_weights* w;
  char* ws;
  Layout lay;
  cudaStream_t st;
  int nR;
  bool tc;
  size_t es;
  template <typename T> T* buf(Buf b) const { return reinterpret_cast<T*>(ws + lay.off[b]); }
  const char* wp(const void* p, long long elems) const {
    return static_cast<const char*>(p) + elems * (long long)es;
  }
  uint32_t* flags() const { return buf<uint32_t>(B_FLAGS); }
};

Ctx make_ctx(const wm_config* c, const wm_weights* w, void* ws, long long N, long long Tmax,
             void* stream) {
  Ctx x;
  x.c = c;
  x.w = w;
  x.ws = static_cast<char*>(ws);
  x.lay = make_layout(*c, N, Tmax);
  x.st = static_cast<cudaStream_t>(stream);
  x.nR = count_nR(*c);
  x.tc = c->dtype == WM_BF16 && !(c->flags & WM_FLAG_SIMT_GEMM);
  x.es = elem_size(c->dtype);
  return x;
}

// Measurement hook: event pair around one launch of the traced kernel class.
int trace_begin(const Ctx& x, int kind) {
  wm_trace* t = x.c->trace;
  if (!t || t->kind != kind || t->count >= t->capacity || !t->begin || !t->end) return -1;
  cudaEventRecord(static_cast<cudaEvent_t>(t->begin[t->count]), x.st);
  return t->count;
}
void trace_end(const Ctx& x, int idx, double work) {
  if (idx < 0) return;
  wm_trace* t = x.c->trace;
  cudaEventRecord(static_cast<cudaEvent_t>(t->end[idx]), x.st);
  if (t->work) t->work[idx] = work;
  t->count = idx + 1;
}

// bf16 contractions run on the tensor-core engine; shapes it cannot express
// (operand strides not 16-byte multiples) and the fp32 mode run on CUDA cores.
void gemm(const Ctx& x, const GemmDesc& gd) {
  const int tr = trace_begin(x, WM_TRACE_GEMM);
  GemmDesc g = gd;
  g.b_const = true;  // every product of the model multiplies by a weight matrix
  g.no_cluster = (x.c->flags & WM_FLAG_NO_CLUSTER) != 0;
  g.wait_probe = (x.c->flags & WM_FLAG_WAIT_PROBE) != 0;
  g.partial = x.buf<float>(B_PARTIAL);
  g.partial_elems = (long long)(x.lay.off[B_PARTIAL + 1] - x.lay.off[B_PARTIAL]) / 4;
  if (g.partial_elems <= 0) g.partial = nullptr;
  if (x.tc && gemm_tc_supported(g)) {
    int n = 0;
    const cudaError_t e = launch_gemm_tc(g, x.st, &n);
    x.launches += n - 1;
    if (e != cudaSuccess && x.err == cudaSuccess) x.err = e;
  } else {
    launch_gemm_simt(x.c->dtype, g, x.st);
  }
  trace_end(x, tr, 2.0 * g.M * g.N * (double)g.K * g.batch * (g.B2 ? 2 : 1));
}

// The mixer's coefficient-tile scratch, or null where the layout has none.
void* mix_atile(const Ctx& x) {
  return x.lay.off[B_ATILE + 1] > x.lay.off[B_ATILE] ? x.buf<void>(B_ATILE) : nullptr;
}

Epi base_epi(const Ctx& x) {
  Epi e;
  e.flags = x.flags();
  e.eps = x.c->eps;
  e.d = x.c->d;
  e.rope = x.buf<float2>(B_ROPE);
  return e;
}

// Layer stack of N rows whose h^0 is already in stash[:, 0]. Layer l reads
// stash[:, l], writes stash[:, l+1] (or h^L), and emits inv_rms / router
// inputs of its input state. The last layer's body runs only if requested.
void run_pool_channel(const Ctx& x, int N, int l, void* cache_k, void* cache_v, int B, int Tmax);

// The consumer stack over N rows. With ``feedback_free``, channel l of every
// row is pooled from its states 0..l right before layer l (k = L).
void run_stack(const Ctx& x, int N, int nq, double pos_sum, bool last_layer, void* cache_k,
               void* cache_v, int B, int Tmax, bool emit_rin, bool feedback_free = false) {
  const wm_config& c = *x.c;
  const wm_weights& w = *x.w;
  const long long LD = (long long)c.L * c.D;
  const int Hd = c.Hq * c.d;
  char* stash = x.buf<char>(B_STASH);
  // One row per sequence (decode): each product is a short weight stream, so
  // it prefetches the next product's weights into L2 behind its own loads.
  const bool pf = nq == 1;
  const long long DHb = (long long)c.D * Hd * (long long)x.es, FDb = (long long)c.F * c.D * (long long)x.es;
  for (int l = 0; l < c.L; ++l) {
    const bool body = l < c.L - 1 || last_layer;
    char* h_in = stash + (long long)l * c.D * x.es;
    ++x.launches;
    launch_norm_emit(c.dtype, stash, LD, c.D, N, l, 1, c.D, c.L, w.in_norm,
                     body ? x.buf<void>(B_XN) : nullptr, x.buf<float>(B_INV), w.src_norm,
                     emit_rin ? x.buf<void>(B_RIN) : nullptr, x.nR, c.p, c.p_offset, c.eps, x.st);
    if (feedback_free) run_pool_channel(x, N, l, cache_k, cache_v, B, Tmax);
    if (!body) break;
    {  // Q projection + per-head q-norm + RoPE
      GemmDesc g;
      g.M = N; g.N = Hd; g.K = c.D;
      g.A = x.buf<void>(B_XN); g.lda = c.D;
      g.B = x.wp(w.Wq, (long long)l * Hd * c.D); g.ldb = c.D;
      g.epi = base_epi(x);
      g.epi.mode = EPI_QNORM_ROPE;
      g.epi.C = x.buf<void>(B_Q); g.epi.ldc = Hd;
      g.epi.gain = x.wp(w.q_norm, (long long)l * c.d);
      g.epi.pos = x.buf<int>(B_POS);
      g.epi.Tmax = Tmax;
      if (pf) {
        g.pf[0] = x.wp(w.Wo, (long long)l * c.D * Hd);
        g.pf_bytes[0] = DHb;
      }
      ++x.launches;
      gemm(x, g);
    }
    {  // attention to channel l mod k over s < pos
      AttnArgs a;
      a.q = x.buf<void>(B_Q); a.N = N; a.seq = x.buf<int32_t>(B_SEQ); a.pos = x.buf<int32_t>(B_POS);
      a.channel = l % c.k; a.cache_k = cache_k; a.cache_v = cache_v;
      a.B = B; a.k = c.k; a.Hq = c.Hq; a.Hkv = c.Hkv; a.d = c.d; a.Tmax = Tmax;
      a.out = x.buf<void>(B_O); a.flags = x.flags();
      a.counters = x.buf<int>(B_CNT);
      a.counter_elems = (long long)(x.lay.off[B_CNT + 1] - x.lay.off[B_CNT]) / 4;
      const int tr = trace_begin(x, WM_TRACE_ATTN);
      const long long pe = (long long)(x.lay.off[B_ATTNP + 1] - x.lay.off[B_ATTNP]) / 4;
      x.launches += launch_attention(c.dtype, a, !x.tc, x.st, nq, nq == 1 ? (int)(pos_sum / B) : 0,
                                     x.buf<float>(B_ATTNP), pe);
      trace_end(x, tr, 4.0 * c.Hq * c.d * pos_sum);
    }
    {  // O projection + residual
      GemmDesc g;
      g.M = N; g.N = c.D; g.K = Hd;
      g.A = x.buf<void>(B_O); g.lda = Hd;
      g.B = x.wp(w.Wo, (long long)l * c.D * Hd); g.ldb = Hd;
      g.epi = base_epi(x);
      g.epi.mode = EPI_RESID;
      g.epi.R = h_in; g.epi.ldr = LD;
      g.epi.C = x.buf<void>(B_HMID); g.epi.ldc = c.D;
      if (pf) {
        g.pf[0] = x.wp(w.Wgate, (long long)l * c.F * c.D);
        g.pf[1] = x.wp(w.Wup, (long long)l * c.F * c.D);
        g.pf_bytes[0] = g.pf_bytes[1] = FDb;
      }
      ++x.launches;
      gemm(x, g);
    }
    ++x.launches;
    launch_rmsnorm(c.dtype, x.buf<void>(B_HMID), c.D, 0, 1, N, c.D,
                   x.wp(w.post_norm, (long long)l * c.D), x.buf<void>(B_XN), c.eps, x.st);
    {  // gate/up + SwiGLU
      GemmDesc g;
      g.M = N; g.N = c.F; g.K = c.D;
      g.A = x.buf<void>(B_XN); g.lda = c.D;
      g.B = x.wp(w.Wgate, (long long)l * c.F * c.D); g.ldb = c.D;
      g.B2 = x.wp(w.Wup, (long long)l * c.F * c.D);
      g.epi = base_epi(x);
      g.epi.mode = EPI_SWIGLU;
      g.epi.C = x.buf<void>(B_ACT); g.epi.ldc = c.F;
      if (pf) {
        g.pf[0] = x.wp(w.Wdown, (long long)l * c.D * c.F);
        g.pf_bytes[0] = FDb;
      }
      ++x.launches;
      gemm(x, g);
    }
    {  // down + residual -> next state
      GemmDesc g;
      g.M = N; g.N = c.D; g.K = c.F;
      g.A = x.buf<void>(B_ACT); g.lda = c.F;
      g.B = x.wp(w.Wdown, (long long)l * c.D * c.F); g.ldb = c.F;
      g.epi = base_epi(x);
      g.epi.mode = EPI_RESID;
      g.epi.R = x.buf<void>(B_HMID); g.epi.ldr = c.D;
      if (l + 1 < c.L) {
        g.epi.C = stash + (long long)(l + 1) * c.D * x.es; g.epi.ldc = LD;
      } else {
        g.epi.C = x.buf<void>(B_HL); g.epi.ldc = c.D;
      }
      if (pf && l + 1 < c.L && (l + 1 < c.L - 1 || last_layer)) {
        g.pf[0] = x.wp(w.Wq, (long long)(l + 1) * Hd * c.D);
        g.pf_bytes[0] = DHb;
      }
      ++x.launches;
      gemm(x, g);
    }
  }
}

// Router, mixer and K/V projections for N rows. Returns the mixer's deferred
// norm part count (0: ``mixed`` holds the normed channels; P > 0: it holds
// u = tau (.) m and the projections applied the norm factor).
int run_pool(const Ctx& x, int N, const void* states, long long ld_row, float* coeff,
             void* mixed, void* cache_k, void* cache_v, int B, int Tmax) {
  const wm_config& c = *x.c;
  const wm_weights& w = *x.w;
  const int kL = c.k * c.L;
  if (w.static_coeff) {
    ++x.launches;
    launch_broadcast_coeff(w.static_coeff, N, 2 * kL, coeff, x.st);
  } else {
    GemmDesc g;
    g.M = N; g.N = kL; g.K = x.nR * c.D; g.batch = 2;
    g.A = x.buf<void>(B_RIN); g.lda = (long long)x.nR * c.D; g.a_bstride = (long long)N * x.nR * c.D;
    g.B = w.Wr; g.ldb = (long long)x.nR * c.D; g.b_bstride = (long long)kL * x.nR * c.D;
    g.epi = base_epi(x);
    g.epi.mode = EPI_STORE;
    g.epi.out_f32 = 1;
    g.epi.C = coeff; g.epi.ldc = 2LL * kL; g.epi.c_bstride = kL;
    ++x.launches;
    gemm(x, g);
  }
  MixArgs m;
  m.stash = states; m.ld_row = ld_row; m.inv = x.buf<float>(B_INV); m.coeff = coeff;
  m.src_norm = w.src_norm; m.chan_norm = w.chan_norm; m.mixed = mixed;
  m.chan_ss = x.buf<float>(B_CHSS);
  m.atile = mix_atile(x);
  m.N = N; m.L = c.L; m.D = c.D; m.k = c.k; m.eps = c.eps;
  m.inv_ld = c.L; m.sn_layers = c.L; m.cn_channels = c.k;
  const int tr = trace_begin(x, WM_TRACE_MIX);
  ++x.launches;
  int parts = launch_mix(c.dtype, m, !x.tc, x.st, x.flags());
  if (parts < 0) {
    if (x.err == cudaSuccess) x.err = cudaErrorLaunchFailure;
    parts = 0;
  }
  trace_end(x, tr, (double)N * ((double)c.L * c.D * x.es + 2.0 * c.k * c.L * 4 + c.L * 4.0 +
                                 2.0 * c.k * c.D * x.es));
  for (int branch = 0; branch < 2; ++branch) {
    GemmDesc g;
    g.M = N; g.N = c.Hkv * c.d; g.K = c.D; g.batch = c.k;
    g.A = static_cast<const char*>(mixed) + (long long)branch * c.k * N * c.D * x.es;
    g.lda = c.D; g.a_bstride = (long long)N * c.D;
    g.B = branch == 0 ? w.Wk : w.Wv; g.ldb = c.D; g.b_bstride = (long long)c.Hkv * c.d * c.D;
    g.epi = base_epi(x);
    g.epi.mode = EPI_KV;
    g.epi.kv_branch = branch;
    g.epi.gain = w.k_norm; g.epi.gain_bstride = c.d;
    g.epi.pos = x.buf<int>(B_POS); g.epi.seq = x.buf<int>(B_SEQ);
    g.epi.cache_k = cache_k; g.epi.cache_v = cache_v;
    g.epi.k = c.k; g.epi.Hkv = c.Hkv; g.epi.Tmax = Tmax; g.epi.B = B;
    if (parts) {
      g.epi.chan_ss = x.buf<float>(B_CHSS);
      g.epi.chan_parts = parts;
      g.epi.chan_ss_k = c.k;
      g.epi.chan_D = (float)c.D;
    }
    ++x.launches;
    gemm(x, g);
  }
  return parts;
}

// The caller asked for the channels themselves: apply a deferred norm in place.
void finish_mixed(const Ctx& x, int N, void* mixed, int parts) {
  if (!parts) return;
  MixArgs m{};
  m.mixed = mixed; m.chan_ss = x.buf<float>(B_CHSS);
  m.N = N; m.D = x.c->D; m.k = x.c->k; m.L = x.c->L; m.eps = x.c->eps;
  m.inv_ld = x.c->L; m.sn_layers = x.c->L; m.cn_channels = x.c->k;
  ++x.launches;
  launch_mix_normalize(m, parts, x.st);
}

// Feedback-free channel l (k = L; [PL 5 ANALYSIS, "Deep-to-shallow feedback"]):
// the pool restricted to the sources 0..l of each row, computed before layer
// l runs, so that layer l reads only states its own pass has produced. The
// router reads the sources of R inside 0..l (a prefix of its input) through
// rows l*L + 0..l of W_R; the mixer takes the first l + 1 states; channel l's
// projections write cache channel l.
void run_pool_channel(const Ctx& x, int N, int l, void* cache_k, void* cache_v, int B, int Tmax) {
  const wm_config& c = *x.c;
  const wm_weights& w = *x.w;
  const int Ls = l + 1;
  float* coeff = x.buf<float>(B_COEFF);  // [N][2][1][Ls]
  if (w.static_coeff) {
    // the row's constants static[b][l][0..l], gathered once, then broadcast
    float* tmp = x.buf<float>(B_CHSS);
    for (int b = 0; b < 2; ++b)
      cudaMemcpyAsync(tmp + b * Ls, w.static_coeff + ((long long)b * c.k + l) * c.L,
                      (size_t)Ls * sizeof(float), cudaMemcpyDeviceToDevice, x.st);
    ++x.launches;
    launch_broadcast_coeff(tmp, N, 2 * Ls, coeff, x.st);
  } else {
    int r = 0;  // router sources inside 0..l
    for (int s = 0; s <= l; ++s) r += (s % c.p) == c.p_offset;
    if (r == 0) {
      cudaMemsetAsync(coeff, 0, (size_t)N * 2 * Ls * sizeof(float), x.st);
    } else {
      const long long in = (long long)x.nR * c.D;
      GemmDesc g;
      g.M = N; g.N = Ls; g.K = r * c.D; g.batch = 2;
      g.A = x.buf<void>(B_RIN); g.lda = in; g.a_bstride = (long long)N * in;
      g.B = x.wp(w.Wr, (long long)l * c.L * in); g.ldb = in; g.b_bstride = (long long)c.k * c.L * in;
      g.epi = base_epi(x);
      g.epi.mode = EPI_STORE;
      g.epi.out_f32 = 1;
      g.epi.C = coeff; g.epi.ldc = 2LL * Ls; g.epi.c_bstride = Ls;
      ++x.launches;
      gemm(x, g);
    }
  }
  MixArgs m;
  m.stash = x.buf<void>(B_STASH); m.ld_row = (long long)c.L * c.D; m.inv = x.buf<float>(B_INV);
  m.coeff = coeff; m.src_norm = w.src_norm; m.chan_norm = x.wp(w.chan_norm, (long long)l * c.D);
  m.mixed = x.buf<void>(B_MIXED); m.chan_ss = x.buf<float>(B_CHSS);
  m.atile = mix_atile(x);
  m.N = N; m.L = Ls; m.D = c.D; m.k = 1; m.eps = c.eps;
  m.inv_ld = c.L; m.sn_layers = c.L; m.cn_channels = c.k;
  const int tr = trace_begin(x, WM_TRACE_MIX);
  ++x.launches;
  int parts = launch_mix(c.dtype, m, !x.tc, x.st, x.flags());
  if (parts < 0) {
    if (x.err == cudaSuccess) x.err = cudaErrorLaunchFailure;
    parts = 0;
  }
  trace_end(x, tr, (double)N * ((double)Ls * c.D * x.es + 2.0 * Ls * 4 + Ls * 4.0 + 2.0 * c.D * x.es));
  for (int branch = 0; branch < 2; ++branch) {
    GemmDesc g;
    g.M = N; g.N = c.Hkv * c.d; g.K = c.D; g.batch = 1;
    g.A = x.buf<char>(B_MIXED) + (long long)branch * N * c.D * x.es; g.lda = c.D;
    g.B = x.wp(branch == 0 ? w.Wk : w.Wv, (long long)l * c.Hkv * c.d * c.D); g.ldb = c.D;
    g.epi = base_epi(x);
    g.epi.mode = EPI_KV;
    g.epi.kv_branch = branch;
    g.epi.gain = x.wp(w.k_norm, (long long)l * c.d); g.epi.gain_bstride = c.d;
    g.epi.pos = x.buf<int>(B_POS); g.epi.seq = x.buf<int>(B_SEQ);
    g.epi.cache_k = cache_k; g.epi.cache_v = cache_v;
    g.epi.k = c.k; g.epi.Hkv = c.Hkv; g.epi.Tmax = Tmax; g.epi.B = B;
    g.epi.chan0 = l;
    if (parts) {
      g.epi.chan_ss = x.buf<float>(B_CHSS);
      g.epi.chan_parts = parts;
      g.epi.chan_ss_k = 1;
      g.epi.chan_D = (float)c.D;
    }
    ++x.launches;
    gemm(x, g);
  }
}

// The split-K partial sums and the arrival counters start at zero in every
// call (their consumers re-zero what they used).
void zero_partials(const Ctx& x) {
  const size_t n = x.lay.off[B_CNT + 1] - x.lay.off[B_PARTIAL];
  if (n) cudaMemsetAsync(x.buf<char>(B_PARTIAL), 0, n, x.st);
}

// One decode step of B single-token rows whose tok/seq/pos rows and RoPE
// table rows are in place: embed, layer stack, final norm + LM head, then the
// pool appends every row's channels. pos_sum: sum of the rows' positions (or
// B * Tmax when only the bound is known on the host).
void decode_body(const Ctx& x, int B, double pos_sum, void* cache_k, void* cache_v, int Tmax,
                 float* logits) {
  const wm_config& c = *x.c;
  const wm_weights* w = x.w;
  zero_partials(x);
  ++x.launches;
  launch_embed(c.dtype, x.buf<int32_t>(B_TOK), B, w->embed, c.V, c.D, x.buf<void>(B_STASH),
               (long long)c.L * c.D, x.flags(), x.st);
  run_stack(x, B, 1, pos_sum, true, cache_k, cache_v, B, Tmax, w->static_coeff == nullptr);
  ++x.launches;
  launch_rmsnorm(c.dtype, x.buf<void>(B_HL), c.D, 0, 1, B, c.D, w->final_norm,
                 x.buf<void>(B_LASTX), c.eps, x.st);
  GemmDesc lg;
  lg.M = B; lg.N = c.V; lg.K = c.D;
  lg.A = x.buf<void>(B_LASTX); lg.lda = c.D;
  lg.B = w->lm_head; lg.ldb = c.D;
  lg.epi = base_epi(x);
  lg.epi.mode = EPI_STORE;
  lg.epi.out_f32 = 1;
  lg.epi.C = logits; lg.epi.ldc = c.V;
  ++x.launches;
  gemm(x, lg);
  run_pool(x, B, x.buf<void>(B_STASH), (long long)c.L * c.D, x.buf<float>(B_COEFF),
           x.buf<void>(B_MIXED), cache_k, cache_v, B, Tmax);
}

// The caller's per-row sequence and position arrays into the workspace.
cudaError_t copy_rows(const Ctx& x, const int32_t* seq, const int32_t* pos, int N) {
  cudaError_t e = cudaMemcpyAsync(x.buf<int32_t>(B_SEQ), seq, (size_t)N * 4,
                                  cudaMemcpyDeviceToDevice, x.st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(x.buf<int32_t>(B_POS), pos, (size_t)N * 4, cudaMemcpyDeviceToDevice, x.st);
  return e;
}

wm_status finish(const Ctx& x) {
  if (x.c->trace) x.c->trace->launches += x.launches;
  const cudaError_t e = cudaGetLastError();
  return (e == cudaSuccess && x.err == cudaSuccess) ? WM_OK : WM_ERR_CUDA;
}

// Device address of the allocation-free pool call's flag word (the first 256
// bytes of its scratch array), defined with that array at the end of the file.
void* pool_static_flags();

}  // namespace

extern "C" {

int32_t wm_abi_version(void) { return WM_ABI_VERSION; }

const char* wm_status_string(wm_status s) {
  switch (s) {
    case WM_OK: return "ok";
    case WM_ERR_INVALID_ARG: return "invalid argument";
    case WM_ERR_UNSUPPORTED: return "unsupported configuration";
    case WM_ERR_WORKSPACE: return "workspace too small or misaligned";
    case WM_ERR_CUDA: return "CUDA error";
    case WM_ERR_TIMEOUT: return "device-side wait timed out";
    case WM_ERR_DEVICE_BOUNDS: return "device-side index check failed";
  }
  return "unknown status";
}

size_t wm_workspace_size(const wm_config* cfg, int32_t max_rows, int32_t Tmax) {
  if (check_config(cfg) != WM_OK || max_rows < 1 || Tmax < 1) return 0;
  return make_layout(*cfg, max_rows, Tmax).total;
}

wm_status wm_pool_mix(const wm_config* cfg, const wm_weights* w, const void* states, int32_t N,
                      const int32_t* seq, const int32_t* pos, void* cache_k, void* cache_v,
                      int32_t B, int32_t Tmax, float* coeff_out, void* mixed_out, void* ws,
                      size_t ws_bytes, void* stream) {
  wm_status s;
  if ((s = check_config(cfg)) != WM_OK) return s;
  if ((s = check_weights(w)) != WM_OK) return s;
  if (N < 1 || B < 1 || Tmax < 1 || !states || !seq || !pos || !cache_k || !cache_v)
    return WM_ERR_INVALID_ARG;
  if (!aligned16(states) || !aligned16(cache_k) || !aligned16(cache_v) ||
      (coeff_out && !aligned16(coeff_out)) || (mixed_out && !aligned16(mixed_out)))
    return WM_ERR_INVALID_ARG;
  if ((s = check_ws(*cfg, ws, ws_bytes, N, Tmax)) != WM_OK) return s;
  Ctx x = make_ctx(cfg, w, ws, N, Tmax, stream);
  const wm_config& c = *cfg;
  if (copy_rows(x, seq, pos, N) != cudaSuccess) return WM_ERR_CUDA;
  ++x.launches;
  launch_rope_table(x.buf<float2>(B_ROPE), 0, Tmax, c.d, c.rope_base, x.st);
  zero_partials(x);
  ++x.launches;
  launch_norm_emit(c.dtype, states, (long long)c.L * c.D, c.D, N, 0, c.L, c.D, c.L, nullptr,
                   nullptr, x.buf<float>(B_INV), w->src_norm,
                   w->static_coeff ? nullptr : x.buf<void>(B_RIN), x.nR, c.p, c.p_offset, c.eps,
                   x.st);
  const int parts =
      run_pool(x, N, states, (long long)c.L * c.D, coeff_out ? coeff_out : x.buf<float>(B_COEFF),
               mixed_out ? mixed_out : x.buf<void>(B_MIXED), cache_k, cache_v, B, Tmax);
  if (mixed_out) finish_mixed(x, N, mixed_out, parts);
  return finish(x);
}

wm_status wm_channel_attn(const wm_config* cfg, const void* q, int32_t N, const int32_t* seq,
                          const int32_t* pos, int32_t channel, const void* cache_k,
                          const void* cache_v, int32_t B, int32_t Tmax, void* out,
                          int32_t rows_per_seq, void* ws, size_t ws_bytes, void* stream) {
  wm_status s;
  if ((s = check_config(cfg)) != WM_OK) return s;
  if (N < 1 || B < 1 || Tmax < 1 || !q || !seq || !pos || !cache_k || !cache_v || !out)
    return WM_ERR_INVALID_ARG;
  if (channel < 0 || channel >= cfg->k) return WM_ERR_INVALID_ARG;
  if (rows_per_seq < 0 || (rows_per_seq > 0 && N % rows_per_seq)) return WM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned16(cache_k) || !aligned16(cache_v))
    return WM_ERR_INVALID_ARG;
  if ((s = check_ws(*cfg, ws, ws_bytes, N, Tmax)) != WM_OK) return s;
  Ctx x = make_ctx(cfg, nullptr, ws, N, Tmax, stream);
  AttnArgs a;
  a.q = q; a.N = N; a.seq = seq; a.pos = pos; a.channel = channel;
  a.cache_k = cache_k; a.cache_v = cache_v; a.B = B; a.k = cfg->k; a.Hq = cfg->Hq;
  a.Hkv = cfg->Hkv; a.d = cfg->d; a.Tmax = Tmax; a.out = out; a.flags = x.flags();
  a.counters = x.buf<int>(B_CNT);
  a.counter_elems = (long long)(x.lay.off[B_CNT + 1] - x.lay.off[B_CNT]) / 4;
  cudaMemsetAsync(a.counters, 0, (size_t)a.counter_elems * 4, x.st);
  const int tr = trace_begin(x, WM_TRACE_ATTN);
  // one row per sequence: the decode engine, with Tmax as the bound on visible keys
  const long long pe = (long long)(x.lay.off[B_ATTNP + 1] - x.lay.off[B_ATTNP]) / 4;
  x.launches += launch_attention(cfg->dtype, a, !x.tc, x.st, rows_per_seq,
                                 rows_per_seq == 1 ? Tmax : 0, x.buf<float>(B_ATTNP), pe);
  trace_end(x, tr, 0.0);  // visible-key count is not known on the host here
  return finish(x);
}

wm_status wm_cyclic_pass(const wm_config* cfg, const wm_weights* w, const int32_t* tokens,
                         int32_t B, int32_t T, int32_t g, int32_t q_begin, int32_t q_end,
                         void* cache_k, void* cache_v, int32_t Tmax, float* logits,
                         int32_t logits_mode, void* ws, size_t ws_bytes, void* stream) {
  wm_status s;
  if ((s = check_config(cfg)) != WM_OK) return s;
  if ((s = check_weights(w)) != WM_OK) return s;
  if (!tokens || !cache_k || !cache_v || B < 1 || T < 1 || T > Tmax || g < 1 || g > T)
    return WM_ERR_INVALID_ARG;
  if (q_begin < 0 || q_end < q_begin || q_end > g) return WM_ERR_INVALID_ARG;
  if (logits_mode < WM_LOGITS_NONE || logits_mode > WM_LOGITS_ALL) return WM_ERR_INVALID_ARG;
  if (logits_mode != WM_LOGITS_NONE && (!logits || !aligned16(logits))) return WM_ERR_INVALID_ARG;
  if (!aligned16(cache_k) || !aligned16(cache_v)) return WM_ERR_INVALID_ARG;
  const long long nq_max = (T + g - 1) / g;
  if ((long long)B * nq_max > (1LL << 26)) return WM_ERR_INVALID_ARG;
  if ((s = check_ws(*cfg, ws, ws_bytes, B * nq_max, Tmax)) != WM_OK) return s;
  Ctx x = make_ctx(cfg, w, ws, B * nq_max, Tmax, stream);
  const wm_config& c = *cfg;
  ++x.launches;
  launch_rope_table(x.buf<float2>(B_ROPE), 0, T, c.d, c.rope_base, x.st);
  zero_partials(x);
  for (int q = q_begin; q < q_end; ++q) {
    const int nq = (T - q + g - 1) / g;
    const int N = B * nq;
    ++x.launches;
    launch_group_rows(tokens, B, T, g, q, nq, x.buf<int32_t>(B_TOK), x.buf<int32_t>(B_SEQ),
                      x.buf<int32_t>(B_POS), x.buf<int32_t>(B_ROWMAP), x.st);
    ++x.launches;
    launch_embed(c.dtype, x.buf<int32_t>(B_TOK), N, w->embed, c.V, c.D, x.buf<void>(B_STASH),
                 (long long)c.L * c.D, x.flags(), x.st);
    const bool has_last = (T - 1) % g == q;
    const bool want = logits_mode == WM_LOGITS_ALL || (logits_mode == WM_LOGITS_LAST && has_last);
    const double pos_sum = (double)B * ((double)nq * q + (double)g * nq * (nq - 1) / 2.0);
    run_stack(x, N, nq, pos_sum, want, cache_k, cache_v, B, Tmax, w->static_coeff == nullptr);
    if (want) {
      GemmDesc lg;
      lg.N = c.V; lg.K = c.D; lg.B = w->lm_head; lg.ldb = c.D;
      lg.epi = base_epi(x);
      lg.epi.mode = EPI_STORE;
      lg.epi.out_f32 = 1;
      lg.epi.C = logits; lg.epi.ldc = c.V;
      if (logits_mode == WM_LOGITS_ALL) {
        ++x.launches;
        launch_rmsnorm(c.dtype, x.buf<void>(B_HL), c.D, 0, 1, N, c.D, w->final_norm,
                       x.buf<void>(B_LASTX), c.eps, x.st);
        lg.M = N; lg.A = x.buf<void>(B_LASTX); lg.lda = c.D;
        lg.epi.rowmap = x.buf<int>(B_ROWMAP);
      } else {
        ++x.launches;
        launch_rmsnorm(c.dtype, x.buf<void>(B_HL), c.D, (T - 1 - q) / g, nq, B, c.D,
                       w->final_norm, x.buf<void>(B_LASTX), c.eps, x.st);
        lg.M = B; lg.A = x.buf<void>(B_LASTX); lg.lda = c.D;
      }
      ++x.launches;
      gemm(x, lg);
    }
    run_pool(x, N, x.buf<void>(B_STASH), (long long)c.L * c.D, x.buf<float>(B_COEFF),
             x.buf<void>(B_MIXED), cache_k, cache_v, B, Tmax);
  }
  return finish(x);
}

wm_status wm_feedforward_pass(const wm_config* cfg, const wm_weights* w, const int32_t* tokens,
                              int32_t B, int32_t T, int32_t pos0, void* cache_k, void* cache_v,
                              int32_t Tmax, float* logits, int32_t logits_mode, void* ws,
                              size_t ws_bytes, void* stream) {
  wm_status s;
  if ((s = check_config(cfg)) != WM_OK) return s;
  if ((s = check_weights(w)) != WM_OK) return s;
  if (cfg->k != cfg->L) return WM_ERR_INVALID_ARG;  // one channel per layer
  if (!tokens || !cache_k || !cache_v || B < 1 || T < 1 || pos0 < 0 || (long long)pos0 + T > Tmax)
    return WM_ERR_INVALID_ARG;
  if (logits_mode < WM_LOGITS_NONE || logits_mode > WM_LOGITS_ALL) return WM_ERR_INVALID_ARG;
  if (logits_mode != WM_LOGITS_NONE && (!logits || !aligned16(logits))) return WM_ERR_INVALID_ARG;
  if (!aligned16(cache_k) || !aligned16(cache_v)) return WM_ERR_INVALID_ARG;
  if ((long long)T > (1LL << 26)) return WM_ERR_INVALID_ARG;
  // sequences per chunk: as many as the workspace holds rows for (at least one)
  int nb = B;
  while (nb > 1 && make_layout(*cfg, (long long)nb * T, Tmax).total > ws_bytes) nb = (nb + 1) / 2;
  if ((s = check_ws(*cfg, ws, ws_bytes, (long long)nb * T, Tmax)) != WM_OK) return s;
  Ctx x = make_ctx(cfg, w, ws, (long long)nb * T, Tmax, stream);
  const wm_config& c = *cfg;
  ++x.launches;
  launch_rope_table(x.buf<float2>(B_ROPE), pos0, pos0 + T, c.d, c.rope_base, x.st);
  zero_partials(x);
  const long long seq_bytes = (long long)c.k * c.Hkv * Tmax * c.d * x.es;
  for (int b0 = 0; b0 < B; b0 += nb) {
    const int nbc = B - b0 < nb ? B - b0 : nb;
    const int N = nbc * T;
    char* ck = static_cast<char*>(cache_k) + b0 * seq_bytes;
    char* cv = static_cast<char*>(cache_v) + b0 * seq_bytes;
    ++x.launches;
    launch_group_rows(tokens + (long long)b0 * T, nbc, T, 1, 0, T, x.buf<int32_t>(B_TOK),
                      x.buf<int32_t>(B_SEQ), x.buf<int32_t>(B_POS), x.buf<int32_t>(B_ROWMAP), x.st,
                      pos0);
    ++x.launches;
    launch_embed(c.dtype, x.buf<int32_t>(B_TOK), N, w->embed, c.V, c.D, x.buf<void>(B_STASH),
                 (long long)c.L * c.D, x.flags(), x.st);
    const bool want = logits_mode != WM_LOGITS_NONE;
    const double pos_sum = (double)nbc * ((double)T * pos0 + (double)T * (T - 1) / 2.0);
    run_stack(x, N, T, pos_sum, want, ck, cv, nbc, Tmax, w->static_coeff == nullptr, true);
    if (want) {
      GemmDesc lg;
      lg.N = c.V; lg.K = c.D; lg.B = w->lm_head; lg.ldb = c.D;
      lg.epi = base_epi(x);
      lg.epi.mode = EPI_STORE;
      lg.epi.out_f32 = 1;
      lg.epi.ldc = c.V;
      if (logits_mode == WM_LOGITS_ALL) {
        ++x.launches;
        launch_rmsnorm(c.dtype, x.buf<void>(B_HL), c.D, 0, 1, N, c.D, w->final_norm,
                       x.buf<void>(B_LASTX), c.eps, x.st);
        lg.M = N; lg.A = x.buf<void>(B_LASTX); lg.lda = c.D;
        lg.epi.rowmap = x.buf<int>(B_ROWMAP);
        lg.epi.C = logits + (long long)b0 * T * c.V;
      } else {
        ++x.launches;
        launch_rmsnorm(c.dtype, x.buf<void>(B_HL), c.D, T - 1, T, nbc, c.D, w->final_norm,
                       x.buf<void>(B_LASTX), c.eps, x.st);
        lg.M = nbc; lg.A = x.buf<void>(B_LASTX); lg.lda = c.D;
        lg.epi.C = logits + (long long)b0 * c.V;
      }
      ++x.launches;
      gemm(x, lg);
    }
  }
  return finish(x);
}

size_t wm_pool_backward_workspace_size(const wm_config* cfg, int32_t max_rows) {
  if (check_config(cfg) != WM_OK || max_rows < 1) return 0;
  return pool_bwd_layout(*cfg, max_rows).total;
}

wm_status wm_pool_backward(const wm_config* cfg, const wm_weights* w, const void* states,
                           int32_t N, const int32_t* pos, const void* dK, const void* dV,
                           float* dstates, const wm_pool_grads* grads, void* ws, size_t ws_bytes,
                           void* stream) {
  wm_status s;
  if ((s = check_config(cfg)) != WM_OK) return s;
  if ((s = check_weights(w)) != WM_OK) return s;
  if (N < 1 || !states || !pos || !dK || !dV || !dstates || !grads) return WM_ERR_INVALID_ARG;
  if (!grads->dWk || !grads->dWv || !grads->dsrc_norm || !grads->dchan_norm || !grads->dk_norm)
    return WM_ERR_INVALID_ARG;
  if ((long long)cfg->k * cfg->L > 1024 || cfg->D > 8192) return WM_ERR_INVALID_ARG;
  if (!aligned16(states) || !aligned16(dK) || !aligned16(dV) || !aligned16(dstates))
    return WM_ERR_INVALID_ARG;
  const PoolBwdLayout lay = pool_bwd_layout(*cfg, N);
  if (!ws || ((uintptr_t)ws & 255u) || ws_bytes < lay.total) return WM_ERR_WORKSPACE;
  PoolBwdArgs q;
  q.cfg = cfg; q.w = w; q.states = states; q.N = N; q.pos = pos; q.dK = dK; q.dV = dV;
  q.dstates = dstates; q.g = *grads; q.ws = ws; q.lay = lay;
  const cudaError_t e = run_pool_backward(q, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WM_OK : WM_ERR_CUDA;
}

wm_status wm_decode_step(const wm_config* cfg, const wm_weights* w, const int32_t* tokens,
                         int32_t B, int32_t pos, void* cache_k, void* cache_v, int32_t Tmax,
                         float* logits, void* ws, size_t ws_bytes, void* stream) {
  wm_status s;
  if ((s = check_config(cfg)) != WM_OK) return s;
  if ((s = check_weights(w)) != WM_OK) return s;
  if (!tokens || !cache_k || !cache_v || !logits || B < 1 || pos < 0 || pos >= Tmax)
    return WM_ERR_INVALID_ARG;
  if (!aligned16(cache_k) || !aligned16(cache_v) || !aligned16(logits)) return WM_ERR_INVALID_ARG;
  if ((s = check_ws(*cfg, ws, ws_bytes, B, Tmax)) != WM_OK) return s;
  Ctx x = make_ctx(cfg, w, ws, B, Tmax, stream);
  const wm_config& c = *cfg;
  ++x.launches;
  launch_rope_table(x.buf<float2>(B_ROPE), pos, pos + 1, c.d, c.rope_base, x.st);
  ++x.launches;
  launch_decode_rows(tokens, B, pos, x.buf<int32_t>(B_TOK), x.buf<int32_t>(B_SEQ),
                     x.buf<int32_t>(B_POS), x.st);
  decode_body(x, B, (double)B * pos, cache_k, cache_v, Tmax, logits);
  return finish(x);
}

wm_status wm_decode_batch(const wm_config* cfg, const wm_weights* w, const int32_t* tokens,
                          const int32_t* pos, int32_t B, void* cache_k, void* cache_v, int32_t Tmax,
                          float* logits, void* ws, size_t ws_bytes, void* stream) {
  wm_status s;
  if ((s = check_config(cfg)) != WM_OK) return s;
  if ((s = check_weights(w)) != WM_OK) return s;
  if (!tokens || !pos || !cache_k || !cache_v || !logits || B < 1 || Tmax < 1)
    return WM_ERR_INVALID_ARG;
  if (!aligned16(cache_k) || !aligned16(cache_v) || !aligned16(logits)) return WM_ERR_INVALID_ARG;
  if ((s = check_ws(*cfg, ws, ws_bytes, B, Tmax)) != WM_OK) return s;
  Ctx x = make_ctx(cfg, w, ws, B, Tmax, stream);
  const wm_config& c = *cfg;
  ++x.launches;
  launch_decode_rows_dev(tokens, pos, B, c.d, c.rope_base, x.buf<int32_t>(B_TOK),
                         x.buf<int32_t>(B_SEQ), x.buf<int32_t>(B_POS), x.buf<float2>(B_ROPE), Tmax,
                         x.st);
  // the host knows only the bound on visible keys
  decode_body(x, B, (double)B * Tmax, cache_k, cache_v, Tmax, logits);
  return finish(x);
}

wm_status wm_check_flags(void* ws, size_t ws_bytes, uint32_t* flags_out, void* stream) {
  if (!flags_out) return WM_ERR_INVALID_ARG;
  if (!ws && ws_bytes == 0) {
    // the flag word of the allocation-free pool call (wm_pool_mix_static)
    ws = pool_static_flags();
    if (!ws) return WM_ERR_CUDA;
    ws_bytes = 256;
  }
  if (!ws || ws_bytes < 256 || ((uintptr_t)ws & 255u)) return WM_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t f = 0;
  if (cudaMemcpyAsync(&f, ws, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess) return WM_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return WM_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, 4, st) != cudaSuccess) return WM_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return WM_ERR_CUDA;
  *flags_out = f;
  if (f & FLAG_TIMEOUT) return WM_ERR_TIMEOUT;
  if (f & (FLAG_BAD_TOKEN | FLAG_BAD_SEQ | FLAG_BAD_POS)) return WM_ERR_DEVICE_BOUNDS;
  return WM_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// wm_pool_mix_static: the pool without a caller workspace.
//
// For callers that cannot allocate device memory themselves: a plug-in host
// that hands the library nothing but its input and output pointers, or a
// latency-bound loop that must not call cudaMalloc (which synchronises the
// device). The pool's scratch (router inputs, per-source inverse RMS,
// coefficients, mixed channels, RoPE table, flag word) lives instead in one
// file-scope device array of WM_POOL_STATIC_SCRATCH_BYTES, which every GPU
// that loads the library holds until the process exits.
// ---------------------------------------------------------------------------
namespace {

__device__ __align__(256) unsigned char g_pool_scratch[WM_POOL_STATIC_SCRATCH_BYTES];

// Device address of g_pool_scratch on the current device. In host code the
// symbol is only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress, once per device, with that device current.
void* pool_scratch_address() {
  static std::mutex mu;
  static void* addr[256] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pool_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

void* pool_static_flags() { return pool_scratch_address(); }

// Compact layout: only the buffers the pool touches.
Layout pool_static_layout(const wm_config& c, long long N, long long Tmax) {
  const size_t es = elem_size(c.dtype);
  const long long nR = count_nR(c);
  Layout lay;
  for (int i = 0; i < NBUF; ++i) lay.off[i] = 0;
  size_t o = 0;
  auto put = [&](Buf b, size_t bytes) {
    lay.off[b] = o;
    o += align256(bytes);
  };
  put(B_FLAGS, 256);
  put(B_ROPE, (size_t)Tmax * (c.d / 2) * sizeof(float2));
  put(B_SEQ, (size_t)N * 4);
  put(B_POS, (size_t)N * 4);
  put(B_RIN, (size_t)2 * N * nR * c.D * es);
  put(B_INV, (size_t)N * c.L * 4);
  put(B_COEFF, (size_t)N * 2 * c.k * c.L * 4);
  put(B_MIXED, (size_t)N * 2 * c.k * c.D * es);
  put(B_CHSS, (size_t)N * 2 * c.k * 8 * 4);
  put(B_ATILE, c.dtype == WM_BF16 ? (size_t)N * MIX_ATILE_BYTES : 0);
  lay.off[B_ATILE + 1] = o;  // marks the end of the tile scratch
  lay.total = o;
  return lay;
}

}  // namespace

extern "C" wm_status wm_pool_mix_static(const wm_config* cfg, const wm_weights* w,
                                        const void* states, int32_t N, const int32_t* seq,
                                        const int32_t* pos, void* cache_k, void* cache_v,
                                        int32_t B, int32_t Tmax, float* coeff_out,
                                        void* mixed_out, void* stream) {
  wm_status s;
  if ((s = check_config(cfg)) != WM_OK) return s;
  if ((s = check_weights(w)) != WM_OK) return s;
  if (N < 1 || B < 1 || Tmax < 1 || !states || !seq || !pos || !cache_k || !cache_v)
    return WM_ERR_INVALID_ARG;
  if (!aligned16(states) || !aligned16(cache_k) || !aligned16(cache_v) ||
      (coeff_out && !aligned16(coeff_out)) || (mixed_out && !aligned16(mixed_out)))
    return WM_ERR_INVALID_ARG;
  const Layout lay = pool_static_layout(*cfg, N, Tmax);
  if (lay.total > (size_t)WM_POOL_STATIC_SCRATCH_BYTES) return WM_ERR_WORKSPACE;
  void* base = pool_scratch_address();
  if (!base) return WM_ERR_CUDA;
  Ctx x = make_ctx(cfg, w, base, N, Tmax, stream);
  x.lay = lay;
  const wm_config& c = *cfg;
  // the previous call's flag bits must not leak into this one
  if (cudaMemsetAsync(x.flags(), 0, 256, x.st) != cudaSuccess) return WM_ERR_CUDA;
  if (copy_rows(x, seq, pos, N) != cudaSuccess) return WM_ERR_CUDA;
  ++x.launches;
  launch_rope_table(x.buf<float2>(B_ROPE), 0, Tmax, c.d, c.rope_base, x.st);
  ++x.launches;
  launch_norm_emit(c.dtype, states, (long long)c.L * c.D, c.D, N, 0, c.L, c.D, c.L, nullptr,
                   nullptr, x.buf<float>(B_INV), w->src_norm,
                   w->static_coeff ? nullptr : x.buf<void>(B_RIN), x.nR, c.p, c.p_offset, c.eps,
                   x.st);
  const int parts =
      run_pool(x, N, states, (long long)c.L * c.D, coeff_out ? coeff_out : x.buf<float>(B_COEFF),
               mixed_out ? mixed_out : x.buf<void>(B_MIXED), cache_k, cache_v, B, Tmax);
  if (mixed_out) finish_mixed(x, N, mixed_out, parts);
  return finish(x);
}
