/*
 * wm.h - C ABI of libwm, the B300 (sm_103a) implementation of the WhiteMatter
 * cross-layer KV pool and its cyclic Gauss-Seidel prefill / decode schedule.
 *
 * Sources (public pages about arXiv 2608.18486, "WhiteMatter: All-to-All
 * Cross-Layer Connections via KV Mixing"), cited by tag and section:
 *   [PL] paperlayer.ai summary, sections "3 METHOD" and "5 ANALYSIS";
 *   [OD] onedev.kr review "WhiteMatter가 모든 층의 KV 재사용으로 캐시를 절반으로
 *        줄인다", sections "How it works" (어떻게 동작하나), "How it differs"
 *        (무엇과 다른가) and "How it is used" (어떻게 쓰나).
 *
 * Conventions for every entry point
 *  - Pointers named in a weights struct or as tensors are DEVICE pointers,
 *    caller-owned, row-major, 16-byte aligned, in the storage type chosen by
 *    wm_config.dtype (fp32 or bf16) unless stated otherwise. Integer arrays are
 *    int32 device arrays. ``stream`` is a cudaStream_t (NULL = legacy stream).
 *  - The library allocates no memory and keeps no state between calls. All
 *    scratch lives in the caller's workspace ``ws`` of ``ws_bytes`` bytes
 *    (device memory, 256-byte aligned, size from wm_workspace_size). Calls
 *    that share one workspace must not overlap on the GPU.
 *  - Calls are asynchronous on ``stream``. The returned status covers argument
 *    validation and kernel launch only; on any error nothing is launched.
 *    Device-side checks (token ids, sequence indices, positions out of range)
 *    skip the offending access and set bits in the workspace's flag word, read
 *    (and cleared) by wm_check_flags after the work.
 *  - Every device-side wait is bounded (4 s). A wait that gives up sets the
 *    timeout bit of the flag word; each later kernel of the same call that
 *    holds bounded waits reads that bit at entry and returns without work, so
 *    one timeout costs at most one wait limit per kernel in flight, not one
 *    per launch. Results of a call that timed out are unspecified.
 *  - Cache layout: cache_k and cache_v are [B][k][Hkv][Tmax][d] each. Keys are
 *    stored after K-norm and RoPE, values raw ([PL 3 METHOD, "Cross-layer KV
 *    pool"]: stored keys are rotated and K-normalised, values stay raw; the
 *    cache holds k*T*Hkv*d elements). The caller initialises the cache (zeros
 *    for a fresh prefill); entry points write only the positions they process.
 */
#ifndef WM_H
#define WM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define WM_ABI_VERSION 1

typedef enum {
    WM_OK = 0,
    WM_ERR_INVALID_ARG = 1,   /* null pointer, bad size or range, misalignment */
    WM_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. d not 64/128)  */
    WM_ERR_WORKSPACE = 3,     /* ws too small or misaligned                     */
    WM_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed              */
    WM_ERR_TIMEOUT = 5,       /* a bounded device-side wait gave up             */
    WM_ERR_DEVICE_BOUNDS = 6  /* device-side index check failed (wm_check_flags) */
} wm_status;

typedef enum { WM_F32 = 0, WM_BF16 = 1 } wm_dtype;

typedef enum {
    WM_LOGITS_NONE = 0,       /* no logits                                       */
    WM_LOGITS_LAST = 1,       /* logits of position T-1 of each sequence, [B][V] */
    WM_LOGITS_ALL = 2         /* logits of every position, [B][T][V]             */
} wm_logits_mode;

/* Engine flags (wm_config.flags). */
#define WM_FLAG_SIMT_GEMM 1u  /* run every contraction on CUDA cores (debug aid) */
#define WM_FLAG_NO_CLUSTER 2u /* few-row products split K with fp32 atomics and a
                                 finalize kernel instead of a thread-block
                                 cluster (the path taken where a cluster does
                                 not fit; a test aid elsewhere) */
#define WM_FLAG_WAIT_PROBE 4u /* test aid for the timeout path: before its first
                                 product, each CTA of the tensor-core GEMM
                                 engine waits on a barrier that nothing
                                 completes, with a 2 ms limit. The wait runs
                                 out, the kernel raises the timeout bit, drains
                                 its copies and returns; every later kernel of
                                 the call that holds bounded waits finds the
                                 bit at entry and returns at once. The call's
                                 results are then unspecified and
                                 wm_check_flags reports WM_ERR_TIMEOUT. */

/* Optional measurement hook (wm_config.trace, nullable). While entries
 * remain, an entry point records begin[i] / end[i] (caller-created
 * cudaEvent_t handles) on its stream immediately before and after each launch
 * of the selected kernel class, stores the launch's algorithmic work in
 * work[i] and advances ``count``. Work is FLOPs for the contraction engine
 * (2*M*N*K per product) and for attention (4*Hq*d per visible key of every
 * row), and bytes read plus written for the mixer. */
typedef enum { WM_TRACE_GEMM = 0, WM_TRACE_MIX = 1, WM_TRACE_ATTN = 2 } wm_trace_kind;
typedef struct {
    int32_t kind;        /* wm_trace_kind                                       */
    int32_t capacity;    /* event pairs available                               */
    int32_t count;       /* in/out: entries used                                */
    int32_t reserved;
    void* const* begin;  /* cudaEvent_t[capacity]                               */
    void* const* end;    /* cudaEvent_t[capacity]                               */
    double* work;        /* [capacity] algorithmic work of each traced launch   */
    int64_t launches;    /* in/out: every kernel launched by calls that carry
                          * this trace (all classes) is counted here          */
} wm_trace;

/* Model shape. The router reads the source states l < L with
 * l % p == p_offset ([OD How it works]: the router reads every p-th layer's
 * state, stride p = 2, yet emits weights for all L layers). */
typedef struct {
    int32_t L;          /* layers = source states per token                    */
    int32_t D;          /* model width, multiple of 64, at most 8192           */
    int32_t k;          /* pool channels, 1 <= k <= L                          */
    int32_t p;          /* router stride, >= 1                                 */
    int32_t p_offset;   /* first router source, 0 <= p_offset < p             */
    int32_t Hq;         /* query heads                                         */
    int32_t Hkv;        /* KV heads, divides Hq                                */
    int32_t d;          /* head size, 64 or 128                                */
    int32_t F;          /* SwiGLU width, multiple of 64                        */
    int32_t V;          /* vocabulary                                          */
    float eps;          /* RMSNorm epsilon                                     */
    float rope_base;    /* RoPE base                                           */
    int32_t dtype;      /* wm_dtype: storage and GEMM operand type             */
    uint32_t flags;     /* WM_FLAG_* engine flags                              */
    wm_trace* trace;    /* nullable measurement hook (host memory)            */
} wm_config;

/* Weights (device pointers, storage type). nR = number of router sources.
 * Matrices are [out][in]: y = W x. Gains are RMSNorm weights. */
typedef struct {
    const void* embed;       /* [V][D]                                          */
    const void* lm_head;     /* [V][D]                                          */
    const void* final_norm;  /* [D]                                             */
    const void* in_norm;     /* [L][D]   layer input norm                       */
    const void* post_norm;   /* [L][D]   norm before the FFN                    */
    const void* q_norm;      /* [L][d]   per-head query norm                    */
    const void* Wq;          /* [L][Hq*d][D]                                    */
    const void* Wo;          /* [L][D][Hq*d]                                    */
    const void* Wgate;       /* [L][F][D]                                       */
    const void* Wup;         /* [L][F][D]                                       */
    const void* Wdown;       /* [L][D][F]                                       */
    const void* src_norm;    /* [2][L][D]  per-source gains, branch 0 = K, 1 = V */
    const void* Wr;          /* [2][k*L][nR*D]  router, output index j*L + l    */
    const void* chan_norm;   /* [2][k][D]  per-channel gains                    */
    const void* Wk;          /* [k][Hkv*d][D]  channel key projections           */
    const void* Wv;          /* [k][Hkv*d][D]  channel value projections         */
    const void* k_norm;      /* [k][d]   per-channel key norm gains             */
    const float* static_coeff; /* nullable fp32 [2][k][L]: when set, these
                              * constant mixing weights replace the router for
                              * every token (static-mixing variant, [PL 5
                              * ANALYSIS, "Dynamic routing"])                   */
} wm_weights;

/* Bytes of workspace needed by calls that process up to ``max_rows`` token
 * rows at once against a cache of ``Tmax`` positions. For wm_cyclic_pass the
 * rows of one group are B * ceil(T/g); for wm_decode_step they are B. */
size_t wm_workspace_size(const wm_config* cfg, int32_t max_rows, int32_t Tmax);

/* The cross-layer KV pool for N token rows ([OD How it works]; [PL 3 METHOD,
 * "Cross-layer KV pool"]). For each row n, with states[n] = its L layer
 * states [L][D] (the inputs of layers 0..L-1), per branch b in {K, V}:
 *   n_l   = RMSNorm(h_l; src_norm[b][l])
 *   a     = Wr[b] . concat_{l in R} n_l   viewed [k][L]  (signed, no softmax)
 *   m_j   = sum_l a[j][l] n_l ;  c_j = RMSNorm(m_j; chan_norm[b][j])
 * then K_j = RoPE_pos(RMSNorm_d(Wk[j] c^K_j per head; k_norm[j])) and
 * V_j = Wv[j] c^V_j are written to cache_{k,v}[seq[n]][j][:][pos[n]][:].
 * states: [N][L][D]; seq, pos: [N] with seq < B, pos < Tmax.
 * coeff_out (nullable): fp32 [N][2][k][L] router output (or static weights).
 * mixed_out (nullable): [2][k][N][D] channel-normed mixtures c, channel-major
 * (branch, channel, row), the operand layout of the channel projections.
 * Rows must have distinct (seq, pos) pairs. */
wm_status wm_pool_mix(const wm_config* cfg, const wm_weights* w,
                      const void* states, int32_t N,
                      const int32_t* seq, const int32_t* pos,
                      void* cache_k, void* cache_v, int32_t B, int32_t Tmax,
                      float* coeff_out, void* mixed_out,
                      void* ws, size_t ws_bytes, void* stream);

/* Strictly causal attention of N query rows to one cache channel ([OD How it
 * differs]: token i attends only to s < i; [PL 3 METHOD, "Per-layer channel
 * selection"]: layer l reads channel l mod k, which the caller passes here).
 * q: [N][Hq][d], already q-normed and rotated; row n sees keys s < pos[n] of
 * sequence seq[n]; query head h reads KV head h*Hkv/Hq; scale 1/sqrt(d); a row
 * with pos = 0 gets 0. out: [N][Hq*d].
 * rows_per_seq: 0, or a declaration that the rows come as N / rows_per_seq
 * runs of rows_per_seq consecutive rows of one sequence each (the shape of a
 * cyclic group); it selects the tensor-core kernel. If the declaration is
 * false the results are unspecified, but no access leaves the given arrays. */
wm_status wm_channel_attn(const wm_config* cfg, const void* q, int32_t N,
                          const int32_t* seq, const int32_t* pos, int32_t channel,
                          const void* cache_k, const void* cache_v,
                          int32_t B, int32_t Tmax, void* out, int32_t rows_per_seq,
                          void* ws, size_t ws_bytes, void* stream);

/* Groups q_begin..q_end-1 of one cyclic Gauss-Seidel pass over tokens [B][T]
 * ([OD How it differs]: positions split into G_q = {i : i mod g = q}, groups in
 * order q = 0..g-1, parallel inside a group, the cache updated after every
 * group). Each group runs the whole layer stack of its B*|G_q| rows against
 * the cache as it stood before the group, then writes their pooled channels
 * at their positions. g = 1 is a Jacobi pass, g = T exact autoregressive
 * evaluation. 1 <= g <= T <= Tmax; 0 <= q_begin <= q_end <= g.
 * logits (fp32, nullable unless logits_mode != NONE): LAST -> [B][V] for
 * position T-1, computed by the group that holds it; ALL -> [B][T][V].
 * When logits_mode is NONE the last layer, whose output feeds only the LM
 * head, is not evaluated. */
wm_status wm_cyclic_pass(const wm_config* cfg, const wm_weights* w,
                         const int32_t* tokens, int32_t B, int32_t T, int32_t g,
                         int32_t q_begin, int32_t q_end,
                         void* cache_k, void* cache_v, int32_t Tmax,
                         float* logits, int32_t logits_mode,
                         void* ws, size_t ws_bytes, void* stream);

/* The feedback-free variant ([PL 5 ANALYSIS, "Deep-to-shallow feedback"]: a
 * full cache, one channel per layer, no deep-to-shallow pathway, no
 * iteration). Requires k = L. Channel l of a token mixes only its states
 * h^0..h^l: the router reads the sources of R inside 0..l (rows l*L + 0..l of
 * W_R, the other inputs unused) or static_coeff[b][l][0..l], and the channel is
 * pooled and written to the cache right before layer l runs, for all rows;
 * layer l then attends to channel l at positions s < pos. One call is one
 * exact evaluation of tokens [B][T] at positions pos0..pos0+T-1 against a
 * cache already holding positions < pos0 (T = 1 is a decode step).
 * logits as for wm_cyclic_pass (LAST -> [B][V] at pos0+T-1, ALL -> [B][T][V]).
 * The workspace may hold fewer rows than B*T: whole sequences are processed
 * in chunks that fit (at least one sequence, T rows). Errors as for
 * wm_cyclic_pass; k != L is WM_ERR_INVALID_ARG. */
wm_status wm_feedforward_pass(const wm_config* cfg, const wm_weights* w,
                              const int32_t* tokens, int32_t B, int32_t T, int32_t pos0,
                              void* cache_k, void* cache_v, int32_t Tmax,
                              float* logits, int32_t logits_mode,
                              void* ws, size_t ws_bytes, void* stream);

/* Gradient accumulators of the pool's parameters (fp32 device pointers, added
 * to, so a caller may sum over groups and steps; zero them to start). */
typedef struct {
    float* dWr;          /* [2][k*L][nR*D]  nullable: router gradient skipped  */
    float* dWk;          /* [k][Hkv*d][D]                                      */
    float* dWv;          /* [k][Hkv*d][D]                                      */
    float* dsrc_norm;    /* [2][L][D]                                          */
    float* dchan_norm;   /* [2][k][D]                                          */
    float* dk_norm;      /* [k][d]                                             */
} wm_pool_grads;

/* Bytes of workspace wm_pool_backward needs for up to ``max_rows`` rows; 0
 * for an invalid configuration. */
size_t wm_pool_backward_workspace_size(const wm_config* cfg, int32_t max_rows);

/* Backward pass of the pool ([PL 3 METHOD, "Cross-layer KV pool"]; the
 * gradients of a training schedule, [PL 4 EXPERIMENTS]) for N token rows:
 * given the layer states the pool read (states [N][L][D], storage type), the
 * rows' positions (pos [N], for RoPE) and the upstream gradients of their
 * cached channels (dK, dV [N][k][Hkv][d], storage type), recompute the pool in
 * fp32 and write dstates [N][L][D] (fp32, overwritten: the gradient of the
 * pool's outputs with respect to every layer state of each row) and add the
 * parameter gradients to ``grads``. With static_coeff set the router is not
 * used and dWr is left alone. Every step runs in this library's kernels; the
 * router and channel-projection products run on the tensor cores with exact
 * bf16 hi/lo operand splits (three bf16 products per fp32 one, summed in
 * fp32: within ~1e-5 of fp32 products). The workspace begins with a flag word
 * (wm_check_flags reads and clears it): a bounded wait of those products that
 * gives up sets its timeout bit. Errors: WM_ERR_INVALID_ARG (null or
 * misaligned pointers, N < 1, k * L > 1024, D > 8192), WM_ERR_WORKSPACE,
 * WM_ERR_CUDA (a failed launch). */
wm_status wm_pool_backward(const wm_config* cfg, const wm_weights* w,
                           const void* states, int32_t N, const int32_t* pos,
                           const void* dK, const void* dV, float* dstates,
                           const wm_pool_grads* grads,
                           void* ws, size_t ws_bytes, void* stream);

/* One autoregressive decode step at position ``pos`` for tokens [B]
 * ([PL 3 METHOD, "Execution schedules"]: a token's pooled channels are
 * appended only after its layer stack). The stack attends to s < pos, then
 * the token's channels are written at pos. logits: fp32 [B][V]. */
wm_status wm_decode_step(const wm_config* cfg, const wm_weights* w,
                         const int32_t* tokens, int32_t B, int32_t pos,
                         void* cache_k, void* cache_v, int32_t Tmax,
                         float* logits, void* ws, size_t ws_bytes, void* stream);

/* wm_decode_step with per-sequence positions read on the device: sequence b
 * of the batch appends its token tokens[b] at pos[b] (both int32 device
 * arrays [B]), attends to its keys s < pos[b] and gets logits[b]. Sequences
 * may sit at different positions. No host-side value depends on the device
 * arrays, so the call can be recorded once into a CUDA graph and replayed,
 * the caller updating tokens and pos in place between replays. A pos[b]
 * outside [0, Tmax) sets the position check bit (see wm_check_flags) and
 * that sequence's cache is left alone. */
wm_status wm_decode_batch(const wm_config* cfg, const wm_weights* w,
                          const int32_t* tokens, const int32_t* pos, int32_t B,
                          void* cache_k, void* cache_v, int32_t Tmax,
                          float* logits, void* ws, size_t ws_bytes, void* stream);

/* Waits for ``stream``, copies the workspace flag word to *flags_out (host)
 * and clears it. Returns WM_ERR_DEVICE_BOUNDS if an index check failed and
 * WM_ERR_TIMEOUT if a bounded wait gave up since the last call.
 * ws = NULL with ws_bytes = 0 selects the flag word that wm_pool_mix_static
 * keeps in its internal scratch (on the current device). */
wm_status wm_check_flags(void* ws, size_t ws_bytes, uint32_t* flags_out, void* stream);

/* wm_pool_mix without a workspace, for callers that cannot allocate device
 * memory: a plug-in host that hands the library only its input and output
 * pointers, or a loop that must not call cudaMalloc because that
 * synchronises the device. (The pages have no counterpart of this call; it
 * computes exactly what wm_pool_mix computes, with the same arguments minus
 * ws / ws_bytes.)
 *
 * Scratch: one device array of WM_POOL_STATIC_SCRATCH_BYTES inside the
 * library, held by every GPU that loads the library until the process exits.
 * It holds a 256-byte flag word, the RoPE table (4*d*Tmax bytes) and, per
 * row, 8 + 2*e*nR*D + 4*L + 8*k*L + 2*e*k*D + 64*k bytes, where e is the
 * storage element size (2 for bf16, 4 for fp32); each of those seven
 * per-row buffers is rounded up to a multiple of 256 bytes (at most 7*255
 * more in all). Calls whose rows do not fit return WM_ERR_WORKSPACE before
 * anything is launched. The call itself allocates
 * nothing: no cudaMalloc, cudaFree or allocating library routine.
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture. Every call shares the one array and finds the
 * previous call's contents there; the call clears what must start at zero
 * (its flag word) itself. Calls that overlap on the GPU - on different
 * streams, or from different host threads - race on the array and must be
 * serialised by the caller. Device-side checks of this call (index bounds,
 * bounded waits) set bits in its internal flag word, which the call clears
 * at its start; read it with wm_check_flags(NULL, 0, &flags, stream). */
#define WM_POOL_STATIC_SCRATCH_BYTES (32u << 20)
wm_status wm_pool_mix_static(const wm_config* cfg, const wm_weights* w,
                             const void* states, int32_t N,
                             const int32_t* seq, const int32_t* pos,
                             void* cache_k, void* cache_v, int32_t B, int32_t Tmax,
                             float* coeff_out, void* mixed_out, void* stream);

const char* wm_status_string(wm_status s);
int32_t wm_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* WM_H */
