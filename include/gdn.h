/*
 * gdn.h -- C ABI of libgdn.so: the Gated DeltaNet forward on one NVIDIA
 * GB300 (sm_103a), chunk-wise parallel prefill and single-token decode step.
 *
 * Sources (web pages on Gated DeltaNet):
 *  [Lab3]  "Lab3 GDN Prefill" (hpc101.zjusct.io).
 *          Section "Linear Attention 与 Gated DeltaNet": the gated delta rule
 *            S_t = alpha_t (I - beta_t k_t^T k_t) S_{t-1} + beta_t k_t^T v_t,
 *            o_t = q_t S_t (row vectors; S is dk x dv).
 *          Section "计算过程描述": the chunk form with C = 64,
 *            A = (I + StrictLower(B Gamma K K^T Gamma^-1))^-1,
 *            U = A B V, W = A B Gamma K,
 *            S_[c+1] = gamma_l S_[c] + gamma_l K^T Gamma^-1 (U - W S_[c]),
 *            O_[c] = (1/sqrt dk)[Gamma Q S_[c] + Gamma Lower(Q K^T) Gamma^-1 (U - W S_[c])],
 *            valid chunk length l_c = min(C, L - cC), tail columns masked.
 *          Section "输入输出定义": tensor interface, raw_g = log(alpha) with a
 *            prefix sum restarted at every chunk, optional initial state,
 *            GVA head map h_qk = floor(h_v / (Hv / Hq)).
 *  [SGL]   "sgl-qwen3-5-moe" (rainlin-net), decode node 7
 *          (gdn_packed_recurrent_qk_norm_gating_state_update): one token,
 *          decay -> predict -> correct -> read, state held in f32; its
 *          steps one and two: q/k L2 norm with eps 1e-6 inside the root and
 *          the query scale, gates g = -exp(A_log) softplus(a + dt_bias),
 *          beta = sigmoid(b).
 *  [Kestrel] "Kestrel_VLLM-24 · GDN 线性注意力上 GPU" (wsisp.com), its
 *          CPU-versus-kernel table: softplus with linear / exponential
 *          branches beyond +-20, q/k normalised per k-head before the
 *          v-heads are expanded.
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller. The library
 *    never allocates, frees or synchronises; all work is enqueued on `stream`
 *    (a cudaStream_t passed as void*, NULL = the legacy default stream).
 *  - Layouts are contiguous and row-major, token-major:
 *      q, k   [total_tokens, hq, dk]      io_dtype
 *      v, out [total_tokens, hv, dv]      io_dtype
 *      g, beta[total_tokens, hv]          float32 (g is the raw log-decay)
 *      state  [num_seqs or slots, hv, dk, dv] float32
 *    Every pointer must be 16-byte aligned (the per-head gate inputs of
 *    gdn_recurrent_step_gated only 4-byte aligned).
 *  - Supported: dk = dv = 128, chunk size 64 (fixed), hv % hq == 0,
 *    io_dtype GDN_DT_F32 (SIMT f32 arithmetic) or GDN_DT_BF16 (tensor-core
 *    bf16 operands with f32 accumulation and f32 state). Anything else returns
 *    GDN_EUNSUPPORTED without launching.
 *  - Every argument is checked before the first launch; on a non-zero return
 *    nothing was enqueued and no output was touched.
 *  - Checks that need device data (cu_seqlens, state_indices) run on the
 *    device; a failure there is recorded in a device status word (read it with
 *    gdn_read_device_status) and the affected work is skipped.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_EINVAL = 1,        /* bad pointer, shape, size or alignment */
    GDN_EUNSUPPORTED = 2,  /* valid but not implemented (dk/dv != 128, flags) */
    GDN_ECUDA = 3,         /* a CUDA runtime call or launch failed */
    GDN_ETIMEOUT = 4,      /* a bounded device-side wait gave up */
    GDN_EDEVICE_INPUT = 5, /* device-side check failed (cu_seqlens, slot index) */
    GDN_ETOOBIG = 6        /* problem exceeds the fixed scratch of gdn_chunk_fwd_noalloc */
} gdn_status;

typedef enum gdn_dtype {
    GDN_DT_F32 = 0,
    GDN_DT_BF16 = 1
} gdn_dtype;

/* gdn_problem.flags: options of the decode entry points, the precision of
 * [SGL]'s packed decode kernel (node 7). Prefill entry points want 0. */
#define GDN_FLAG_BETA_BF16 (1u << 1)  /* beta rounded to the nearest bf16 (ties to even) before use */
#define GDN_FLAG_STATE_BF16 (1u << 2) /* the state array holds bf16: loaded to f32, the updated state
                                          rounded to bf16 when written back */

/* Problem descriptor.
 *  Dense prefill  : batch = B, seqlen = T, num_seqs = B, total_tokens = B*T,
 *                   cu_seqlens = NULL (sequence b = rows [b*T, (b+1)*T)).
 *  Packed prefill : batch = 1, seqlen = 0, num_seqs = N, total_tokens = rows,
 *                   cu_seqlens = device int32 [N+1].
 *  Decode step    : num_seqs = N tokens (one per sequence), total_tokens = N,
 *                   num_state_slots = rows of the state array.
 */
typedef struct gdn_problem {
    int32_t batch;
    int32_t seqlen;
    int32_t num_seqs;
    int32_t total_tokens;
    int32_t hq;
    int32_t hv;
    int32_t dk;
    int32_t dv;
    int32_t io_dtype;         /* gdn_dtype of q, k, v and out */
    uint32_t flags;           /* GDN_FLAG_* bits (decode only); 0 for prefill */
    int32_t num_state_slots;  /* decode only */
} gdn_problem;

/* Workspace bytes gdn_chunk_fwd needs for problem `p` (0 if `p` is invalid).
 * Sized from an upper bound on the number of 64-token chunks,
 * total_tokens / 64 + num_seqs, so it does not depend on cu_seqlens values. */
size_t gdn_chunk_fwd_workspace_size(const gdn_problem *p);

/* Chunk-wise parallel prefill forward ([Lab3] "计算过程描述").
 *   q, k          [total_tokens, hq, 128]  L2-normalised by the caller
 *   v             [total_tokens, hv, 128]
 *   g             [total_tokens, hv] raw per-token log-decay (log alpha);
 *                 the library does the per-chunk prefix sum
 *   beta          [total_tokens, hv]
 *   scale         multiplies every read-out term (1/sqrt(dk) on the pages)
 *   initial_state [num_seqs, hv, 128, 128] f32, or NULL for zeros
 *   cu_seqlens    int32 [num_seqs+1] packed offsets, or NULL (dense layout).
 *                 Must start at 0, be non-decreasing and end at total_tokens
 *                 (checked on the device). Each sequence starts its own chunk
 *                 grid; chunks never straddle sequences.
 *   out           [total_tokens, hv, 128] written for every token
 *   final_state   [num_seqs, hv, 128, 128] f32, or NULL to skip. A sequence
 *                 of length 0 copies its initial state (or zeros).
 *   workspace     device scratch of at least gdn_chunk_fwd_workspace_size(p)
 *                 bytes, 256-byte aligned; contents need no initialisation
 *                 and are garbage afterwards. Calls that share a workspace
 *                 must be ordered on one stream.
 * Returns GDN_OK once everything is enqueued. */
int gdn_chunk_fwd(const gdn_problem *p, const void *q, const void *k, const void *v,
                  const float *g, const float *beta, float scale,
                  const float *initial_state, const int32_t *cu_seqlens,
                  void *out, float *final_state,
                  void *workspace, size_t workspace_bytes, void *stream);

/* gdn_chunk_fwd followed by the layer's output gate ([SGL] node
 * output_rmsnorm_silu_gate; the gated-RMSNorm row of [Kestrel]): out receives,
 * for every token t and v-head h,
 *   y[t,h] = o[t,h] / sqrt(mean_j o[t,h,j]^2 + norm_eps) * norm_weight * silu(z[t,h])
 * where o is what gdn_chunk_fwd would have written (rounded to the io dtype
 * first, as [SGL]'s node reads it). The other arguments and results are
 * gdn_chunk_fwd's (same workspace size).
 *   z           [total_tokens, hv, 128] io dtype, 16-byte aligned (not NULL)
 *   norm_weight [128] f32, 16-byte aligned; norm_eps >= 0
 * The bf16 path applies the gate inside its fused kernel, on the prepare
 * CTAs once their units are done, tile by tile as the walks finish them; the
 * f32 path runs the gdn_gated_rmsnorm pass after its output kernel. */
int gdn_chunk_fwd_gated(const gdn_problem *p, const void *q, const void *k, const void *v,
                        const float *g, const float *beta, float scale,
                        const float *initial_state, const int32_t *cu_seqlens,
                        const void *z, const float *norm_weight, float norm_eps,
                        void *out, float *final_state,
                        void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of the static device scratch array behind gdn_chunk_fwd_noalloc. */
#define GDN_NOALLOC_SCRATCH_BYTES (32u << 20)

/* gdn_chunk_fwd for callers that cannot allocate device memory.
 * The method itself has no counterpart of this entry point on the pages; it
 * exists for callers that are not allowed to call cudaMalloc (for example
 * code running inside a memory allocator's own hooks, a host callback, or a
 * runtime that fixes its memory footprint after start-up) and so cannot hand
 * over a workspace. Same arguments and results as gdn_chunk_fwd, minus the
 * workspace: the scratch lives in one file-scope device array of
 * GDN_NOALLOC_SCRATCH_BYTES (32 MiB) that every GPU loading the library holds
 * until the process exits. No call allocates or frees anything.
 *  - Returns GDN_ETOOBIG, without launching, when
 *    gdn_chunk_fwd_workspace_size(p) > GDN_NOALLOC_SCRATCH_BYTES. With the
 *    Qwen3.5-style layer (hq = 16, hv = 32) one sequence fits up to 959
 *    tokens on the bf16 path and 447 on the f32 path (the workspace grows by
 *    about 2.1 MB (bf16) or 4.7 MB (f32) per 64-token chunk at hv = 32;
 *    fewer v-heads fit proportionally more tokens). Larger prefills use
 *    gdn_chunk_fwd with a caller workspace.
 *  - The first call on a device (and the first after a cudaDeviceReset of
 *    it) looks up the array's device address with cudaGetSymbolAddress, with
 *    that device current; later calls reuse the address.
 *  - All calls share the one array and it keeps the last call's contents;
 *    nothing in it needs to start at zero. Calls whose work overlaps on the
 *    GPU (different streams, different host threads without ordering) race
 *    on it: order them on one stream. */
int gdn_chunk_fwd_noalloc(const gdn_problem *p, const void *q, const void *k, const void *v,
                          const float *g, const float *beta, float scale,
                          const float *initial_state, const int32_t *cu_seqlens,
                          void *out, float *final_state, void *stream);

/* Single-token recurrent decode step, state updated in place
 * ([Lab3] gated delta rule; [SGL] decode node 7 operation order).
 * For each sequence n < num_seqs and v-head h, with slot s = state_indices[n]
 * (or n when state_indices is NULL) and alpha = exp(g[n,h]):
 *   S = alpha * state[s,h];  p = k_n S;  d = beta (v_n - p);
 *   state[s,h] = S + k_n^T d;  out[n,h] = scale * q_n state[s,h].
 *   q, k [num_seqs, hq, 128]; v, out [num_seqs, hv, 128]; g, beta [num_seqs, hv]
 *   state [num_state_slots, hv, 128, 128] f32 (bf16 with GDN_FLAG_STATE_BF16),
 *   read and written in place; arithmetic is f32 either way.
 *   p->flags may hold GDN_FLAG_BETA_BF16 and GDN_FLAG_STATE_BF16 (any other
 *   bit: GDN_EUNSUPPORTED).
 *   state_indices int32 [num_seqs] or NULL. A negative index skips the
 *   sequence (its out rows are not written: a padding slot). An index
 *   >= num_state_slots is skipped and recorded as GDN_EDEVICE_INPUT.
 *   Two sequences must not name the same slot (their updates would race). */
int gdn_recurrent_step(const gdn_problem *p, const void *q, const void *k, const void *v,
                       const float *g, const float *beta, float scale,
                       void *state, const int32_t *state_indices,
                       void *out, void *stream);

/* Decode step from the raw projections: gdn_recurrent_step with its
 * front-end fused in (decode node 7 of [SGL], steps one and two; the gating
 * kernel of [Kestrel]). For each sequence n and v-head h (k-head
 * kh = h / (hv / hq)):
 *   k_bar = k[n,kh] / sqrt(sum_j k[n,kh,j]^2 + 1e-6)
 *   q_bar = scale * q[n,kh] / sqrt(sum_j q[n,kh,j]^2 + 1e-6)
 *   g     = -exp(A_log[h]) * softplus(a[n,h] + dt_bias[h]),  alpha = exp(g)
 *   beta  = 1 / (1 + exp(-b[n,h]))
 * where softplus(x) is x above 20, exp(x) below -20, log1p(exp(x)) between.
 * Then, as gdn_recurrent_step with scale 1 on q_bar:
 *   S = alpha * state[s,h];  d = beta (v[n,h] - k_bar S);
 *   state[s,h] = S + k_bar^T d;  out[n,h] = q_bar state[s,h].
 *   q, k      [num_seqs, hq, 128] raw (not normalised), io dtype
 *   v, out    [num_seqs, hv, 128], io dtype
 *   a, b      [num_seqs, hv] f32: the gate projections (a drives the decay,
 *             b the write strength)
 *   A_log, dt_bias [hv] f32: per-head parameters
 *   scale     the query scale, 1/sqrt(128) on the pages; applied once
 *   state, state_indices, flags: as gdn_recurrent_step (in place; negative
 *             index = padding slot, skipped; index >= num_state_slots is
 *             skipped and recorded as GDN_EDEVICE_INPUT).
 * All pointers are caller-owned device memory; q, k, v, out, state and
 * state_indices 16-byte aligned, a, b, A_log, dt_bias 4-byte aligned.
 *   z, norm_weight, norm_eps: optional output gate. With z non-NULL
 *             ([num_seqs, hv, 128] io dtype, 16-byte aligned; norm_weight
 *             [128] f32, 16-byte aligned) out receives
 *             y = o / sqrt(mean(o^2) + norm_eps) * norm_weight * silu(z)
 *             per head, computed from the f32 o (as gdn_gated_rmsnorm, but
 *             without rounding o first); with z NULL out receives o and
 *             norm_weight is ignored.
 * Returns GDN_EINVAL (nothing launched) on a bad descriptor or pointer.
 * beta is used in f32 unless p->flags holds GDN_FLAG_BETA_BF16 (the bf16
 * rounding of [SGL]'s packed kernel). */
int gdn_recurrent_step_gated(const gdn_problem *p, const void *q, const void *k, const void *v,
                             const float *a, const float *b, const float *A_log, const float *dt_bias,
                             float scale, void *state, const int32_t *state_indices,
                             const void *z, const float *norm_weight, float norm_eps,
                             void *out, void *stream);

/* Output gate of the GDN layer ([SGL] node output_rmsnorm_silu_gate; the
 * gated-RMSNorm row of [Kestrel]): for every token t and v-head h,
 *   y[t,h] = o[t,h] / sqrt(mean_j o[t,h,j]^2 + eps) * weight * silu(z[t,h])
 * over the head's 128 channels, normalised before the gate; silu(x) =
 * x / (1 + exp(-x)); the weight multiplies directly.
 *   o, z, y  [total_tokens, hv, 128] io dtype (16-byte aligned); y may be o
 *            (in place)
 *   weight   [128] f32 (16-byte aligned), shared by the heads
 *   eps      the RMSNorm epsilon (the pages leave it symbolic)
 * Only total_tokens, hv, dv and io_dtype of `p` are used (dv must be 128).
 * Returns GDN_EINVAL (nothing launched) on a bad descriptor or pointer. */
int gdn_gated_rmsnorm(const gdn_problem *p, const void *o, const void *z, const float *weight, float eps,
                      void *y, void *stream);

/* Short causal depthwise convolution + SiLU with its state, and the split of
 * its output into q, k, v ([Kestrel] conv+SiLU row: window [s0, s1, s2, x_t]
 * oldest first, the state holding the convolution's inputs; [SGL] node 6:
 * x~[t,c] = SiLU(sum_l w[c,l] x[t-l,c] + b[c]), and its layout step).
 * Channels c < C = (2 hq + hv) * 128, taps K = 4, for every packed token t
 * of sequence n (cu_seqlens) at position p:
 *   y[t,c] = SiLU(bias[c] + sum_j weight[c,j] * e[p + j, c]),  j = 0 .. 3,
 * where e = [state of n (3 rows, oldest first) ; the sequence's inputs x], so
 * weight[c,3] multiplies x[t] and weight[c,0] the input three steps back
 * ([SGL]'s lag-l weight is weight[c, 3 - l]). Then q[t] = y[t, 0 : hq*128),
 * k[t] = y[t, hq*128 : 2*hq*128), v[t] = y[t, 2*hq*128 : C), each as
 * [hq or hv, 128] rows; with norm_qk != 0 each q and k head row is divided
 * by sqrt(its sum of squares + 1e-6) ([SGL] node 7 step one, without the
 * query scale). The state of sequence n becomes the last 3 rows of e (the
 * last three inputs; part of the old state when the sequence is shorter).
 *   x          [total_tokens, C] io dtype, 16-byte aligned
 *   weight     [C, 4] f32, bias [C] f32 or NULL (zero), 16-byte aligned
 *   conv_state [num_state_slots, 3, C] io dtype, read and written in place,
 *              or NULL (zero history, nothing written)
 *   state_indices int32 [num_seqs] or NULL (sequence n uses slot n); a
 *              negative index means zero history and no state write; an
 *              index >= num_state_slots is treated the same and recorded as
 *              GDN_EDEVICE_INPUT
 *   cu_seqlens int32 [num_seqs + 1] packed offsets (checked on the device),
 *              or NULL for one sequence of total_tokens (num_seqs must be 1).
 *              Decode: one token per sequence, cu_seqlens = 0, 1, ..., N.
 *   q, k       [total_tokens, hq, 128], v [total_tokens, hv, 128], io dtype
 * Two sequences must not name the same slot. Returns GDN_EINVAL (nothing
 * launched) on a bad descriptor or pointer. */
int gdn_causal_conv1d_silu(const gdn_problem *p, const void *x, const float *weight, const float *bias,
                           void *conv_state, const int32_t *state_indices, const int32_t *cu_seqlens,
                           int norm_qk, void *q, void *k, void *v, void *stream);

/* gdn_causal_conv1d_silu for one token per sequence (decode): sequence n is
 * token n (total_tokens == num_seqs, no offsets); the same arguments
 * otherwise, with x [num_seqs, C] and q, k, v [num_seqs, h, 128]. Its state
 * moves on by one input: [s1, s2, x]. */
int gdn_causal_conv1d_silu_step(const gdn_problem *p, const void *x, const float *weight, const float *bias,
                                void *conv_state, const int32_t *state_indices, int norm_qk,
                                void *q, void *k, void *v, void *stream);

/* Gates of every token from the gate projections ([SGL] gdn_gating node;
 * [Kestrel] gating kernel, softplus linear above 20 and exponential below
 * -20): for t < total_tokens, h < hv,
 *   g[t,h] = -exp(A_log[h]) * softplus(a[t,h] + dt_bias[h]),
 *   beta[t,h] = 1 / (1 + exp(-b[t,h])),
 * ready for gdn_chunk_fwd (g is the raw per-token log-decay).
 *   a, b, g, beta [total_tokens, hv] f32; A_log, dt_bias [hv] f32; all
 *   4-byte aligned. */
int gdn_gating(const gdn_problem *p, const float *a, const float *b, const float *A_log, const float *dt_bias,
               float *g, float *beta, void *stream);

/* Synchronises `stream`, returns the device status word (GDN_OK or the first
 * device-side error recorded since the last clear) and clears it when
 * `clear` is non-zero. Returns GDN_ECUDA if the CUDA calls themselves fail. */
int gdn_read_device_status(void *stream, int clear);

/* The status read under the name the library's boundary was specified with:
 * gdn_read_device_status(stream, 1). Synchronises `stream`, returns the first
 * device-side error (GDN_ETIMEOUT, GDN_EDEVICE_INPUT) recorded since the last
 * read, or GDN_OK, and resets the word, the way cudaGetLastError resets the
 * runtime's last error. Returns GDN_ECUDA if the CUDA calls themselves fail. */
int gdn_get_device_status(void *stream);

/* Static, human-readable name of a gdn_status value. */
const char *gdn_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int gdn_version(void);

/* ---- measurement hooks (not part of the method; used by benchmarks) ---- */

/* Kernels the library launches, as indices of the gdn_profile_collect arrays. */
typedef enum gdn_kernel {
    GDN_K_CHUNK_TABLE = 0,        /* chunk table from cu_seqlens */
    GDN_K_PREP_SIMT = 1,          /* f32: gate cumsum + KK^T solve + W, U */
    GDN_K_STATE_SIMT = 2,         /* f32: sequential state pass */
    GDN_K_OUTPUT_SIMT = 3,        /* f32: chunk output */
    GDN_K_RECURRENT_STEP = 4,     /* decode step */
    GDN_K_CHUNK_FUSED_TC = 5,     /* bf16: chunk preparation and state walk, one co-resident grid (tensor cores) */
    GDN_K_RECURRENT_STEP_GATED = 6, /* decode step with the gate / q-k norm front-end */
    GDN_K_GATED_RMSNORM = 7,      /* output gate (head-wise RMSNorm, SiLU(z)) over a whole tensor */
    GDN_K_CONV1D_SILU = 8,        /* short causal convolution + SiLU with conv state, split into q, k, v */
    GDN_K_GATING = 9,             /* g and beta from the gate projections, every token */
    GDN_K_CONV1D_STEP = 10,       /* short convolution, one token per sequence (decode) */
    GDN_K_COUNT = 11
} gdn_kernel;

/* Turns per-kernel CUDA-event timing on (non-zero) or off for every later
 * launch (process-wide). Launch counting is always on. */
int gdn_profile_enable(int enable);

/* Synchronises the recorded events and copies, for the first `count` kernel
 * ids, the number of launches, the summed event time in ms and the number of
 * timed launches into the caller's host arrays (any may be NULL). Clears all
 * counters when `reset` is non-zero. */
int gdn_profile_collect(long long *launches, double *ms, long long *timed, int count, int reset);

/* Static name of a gdn_kernel id. */
const char *gdn_kernel_name(int kernel);

/* Sets, process-wide, the limit of every bounded device-side wait in the
 * prefill kernels launched after the call (the tensor-core kernel's copy,
 * MMA and ready-flag waits), in nanoseconds of wall time; 0 restores the
 * default of 2 s. A wait that runs out records GDN_ETIMEOUT in the device
 * status word; the kernel then drains what it has in flight (copies and
 * MMAs, each drain bounded too), frees its tensor memory and returns, so the
 * context stays usable and the call's outputs are unspecified. Meant for
 * tests of that path: a limit of a few microseconds makes the waits on
 * not-yet-prepared chunks run out. Returns GDN_OK. */
int gdn_set_wait_limit_ns(unsigned long long ns);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
