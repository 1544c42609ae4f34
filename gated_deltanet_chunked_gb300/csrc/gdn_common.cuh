// Shared device-side definitions of libgdn (not part of the public ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn.h"

namespace gdn {

constexpr int kChunk = 64;   // chunk size C fixed by the Lab3 GDN Prefill page
constexpr int kHeadDim = 128;  // d_k = d_v = 128 on every configuration

// One 64-token chunk of one sequence (built on the device from cu_seqlens).
struct ChunkInfo {
    int seq;    // sequence index
    int start;  // first token row of the chunk
    int len;    // valid length l_c = min(64, L - c*64), 1..64
    int idx;    // chunk index inside its sequence
};

// Per-sequence range of chunks in the global chunk list.
struct SeqInfo {
    int first_chunk;
    int num_chunks;
    int start;  // first token row of the sequence
    int len;    // tokens in the sequence
};

// Everything a prefill launch needs; built once on the host per call.
struct PrefillArgs {
    const void *q, *k, *v;
    const float *g, *beta;
    const float *s0;
    float *final_state;
    void *out;
    float scale;
    int hq, hv, group;  // group = hv / hq
    int num_seqs, total_tokens;
    int dense_batch, dense_seqlen;  // used when cu == nullptr
    const int *cu;
    int max_chunks;
    // workspace regions
    int *n_chunks;  // [1]
    SeqInfo *seq_info;  // [num_seqs]
    ChunkInfo *chunk_info;  // [max_chunks]
    int *status;  // device status word
    int *ready;       // per-unit ready flags of the tensor-core path (zeroed by the chunk table), or null
    int ready_count;  // flags the chunk table zeroes (ready flags, then the output counters)
    // optional output gate (z null: none): out = RMSNorm(o) * weight * silu(z)
    const void *z;
    const float *norm_weight;
    float norm_eps;
    int *done;        // per-unit count of math warps whose output block has landed (tensor-core path)
    // limit of every bounded wait of the launch, in ns of wall time (2 s
    // unless a test lowers it through gdn_set_wait_limit_ns)
    unsigned long long wait_ns;
};

__device__ __forceinline__ void record_status(int *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Counts a kernel launch and, when profiling is enabled, brackets it with
// CUDA events on `s` (construct right before the launch, destroy right after).
class LaunchScope {
  public:
    LaunchScope(int kernel, cudaStream_t s);
    ~LaunchScope();
    LaunchScope(const LaunchScope &) = delete;
    LaunchScope &operator=(const LaunchScope &) = delete;

  private:
    int kernel_;
    cudaStream_t stream_;
    cudaEvent_t start_;
};

// Host-side launchers implemented in the kernel translation units.
cudaError_t launch_chunk_table(const PrefillArgs &a, cudaStream_t s);
cudaError_t launch_conv1d_silu(const gdn_problem &p, const void *x, const float *weight, const float *bias,
                               void *conv_state, const int32_t *state_indices, const int32_t *cu_seqlens,
                               int norm_qk, void *out_q, void *out_k, void *out_v, int *status, cudaStream_t s);
cudaError_t launch_conv1d_step(const gdn_problem &p, const void *x, const float *weight, const float *bias,
                               void *conv_state, const int32_t *state_indices, int norm_qk, void *out_q,
                               void *out_k, void *out_v, int *status, cudaStream_t s);
cudaError_t launch_gating(const float *a, const float *b, const float *A_log, const float *dt_bias, float *g,
                          float *beta, long long n, int hv, cudaStream_t s);
cudaError_t launch_gated_rmsnorm(const void *o, const void *z, const float *weight, float eps, void *y,
                                 long long rows, int io_dtype, int *status, cudaStream_t s);
cudaError_t launch_prefill_simt(const PrefillArgs &a, void *ws_data, cudaStream_t s);
size_t prefill_simt_workspace(int max_chunks, int hv);
cudaError_t launch_prefill_tc(const PrefillArgs &a, void *ws_data, cudaStream_t s);
int *prefill_tc_ready_flags(void *ws_data, int max_chunks, int hv);
size_t prefill_tc_workspace(int max_chunks, int hv);
// Raw inputs of the decode front-end (gdn_recurrent_step_gated): gate
// projections a, b [num_seqs, hv] and per-head A_log, dt_bias [hv]; and the
// optional output gate: z [num_seqs, hv, 128] (io dtype) with the RMSNorm
// weight [128] and eps (z null: no output gate).
struct DecodeFront {
    const float *a, *b, *A_log, *dt_bias;
    const void *z;
    const float *norm_weight;
    float norm_eps;
};

// log(1 + e^x), linear above 20 and e^x below -20 (no overflow of e^x)
__device__ __forceinline__ float softplus_f(float x) {
    if (x > 20.f) return x;
    if (x < -20.f) return expf(x);
    return log1pf(expf(x));
}

// x * sigmoid(x) = x / (1 + e^-x), the output gate's activation. e^-x is
// taken as 2^(-x log2 e) on the base-2 exponential unit and the quotient
// through the approximate reciprocal (both relative errors ~1e-7): x = -inf
// side gives x * 0, the +inf side x * 1.
__device__ __forceinline__ float silu_f(float x) {
    float e, r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(x * -1.4426950408889634f));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + e));
    return x * r;
}

// silu_f on two values, the multiplies and the add as packed f32x2 operations
// (one IEEE operation per lane, so the same results as silu_f; half the
// issue slots for that part)
__device__ __forceinline__ float2 silu2_f(float2 x) {
    const float2 t = __fmul2_rn(x, make_float2(-1.4426950408889634f, -1.4426950408889634f));
    float2 e, r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.x) : "f"(t.x));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.y) : "f"(t.y));
    e = __fadd2_rn(e, make_float2(1.f, 1.f));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.x) : "f"(e.x));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.y) : "f"(e.y));
    return __fmul2_rn(x, r);
}
// `front` null: g and beta are given and q, k are used as they are.
// `front` set: g and beta are null and computed from it, q and k are
// L2-normalised in the kernel.
cudaError_t launch_recurrent_step(const gdn_problem &p, const void *q, const void *k, const void *v,
                                  const float *g, const float *beta, const DecodeFront *front, float scale,
                                  void *state, const int32_t *state_indices, void *out, int *status,
                                  cudaStream_t s);

}  // namespace gdn
