// Single-token recurrent decode step (gdn_recurrent_step).
//
// The gated delta rule of the Lab3 GDN Prefill page (section "Linear
// Attention 与 Gated DeltaNet"), applied once per sequence with the operation
// order of decode node 7 on the sgl-qwen3-5-moe page: decay the old state,
// predict with the key, write the beta-weighted correction, read with the
// query from the UPDATED state.
//
// The step is HBM-bound: every (sequence, v-head) streams its 64 KiB f32 state
// in and out once (2 x 64 KiB per pair, 1.07 GB per step at 256 x 32 pairs).
// One CTA of 256 threads owns one pair. Thread t holds columns 4*(t%32)..+3 of
// rows t/32 + 8i (i < 16) as 16 float4 registers, so each warp moves whole
// 512-byte rows (fully coalesced 128-bit accesses) and the state is read and
// written exactly once.
//
// Both reductions over dk are taken in one pass from the OLD state:
//   p   = k S_old                    (prediction before decay: k S_bar = alpha p)
//   r   = q S_old,  qk = q . k
//   d   = beta (v - alpha p)
//   o   = scale (alpha r + qk d)     (= scale q (alpha S_old + k^T d) exactly)
//   S'  = alpha S_old + k^T d
// so the new state never has to be re-read to produce the output.
//
// The gated variant (gdn_recurrent_step_gated) adds the front-end of decode
// node 7 on the sgl-qwen3-5-moe page, steps one and two, with the softplus
// branches of the Kestrel_VLLM-24 page's gating kernel:
//   k_bar = k / sqrt(|k|^2 + 1e-6),  q_bar = scale * q / sqrt(|q|^2 + 1e-6)
//   g = -exp(A_log) softplus(a + dt_bias),  alpha = exp(g),  beta = sigmoid(b)
// The norms are taken over the raw rows already in shared memory; instead of
// rescaling the rows, rk = 1/|k| and rq = 1/|q| fold into the scalars:
//   d' = rk beta (v - alpha rk p),  S' = alpha S_old + k^T d',
//   o  = scale rq (alpha r + qk d')
// with p, r, qk the raw-row reductions above. The state traffic is unchanged.
// The SGLang parity options of that page: a bf16 state cache (loaded to f32,
// written back rounded to bf16: half the traffic) and beta rounded to bf16
// before use.
// With an output gate z (the sgl-qwen3-5-moe page's output_rmsnorm_silu_gate,
// norm before gate), warp 0, which holds the head's 128 outputs, finishes
//   y = o / sqrt(mean(o^2) + eps) * weight * silu(z)
// in f32 before the single rounding to the output dtype.
#include "gdn_common.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

constexpr int kRThreads = 256;
constexpr int kRowsPerThread = kHeadDim / (kRThreads / 32);  // 16

template <typename T>
__device__ __forceinline__ float ldx(const void *p, size_t i) {
    return to_f32<T>(static_cast<const T *>(p)[i]);
}

// four consecutive elements starting at a multiple of 4 (one 8- or 16-byte store)
template <typename T>
__device__ __forceinline__ void st4(void *p, size_t i, const float4 &x);
template <>
__device__ __forceinline__ void st4<float>(void *p, size_t i, const float4 &x) {
    *reinterpret_cast<float4 *>(static_cast<float *>(p) + i) = x;
}
template <>
__device__ __forceinline__ void st4<__nv_bfloat16>(void *p, size_t i, const float4 &x) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y), hi = __floats2bfloat162_rn(x.z, x.w);
    *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p) + i) =
        make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
}

// four consecutive elements starting at a multiple of 4 (one 8- or 16-byte load)
template <typename T>
__device__ __forceinline__ float4 ld4(const void *p, size_t i);
template <>
__device__ __forceinline__ float4 ld4<float>(const void *p, size_t i) {
    return *reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i);
}
template <>
__device__ __forceinline__ float4 ld4<__nv_bfloat16>(const void *p, size_t i) {
    const uint2 u = *reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(p) + i);
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}

// state words as loaded: float4 (f32 cache) or 4 packed bf16 (bf16 cache,
// widened where used, so that the registers hold twice the rows in flight)
template <typename ST>
struct StateWords;
template <>
struct StateWords<float> {
    using raw = float4;
    static __device__ __forceinline__ raw load(const float *p) { return *reinterpret_cast<const float4 *>(p); }
    static __device__ __forceinline__ float4 f(const raw &r) { return r; }
};
template <>
struct StateWords<__nv_bfloat16> {
    using raw = uint2;
    static __device__ __forceinline__ raw load(const __nv_bfloat16 *p) { return *reinterpret_cast<const uint2 *>(p); }
    static __device__ __forceinline__ float4 f(const raw &r) {
        const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.x));
        const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.y));
        return make_float4(lo.x, lo.y, hi.x, hi.y);
    }
};

// bf16 state cache: the pair's 32 KiB state comes in by one bulk copy into
// shared memory and is read from there where it is used, so that no
// registers hold it in flight and five CTAs fit on an SM (160 KiB in flight
// per SM). The f32 state keeps its words in registers (16 x 16 bytes per
// thread, two CTAs per SM), which already streams at the copy rate.
template <typename ST>
constexpr bool kBulkState = sizeof(ST) == 2;
constexpr uint32_t kBulkStateBytes = kHeadDim * kHeadDim * 2;

template <typename T, typename ST, bool kFront, bool kGateOut>
__global__ void __launch_bounds__(kRThreads, kBulkState<ST> ? 5 : 2)
k_recurrent_step(const void *__restrict__ q, const void *__restrict__ k, const void *__restrict__ v,
                 const float *__restrict__ g, const float *__restrict__ beta, DecodeFront front, float scale,
                 void *__restrict__ state, const int32_t *__restrict__ idx, void *__restrict__ out,
                 int num_seqs, int hq, int hv, int slots, int beta_bf16, int *status) {
    __shared__ float ks[kHeadDim], qs[kHeadDim];
    __shared__ float4 red_p[kRThreads / 32][32], red_r[kRThreads / 32][32];
    __shared__ float qk_s, rk_s, rq_s, alpha_s, beta_s;
    __shared__ float4 gz_s[32];  // weight * silu(z), 4 channels per lane
    __shared__ uint64_t st_bar;
    extern __shared__ __align__(128) uint8_t st_sm[];  // bf16 cache: the pair's state [128][128]
    constexpr bool kBulk = kBulkState<ST>;
    const int pair = blockIdx.x;
    const int n = pair / hv, h = pair % hv, hk = h / (hv / hq);
    const int tid = threadIdx.x, lane = tid & 31, wrow = tid >> 5;
    int slot = idx ? idx[n] : n;
    if (slot < 0) return;  // padding slot: nothing read, nothing written
    if (slot >= slots) {
        if (tid == 0) record_status(status, GDN_EDEVICE_INPUT);
        return;
    }
    ST *S = static_cast<ST *>(state) + (size_t(slot) * hv + h) * kHeadDim * kHeadDim;
    if (kBulk && tid == 0) {
        tc::mbar_init(&st_bar, 1);
        tc::fence_mbar_init();
        tc::mbar_arrive_expect_tx(&st_bar, kBulkStateBytes);
        tc::bulk_load(st_sm, S, kBulkStateBytes, &st_bar);
    }
    // The small inputs are issued first, each by the warp that uses it, so that
    // they arrive while the 64 KiB state read is still in flight. Nothing but
    // the q/k staging stands before the first barrier: the front-end's scalar
    // work runs in warps that would otherwise wait at the second one.
    constexpr bool gate_out = kFront && kGateOut;
    constexpr int kGateWarp = 3, kZWarp = 4;
    const size_t nh = size_t(n) * hv + h;
    const size_t vo = nh * kHeadDim + 4 * lane;
    float ga = 0.f, gb = 0.f, gA = 0.f, gdt = 0.f;
    if (kFront && wrow == kGateWarp) {
        ga = front.a[nh];
        gb = front.b[nh];
        gA = front.A_log[h];
        gdt = front.dt_bias[h];
    } else if (!kFront) {
        ga = g[nh];
        gb = beta[nh];
    }
    const float4 vv = ld4<T>(v, vo);
    float4 zz = make_float4(0.f, 0.f, 0.f, 0.f), nw = zz;
    if (gate_out && wrow == kZWarp) {
        zz = ld4<T>(front.z, vo);
        nw = *reinterpret_cast<const float4 *>(front.norm_weight + 4 * lane);
    }
    float kq_k = 0.f, kq_q = 0.f;
    if (tid < kHeadDim) {
        const size_t qk_off = (size_t(n) * hq + hk) * kHeadDim + tid;
        kq_k = ldx<T>(k, qk_off);
        kq_q = ldx<T>(q, qk_off);
    }
    // f32 cache: all state loads, 16 independent 128-bit loads per thread
    typename StateWords<ST>::raw s[kBulk ? 1 : kRowsPerThread];
    if constexpr (!kBulk) {
#pragma unroll
        for (int i = 0; i < kRowsPerThread; ++i)
            s[i] = StateWords<ST>::load(S + size_t(wrow + 8 * i) * kHeadDim + 4 * lane);
    }
    // this thread's 4 columns of state row wrow + 8 i
    auto state_row = [&](int i) -> float4 {
        if constexpr (kBulk)
            return StateWords<ST>::f(
                StateWords<ST>::load(reinterpret_cast<const ST *>(st_sm) + size_t(wrow + 8 * i) * kHeadDim + 4 * lane));
        else
            return StateWords<ST>::f(s[i]);
    };
    if (tid < kHeadDim) {
        ks[tid] = kq_k;
        qs[tid] = kq_q;
    }
    __syncthreads();
    // q . k by warp 0; for the front-end |k|^2 by warp 1 and |q|^2 by warp 2,
    // the gates by warp 3 and weight * silu(z) by warp 4
    if (wrow < (kFront ? 3 : 1)) {
        const float *x = wrow == 2 ? qs : ks, *y = wrow == 0 ? qs : x;
        float acc = 0.f;
        for (int d = lane; d < kHeadDim; d += 32) acc = fmaf(x[d], y[d], acc);
        for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) {
            if (wrow == 0) qk_s = acc;
            else if (wrow == 1) rk_s = rsqrtf(acc + 1e-6f);
            else rq_s = rsqrtf(acc + 1e-6f);
        }
    }
    if (kFront && wrow == kGateWarp && lane == 0) {
        alpha_s = expf(-expf(gA) * softplus_f(ga + gdt));
        beta_s = 1.f / (1.f + expf(-gb));
    }
    if (gate_out && wrow == kZWarp)
        gz_s[lane] = make_float4(nw.x * silu_f(zz.x), nw.y * silu_f(zz.y), nw.z * silu_f(zz.z), nw.w * silu_f(zz.w));
    if constexpr (kBulk) {  // the state copy has landed (a bounded wait; a timeout skips the pair)
        const bool landed = tc::mbar_wait_spin(&st_bar, 0);
        if (__syncthreads_or(!landed)) {
            if (tid == 0) record_status(status, GDN_ETIMEOUT);
            return;
        }
    }
    float4 p = make_float4(0.f, 0.f, 0.f, 0.f), r = p;
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) {
        const float kd = ks[wrow + 8 * i], qd = qs[wrow + 8 * i];
        const float4 si = state_row(i);
        p.x = fmaf(kd, si.x, p.x); p.y = fmaf(kd, si.y, p.y);
        p.z = fmaf(kd, si.z, p.z); p.w = fmaf(kd, si.w, p.w);
        r.x = fmaf(qd, si.x, r.x); r.y = fmaf(qd, si.y, r.y);
        r.z = fmaf(qd, si.z, r.z); r.w = fmaf(qd, si.w, r.w);
    }
    red_p[wrow][lane] = p;
    red_r[wrow][lane] = r;
    __syncthreads();
    p = make_float4(0.f, 0.f, 0.f, 0.f);
    r = p;
#pragma unroll
    for (int w = 0; w < kRThreads / 32; ++w) {
        const float4 a = red_p[w][lane], b = red_r[w][lane];
        p.x += a.x; p.y += a.y; p.z += a.z; p.w += a.w;
        r.x += b.x; r.y += b.y; r.z += b.z; r.w += b.w;
    }
    float alpha, b;
    if (kFront) {
        alpha = alpha_s;
        b = beta_s;
    } else {
        alpha = expf(ga);
        b = gb;
    }
    if (beta_bf16) b = __bfloat162float(__float2bfloat16_rn(b));  // the packed SGLang kernel's rounding
    float rk = 1.f, oscale = scale;
    if (kFront) {
        rk = rk_s;
        oscale = scale * rq_s;
    }
    const float ak = alpha * rk, bk = b * rk;  // d' = rk beta (v - alpha rk p)
    float4 d;
    d.x = bk * (vv.x - ak * p.x);
    d.y = bk * (vv.y - ak * p.y);
    d.z = bk * (vv.z - ak * p.z);
    d.w = bk * (vv.w - ak * p.w);
    // the read-out (warp 0 holds the head's 128 outputs), then the state
    if (wrow == 0) {
        const float qk = qk_s;
        float4 y;
        y.x = oscale * fmaf(alpha, r.x, qk * d.x);
        y.y = oscale * fmaf(alpha, r.y, qk * d.y);
        y.z = oscale * fmaf(alpha, r.z, qk * d.z);
        y.w = oscale * fmaf(alpha, r.w, qk * d.w);
        if (gate_out) {  // y = o / rms(o) * weight * silu(z), the head's 128 values in this warp
            float ss = y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w;
            for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float inv = rsqrtf(ss * (1.f / kHeadDim) + front.norm_eps);
            const float4 gz = gz_s[lane];
            y.x *= inv * gz.x;
            y.y *= inv * gz.y;
            y.z *= inv * gz.z;
            y.w *= inv * gz.w;
        }
        st4<T>(out, vo, y);
    }
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) {
        const float kd = ks[wrow + 8 * i];
        const float4 si = state_row(i);
        float4 t;
        t.x = fmaf(alpha, si.x, kd * d.x);
        t.y = fmaf(alpha, si.y, kd * d.y);
        t.z = fmaf(alpha, si.z, kd * d.z);
        t.w = fmaf(alpha, si.w, kd * d.w);
        st4<ST>(S, size_t(wrow + 8 * i) * kHeadDim + 4 * lane, t);
    }
}

}  // namespace

namespace {
using StepKernel = void (*)(const void *, const void *, const void *, const float *, const float *, DecodeFront,
                            float, void *, const int32_t *, void *, int, int, int, int, int, int *);

template <typename T, typename ST>
StepKernel pick_step(bool front, bool gate) {
    return gate ? k_recurrent_step<T, ST, true, true>
                : front ? k_recurrent_step<T, ST, true, false> : k_recurrent_step<T, ST, false, false>;
}
}  // namespace

cudaError_t launch_recurrent_step(const gdn_problem &p, const void *q, const void *k, const void *v,
                                  const float *g, const float *beta, const DecodeFront *front, float scale,
                                  void *state, const int32_t *state_indices, void *out, int *status,
                                  cudaStream_t s) {
    const unsigned pairs = unsigned(p.num_seqs) * unsigned(p.hv);
    if (pairs == 0) return cudaSuccess;
    LaunchScope scope(front ? GDN_K_RECURRENT_STEP_GATED : GDN_K_RECURRENT_STEP, s);
    const DecodeFront f = front ? *front : DecodeFront{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, 0.f};
    const bool gate = front && front->z;
    const bool st_bf = (p.flags & GDN_FLAG_STATE_BF16) != 0;
    const StepKernel kern =
        p.io_dtype == GDN_DT_BF16
            ? (st_bf ? pick_step<__nv_bfloat16, __nv_bfloat16>(front, gate)
                     : pick_step<__nv_bfloat16, float>(front, gate))
            : (st_bf ? pick_step<float, __nv_bfloat16>(front, gate) : pick_step<float, float>(front, gate));
    kern<<<pairs, kRThreads, st_bf ? kBulkStateBytes : 0, s>>>(q, k, v, g, beta, f, scale, state, state_indices, out,
                                                              p.num_seqs, p.hq,
                                    p.hv, p.num_state_slots, (p.flags & GDN_FLAG_BETA_BF16) ? 1 : 0, status);
    return cudaGetLastError();
}

}  // namespace gdn
