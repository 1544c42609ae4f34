// Front-end kernels of a GDN layer ahead of the chunk-wise core:
//
//  k_conv1d_silu -- the short causal depthwise convolution with its state
//    (the Kestrel_VLLM-24 page's conv+SiLU row: window [s0, s1, s2, x_t],
//    oldest first, the history holding the convolution's inputs; the
//    sgl-qwen3-5-moe page's node 6 with the split of its output into q, k, v),
//    optionally followed by the per-head L2 norm of q and k (decode node 7,
//    step one, without the query scale, which the chunk form applies).
//  k_gating -- g = -exp(A_log) softplus(a + dt_bias) and beta = sigmoid(b) for
//    every token (the sgl-qwen3-5-moe page's gdn_gating node; the softplus
//    branches of the Kestrel page's gating kernel).
//
// Both are HBM-bound elementwise passes.
//
// k_conv1d_silu: a thread owns 4 consecutive channels (one 8- or 16-byte
// access per token), so a warp covers exactly one 128-channel head and the
// q/k norm is one warp reduction. A CTA (grid x: token tiles, y: channel
// blocks) takes 1024 channels over a tile of tokens of the packed token axis
// and slides the window down it in registers; tiles may span several
// sequences (the window restarts from each sequence's state).
// In-place state update without a race: a tile never starts at the second or
// third token of a sequence (its start moves to the fourth), so the old state
// of a sequence is read only by the thread that processes the sequence's
// first token, and that same thread writes the new state (the last K-1
// inputs) after it has read the old one.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kConvK = 4;  // taps
constexpr int kCThreads = 256;
constexpr int kCPerThread = 4;
constexpr int kCPerBlock = kCThreads * kCPerThread;  // 1024 channels

template <typename T>
__device__ __forceinline__ float4 ld4v(const T *p);
template <>
__device__ __forceinline__ float4 ld4v<float>(const float *p) { return *reinterpret_cast<const float4 *>(p); }
template <>
__device__ __forceinline__ float4 ld4v<__nv_bfloat16>(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}
template <typename T>
__device__ __forceinline__ void st4v(T *p, const float4 &x);
template <>
__device__ __forceinline__ void st4v<float>(float *p, const float4 &x) { *reinterpret_cast<float4 *>(p) = x; }
template <>
__device__ __forceinline__ void st4v<__nv_bfloat16>(__nv_bfloat16 *p, const float4 &x) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y), hi = __floats2bfloat162_rn(x.z, x.w);
    *reinterpret_cast<uint2 *>(p) =
        make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
}

struct ConvArgs {
    const void *x;            // [T, C]
    const float *weight;      // [C, 4] oldest first
    const float *bias;        // [C] or null
    void *state;              // [slots, 3, C] or null
    const int32_t *idx;       // [N] or null
    const int32_t *cu;        // [N+1] or null (one sequence)
    void *oq, *ok, *ov;       // [T, hq, 128], [T, hq, 128], [T, hv, 128]
    int T, C, N, slots, hq, hv, tile, norm_qk;
    int *status;
};

// sequence holding token t (cu[s] <= t < cu[s+1]); the last non-empty one for t = T
__device__ __forceinline__ int seq_of(const int32_t *cu, int N, int t) {
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// start of the tile that nominally starts at t: moved from the 2nd/3rd token
// of a sequence to its 4th (or to the sequence's end)
__device__ __forceinline__ int tile_start(const int32_t *cu, int N, int T, int t) {
    if (t >= T) return T;
    const int s = seq_of(cu, N, t);
    const int p = t - cu[s];
    if (p == 1 || p == 2) return min(cu[s] + kConvK - 1, cu[s + 1]);
    return t;
}

template <typename T>
__global__ void __launch_bounds__(kCThreads) k_conv1d_silu(ConvArgs a) {
    const int lane = threadIdx.x & 31;
    const int c0 = blockIdx.y * kCPerBlock + threadIdx.x * kCPerThread;
    const int32_t one_seq[2] = {0, a.T};
    const int32_t *cu = a.cu ? a.cu : one_seq;
    const int N = a.cu ? a.N : 1;
    if (a.cu) {  // the offsets must start at 0, never decrease and end at T
        bool bad = false;
        for (int i = threadIdx.x; i < N; i += kCThreads) bad |= cu[i] > cu[i + 1];
        bad |= cu[0] != 0 || cu[N] != a.T;
        if (__syncthreads_or(bad)) {
            if (threadIdx.x == 0) record_status(a.status, GDN_EDEVICE_INPUT);
            return;
        }
    }
    if (c0 >= a.C) return;  // whole warps: C is a multiple of 128
    const int t_nominal = int(blockIdx.x) * a.tile;
    const int t_begin = tile_start(cu, N, a.T, t_nominal);
    const int t_end = tile_start(cu, N, a.T, min(t_nominal + a.tile, a.T));
    if (t_begin >= t_end) return;
    const T *X = static_cast<const T *>(a.x);
    T *S = static_cast<T *>(a.state);
    float4 w[kConvK];  // w[j] = taps j of the 4 channels
    {
        float4 r[kCPerThread];
#pragma unroll
        for (int i = 0; i < kCPerThread; ++i) r[i] = reinterpret_cast<const float4 *>(a.weight)[c0 + i];
        w[0] = make_float4(r[0].x, r[1].x, r[2].x, r[3].x);
        w[1] = make_float4(r[0].y, r[1].y, r[2].y, r[3].y);
        w[2] = make_float4(r[0].z, r[1].z, r[2].z, r[3].z);
        w[3] = make_float4(r[0].w, r[1].w, r[2].w, r[3].w);
    }
    const float4 bias = a.bias ? *reinterpret_cast<const float4 *>(a.bias + c0) : make_float4(0.f, 0.f, 0.f, 0.f);
    // output tensor and column of these channels
    const int qk_c = a.hq * kHeadDim;
    T *dst;
    int dcol, drow;
    if (c0 < qk_c) dst = static_cast<T *>(a.oq), dcol = c0, drow = qk_c;
    else if (c0 < 2 * qk_c) dst = static_cast<T *>(a.ok), dcol = c0 - qk_c, drow = qk_c;
    else dst = static_cast<T *>(a.ov), dcol = c0 - 2 * qk_c, drow = a.hv * kHeadDim;
    const bool norm = a.norm_qk && c0 < 2 * qk_c;  // uniform over the warp (one head)

    int s = seq_of(cu, N, t_begin);
    int s_end = cu[s + 1];
    float4 h0, h1, h2;  // x_{t-3}, x_{t-2}, x_{t-1}
    // history at the first token of the tile (position p of sequence s)
    auto load_history = [&](int t) {
        const int ss = cu[s], p = t - ss;
        float4 e[kConvK - 1];
        int slot = -1;
        if (p < kConvK - 1 && S) {
            slot = a.idx ? a.idx[s] : s;
            if (slot >= a.slots) {
                if (lane == 0) record_status(a.status, GDN_EDEVICE_INPUT);
                slot = -1;
            }
        }
#pragma unroll
        for (int i = 0; i < kConvK - 1; ++i) {
            const int j = p + i;  // index in [state ; x of the sequence]
            if (j >= kConvK - 1) e[i] = ld4v<T>(X + size_t(ss + j - (kConvK - 1)) * a.C + c0);
            else if (slot >= 0) e[i] = ld4v<T>(S + (size_t(slot) * (kConvK - 1) + j) * a.C + c0);
            else e[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        h0 = e[0], h1 = e[1], h2 = e[2];
        if (p == 0 && slot >= 0) {
            // this thread alone reads the old state of sequence s: write the new one
            const int L = s_end - ss;
#pragma unroll
            for (int i = 0; i < kConvK - 1; ++i) {
                const int j = L + i;  // last K-1 entries of [state ; x]
                const float4 v = j >= kConvK - 1 ? ld4v<T>(X + size_t(ss + j - (kConvK - 1)) * a.C + c0) : e[j];
                st4v<T>(S + (size_t(slot) * (kConvK - 1) + i) * a.C + c0, v);
            }
        }
    };
    load_history(t_begin);
    for (int t = t_begin; t < t_end; ++t) {
        if (t == s_end) {  // next non-empty sequence starts here
            while (cu[s + 1] <= t) ++s;
            s_end = cu[s + 1];
            load_history(t);
        }
        const float4 xv = ld4v<T>(X + size_t(t) * a.C + c0);
        float4 y;
        y.x = silu_f(fmaf(w[3].x, xv.x, fmaf(w[2].x, h2.x, fmaf(w[1].x, h1.x, fmaf(w[0].x, h0.x, bias.x)))));
        y.y = silu_f(fmaf(w[3].y, xv.y, fmaf(w[2].y, h2.y, fmaf(w[1].y, h1.y, fmaf(w[0].y, h0.y, bias.y)))));
        y.z = silu_f(fmaf(w[3].z, xv.z, fmaf(w[2].z, h2.z, fmaf(w[1].z, h1.z, fmaf(w[0].z, h0.z, bias.z)))));
        y.w = silu_f(fmaf(w[3].w, xv.w, fmaf(w[2].w, h2.w, fmaf(w[1].w, h1.w, fmaf(w[0].w, h0.w, bias.w)))));
        if (norm) {
            float ss = y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w;
            for (int m = 16; m; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
            const float inv = rsqrtf(ss + 1e-6f);
            y.x *= inv; y.y *= inv; y.z *= inv; y.w *= inv;
        }
        st4v<T>(dst + size_t(t) * drow + dcol, y);
        h0 = h1, h1 = h2, h2 = xv;
    }
}

// g, beta [T, hv] from a, b [T, hv] and A_log, dt_bias [hv]
__global__ void __launch_bounds__(256) k_gating(const float *__restrict__ ga, const float *__restrict__ gb,
                                                const float *__restrict__ A_log, const float *__restrict__ dt_bias,
                                                float *__restrict__ g, float *__restrict__ beta, long long n,
                                                int hv) {
    for (long long i = blockIdx.x * 256ll + threadIdx.x; i < n; i += (long long)gridDim.x * 256) {
        const int h = int(i % hv);
        g[i] = -expf(A_log[h]) * softplus_f(ga[i] + dt_bias[h]);
        beta[i] = 1.f / (1.f + expf(-gb[i]));
    }
}

}  // namespace

cudaError_t launch_conv1d_silu(const gdn_problem &p, const void *x, const float *weight, const float *bias,
                               void *conv_state, const int32_t *state_indices, const int32_t *cu_seqlens,
                               int norm_qk, void *out_q, void *out_k, void *out_v, int *status, cudaStream_t s) {
    const int C = (2 * p.hq + p.hv) * kHeadDim;
    if (p.total_tokens == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    int tile = 1;  // tokens per tile: about two token tiles per SM, 1 .. 64
    while (tile < 64 && tile * 2 <= p.total_tokens / sms) tile *= 2;
    ConvArgs a{x, weight, bias, conv_state, state_indices, cu_seqlens, out_q, out_k, out_v,
               p.total_tokens, C, p.num_seqs, p.num_state_slots, p.hq, p.hv, tile, norm_qk, status};
    const dim3 grid((p.total_tokens + tile - 1) / tile, (C + kCPerBlock - 1) / kCPerBlock);
    LaunchScope scope(GDN_K_CONV1D_SILU, s);
    if (p.io_dtype == GDN_DT_BF16) k_conv1d_silu<__nv_bfloat16><<<grid, kCThreads, 0, s>>>(a);
    else k_conv1d_silu<float><<<grid, kCThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_gating(const float *a, const float *b, const float *A_log, const float *dt_bias, float *g,
                          float *beta, long long n, int hv, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long blocks = (n + 255) / 256;
    LaunchScope scope(GDN_K_GATING, s);
    k_gating<<<unsigned(blocks < 8ll * sms ? blocks : 8ll * sms), 256, 0, s>>>(a, b, A_log, dt_bias, g, beta, n, hv);
    return cudaGetLastError();
}

}  // namespace gdn
