// Front-end kernels of a GDN layer ahead of the chunk-wise core:
//
//  k_conv1d_silu -- the short causal depthwise convolution with its state
//    (the Kestrel_VLLM-24 page's conv+SiLU row: window [s0, s1, s2, x_t],
//    oldest first, the history holding the convolution's inputs; the
//    sgl-qwen3-5-moe page's node 6 with the split of its output into q, k, v),
//    optionally followed by the per-head L2 norm of q and k (decode node 7,
//    step one, without the query scale, which the chunk form applies).
//  k_conv1d_step -- the same for one token per sequence (decode), the state
//    shifted in place by the thread that owns the channels.
//  k_gating -- g = -exp(A_log) softplus(a + dt_bias) and beta = sigmoid(b) for
//    every token (the sgl-qwen3-5-moe page's gdn_gating node; the softplus
//    branches of the Kestrel page's gating kernel).
//
// Both are HBM-bound elementwise passes.
//
// k_conv1d_silu: a thread owns 4 consecutive channels (one 8- or 16-byte
// access per token), so a warp covers exactly one 128-channel head and the
// q/k norm is one warp reduction. A CTA (linear grid, the channel block
// varying fastest) takes 512 channels over a tile of tokens of the packed token axis
// and slides the window down it in registers. The tile's rows of x (2 KiB per
// token for bf16) come into shared memory by bulk copies issued at once by one
// thread, so that a whole tile is in flight per CTA without holding
// registers (loads issued token by token left the kernel bound by load
// latency at 0.3 of HBM); tiles may span several sequences (the window
// restarts from each sequence's state). The copies also bring the K-1 rows
// before the tile, the history of a tile that starts inside a sequence: as
// plain loads issued after the tile's copies they arrived after the whole
// tile. A token that is a whole sequence (decode) finds its sequence without
// a search.
// In-place state update without a race: a tile never starts at the second or
// third token of a sequence (its start moves to the fourth), so the old state
// of a sequence is read only by the thread that processes the sequence's
// first token, and that same thread writes the new state (the last K-1
// inputs) after it has read the old one.
#include "gdn_common.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

constexpr int kConvK = 4;  // taps
constexpr int kCThreads = 128;
constexpr int kCPerThread = 4;
constexpr int kCPerBlock = kCThreads * kCPerThread;  // 512 channels
constexpr int kMaxTileBytes = 16 * 1024;            // x rows staged per CTA (plus five rows)

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
    int T, C, N, slots, hq, hv, tile, norm_qk, cblocks;
    int *status;
};

// sequence holding token t (cu[s] <= t < cu[s+1]); the last non-empty one for t = T
__device__ __forceinline__ int seq_of(const int32_t *cu, int N, int t) {
    if (t < N && cu[t] == t && cu[t + 1] == t + 1) return t;  // one token per sequence (decode)
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
    using namespace tc;
    extern __shared__ __align__(128) uint8_t xs_raw[];  // the tile's rows of x: [rows][512] T
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    const int lane = threadIdx.x & 31;
    // channel block fastest: CTAs that run together cover whole token rows
    const int cblock = int(blockIdx.x % a.cblocks), ctile = int(blockIdx.x / a.cblocks);
    const int c0 = cblock * kCPerBlock + threadIdx.x * kCPerThread;
    const int32_t one_seq[2] = {0, a.T};
    const int32_t *cu = a.cu ? a.cu : one_seq;
    const int N = a.cu ? a.N : 1;
    const bool active = c0 < a.C;  // whole warps: C is a multiple of 128
    // the taps and bias first: their loads then overlap the tile bounds'
    // dependent reads of cu_seqlens instead of queueing behind the tile's copies
    float4 wr[kCPerThread], bias = make_float4(0.f, 0.f, 0.f, 0.f);
    if (active) {
#pragma unroll
        for (int i = 0; i < kCPerThread; ++i) wr[i] = reinterpret_cast<const float4 *>(a.weight)[c0 + i];
        if (a.bias) bias = *reinterpret_cast<const float4 *>(a.bias + c0);
    }
    if (a.cu) {  // the offsets must start at 0, never decrease and end at T
        bool bad = false;
        for (int i = threadIdx.x; i < N; i += kCThreads) bad |= cu[i] > cu[i + 1];
        bad |= cu[0] != 0 || cu[N] != a.T;
        if (__syncthreads_or(bad)) {
            if (threadIdx.x == 0) record_status(a.status, GDN_EDEVICE_INPUT);
            return;
        }
    }
    const int t_nominal = ctile * a.tile;
    const int t_begin = tile_start(cu, N, a.T, t_nominal);
    const int t_end = tile_start(cu, N, a.T, min(t_nominal + a.tile, a.T));
    if (t_begin >= t_end) return;  // uniform over the CTA
    const T *X = static_cast<const T *>(a.x);
    // the tile's rows of x for these 512 channels and the K-1 rows before it
    // (a mid-sequence tile's history), by bulk copies (one per token)
    const int h_begin = max(t_begin - (kConvK - 1), 0);
    const int cb0 = cblock * kCPerBlock;
    const uint32_t row_bytes = uint32_t(min(kCPerBlock, a.C - cb0)) * sizeof(T);
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
        mbar_arrive_expect_tx(&bar, uint32_t(t_end - h_begin) * row_bytes);
        for (int t = h_begin; t < t_end; ++t)
            bulk_load(xs_raw + size_t(t - h_begin) * kCPerBlock * sizeof(T), X + size_t(t) * a.C + cb0, row_bytes,
                      &bar);
    }
    __syncthreads();
    T *S = static_cast<T *>(a.state);
    if (!active) {  // still waits for the copies into this CTA's shared memory
        if (threadIdx.x == 0 && !mbar_wait(&bar, 0)) record_status(a.status, GDN_ETIMEOUT);
        return;
    }
    float4 w[kConvK];  // w[j] = taps j of the 4 channels
    w[0] = make_float4(wr[0].x, wr[1].x, wr[2].x, wr[3].x);
    w[1] = make_float4(wr[0].y, wr[1].y, wr[2].y, wr[3].y);
    w[2] = make_float4(wr[0].z, wr[1].z, wr[2].z, wr[3].z);
    w[3] = make_float4(wr[0].w, wr[1].w, wr[2].w, wr[3].w);
    // taps and bias as channel pairs (0, 1) and (2, 3) for the packed f32x2 arithmetic
    float2 wl[kConvK], wh[kConvK];
#pragma unroll
    for (int j = 0; j < kConvK; ++j) wl[j] = make_float2(w[j].x, w[j].y), wh[j] = make_float2(w[j].z, w[j].w);
    const float2 bl = make_float2(bias.x, bias.y), bh = make_float2(bias.z, bias.w);
    // output tensor and column of these channels
    const int qk_c = a.hq * kHeadDim;
    T *dst;
    int dcol, drow;
    if (c0 < qk_c) dst = static_cast<T *>(a.oq), dcol = c0, drow = qk_c;
    else if (c0 < 2 * qk_c) dst = static_cast<T *>(a.ok), dcol = c0 - qk_c, drow = qk_c;
    else dst = static_cast<T *>(a.ov), dcol = c0 - 2 * qk_c, drow = a.hv * kHeadDim;
    const bool norm = a.norm_qk && c0 < 2 * qk_c;  // uniform over the warp (one head)

    const T *XS = reinterpret_cast<const T *>(xs_raw) + threadIdx.x * kCPerThread;
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
            const int row = ss + j - (kConvK - 1);  // token of an x entry
            if (j >= kConvK - 1)
                e[i] = row >= h_begin ? ld4v<T>(XS + size_t(row - h_begin) * kCPerBlock)  // copied with the tile
                                      : ld4v<T>(X + size_t(row) * a.C + c0);
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
                const float4 v = j >= kConvK - 1 ? ld4v<T>(X + size_t(ss + j - (kConvK - 1)) * a.C + c0)
                                 : j == 0          ? e[0]
                                 : j == 1          ? e[1]
                                                   : e[2];
                st4v<T>(S + (size_t(slot) * (kConvK - 1) + i) * a.C + c0, v);
            }
        }
    };
    // one token's 4 channels: taps oldest first, bias innermost, then SiLU,
    // two channels per packed f32x2 operation (the same result per channel;
    // measured 41.8 -> 40.4 us on the T=4096 projections)
    auto conv1 = [&](const float4 &a0, const float4 &a1, const float4 &a2, const float4 &a3) {
        float2 lo = __ffma2_rn(wl[3], make_float2(a3.x, a3.y),
                               __ffma2_rn(wl[2], make_float2(a2.x, a2.y),
                                          __ffma2_rn(wl[1], make_float2(a1.x, a1.y),
                                                     __ffma2_rn(wl[0], make_float2(a0.x, a0.y), bl))));
        float2 hi = __ffma2_rn(wh[3], make_float2(a3.z, a3.w),
                               __ffma2_rn(wh[2], make_float2(a2.z, a2.w),
                                          __ffma2_rn(wh[1], make_float2(a1.z, a1.w),
                                                     __ffma2_rn(wh[0], make_float2(a0.z, a0.w), bh))));
        lo = silu2_f(lo);
        hi = silu2_f(hi);
        return make_float4(lo.x, lo.y, hi.x, hi.y);
    };
    auto emit = [&](int t, const float4 &xv) {
        float4 y = conv1(h0, h1, h2, xv);
        if (norm) {
            float ss = y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w;
            for (int m = 16; m; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
            const float inv = rsqrtf(ss + 1e-6f);
            y.x *= inv; y.y *= inv; y.z *= inv; y.w *= inv;
        }
        st4v<T>(dst + size_t(t) * drow + dcol, y);
        h0 = h1, h1 = h2, h2 = xv;
    };
    // four tokens at once: their windows [h0 h1 h2 x0], [h1 h2 x0 x1],
    // [h2 x0 x1 x2], [x0 x1 x2 x3] and four independent norm reductions
    auto emit4 = [&](int t, const float4 &x0, const float4 &x1, const float4 &x2, const float4 &x3) {
        float4 y[4] = {conv1(h0, h1, h2, x0), conv1(h1, h2, x0, x1), conv1(h2, x0, x1, x2), conv1(x0, x1, x2, x3)};
        if (norm) {
            float ss[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) ss[j] = y[j].x * y[j].x + y[j].y * y[j].y + y[j].z * y[j].z + y[j].w * y[j].w;
#pragma unroll
            for (int m = 16; m; m >>= 1)
#pragma unroll
                for (int j = 0; j < 4; ++j) ss[j] += __shfl_xor_sync(0xffffffffu, ss[j], m);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float inv = rsqrtf(ss[j] + 1e-6f);
                y[j].x *= inv; y[j].y *= inv; y[j].z *= inv; y[j].w *= inv;
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) st4v<T>(dst + size_t(t + j) * drow + dcol, y[j]);
        h0 = x1, h1 = x2, h2 = x3;
    };
    // a tile at a sequence's start takes its history from the conv state (plain
    // loads, issued before the wait); a mid-sequence tile from the copied rows
    const bool at_start = t_begin == cu[s];
    if (at_start) load_history(t_begin);
    const bool landed = mbar_wait(&bar, 0);
    if (!__all_sync(0xffffffffu, landed)) {
        if (lane == 0) record_status(a.status, GDN_ETIMEOUT);
        return;
    }
    if (!at_start) load_history(t_begin);
    for (int t = t_begin; t < t_end;) {
        if (t == s_end) {  // next non-empty sequence starts here
            while (cu[s + 1] <= t) ++s;
            s_end = cu[s + 1];
            load_history(t);
        }
        const int run_end = min(t_end, s_end);  // tokens of sequence s in this tile
        for (; t + 4 <= run_end; t += 4) {
            const T *xr = XS + size_t(t - h_begin) * kCPerBlock;
            emit4(t, ld4v<T>(xr), ld4v<T>(xr + kCPerBlock), ld4v<T>(xr + 2 * kCPerBlock), ld4v<T>(xr + 3 * kCPerBlock));
        }
        for (; t < run_end; ++t) emit(t, ld4v<T>(XS + size_t(t - h_begin) * kCPerBlock));
    }
}

// One token per sequence (decode). A thread owns 8 consecutive channels (one
// 16-byte access per row for bf16) of kStepSeqs sequences: the CTA reads its
// channels' weights and bias once, then issues the x rows and (after the slot
// indices) the three state rows of all its sequences before any arithmetic,
// so that a thread has a dozen independent loads in flight instead of one
// dependent chain per sequence.
constexpr int kStepCh = 8;
constexpr int kStepThreads = 128;                          // 1024 channels per CTA
constexpr int kStepSeqs = 4;

// 8 consecutive values of a row as loaded (one 16-byte access for bf16, two
// for f32), widened to f32 only when used, so that the loads in flight hold
// as few registers as possible
template <typename T>
struct Row8;
template <>
struct Row8<__nv_bfloat16> {
    uint4 u;
    __device__ __forceinline__ void zero() { u = make_uint4(0, 0, 0, 0); }
    __device__ __forceinline__ void load(const __nv_bfloat16 *p) { u = *reinterpret_cast<const uint4 *>(p); }
    __device__ __forceinline__ void store(__nv_bfloat16 *p) const { *reinterpret_cast<uint4 *>(p) = u; }
    __device__ __forceinline__ float get(int i) const {
        const uint32_t w = i < 2 ? u.x : i < 4 ? u.y : i < 6 ? u.z : u.w;
        return __uint_as_float((i & 1) ? (w & 0xffff0000u) : (w << 16));
    }
};
template <>
struct Row8<float> {
    float4 a, b;
    __device__ __forceinline__ void zero() { a = b = make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ __forceinline__ void load(const float *p) {
        a = reinterpret_cast<const float4 *>(p)[0];
        b = reinterpret_cast<const float4 *>(p)[1];
    }
    __device__ __forceinline__ void store(float *p) const {
        reinterpret_cast<float4 *>(p)[0] = a;
        reinterpret_cast<float4 *>(p)[1] = b;
    }
    __device__ __forceinline__ float get(int i) const {
        const float4 &v = i < 4 ? a : b;
        const int j = i & 3;
        return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
    }
};

template <typename T>
__device__ __forceinline__ void st8(T *p, const float (&v)[8]);
template <>
__device__ __forceinline__ void st8<float>(float *p, const float (&v)[8]) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
template <>
__device__ __forceinline__ void st8<__nv_bfloat16>(__nv_bfloat16 *p, const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
        w[q] = *reinterpret_cast<const uint32_t *>(&h);
    }
    *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename T>
__global__ void __launch_bounds__(kStepThreads) k_conv1d_step(ConvArgs a) {
    const int n0 = blockIdx.x * kStepSeqs;
    const int c0 = blockIdx.y * (kStepThreads * kStepCh) + threadIdx.x * kStepCh;
    // heads are 128 channels = 16 threads, so a head is wholly valid or not;
    // invalid threads still join the half-warp reductions below
    const bool cvalid = c0 < a.C;
    const T *X = static_cast<const T *>(a.x);
    T *S = static_cast<T *>(a.state);
    int slot[kStepSeqs];
#pragma unroll
    for (int k = 0; k < kStepSeqs; ++k) {
        const int n = n0 + k;
        slot[k] = (n < a.N && S) ? (a.idx ? a.idx[n] : n) : -1;
    }
    Row8<T> xv[kStepSeqs];
#pragma unroll
    for (int k = 0; k < kStepSeqs; ++k) {
        xv[k].zero();
        if (cvalid && n0 + k < a.N) xv[k].load(X + size_t(n0 + k) * a.C + c0);
    }
    float4 w[8];
    float bias[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        w[i] = cvalid ? reinterpret_cast<const float4 *>(a.weight)[c0 + i] : make_float4(0.f, 0.f, 0.f, 0.f);
        bias[i] = (cvalid && a.bias) ? a.bias[c0 + i] : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kStepSeqs; ++k) {
        if (slot[k] >= a.slots) {
            if (threadIdx.x == 0 && blockIdx.y == 0) record_status(a.status, GDN_EDEVICE_INPUT);
            slot[k] = -1;
        }
    }
    Row8<T> h[kStepSeqs][kConvK - 1];
#pragma unroll
    for (int k = 0; k < kStepSeqs; ++k)
#pragma unroll
        for (int j = 0; j < kConvK - 1; ++j) {
            h[k][j].zero();
            if (cvalid && slot[k] >= 0) h[k][j].load(S + (size_t(slot[k]) * (kConvK - 1) + j) * a.C + c0);
        }
    const int qk_c = a.hq * kHeadDim;
    const bool norm = a.norm_qk && c0 < 2 * qk_c;  // uniform over a head (16 threads)
#pragma unroll
    for (int k = 0; k < kStepSeqs; ++k) {
        const int n = n0 + k;
        float y[8];
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            // taps oldest first: w.x x[t-3], w.y x[t-2], w.z x[t-1], w.w x[t]
            y[i] = silu_f(fmaf(w[i].w, xv[k].get(i),
                               fmaf(w[i].z, h[k][2].get(i),
                                    fmaf(w[i].y, h[k][1].get(i), fmaf(w[i].x, h[k][0].get(i), bias[i])))));
            ss = fmaf(y[i], y[i], ss);
        }
        // sum over the head's 16 threads (lanes of one half-warp)
#pragma unroll
        for (int m = 8; m; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
        if (!cvalid || n >= a.N) continue;
        if (norm) {
            const float inv = rsqrtf(ss + 1e-6f);
#pragma unroll
            for (int i = 0; i < 8; ++i) y[i] *= inv;
        }
        if (c0 < qk_c) st8<T>(static_cast<T *>(a.oq) + size_t(n) * qk_c + c0, y);
        else if (c0 < 2 * qk_c) st8<T>(static_cast<T *>(a.ok) + size_t(n) * qk_c + c0 - qk_c, y);
        else st8<T>(static_cast<T *>(a.ov) + size_t(n) * a.hv * kHeadDim + c0 - 2 * qk_c, y);
        if (slot[k] >= 0) {  // the window moves on by one input
            T *srow = S + size_t(slot[k]) * (kConvK - 1) * a.C + c0;
            h[k][1].store(srow);
            h[k][2].store(srow + a.C);
            xv[k].store(srow + 2 * size_t(a.C));
        }
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
    // tokens per tile (a power of two, up to 16 for bf16): the largest that
    // still gives at least six CTAs per SM over the grid (128-thread CTAs on
    // 16-token tiles measured best: their load and compute phases interleave
    // across the SM's CTAs)
    const int cblocks = (C + kCPerBlock - 1) / kCPerBlock;
    const int esize = p.io_dtype == GDN_DT_BF16 ? 2 : 4;
    const int max_tile = kMaxTileBytes / (kCPerBlock * esize);  // 16 (bf16) or 8 (f32)
    int tile = 1;
    while (tile < max_tile && int64_t(tile) * 2 * 3 * sms <= int64_t(p.total_tokens) * cblocks) tile *= 2;
    // a tile may grow by two rows and takes the K-1 rows before it
    const size_t smem = size_t(tile + kConvK - 2 + kConvK - 1) * kCPerBlock * esize;
    const void *fn = p.io_dtype == GDN_DT_BF16 ? reinterpret_cast<const void *>(k_conv1d_silu<__nv_bfloat16>)
                                               : reinterpret_cast<const void *>(k_conv1d_silu<float>);
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    ConvArgs a{x, weight, bias, conv_state, state_indices, cu_seqlens, out_q, out_k, out_v,
               p.total_tokens, C, p.num_seqs, p.num_state_slots, p.hq, p.hv, tile, norm_qk, cblocks, status};
    const long long nblk = (long long)((p.total_tokens + tile - 1) / tile) * cblocks;
    if (nblk >= (1ll << 31)) return cudaErrorInvalidConfiguration;
    const unsigned grid = unsigned(nblk);
    LaunchScope scope(GDN_K_CONV1D_SILU, s);
    if (p.io_dtype == GDN_DT_BF16) k_conv1d_silu<__nv_bfloat16><<<grid, kCThreads, smem, s>>>(a);
    else k_conv1d_silu<float><<<grid, kCThreads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_conv1d_step(const gdn_problem &p, const void *x, const float *weight, const float *bias,
                               void *conv_state, const int32_t *state_indices, int norm_qk, void *out_q,
                               void *out_k, void *out_v, int *status, cudaStream_t s) {
    const int C = (2 * p.hq + p.hv) * kHeadDim;
    if (p.num_seqs == 0) return cudaSuccess;
    ConvArgs a{x, weight, bias, conv_state, state_indices, nullptr, out_q, out_k, out_v,
               p.num_seqs, C, p.num_seqs, p.num_state_slots, p.hq, p.hv, 1, norm_qk, 1, status};
    const int per_block = kStepThreads * kStepCh;
    const dim3 grid((p.num_seqs + kStepSeqs - 1) / kStepSeqs, (C + per_block - 1) / per_block);
    LaunchScope scope(GDN_K_CONV1D_STEP, s);
    if (p.io_dtype == GDN_DT_BF16) k_conv1d_step<__nv_bfloat16><<<grid, kStepThreads, 0, s>>>(a);
    else k_conv1d_step<float><<<grid, kStepThreads, 0, s>>>(a);
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
