// Output gate over whole tensors (gdn_gated_rmsnorm).
//
// The sgl-qwen3-5-moe page's output_rmsnorm_silu_gate node (the gated-RMSNorm
// row of the Kestrel_VLLM-24 page's kernel table): per token and v-head,
//   y = o / sqrt(mean_j o_j^2 + eps) * weight * silu(z)
// over the head's d_v = 128 channels, norm before gate, the weight applied
// directly. It follows the prefill as its own pass over o, like the page's
// node, which also reads the read-out after it was rounded to the output
// dtype.
//
// HBM-bound: per (token, head) row it reads o and z and writes y
// (3 x 128 elements). Rows are contiguous, so a block of rows of o (and of z)
// is one linear range: each CTA streams blocks of kBlockRows rows per tensor
// into shared memory with bulk copies (cp.async.bulk, completing on an
// mbarrier), kStages blocks deep, from one producer thread, while eight
// consumer warps take four rows at a time (4 channels per lane; four independent chains, as
// the kernel is otherwise bound by the latency of its reductions), reduce each
// row's sum of squares with shuffles and store y straight to global memory
// (fully coalesced, one 8- or 16-byte store per lane). The grid is kCtasPerSm
// CTAs per SM; CTA b takes blocks b, b + grid, ...
#include "gdn_common.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kNThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kStages = 3;
constexpr int kBlockRows = 64;  // rows per block, a multiple of 4 x kConsumerWarps (32 .. 64 measured alike)
constexpr int kCtasPerSm = 2;

// bytes of one block of one tensor
template <typename T>
__host__ __device__ constexpr uint32_t block_bytes() { return uint32_t(kBlockRows) * kHeadDim * sizeof(T); }
template <typename T>
__host__ __device__ constexpr size_t smem_bytes() { return size_t(2) * kStages * block_bytes<T>() + 128; }

template <typename T>
struct Vec4;
template <>
struct Vec4<float> {
    using type = float4;
    static __device__ __forceinline__ float4 to_f(const float4 &v) { return v; }
    static __device__ __forceinline__ float4 from_f(const float4 &v) { return v; }
};
template <>
struct Vec4<__nv_bfloat16> {
    using type = uint2;
    static __device__ __forceinline__ float4 to_f(const uint2 &v) {
        const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.x));
        const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.y));
        return make_float4(lo.x, lo.y, hi.x, hi.y);
    }
    static __device__ __forceinline__ uint2 from_f(const float4 &v) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
        return make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
    }
};

template <typename T>
__global__ void __launch_bounds__(kNThreads, kCtasPerSm)
k_gated_rmsnorm(const void *__restrict__ o, const void *__restrict__ z, const float *__restrict__ weight,
                float eps, void *y, long long rows, int *status) {
    using namespace tc;
    using V = typename Vec4<T>::type;
    constexpr uint32_t kRowBytes = kHeadDim * sizeof(T);
    constexpr int kRows = kBlockRows;
    constexpr uint32_t kBlockBytes = block_bytes<T>();
    constexpr int kRowsPerWarp = kRows / kConsumerWarps;
    static_assert(kRowsPerWarp % 4 == 0, "rows are taken four at a time");
    extern __shared__ __align__(128) uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 127) & ~uintptr_t(127));
    uint8_t *so = sm, *sz = sm + kStages * kBlockBytes;
    __shared__ uint64_t full[kStages], empty[kStages];
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long nblocks = (rows + kRows - 1) / kRows;
    const long long mine = blockIdx.x < nblocks ? (nblocks - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == kConsumerWarps) {  // producer
        if (lane == 0) {
            long long i = 0;
            for (; i < mine; ++i) {
                const int st = int(i % kStages);
                if (i >= kStages && !mbar_wait_spin(&empty[st], uint32_t((i / kStages - 1) & 1))) {
                    abort_flag = 1;
                    break;
                }
                const long long b = blockIdx.x + i * gridDim.x;
                const long long r0 = b * kRows;
                const uint32_t bytes = uint32_t((rows - r0 < kRows ? rows - r0 : kRows) * kRowBytes);
                mbar_arrive_expect_tx(&full[st], 2 * bytes);
                bulk_load(so + st * kBlockBytes, static_cast<const uint8_t *>(o) + r0 * kRowBytes, bytes, &full[st]);
                bulk_load(sz + st * kBlockBytes, static_cast<const uint8_t *>(z) + r0 * kRowBytes, bytes, &full[st]);
            }
            // copies still in flight land before the CTA may exit
            for (long long k = (i > kStages ? i - kStages : 0); k < i; ++k)
                if (!mbar_wait(&full[k % kStages], uint32_t((k / kStages) & 1))) abort_flag = 1;
        }
    } else {  // consumers
        const float4 w = reinterpret_cast<const float4 *>(weight)[lane];
        V *Y = static_cast<V *>(y);  // may alias o: each block of o is in shared memory before y is written
        for (long long i = 0; i < mine; ++i) {
            const int st = int(i % kStages);
            bool ok = mbar_wait_spin(&full[st], uint32_t((i / kStages) & 1));
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) abort_flag = 1;
                break;
            }
            const long long r0 = (blockIdx.x + i * gridDim.x) * kRows;
            const int n = int(rows - r0 < kRows ? rows - r0 : kRows);
            const V *bo = reinterpret_cast<const V *>(so + st * kBlockBytes);
            const V *bz = reinterpret_cast<const V *>(sz + st * kBlockBytes);
            // warp w takes rows w * kRowsPerWarp ... of the block, four at a time so
            // that four independent reduce / scale chains overlap
#pragma unroll
            for (int r4 = 0; r4 < kRowsPerWarp; r4 += 4) {
                const int rb = warp * kRowsPerWarp + r4;
                float4 x[4], g[4];
                float ss[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = rb + j < n ? rb + j : n - 1;  // rows past the end: recomputed, not stored
                    x[j] = Vec4<T>::to_f(bo[r * 32 + lane]);
                    g[j] = Vec4<T>::to_f(bz[r * 32 + lane]);
                    ss[j] = x[j].x * x[j].x + x[j].y * x[j].y + x[j].z * x[j].z + x[j].w * x[j].w;
                }
#pragma unroll
                for (int m = 16; m; m >>= 1)
#pragma unroll
                    for (int j = 0; j < 4; ++j) ss[j] += __shfl_xor_sync(0xffffffffu, ss[j], m);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float inv = rsqrtf(ss[j] * (1.f / kHeadDim) + eps);
                    float4 t;
                    t.x = x[j].x * inv * (w.x * silu_f(g[j].x));
                    t.y = x[j].y * inv * (w.y * silu_f(g[j].y));
                    t.z = x[j].z * inv * (w.z * silu_f(g[j].z));
                    t.w = x[j].w * inv * (w.w * silu_f(g[j].w));
                    if (rb + j < n) Y[(r0 + rb + j) * 32 + lane] = Vec4<T>::from_f(t);
                }
            }
            warp_arrive(&empty[st]);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag) record_status(status, GDN_ETIMEOUT);
}

}  // namespace

cudaError_t launch_gated_rmsnorm(const void *o, const void *z, const float *weight, float eps, void *y,
                                 long long rows, int io_dtype, int *status, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const bool bf = io_dtype == GDN_DT_BF16;
    const void *fn = bf ? reinterpret_cast<const void *>(k_gated_rmsnorm<__nv_bfloat16>)
                        : reinterpret_cast<const void *>(k_gated_rmsnorm<float>);
    const size_t smem = bf ? smem_bytes<__nv_bfloat16>() : smem_bytes<float>();
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    const long long nblocks = (rows + kBlockRows - 1) / kBlockRows;
    const unsigned grid = unsigned(nblocks < (long long)kCtasPerSm * sms ? nblocks : (long long)kCtasPerSm * sms);
    LaunchScope scope(GDN_K_GATED_RMSNORM, s);
    if (bf)
        k_gated_rmsnorm<__nv_bfloat16><<<grid, kNThreads, smem, s>>>(o, z, weight, eps, y, rows, status);
    else
        k_gated_rmsnorm<float><<<grid, kNThreads, smem, s>>>(o, z, weight, eps, y, rows, status);
    return cudaGetLastError();
}

}  // namespace gdn
