// Chunk-form prefill on the tensor cores (the GDN_DT_BF16 path), sm_103a.
//
// Method (Lab3 GDN Prefill page, section "计算过程描述"), per chunk c of valid
// length l_c, with gc the per-chunk prefix sum of the raw gates:
//   A_c = (I + StrictLower(B Gamma K K^T Gamma^-1))^-1,  U_c = A_c B V,
//   W_c = A_c B Gamma K,  V'_c = U_c - W_c S_c,
//   S_{c+1} = gamma_c S_c + K_c^T diag(d_c) V'_c,   d_{c,i} = exp(gc_{l-1} - gc_i)
//   O_c = scale [Gamma Q_c S_c + P_c V'_c],  P_c = Lower(Q K^T) * exp(gc_r - gc_i)
//
// A tcgen05 MMA round trip (issue, completion, wake-up) costs about 900 SM
// cycles on this part whatever its size, so a serial walk with two dependent
// products per chunk (W S, then K^T V') is latency-bound. Substituting the
// state update into the next chunk's V' removes one of them:
//   V'_{c+1} = U_{c+1} - (gamma_c W_{c+1}) S_c - G_c V'_c,
//   G_c = W_{c+1} K_c^T diag(d_c)                    (chunk-parallel)
// so (S_{c+1}, V'_{c+1}, O_c) all follow from (S_c, V'_c) in ONE batch of
// MMAs. Stacking the two 64-row products that share a right operand gives
// M = 128 MMAs (an M = 64 MMA runs at half the rate):
//   D1 = [A_c+1 B ; 0] V_{c+1} + [-gamma_c W_{c+1} ; Gamma_c Q_c] S_c
//        + [-G_c ; P_c] V'_c         rows 0..63 = V'_{c+1}, rows 64..127 = O_c/scale
//   D2 = K_c^T (diag(d_c) V'_c)      S_{c+1} = gamma_c S_c + D2
// The walk starts at a virtual step c = -1 with S_-1 = S0, V'_-1 = 0,
// gamma_-1 = 1 and G_-1 = 0, which yields V'_0 = U_0 - W_0 S0.
//
// k_chunk_prepare_tc (grid: chunk x q/k head, all SMs): gate prefix sums,
//   [K;Q] K^T in one M=128 MMA, the masked gated M and its unit-lower-
//   triangular inverse by blocked (16x16) forward substitution in f32, then
//   W_c and G_{c-1} on the tensor cores. Writes, per (chunk, v-head), bf16
//   tiles already in the 128B-swizzled K-major layout the state kernel's
//   MMAs read: A B, -gamma_{c-1} W_c, -G_{c-1}, P_c; and f32 gc, beta.
// k_chunk_state_output_tc (grid: 64-wide dv tile x v-head x sequence): the
//   serial walk. One producer warp (TMA for q/k/v tiles, bulk copies for the
//   prepared tiles, two step buffers), one MMA warp, four math warps holding
//   the f32 state tile S[128 x 64] in registers (thread t = row t).
//
// Tensor-memory layouts: an M=128 accumulator keeps row m in lane m; an M=64
// accumulator keeps row r in lane 32 (r / 16) + r % 16.
// Every mbarrier wait is bounded; on timeout the CTA records GDN_ETIMEOUT,
// stops, drains its outstanding copies (bounded), frees TMEM and returns.
#include <string.h>

#include "gdn_common.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr uint32_t kTile = 64 * 128;  // bytes of a [64 rows][64 bf16] swizzled tile
constexpr int kFPitch = 68;           // f32 row pitch of the solve matrices

// per (chunk, v-head) outputs of the prepare kernel
constexpr uint32_t kUnitAb = 0;               // A diag(beta)        [i][j]
constexpr uint32_t kUnitW = kTile;            // -gamma_{c-1} W_c    [i][d], two d-halves
constexpr uint32_t kUnitG = 3 * kTile;        // -G_{c-1}            [i][i']
constexpr uint32_t kUnitP = 4 * kTile;        // P_c                 [r][i]
constexpr uint32_t kUnitBytes = 5 * kTile;    // 40 KiB

struct TcWs {
    uint8_t *unit;  // [max_chunks][hv][kUnitBytes]
    float *gb;      // [max_chunks][hv][128]: gc[0..63], beta[0..63]
};

__host__ __device__ inline size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

TcWs tc_carve(void *base, int max_chunks, int hv) {
    char *p = static_cast<char *>(base);
    const size_t units = size_t(max_chunks) * hv;
    TcWs w;
    w.unit = reinterpret_cast<uint8_t *>(p);
    p += al256(units * kUnitBytes);
    w.gb = reinterpret_cast<float *>(p);
    return w;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ uint4 pack8(const float *x) {
    return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                      pack_bf16x2(x[6], x[7]));
}

__device__ __forceinline__ void unpack8(const uint4 u, float *x) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(h[q]);
        x[2 * q] = f.x;
        x[2 * q + 1] = f.y;
    }
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// inclusive prefix sum of 64 values held two per lane (lane l: 2l, 2l+1)
__device__ __forceinline__ void warp_scan64(float &a0, float &a1, int lane) {
    a1 += a0;
    float s = a1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += t;
    }
    const float before = s - a1;
    a0 += before;
    a1 = s;
}

// ===========================================================================
// k_chunk_prepare_tc
// ===========================================================================
constexpr int kPrepThreads = 256;

struct PrepSmem {
    alignas(1024) uint8_t KQ[4 * kTile];  // [K_c ; Q_c] K-major, M = 128: two d-halves of 16 KiB
    alignas(1024) uint8_t Kp[2 * kTile];  // K_{c-1}, two d-halves
    alignas(1024) uint8_t Ag[kTile];      // A diag(beta gamma) bf16 [i][j]
    alignas(1024) uint8_t Wb[2 * kTile];  // W_c bf16 [i][d]
    float M[64 * kFPitch];                // strict lower gated K K^T
    float X[64 * kFPitch];                // (I + M)^-1
    float T[3 * 256];                     // block products of the solve
    float gc[64], beta[64], gcp[64], dprev[64];
    uint64_t bar_load, bar_mma;
    uint32_t tmem;
    int abort;
};

__global__ void __launch_bounds__(kPrepThreads, 2)
k_chunk_prepare_tc(PrefillArgs a, TcWs w, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k) {
    extern __shared__ uint8_t smraw[];
    PrepSmem &s = *reinterpret_cast<PrepSmem *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const int c = blockIdx.x, hk = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (c >= *a.n_chunks) return;  // also a rejected chunk table (-1)
    const ChunkInfo ci = a.chunk_info[c];
    const int l = ci.len;
    const bool has_prev = ci.idx > 0;
    const int prev_start = ci.start - kChunk;

    if (tid == 0) {
        s.abort = 0;
        mbar_init(&s.bar_load, 1);
        mbar_init(&s.bar_mma, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&s.bar_load, (has_prev ? 6u : 4u) * kTile);
        for (int hf = 0; hf < 2; ++hf) {
            tma_load_3d(s.KQ + hf * 2 * kTile, &tm_k, 64 * hf, hk, ci.start, &s.bar_load);
            tma_load_3d(s.KQ + hf * 2 * kTile + kTile, &tm_q, 64 * hf, hk, ci.start, &s.bar_load);
            if (has_prev) tma_load_3d(s.Kp + hf * kTile, &tm_k, 64 * hf, hk, prev_start, &s.bar_load);
        }
    }
    if (warp == 0) {
        tmem_alloc(&s.tmem, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem;
    const uint32_t kTmKK = 0, kTmW = 64, kTmG = 192;
    uint32_t mma_phase = 0;

    // [K;Q] K^T : M=128 (rows 0-63 K K^T, rows 64-127 Q K^T), N=64, K=128
    if (tid == 0) {
        if (mbar_wait(&s.bar_load, 0)) {
            tc_fence_after();
            const uint32_t kq = smem_u32(s.KQ);
            const uint32_t id = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const uint32_t off = (t >> 2) * 2 * kTile + (t & 3) * 32;
                mma_bf16(tmem + kTmKK, sdesc_sw128(kq + off, 16, 1024), sdesc_sw128(kq + off, 16, 1024), id, t > 0);
            }
            mma_commit(&s.bar_mma);
        } else {
            s.abort = 1;
        }
    }
    __syncthreads();
    if (!s.abort && !mbar_wait(&s.bar_mma, mma_phase)) s.abort = 1;
    mma_phase ^= 1;
    __syncthreads();
    tc_fence_after();

    const int q4 = warp & 3, colhalf = warp >> 2;
    for (int hh = 0; !s.abort && hh < a.group; ++hh) {
        const int h = hk * a.group + hh;
        const size_t unit = size_t(c) * a.hv + h;
        uint8_t *uo = w.unit + unit * kUnitBytes;
        // ---- gate prefix sums (this chunk; previous chunk of the sequence) ----
        if (warp < 2) {
            const int base = warp == 0 ? ci.start : prev_start;
            const int len = warp == 0 ? l : (has_prev ? kChunk : 0);
            float a0 = 2 * lane < len ? a.g[size_t(base + 2 * lane) * a.hv + h] : 0.f;
            float a1 = 2 * lane + 1 < len ? a.g[size_t(base + 2 * lane + 1) * a.hv + h] : 0.f;
            warp_scan64(a0, a1, lane);
            float *dst = warp == 0 ? s.gc : s.gcp;
            dst[2 * lane] = a0;
            dst[2 * lane + 1] = a1;
        } else if (warp < 4) {
            const int i = tid - 64;
            s.beta[i] = i < l ? a.beta[size_t(ci.start + i) * a.hv + h] : 0.f;
        }
        __syncthreads();
        if (tid < 64) {
            w.gb[unit * 128 + tid] = s.gc[tid];
            w.gb[unit * 128 + 64 + tid] = s.beta[tid];
            s.dprev[tid] = has_prev ? __expf(s.gcp[63] - s.gcp[tid]) : 0.f;
        }
        // ---- M (from K K^T) and P (from Q K^T), straight out of TMEM ----
        {
            float v[32];
            tmem_ld16(tmem_addr(tmem, 32 * q4, kTmKK + 32 * colhalf), v);
            tmem_ld16(tmem_addr(tmem, 32 * q4, kTmKK + 32 * colhalf + 16), v + 16);
            tmem_ld_wait();
            if (q4 < 2) {
                const int i = 32 * q4 + lane;
                const float bi = s.beta[i], gi = s.gc[i];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int j = 32 * colhalf + e;
                    s.M[i * kFPitch + j] = (j < i && i < l) ? bi * __expf(gi - s.gc[j]) * v[e] : 0.f;
                }
            } else {
                const int r = 32 * (q4 - 2) + lane;
                const float gr = s.gc[r];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int i = 32 * colhalf + e;
                    v[e] = (i <= r && r < l) ? __expf(gr - s.gc[i]) * v[e] : 0.f;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<uint4 *>(uo + kUnitP + sw128_offset(r, 4 * colhalf + q)) = pack8(v + 8 * q);
            }
        }
        __syncthreads();
        // ---- A = (I + M)^-1, blocked 16x16 forward substitution ----
        if (tid < 64) {  // diagonal blocks: thread = (block, column)
            const int b = tid >> 4, jj = tid & 15;
            float x[16];
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) {
                float acc = (ii == jj) ? 1.f : 0.f;
                const float *Mr = s.M + (16 * b + ii) * kFPitch + 16 * b;
#pragma unroll
                for (int m = 0; m < ii; ++m) acc = fmaf(-Mr[m], x[m], acc);
                x[ii] = acc;
            }
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) s.X[(16 * b + ii) * kFPitch + 16 * b + jj] = x[ii];
        } else {  // zero the strictly-upper blocks
            for (int e = tid - 64; e < 6 * 256; e += kPrepThreads - 64) {
                const int blk = e >> 8, ii = (e >> 4) & 15, jj = e & 15;
                const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
                const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
                s.X[(16 * bi + ii) * kFPitch + 16 * bj + jj] = 0.f;
            }
        }
        __syncthreads();
        {
            const int ii = tid >> 4, jj = tid & 15;
#pragma unroll
            for (int L = 1; L < 4; ++L) {
                for (int j = 0; j + L < 4; ++j) {  // T = sum_{k=j}^{i-1} M_ik X_kj
                    const int i = j + L;
                    float acc = 0.f;
                    for (int k = j; k < i; ++k) {
                        const float *Mr = s.M + (16 * i + ii) * kFPitch + 16 * k;
                        const float *Xc = s.X + (16 * k) * kFPitch + 16 * j + jj;
#pragma unroll
                        for (int m = 0; m < 16; ++m) acc = fmaf(Mr[m], Xc[m * kFPitch], acc);
                    }
                    s.T[j * 256 + tid] = acc;
                }
                __syncthreads();
                for (int j = 0; j + L < 4; ++j) {  // X_ij = -X_ii T
                    const int i = j + L;
                    const float *Xr = s.X + (16 * i + ii) * kFPitch + 16 * i;
                    float acc = 0.f;
#pragma unroll
                    for (int m = 0; m < 16; ++m)
                        if (m <= ii) acc = fmaf(Xr[m], s.T[j * 256 + m * 16 + jj], acc);
                    s.X[(16 * i + ii) * kFPitch + 16 * j + jj] = -acc;
                }
                __syncthreads();
            }
        }
        // ---- A diag(beta) -> global; A diag(beta gamma) -> smem operand ----
        for (int p = tid; p < 512; p += kPrepThreads) {
            const int i = p >> 3, ch = p & 7;
            float x[8], y[8];
            const float4 *xr = reinterpret_cast<const float4 *>(s.X + i * kFPitch + 8 * ch);
            const float4 x0 = xr[0], x1 = xr[1];
            x[0] = x0.x; x[1] = x0.y; x[2] = x0.z; x[3] = x0.w;
            x[4] = x1.x; x[5] = x1.y; x[6] = x1.z; x[7] = x1.w;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int j = 8 * ch + e;
                x[e] *= s.beta[j];
                y[e] = x[e] * __expf(s.gc[j]);
            }
            *reinterpret_cast<uint4 *>(uo + kUnitAb + sw128_offset(i, ch)) = pack8(x);
            *reinterpret_cast<uint4 *>(s.Ag + sw128_offset(i, ch)) = pack8(y);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- W_c = Ag K_c : M=64, N=128 (d), K=64 (j); K tile read MN-major ----
        if (tid == 0) {
            tc_fence_after();
            const uint32_t ag = smem_u32(s.Ag), kq = smem_u32(s.KQ);
            const uint32_t id = idesc_bf16_f32(64, 128, false, true);
#pragma unroll
            for (int t = 0; t < 4; ++t)
                mma_bf16(tmem + kTmW, sdesc_sw128(ag + 32 * t, 16, 1024), sdesc_sw128(kq + 2048 * t, 2 * kTile, 1024),
                         id, t > 0);
            mma_commit(&s.bar_mma);
        }
        if (!mbar_wait(&s.bar_mma, mma_phase)) s.abort = 1;
        mma_phase ^= 1;
        tc_fence_after();
        {
            const float gprev = has_prev ? -__expf(s.gcp[63]) : -1.f;
            const int i = 16 * q4 + lane;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float v[16];
                tmem_ld16(tmem_addr(tmem, 32 * q4, kTmW + 64 * colhalf + 16 * j), v);
                tmem_ld_wait();
                if (lane < 16) {
                    uint8_t *wbh = s.Wb + colhalf * kTile;
                    uint8_t *woh = uo + kUnitW + colhalf * kTile;
                    float sv[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) sv[e] = gprev * v[e];
                    *reinterpret_cast<uint4 *>(wbh + sw128_offset(i, 2 * j)) = pack8(v);
                    *reinterpret_cast<uint4 *>(wbh + sw128_offset(i, 2 * j + 1)) = pack8(v + 8);
                    *reinterpret_cast<uint4 *>(woh + sw128_offset(i, 2 * j)) = pack8(sv);
                    *reinterpret_cast<uint4 *>(woh + sw128_offset(i, 2 * j + 1)) = pack8(sv + 8);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- G_{c-1} = W_c K_{c-1}^T diag(d_{c-1}) : M=64, N=64, K=128 ----
        if (has_prev) {
            if (tid == 0) {
                tc_fence_after();
                const uint32_t wb = smem_u32(s.Wb), kp = smem_u32(s.Kp);
                const uint32_t id = idesc_bf16_f32(64, 64, false, false);
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const uint32_t off = (t >> 2) * kTile + (t & 3) * 32;
                    mma_bf16(tmem + kTmG, sdesc_sw128(wb + off, 16, 1024), sdesc_sw128(kp + off, 16, 1024), id, t > 0);
                }
                mma_commit(&s.bar_mma);
            }
            if (!mbar_wait(&s.bar_mma, mma_phase)) s.abort = 1;
            mma_phase ^= 1;
            tc_fence_after();
            const int i = 16 * q4 + lane;
            float v[32];
            tmem_ld16(tmem_addr(tmem, 32 * q4, kTmG + 32 * colhalf), v);
            tmem_ld16(tmem_addr(tmem, 32 * q4, kTmG + 32 * colhalf + 16), v + 16);
            tmem_ld_wait();
            if (lane < 16) {
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = -v[e] * s.dprev[32 * colhalf + e];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<uint4 *>(uo + kUnitG + sw128_offset(i, 4 * colhalf + q)) = pack8(v + 8 * q);
            }
        } else {
            for (int p = tid; p < int(kTile / 16); p += kPrepThreads)
                reinterpret_cast<uint4 *>(uo + kUnitG)[p] = make_uint4(0, 0, 0, 0);
        }
        tc_fence_before();
        __syncthreads();
    }
    if (s.abort && tid == 0) {
        record_status(a.status, GDN_ETIMEOUT);
        mbar_wait(&s.bar_load, 0, 100000000ull);  // bounded drain of the tile copies
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// ===========================================================================
// k_chunk_state_output_tc
// ===========================================================================
constexpr int kMathThreads = 128;
constexpr int kStateThreads = 192;  // 4 math warps + producer warp + MMA warp
constexpr int kDvTile = 64;

struct StepBuf {
    alignas(1024) uint8_t A0[2 * kTile];  // [A_{c+1} B ; 0]          K-major, M=128, K=64
    alignas(1024) uint8_t A1[4 * kTile];  // [-W'_{c+1} ; Gamma_c Q_c] K-major, M=128, K=128 (two d-halves)
    alignas(1024) uint8_t A2[2 * kTile];  // [-G_c ; P_c]             K-major, M=128, K=64
    alignas(1024) uint8_t Bv[kTile];      // V_{c+1}[:, tile]         MN-major B, [j][e]
    alignas(1024) uint8_t Kt[2 * kTile];  // K_c                      MN-major A (K^T), [i][d]
    float gbc[128];                       // gc, beta of chunk c
    float gbn[128];                       // gc, beta of chunk c+1
};

struct StateSmem {
    StepBuf buf[2];
    alignas(1024) uint8_t Sb[2 * kTile];  // S_c bf16 [d][e] (128 rows), MN-major B
    alignas(1024) uint8_t Vp[kTile];      // V'_c bf16 [i][e], MN-major B
    alignas(1024) uint8_t Vd[kTile];      // diag(d_c) V'_c bf16 [i][e], MN-major B
    uint64_t full[2], empty[2], ready, mma_s, mma;
    uint32_t tmem;
    int abort;
};

struct StateArgs {
    PrefillArgs a;
    TcWs w;
};

// dynamic shared memory per block is capped at 227 KiB; one more KiB is
// requested to align the base to 1024 bytes
static_assert(sizeof(StateSmem) + 1024 <= 227 * 1024, "state kernel shared memory");
static_assert(sizeof(StepBuf) % 1024 == 0, "step buffers keep the 1024-byte swizzle alignment");
static_assert(2 * (sizeof(PrepSmem) + 1024) <= 228 * 1024, "two prepare CTAs per SM");

__global__ void __launch_bounds__(kStateThreads, 1)
k_chunk_state_output_tc(StateArgs sa, const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
    extern __shared__ uint8_t smraw[];
    StateSmem &s = *reinterpret_cast<StateSmem *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const PrefillArgs &a = sa.a;
    const TcWs &w = sa.w;
    const int tile = blockIdx.x & 1, n = blockIdx.x >> 1, h = blockIdx.y;
    const int hk = h / a.group, e0 = tile * kDvTile;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (*a.n_chunks < 0) return;  // the chunk table rejected cu_seqlens
    const SeqInfo si = a.seq_info[n];
    const int nc = si.num_chunks;
    const size_t sbase = (size_t(n) * a.hv + h) * kHeadDim * kHeadDim;

    // zero every operand buffer once: regions a step does not load must hold
    // finite values (their products land in rows that are discarded)
    for (uint32_t o = tid * 16; o < sizeof(StateSmem) - 64; o += kStateThreads * 16)
        *reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(&s) + o) = make_uint4(0, 0, 0, 0);
    __syncthreads();
    if (tid == 0) {
        s.abort = 0;
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s.full[b], 1);
            mbar_init(&s.empty[b], 1);
        }
        mbar_init(&s.ready, kMathThreads);
        mbar_init(&s.mma_s, 1);
        mbar_init(&s.mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&s.tmem, 128);
        tmem_relinquish();
    }
    // initial state rows (thread t = row d = t) and its bf16 operand copy
    float Sr[64];
    if (tid < kMathThreads) {
#pragma unroll
        for (int q = 0; q < 64; ++q) Sr[q] = 0.f;
        if (a.s0) {
            const float4 *src = reinterpret_cast<const float4 *>(a.s0 + sbase + size_t(tid) * kHeadDim + e0);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const float4 v = src[q];
                Sr[4 * q] = v.x; Sr[4 * q + 1] = v.y; Sr[4 * q + 2] = v.z; Sr[4 * q + 3] = v.w;
            }
        }
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
            *reinterpret_cast<uint4 *>(s.Sb + sw128_offset(tid, ch)) = pack8(Sr + 8 * ch);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem;
    const uint32_t kTmD1 = 0, kTmD2 = 64;

    if (warp == 4) {
        // ----------------------------- producer -----------------------------
        if (lane == 0 && nc > 0) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
            for (int c = -1; c < nc && !s.abort; ++c) {
                const int b = (c + 1) & 1, use = (c + 1) >> 1;
                if (use > 0 && !mbar_wait(&s.empty[b], (use - 1) & 1)) {
                    s.abort = 1;
                    break;
                }
                StepBuf &B = s.buf[b];
                uint32_t bytes = 0;
                const bool cur = c >= 0, nxt = c + 1 < nc;
                if (cur) bytes += 2 * kTile /*Q*/ + kTile /*P*/ + 2 * kTile /*K*/ + 512;
                if (nxt) bytes += kTile /*Ab*/ + 2 * kTile /*W*/ + kTile /*G*/ + kTile /*V*/ + 512;
                mbar_arrive_expect_tx(&s.full[b], bytes);
                if (cur) {
                    const int cg = si.first_chunk + c;
                    const int start = si.start + kChunk * c;
                    const uint8_t *uo = w.unit + (size_t(cg) * a.hv + h) * kUnitBytes;
                    for (int hf = 0; hf < 2; ++hf) {
                        tma_load_3d(B.A1 + hf * 2 * kTile + kTile, &tm_q, 64 * hf, hk, start, &s.full[b]);
                        tma_load_3d(B.Kt + hf * kTile, &tm_k, 64 * hf, hk, start, &s.full[b]);
                    }
                    bulk_load(B.A2 + kTile, uo + kUnitP, kTile, &s.full[b]);
                    bulk_load(B.gbc, w.gb + (size_t(cg) * a.hv + h) * 128, 512, &s.full[b]);
                }
                if (nxt) {
                    const int cg = si.first_chunk + c + 1;
                    const int start = si.start + kChunk * (c + 1);
                    const uint8_t *uo = w.unit + (size_t(cg) * a.hv + h) * kUnitBytes;
                    bulk_load(B.A0, uo + kUnitAb, kTile, &s.full[b]);
                    bulk_load(B.A1, uo + kUnitW, kTile, &s.full[b]);
                    bulk_load(B.A1 + 2 * kTile, uo + kUnitW + kTile, kTile, &s.full[b]);
                    bulk_load(B.A2, uo + kUnitG, kTile, &s.full[b]);
                    tma_load_3d(B.Bv, &tm_v, e0, h, start, &s.full[b]);
                    bulk_load(B.gbn, w.gb + (size_t(cg) * a.hv + h) * 128, 512, &s.full[b]);
                }
            }
        }
    } else if (warp == 5) {
        // ---------------------------- MMA issuer ----------------------------
        if (lane == 0 && nc > 0) {
            const uint32_t id_kmn = idesc_bf16_f32(128, 64, false, true);
            const uint32_t id_mnmn = idesc_bf16_f32(128, 64, true, true);
            // descriptors of every operand base; a K step only adds its byte
            // offset >> 4 to the start-address field (no carry: < 256 KiB)
            const uint64_t dS = sdesc_sw128(smem_u32(s.Sb), kTile, 1024);
            const uint64_t dVp = sdesc_sw128(smem_u32(s.Vp), kTile, 1024);
            const uint64_t dVd = sdesc_sw128(smem_u32(s.Vd), kTile, 1024);
            // the two step buffers differ by a constant byte offset
            const uint64_t dA0_0 = sdesc_sw128(smem_u32(s.buf[0].A0), 16, 1024);
            const uint64_t dA1_0 = sdesc_sw128(smem_u32(s.buf[0].A1), 16, 1024);
            const uint64_t dA2_0 = sdesc_sw128(smem_u32(s.buf[0].A2), 16, 1024);
            const uint64_t dBv_0 = sdesc_sw128(smem_u32(s.buf[0].Bv), kTile, 1024);
            const uint64_t dKt_0 = sdesc_sw128(smem_u32(s.buf[0].Kt), kTile, 1024);
            const uint64_t dbuf = uint64_t(sizeof(StepBuf) >> 4);
            for (int c = -1; c < nc && !s.abort; ++c) {
                const int b = (c + 1) & 1;
                if (!mbar_wait(&s.ready, (c + 1) & 1)) {
                    s.abort = 1;
                    break;
                }
                tc_fence_after();
                const uint64_t ob = b ? dbuf : 0;
                const uint64_t dA0 = dA0_0 + ob, dA1 = dA1_0 + ob, dA2 = dA2_0 + ob, dBv = dBv_0 + ob,
                               dKt = dKt_0 + ob;
#pragma unroll
                for (int t = 0; t < 4; ++t)  // D2 = K_c^T diag(d_c) V'_c (state update first)
                    mma_bf16(tmem + kTmD2, dKt + (2048 * t >> 4), dVd + (2048 * t >> 4), id_mnmn, t > 0);
                mma_commit(&s.mma_s);
#pragma unroll
                for (int t = 0; t < 4; ++t)  // [A B ; 0] V_{c+1}
                    mma_bf16(tmem + kTmD1, dA0 + (32 * t >> 4), dBv + (2048 * t >> 4), id_kmn, t > 0);
#pragma unroll
                for (int t = 0; t < 8; ++t)  // [-W' ; Gamma Q] S_c
                    mma_bf16(tmem + kTmD1, dA1 + (((t >> 2) * 2 * kTile + (t & 3) * 32) >> 4),
                             dS + (2048 * t >> 4), id_kmn, 1);
#pragma unroll
                for (int t = 0; t < 4; ++t)  // [-G ; P] V'_c
                    mma_bf16(tmem + kTmD1, dA2 + (32 * t >> 4), dVp + (2048 * t >> 4), id_kmn, 1);
                mma_commit(&s.mma);
                mma_commit(&s.empty[b]);
            }
        }
    } else {
        // --------------------------- math warps ----------------------------
        const int t = tid;  // TMEM lane and state row
        const int last_len = si.len - kChunk * (nc - 1);  // valid length of the last chunk
        // Gamma_c Q_c in place (rows 64..127 of A1 of the step's buffer)
        auto scale_q = [&](StepBuf &B) {
#pragma unroll
            for (int k2 = 0; k2 < 8; ++k2) {
                const int p = t + kMathThreads * k2;  // 1024 chunks: 64 rows x 16
                const int r = p >> 4, hf = (p >> 3) & 1, ch = p & 7;
                uint8_t *ptr = B.A1 + hf * 2 * kTile + kTile + sw128_offset(r, ch);
                float x[8];
                unpack8(*reinterpret_cast<const uint4 *>(ptr), x);
                const float gr = __expf(B.gbc[r]);
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] *= gr;
                *reinterpret_cast<uint4 *>(ptr) = pack8(x);
            }
        };
        auto len_of = [&](int c) { return c == nc - 1 ? last_len : kChunk; };
        // A step buffer is handed back to the producer as soon as the step's
        // MMAs complete, so every value the epilogue needs from it (gamma_c,
        // d_{c+1}) is read into registers while the buffer is known to hold
        // this step's data: one step ahead, right after its copies land.
        float gam_cur = 1.f, dn_cur = 0.f;  // gamma_c and d_{c+1}[t] of the current step
        if (nc > 0) {
            if (!mbar_wait(&s.full[0], 0)) s.abort = 1;  // step -1 reads buffer 0 (no Q)
            const int l0 = len_of(0);
            dn_cur = t < l0 ? __expf(s.buf[0].gbn[l0 - 1] - s.buf[0].gbn[t]) : 0.f;
        }
        // an empty sequence has no steps at all (not even the virtual c = -1):
        // its final state is its initial state
        for (int c = -1; nc > 0 && c < nc && !s.abort; ++c) {
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&s.ready);
            // next step's buffer: wait for its copies, scale its Q, take its gates
            float gam_nxt = 1.f, dn_nxt = 0.f;
            if (c + 1 < nc) {
                const int bn = (c + 2) & 1, usen = (c + 2) >> 1;
                if (!mbar_wait(&s.full[bn], usen & 1)) {
                    s.abort = 1;
                    break;
                }
                StepBuf &N = s.buf[bn];
                scale_q(N);
                gam_nxt = __expf(N.gbc[len_of(c + 1) - 1]);
                if (c + 2 < nc) {
                    const int l2 = len_of(c + 2);
                    dn_nxt = t < l2 ? __expf(N.gbn[l2 - 1] - N.gbn[t]) : 0.f;
                }
            }
            const int lc = c < 0 ? 0 : len_of(c);
            // state update: S_{c+1}[t] = gamma_c S_c[t] + D2[t]
            if (!mbar_wait(&s.mma_s, (c + 1) & 1)) {
                s.abort = 1;
                break;
            }
            tc_fence_after();
            {
                float v[64];
#pragma unroll
                for (int j = 0; j < 4; ++j) tmem_ld16(tmem_addr(tmem, 32 * warp, kTmD2 + 16 * j), v + 16 * j);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 64; ++e) Sr[e] = fmaf(gam_cur, Sr[e], v[e]);
            }
            // D1 rows: V'_{c+1} (t < 64) or O_c (t >= 64)
            if (!mbar_wait(&s.mma, (c + 1) & 1)) {
                s.abort = 1;
                break;
            }
            tc_fence_after();
            float d1[64];
#pragma unroll
            for (int j = 0; j < 4; ++j) tmem_ld16(tmem_addr(tmem, 32 * warp, kTmD1 + 16 * j), d1 + 16 * j);
            tmem_ld_wait();
            tc_fence_before();
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
                *reinterpret_cast<uint4 *>(s.Sb + sw128_offset(t, ch)) = pack8(Sr + 8 * ch);
            if (t < 64) {
                if (c + 1 < nc) {
                    float vd[8];
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) vd[e] = dn_cur * d1[8 * ch + e];
                        *reinterpret_cast<uint4 *>(s.Vp + sw128_offset(t, ch)) = pack8(d1 + 8 * ch);
                        *reinterpret_cast<uint4 *>(s.Vd + sw128_offset(t, ch)) = pack8(vd);
                    }
                }
            } else if (c >= 0) {
                const int r = t - 64;
                if (r < lc) {
                    __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(a.out) +
                                          (size_t(si.start + kChunk * c + r) * a.hv + h) * kHeadDim + e0;
                    float o[8];
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[e] = a.scale * d1[8 * ch + e];
                        reinterpret_cast<uint4 *>(orow)[ch] = pack8(o);
                    }
                }
            }
            gam_cur = gam_nxt;
            dn_cur = dn_nxt;
        }
        if (!s.abort && a.final_state) {
            float4 *dst = reinterpret_cast<float4 *>(a.final_state + sbase + size_t(t) * kHeadDim + e0);
#pragma unroll
            for (int q = 0; q < 16; ++q) dst[q] = make_float4(Sr[4 * q], Sr[4 * q + 1], Sr[4 * q + 2], Sr[4 * q + 3]);
        }
    }
    __syncthreads();
    if (s.abort) {
        if (tid == 0) record_status(a.status, GDN_ETIMEOUT);
        if (tid == kMathThreads) {  // bounded drain of copies that may be in flight
            mbar_wait(&s.full[0], 0, 100000000ull);
            mbar_wait(&s.full[1], 0, 100000000ull);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

}  // namespace

size_t prefill_tc_workspace(int max_chunks, int hv) {
    const size_t units = size_t(max_chunks) * hv;
    return al256(units * kUnitBytes) + al256(units * 128 * sizeof(float));
}

cudaError_t launch_prefill_tc(const PrefillArgs &a, void *ws_data, cudaStream_t s) {
    const TcWs w = tc_carve(ws_data, a.max_chunks, a.hv);
    CUtensorMap tq, tk, tv;
    const uint64_t T = uint64_t(a.total_tokens);
    memset(&tq, 0, sizeof(tq));
    memset(&tk, 0, sizeof(tk));
    memset(&tv, 0, sizeof(tv));
    // with no tokens every sequence is empty: the state kernel only copies
    // S0 to the final state and never touches the (then unset) tensor maps
    if (T > 0 &&
        (!make_tmap_bf16_3d(&tq, a.q, kHeadDim, a.hq, T, kHeadDim * 2, uint64_t(a.hq) * kHeadDim * 2, 64, 1, 64) ||
         !make_tmap_bf16_3d(&tk, a.k, kHeadDim, a.hq, T, kHeadDim * 2, uint64_t(a.hq) * kHeadDim * 2, 64, 1, 64) ||
         !make_tmap_bf16_3d(&tv, a.v, kHeadDim, a.hv, T, kHeadDim * 2, uint64_t(a.hv) * kHeadDim * 2, 64, 1, 64)))
        return cudaErrorInvalidValue;
    const size_t prep_smem = sizeof(PrepSmem) + 1024;
    const size_t state_smem = sizeof(StateSmem) + 1024;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(k_chunk_prepare_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, int(prep_smem))))
        return e;
    if ((e = cudaFuncSetAttribute(k_chunk_state_output_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  int(state_smem))))
        return e;
    if (a.max_chunks > 0 && T > 0) {
        LaunchScope scope(GDN_K_CHUNK_PREPARE_TC, s);
        k_chunk_prepare_tc<<<dim3(a.max_chunks, a.hq), kPrepThreads, prep_smem, s>>>(a, w, tq, tk);
    }
    if ((e = cudaGetLastError())) return e;
    {
        LaunchScope scope(GDN_K_STATE_OUTPUT_TC, s);
        StateArgs sa{a, w};
        k_chunk_state_output_tc<<<dim3(2 * a.num_seqs, a.hv), kStateThreads, state_smem, s>>>(sa, tq, tk, tv);
    }
    return cudaGetLastError();
}

}  // namespace gdn
