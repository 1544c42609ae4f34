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
//   D2 = (diag(d_c) K_c)^T V'_c      S_{c+1} = gamma_c S_c + D2
// The walk starts at a virtual step c = -1 with S_-1 = S0, V'_-1 = 0,
// gamma_-1 = 1 and G_-1 = 0, which yields V'_0 = U_0 - W_0 S0.
//
// k_chunk_prepare_tc (grid: chunk x v-head, all SMs): gate prefix sums,
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
// k_chunk_prepare_tc: one CTA per (chunk, v-head), 128 threads, 3 CTAs/SM
// ===========================================================================
constexpr int kPrepThreads = 128;

struct PrepSmem {
    alignas(1024) uint8_t KQ[4 * kTile];  // [K_c ; Q_c] K-major, M = 128 (two d-halves of 16 KiB)
    alignas(1024) uint8_t Kp[2 * kTile];  // K_{c-1}, two d-halves
    // A diag(beta gamma) bf16 [i][j]; before the solve ends it holds the raw
    // gates (g, gp) and the 16x16 block product T of the solve
    alignas(1024) uint8_t Ag[kTile];
    alignas(1024) float MX[64 * kFPitch]; // M, inverted in place into A; later W_c bf16 [i][d]
    float beta[64], gc[64], gcp[64];
    uint64_t bar_load, bar_mma;
    uint32_t tmem;
    int abort;
};

// MX (17 KiB) must also hold the bf16 W tile (16 KiB) once the solve is done
static_assert(64 * kFPitch * sizeof(float) >= 2 * kTile, "W tile reuses the solve buffer");

__global__ void __launch_bounds__(kPrepThreads, 3)
k_chunk_prepare_tc(PrefillArgs a, TcWs w, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k) {
    extern __shared__ uint8_t smraw[];
    PrepSmem &s = *reinterpret_cast<PrepSmem *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const int c = blockIdx.x, h = blockIdx.y, hk = h / a.group;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (c >= *a.n_chunks) return;  // also a rejected chunk table (-1)
    const ChunkInfo ci = a.chunk_info[c];
    const int l = ci.len;
    const bool has_prev = ci.idx > 0;  // chunk c-1 belongs to the same sequence (and is full)
    const int prev_start = ci.start - kChunk;
    const size_t unit = size_t(c) * a.hv + h;
    uint8_t *uo = w.unit + unit * kUnitBytes;
    float *M = s.MX;
    // scratch in the Ag region, all consumed before Ag is written
    float *graw = reinterpret_cast<float *>(s.Ag);  // [64] gates of chunk c
    float *gpraw = graw + 64;                       // [64] gates of chunk c-1
    float *T = graw + 128;                          // [256] block product of the solve
    float *colf = graw + 384;                       // [64]  exp(gc_{e(j)} - gc_j)
    float *rowf = graw + 448;                       // [64][4] exp(gc_i - gc_{e(b)}), b < i/16
    float *DB = graw + 704;                         // [4][16][17] exp(gc_r - gc_i) within a block
    constexpr int kDBp = 17;                        // padded row: lanes of a warp hit distinct banks

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
    // gates of this chunk and of the previous one (independent loads, issued
    // before anything waits)
    if (tid < 64) {
        graw[tid] = tid < l ? a.g[size_t(ci.start + tid) * a.hv + h] : 0.f;
        gpraw[tid] = has_prev ? a.g[size_t(prev_start + tid) * a.hv + h] : 0.f;
    } else {
        const int i = tid - 64;
        s.beta[i] = i < l ? a.beta[size_t(ci.start + i) * a.hv + h] : 0.f;
    }
    if (warp == 0) {
        tmem_alloc(&s.tmem, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem;
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
                mma_bf16(tmem, sdesc_sw128(kq + off, 16, 1024), sdesc_sw128(kq + off, 16, 1024), id, t > 0);
            }
            mma_commit(&s.bar_mma);
        } else {
            s.abort = 1;
        }
    }
    // gate prefix sums while the MMA runs (warp 0: chunk c, warp 1: chunk c-1)
    float gprev = -1.f;  // -gamma_{c-1} (1 for the first chunk of a sequence)
    if (warp < 2) {
        const float *src = warp == 0 ? graw : gpraw;
        float a0 = src[2 * lane], a1 = src[2 * lane + 1];
        warp_scan64(a0, a1, lane);
        float *dst = warp == 0 ? s.gc : s.gcp;
        dst[2 * lane] = a0;
        dst[2 * lane + 1] = a1;
    }
    __syncthreads();
    const float gp63 = s.gcp[63];  // read before gcp is overwritten with d_{c-1}
    if (has_prev) gprev = -__expf(gp63);
    __syncthreads();
    // Decay factors exp(gc_r - gc_i), i <= r, from about 1.5K exponentials
    // instead of one per matrix entry. Within a 16-row block they are taken
    // directly; across blocks, with e(b) = 16 b + 15 the last row of block b,
    //   exp(gc_r - gc_i) = exp(gc_r - gc_e(b_i)) * exp(gc_e(b_i) - gc_i),
    // where both factors are <= 1 because the gates are log-decays (g <= 0,
    // so gc does not increase along the chunk). gamma_j = exp(gc_j) and
    // d_{c-1,i'} = exp(gc_{c-1,63} - gc_{c-1,i'}) are tabulated the same way.
    if (tid < 64) {
        w.gb[unit * 128 + tid] = s.gc[tid];
        w.gb[unit * 128 + 64 + tid] = s.beta[tid];
        colf[tid] = __expf(s.gc[16 * (tid >> 4) + 15] - s.gc[tid]);
#pragma unroll
        for (int b = 0; b < 4; ++b) rowf[4 * tid + b] = b < (tid >> 4) ? __expf(s.gc[tid] - s.gc[16 * b + 15]) : 0.f;
    } else {
        const int j = tid - 64;
        s.gcp[j] = has_prev ? __expf(gp63 - s.gcp[j]) : 0.f;  // becomes d_{c-1}
    }
    for (int e = tid; e < 1024; e += kPrepThreads) {
        const int b = e >> 8, r = (e >> 4) & 15, i = e & 15;
        DB[(b * 16 + r) * kDBp + i] = i <= r ? __expf(s.gc[16 * b + r] - s.gc[16 * b + i]) : 0.f;
    }
    if (!s.abort && !mbar_wait(&s.bar_mma, mma_phase)) s.abort = 1;
    mma_phase ^= 1;
    tc_fence_after();
    // ---- M (rows 0-63: K K^T) and P (rows 64-127: Q K^T), one row per thread ----
    if (!s.abort) {
        float v[64];
#pragma unroll
        for (int j = 0; j < 4; ++j) tmem_ld16(tmem_addr(tmem, 32 * warp, 16 * j), v + 16 * j);
        tmem_ld_wait();
        const int r = tid & 63, br = r >> 4;  // row (of M or P) and its 16-block
        const float *db = DB + (br * 16 + (r & 15)) * kDBp;
        float rf[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) rf[b] = rowf[4 * r + b];
        // decay factor of column i for row r (i <= r), 0 otherwise
        auto decay = [&](int i) {
            const int bi = i >> 4;
            return bi == br ? db[i & 15] : (bi < br ? rf[bi] * colf[i] : 0.f);
        };
        if (warp < 2) {
            const float bi = s.beta[r];
#pragma unroll
            for (int j = 0; j < 64; ++j) v[j] = (j < r && r < l) ? bi * decay(j) * v[j] : 0.f;
            float4 *row = reinterpret_cast<float4 *>(M + r * kFPitch);
#pragma unroll
            for (int q = 0; q < 16; ++q) row[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) v[i] = (i <= r && r < l) ? decay(i) * v[i] : 0.f;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                *reinterpret_cast<uint4 *>(uo + kUnitP + sw128_offset(r, q)) = pack8(v + 8 * q);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tid < 64) s.gc[tid] = __expf(s.gc[tid]);  // gc -> gamma (read only by the A diag(beta gamma) step)
    // ---- A = (I + M)^-1 in place, 16x16 blocks ----

    // diagonal blocks: thread = (block, column); column kept in registers
    if (tid < 64) {
        const int b = tid >> 4, jj = tid & 15;
        float x[16];
#pragma unroll
        for (int ii = 0; ii < 16; ++ii) {
            float acc = (ii == jj) ? 1.f : 0.f;
            const float4 *Mr = reinterpret_cast<const float4 *>(M + (16 * b + ii) * kFPitch + 16 * b);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (4 * q < ii) {
                    const float4 m = Mr[q];
                    if (4 * q + 0 < ii) acc = fmaf(-m.x, x[4 * q + 0], acc);
                    if (4 * q + 1 < ii) acc = fmaf(-m.y, x[4 * q + 1], acc);
                    if (4 * q + 2 < ii) acc = fmaf(-m.z, x[4 * q + 2], acc);
                    if (4 * q + 3 < ii) acc = fmaf(-m.w, x[4 * q + 3], acc);
                }
            }
            x[ii] = acc;
        }
        __syncwarp();
        // every thread of a block has read the block's M rows before any writes
        // (the 16 threads of a block sit in the same warp)
#pragma unroll
        for (int ii = 0; ii < 16; ++ii) M[(16 * b + ii) * kFPitch + 16 * b + jj] = x[ii];
    }
    __syncthreads();
    // off-diagonal blocks, column block j left to right, rows i = j+1..3:

    //   X_ij = -X_ii sum_{k=j}^{i-1} L_ik X_kj; L_ij is overwritten by X_ij,
    //   which is safe because later blocks only read L_ik with k > j
    {
        const int ii = tid >> 3, jj = 2 * (tid & 7);  // two adjacent outputs per thread
#pragma unroll 1
        for (int j = 0; j < 3; ++j) {
#pragma unroll 1
            for (int i = j + 1; i < 4; ++i) {
                float t0 = 0.f, t1 = 0.f;
                for (int k = j; k < i; ++k) {
                    const float4 *Lr = reinterpret_cast<const float4 *>(M + (16 * i + ii) * kFPitch + 16 * k);
                    const float *Xc = M + (16 * k) * kFPitch + 16 * j + jj;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 lq = Lr[q];
                        const float2 x0 = *reinterpret_cast<const float2 *>(Xc + (4 * q + 0) * kFPitch);
                        const float2 x1 = *reinterpret_cast<const float2 *>(Xc + (4 * q + 1) * kFPitch);
                        const float2 x2 = *reinterpret_cast<const float2 *>(Xc + (4 * q + 2) * kFPitch);
                        const float2 x3 = *reinterpret_cast<const float2 *>(Xc + (4 * q + 3) * kFPitch);
                        t0 = fmaf(lq.x, x0.x, t0); t1 = fmaf(lq.x, x0.y, t1);
                        t0 = fmaf(lq.y, x1.x, t0); t1 = fmaf(lq.y, x1.y, t1);
                        t0 = fmaf(lq.z, x2.x, t0); t1 = fmaf(lq.z, x2.y, t1);
                        t0 = fmaf(lq.w, x3.x, t0); t1 = fmaf(lq.w, x3.y, t1);
                    }
                }
                T[ii * 16 + jj] = t0;
                T[ii * 16 + jj + 1] = t1;
                __syncthreads();
                const float4 *Xr = reinterpret_cast<const float4 *>(M + (16 * i + ii) * kFPitch + 16 * i);
                float o0 = 0.f, o1 = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 xq = Xr[q];  // X_ii row (zero above the diagonal)
                    const float2 u0 = *reinterpret_cast<const float2 *>(&T[(4 * q + 0) * 16 + jj]);
                    const float2 u1 = *reinterpret_cast<const float2 *>(&T[(4 * q + 1) * 16 + jj]);
                    const float2 u2 = *reinterpret_cast<const float2 *>(&T[(4 * q + 2) * 16 + jj]);
                    const float2 u3 = *reinterpret_cast<const float2 *>(&T[(4 * q + 3) * 16 + jj]);
                    o0 = fmaf(xq.x, u0.x, o0); o1 = fmaf(xq.x, u0.y, o1);
                    o0 = fmaf(xq.y, u1.x, o0); o1 = fmaf(xq.y, u1.y, o1);
                    o0 = fmaf(xq.z, u2.x, o0); o1 = fmaf(xq.z, u2.y, o1);
                    o0 = fmaf(xq.w, u3.x, o0); o1 = fmaf(xq.w, u3.y, o1);
                }
                *reinterpret_cast<float2 *>(M + (16 * i + ii) * kFPitch + 16 * j + jj) = make_float2(-o0, -o1);
                __syncthreads();
            }
        }
    }
    // ---- A diag(beta) -> global; A diag(beta gamma) -> smem operand ----
    // (entries above the diagonal of A are exactly zero: the strictly upper
    // part of M was never written with anything but zeros)
    for (int p = tid; p < 512; p += kPrepThreads) {
        const int i = p >> 3, ch = p & 7;
        float x[8], y[8];
        const float4 *xr = reinterpret_cast<const float4 *>(M + i * kFPitch + 8 * ch);
        const float4 x0 = xr[0], x1 = xr[1];
        x[0] = x0.x; x[1] = x0.y; x[2] = x0.z; x[3] = x0.w;
        x[4] = x1.x; x[5] = x1.y; x[6] = x1.z; x[7] = x1.w;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int j = 8 * ch + e;
            x[e] = (j <= i) ? x[e] * s.beta[j] : 0.f;
            y[e] = x[e] * s.gc[j];  // gamma_j
        }
        *reinterpret_cast<uint4 *>(uo + kUnitAb + sw128_offset(i, ch)) = pack8(x);
        *reinterpret_cast<uint4 *>(s.Ag + sw128_offset(i, ch)) = pack8(y);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---- W_c = Ag K_c : M=64, N=128 (d), K=64 (j); K tile read MN-major ----
    if (tid == 0 && !s.abort) {
        tc_fence_after();
        const uint32_t ag = smem_u32(s.Ag), kq = smem_u32(s.KQ);
        const uint32_t id = idesc_bf16_f32(64, 128, false, true);
#pragma unroll
        for (int t = 0; t < 4; ++t)
            mma_bf16(tmem, sdesc_sw128(ag + 32 * t, 16, 1024), sdesc_sw128(kq + 2048 * t, 2 * kTile, 1024), id,
                     t > 0);
        mma_commit(&s.bar_mma);
    }
    __syncthreads();
    if (!s.abort && !mbar_wait(&s.bar_mma, mma_phase)) s.abort = 1;
    mma_phase ^= 1;
    tc_fence_after();
    uint8_t *Wb = reinterpret_cast<uint8_t *>(s.MX);  // the solve buffer is free now
    {
        const int i = 16 * warp + lane;  // M=64 accumulator row (lanes 0-15)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float v[16];
            tmem_ld16(tmem_addr(tmem, 32 * warp, 16 * j), v);
            tmem_ld_wait();
            if (lane < 16) {
                uint8_t *wbh = Wb + (j >> 2) * kTile;
                uint8_t *woh = uo + kUnitW + (j >> 2) * kTile;
                float sv[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) sv[e] = gprev * v[e];
                *reinterpret_cast<uint4 *>(wbh + sw128_offset(i, (2 * j) & 7)) = pack8(v);
                *reinterpret_cast<uint4 *>(wbh + sw128_offset(i, (2 * j + 1) & 7)) = pack8(v + 8);
                *reinterpret_cast<uint4 *>(woh + sw128_offset(i, (2 * j) & 7)) = pack8(sv);
                *reinterpret_cast<uint4 *>(woh + sw128_offset(i, (2 * j + 1) & 7)) = pack8(sv + 8);
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---- G_{c-1} = W_c K_{c-1}^T diag(d_{c-1}) : M=64, N=64, K=128 ----
    if (has_prev) {
        if (tid == 0 && !s.abort) {
            tc_fence_after();
            const uint32_t wb = smem_u32(Wb), kp = smem_u32(s.Kp);
            const uint32_t id = idesc_bf16_f32(64, 64, false, false);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const uint32_t off = (t >> 2) * kTile + (t & 3) * 32;
                mma_bf16(tmem, sdesc_sw128(wb + off, 16, 1024), sdesc_sw128(kp + off, 16, 1024), id, t > 0);
            }
            mma_commit(&s.bar_mma);
        }
        __syncthreads();
        if (!s.abort && !mbar_wait(&s.bar_mma, mma_phase)) s.abort = 1;
        mma_phase ^= 1;
        tc_fence_after();
        const int i = 16 * warp + lane;
        float v[64];
#pragma unroll
        for (int j = 0; j < 4; ++j) tmem_ld16(tmem_addr(tmem, 32 * warp, 16 * j), v + 16 * j);
        tmem_ld_wait();
        if (lane < 16) {
#pragma unroll
            for (int e = 0; e < 64; ++e) v[e] = -v[e] * s.gcp[e];  // d_{c-1}
#pragma unroll
            for (int q = 0; q < 8; ++q)
                *reinterpret_cast<uint4 *>(uo + kUnitG + sw128_offset(i, q)) = pack8(v + 8 * q);
        }
    } else {
        for (int p = tid; p < int(kTile / 16); p += kPrepThreads)
            reinterpret_cast<uint4 *>(uo + kUnitG)[p] = make_uint4(0, 0, 0, 0);
    }
    if (s.abort && tid == 0) {
        record_status(a.status, GDN_ETIMEOUT);
        mbar_wait(&s.bar_load, 0, 100000000ull);  // bounded drain of the tile copies
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
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
    alignas(1024) uint8_t Kt[2 * kTile];  // diag(d_c) K_c             MN-major A (K^T), [i][d]
    float gbc[128];                       // gc, beta of chunk c
};

struct StateSmem {
    StepBuf buf[2];
    alignas(1024) uint8_t Sb[2 * kTile];  // S_c bf16 [d][e] (128 rows), MN-major B
    alignas(1024) uint8_t Vp[kTile];      // V'_c bf16 [i][e], MN-major B
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
// three CTAs per SM: 228 KiB per SM, 1 KiB reserved per CTA, 1 KiB alignment slack
static_assert(3 * (sizeof(PrepSmem) + 2048) <= 228 * 1024, "three prepare CTAs per SM");

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
                if (nxt) bytes += kTile /*Ab*/ + 2 * kTile /*W*/ + kTile /*G*/ + kTile /*V*/;
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
                for (int t = 0; t < 4; ++t)  // D2 = (diag(d_c) K_c)^T V'_c (state update first)
                    mma_bf16(tmem + kTmD2, dKt + (2048 * t >> 4), dVp + (2048 * t >> 4), id_mnmn, t > 0);
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
        auto len_of = [&](int c) { return c == nc - 1 ? last_len : kChunk; };
        // Readies a loaded step buffer for its MMAs, in place: rows r of Q_c
        // scaled by gamma_r = exp(gc_r), rows i of K_c by d_{c,i} =
        // exp(gc_{l-1} - gc_i) (zero for i >= l, which also clears rows that
        // belong to the next sequence). Returns gamma_c = exp(gc_{l-1}).
        // A step buffer goes back to the producer as soon as its MMAs
        // complete, so nothing is read from it after that point.
        auto ready_buffer = [&](StepBuf &B, int lc) {
            const float glast = B.gbc[lc - 1];
#pragma unroll
            for (int k2 = 0; k2 < 8; ++k2) {
                const int p = t + kMathThreads * k2;  // 1024 chunks: 64 rows x 16
                const int r = p >> 4, hf = (p >> 3) & 1, ch = p & 7;
                uint8_t *qp = B.A1 + hf * 2 * kTile + kTile + sw128_offset(r, ch);
                uint8_t *kp = B.Kt + hf * kTile + sw128_offset(r, ch);
                float x[8], y[8];
                unpack8(*reinterpret_cast<const uint4 *>(qp), x);
                unpack8(*reinterpret_cast<const uint4 *>(kp), y);
                const float gr = __expf(B.gbc[r]);
                const float dr = r < lc ? __expf(glast - B.gbc[r]) : 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    x[e] *= gr;
                    y[e] *= dr;
                }
                *reinterpret_cast<uint4 *>(qp) = pack8(x);
                *reinterpret_cast<uint4 *>(kp) = pack8(y);
            }
            return __expf(glast);
        };
        float gam_cur = 1.f;  // gamma_c of the current step (1 for the virtual step c = -1)
        if (nc > 0) {
            if (!mbar_wait(&s.full[0], 0)) s.abort = 1;  // step -1: nothing to scale
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&s.ready);
        }
        // an empty sequence has no steps at all (not even the virtual c = -1):
        // its final state is its initial state
        for (int c = -1; nc > 0 && c < nc && !s.abort; ++c) {
            // (A) while step c's MMAs run: ready the next step's buffer
            float gam_nxt = 1.f;
            if (c + 1 < nc) {
                const int bn = (c + 2) & 1, usen = (c + 2) >> 1;
                if (!mbar_wait(&s.full[bn], usen & 1)) {
                    s.abort = 1;
                    break;
                }
                gam_nxt = ready_buffer(s.buf[bn], len_of(c + 1));
            }
            // (B) the chain: S_{c+1} and V'_{c+1} go to their operand buffers
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
            if (!mbar_wait(&s.mma, (c + 1) & 1)) {
                s.abort = 1;
                break;
            }
            tc_fence_after();
            float d1[64];
#pragma unroll
            for (int j = 0; j < 4; ++j) tmem_ld16(tmem_addr(tmem, 32 * warp, kTmD1 + 16 * j), d1 + 16 * j);
            tmem_ld_wait();
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
                *reinterpret_cast<uint4 *>(s.Sb + sw128_offset(t, ch)) = pack8(Sr + 8 * ch);
            if (t < 64 && c + 1 < nc) {
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    *reinterpret_cast<uint4 *>(s.Vp + sw128_offset(t, ch)) = pack8(d1 + 8 * ch);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            if (c + 1 < nc) mbar_arrive(&s.ready);
            // (C) output rows of chunk c, overlapping step c+1's MMAs
            if (t >= 64 && c >= 0) {
                const int r = t - 64;
                if (r < len_of(c)) {
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
        k_chunk_prepare_tc<<<dim3(a.max_chunks, a.hv), kPrepThreads, prep_smem, s>>>(a, w, tq, tk);
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
