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
// cycles, so a serial walk with two dependent products per chunk (W S, then
// K^T V') is latency-bound. Substituting the state update into the next
// chunk's V' removes one of them:
//   V'_{c+1} = U_{c+1} - (gamma_c W_{c+1}) S_c - G_c V'_c,
//   G_c = W_{c+1} K_c^T diag(d_c)                    (chunk-parallel)
// so (S_{c+1}, V'_{c+1}, O_c) all follow from (S_c, V'_c) in one batch of
// MMAs. The walk starts at a virtual step c = -1 with S_-1 = S0, V'_-1 = 0,
// gamma_-1 = 1 and G_-1 = 0, which yields V'_0 = U_0 - W_0 S0.
//
// prep_unit (one unit = chunk c x v-head h): gate prefix sums, [K;Q] K^T in
//   one M=128 MMA, the masked gated M and its unit-lower-triangular inverse
//   by blocked (16x16) substitution in f32, then W_c, U_c^T and K_{c-1} W_c^T
//   on the tensor cores. It writes bf16 tiles in the 128B-swizzled layouts
//   the walk's MMAs read (P_c, -gamma_{c-1} W_c, -K_{c-1} W_c^T, U_c^T), f32
//   Gamma and d tables, then a ready flag.
// state_walk (one walk = sequence x v-head): the serial walk, transposed so
//   that dv is the MMA's M dimension; see the comment above it.
// k_chunk_fused_tc runs both in one cooperative grid, one CTA per SM: a few
//   CTAs walk while the others prepare the later chunks.
//
// Tensor-memory layouts: an M=128 accumulator keeps row m in lane m; an M=64
// accumulator keeps row r in lane 32 (r / 16) + r % 16.
// Every mbarrier and flag wait is bounded; on timeout the CTA records
// GDN_ETIMEOUT, stops, drains its outstanding copies (bounded) and returns.
#include <string.h>

#include <cmath>

#include "gdn_common.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr uint32_t kTile = 64 * 128;  // bytes of a [64 rows][64 bf16] swizzled tile
constexpr int kFPitch = 68;           // f32 row pitch of the solve matrices

// per (chunk, v-head) outputs of the prepare kernel, bf16, 128B-swizzled rows
constexpr uint32_t kUnitP = 0;              // P_c                  [r][j]  64 rows
constexpr uint32_t kUnitW = kTile;          // -gamma_{c-1} W_c     [i][d]  64 rows, two d-halves
constexpr uint32_t kUnitG = 3 * kTile;      // -K_{c-1} W_c^T       [t][i]  64 rows
constexpr uint32_t kUnitU = 4 * kTile;      // U_c^T = (A B V)^T    [e][i] 128 rows
constexpr uint32_t kUnitQ = 6 * kTile;      // scale Gamma Q_c      [r][d]  64 rows, two d-halves
constexpr uint32_t kUnitBytes = 8 * kTile;  // 64 KiB

struct TcWs {
    uint8_t *unit;  // [max_chunks][hv][kUnitBytes]
    float *gb;      // [max_chunks][hv][128]: Gamma_r = exp(gc_r) (r < 64), then d_i (i < 64)
    int *ready;     // [max_chunks][hv]: 1 once the unit is written (zeroed by the chunk table)
};

__host__ __device__ inline size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

TcWs tc_carve(void *base, int max_chunks, int hv) {
    char *p = static_cast<char *>(base);
    const size_t units = size_t(max_chunks) * hv;
    TcWs w;
    w.unit = reinterpret_cast<uint8_t *>(p);
    p += al256(units * kUnitBytes);
    w.gb = reinterpret_cast<float *>(p);
    p += al256(units * 128 * sizeof(float));
    w.ready = reinterpret_cast<int *>(p);
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

// e^x for the decay exponents (x <= 0: sums of log-decay gates), written as
// 2^(x log2 e) on the special-function unit's base-2 exponential (PTX
// ex2.approx.ftz.f32, relative error near 2^-22 per the PTX ISA). Results
// below the smallest normal float flush to zero, which is the limit of a
// decay factor; the product x log2 e adds a relative error of about
// |x| 2^-24, negligible against the bf16 operands these factors scale.
__device__ __forceinline__ float exp_decay(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * 1.4426950408889634f));
    return y;
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
// prep_unit: one (chunk, v-head) unit on a 128-thread engine
// ===========================================================================
constexpr int kPrepThreads = 128;

struct PrepSmem {
    // [K_c ; Q_c] K-major, M = 128 (two d-halves of 16 KiB: K rows, then Q
    // rows). Once [K;Q]K^T is done the Q slots take V_c (for U^T), and once
    // W_c is done the K slots take W_c bf16 (for K_{c-1} W_c^T).
    alignas(1024) uint8_t KQ[4 * kTile];
    alignas(1024) uint8_t Kp[2 * kTile];  // K_{c-1}, two d-halves
    // A diag(beta gamma) bf16 [i][j]; before the solve ends it holds the raw
    // gates (g, gp) and the 16x16 block product T of the solve
    alignas(1024) uint8_t Ag[kTile];
    alignas(1024) float MX[64 * kFPitch]; // M, inverted in place into A; then A diag(beta) bf16 [i][j]
    float beta[64], gc[64], gcp[64];
    uint64_t bar_load, bar_v, bar_mma, bar_drain;
    uint32_t tmem;
    int abort;
};


// One unit (chunk c, v-head h) on a prepare engine: 128 threads (four
// consecutive warps, so warp % 4 is the TMEM lane quarter) synchronised on
// their own named barrier, with their own shared-memory slice and 128 TMEM
// columns. ld_phase / mma_phase carry the engine's mbarrier phases from unit
// to unit.
__device__ __forceinline__ void prep_unit(const PrefillArgs &a, const TcWs &w, const CUtensorMap *tm_q,
                                          const CUtensorMap *tm_k, const CUtensorMap *tm_v, PrepSmem &s,
                                          uint32_t tmem, int bar_id, uint32_t &ld_phase, uint32_t &mma_phase, int c,
                                          int h) {
    const int hk = h / a.group;
    const int tid = threadIdx.x & (kPrepThreads - 1), warp = tid >> 5, lane = tid & 31;
    auto ebar = [&]() { named_bar_sync(bar_id, kPrepThreads); };
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
    float *T = graw + 128;                          // [4][256] per-warp scratch of the solve

    if (tid == 0) {
        mbar_arrive_expect_tx(&s.bar_load, (has_prev ? 6u : 4u) * kTile);
        for (int hf = 0; hf < 2; ++hf) {
            tma_load_3d(s.KQ + hf * 2 * kTile, tm_k, 64 * hf, hk, ci.start, &s.bar_load);
            tma_load_3d(s.KQ + hf * 2 * kTile + kTile, tm_q, 64 * hf, hk, ci.start, &s.bar_load);
            if (has_prev) tma_load_3d(s.Kp + hf * kTile, tm_k, 64 * hf, hk, prev_start, &s.bar_load);
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
    tc_fence_before();
    ebar();
    tc_fence_after();

    // [K;Q] K^T : M=128 (rows 0-63 K K^T, rows 64-127 Q K^T), N=64, K=128
    if (tid == 0) {
        if (mbar_wait(&s.bar_load, ld_phase, a.wait_ns)) {
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
    ebar();
    if (has_prev) gprev = -exp_decay(s.gcp[63]);  // gamma_{c-1} = exp(sum of the gates of chunk c-1)
    // The state walk gets Gamma_r = exp(gc_r) and d_i = exp(gc_{l-1} - gc_i)
    // (zero for i >= l); the gates past l are zero, so gc_63 = gc_{l-1}.
    if (tid < 64) {
        w.gb[unit * 128 + tid] = exp_decay(s.gc[tid]);
    } else {
        const int i = tid - 64;
        w.gb[unit * 128 + 64 + i] = i < l ? exp_decay(s.gc[63] - s.gc[i]) : 0.f;
    }
    // scale Gamma_r Q_r for the walk's output product, while [K;Q]K^T runs
    // (both only read the Q tile). A row scale commutes with the swizzle
    // inside the row, so the copy is linear: thread p moves bytes 16p..16p+15
    // of each 8 KiB half, and every warp writes 512 contiguous bytes.
    if (mbar_wait(&s.bar_load, ld_phase, a.wait_ns)) {
#pragma unroll 2
        for (int k2 = 0; k2 < 8; ++k2) {
            const int p = tid + kPrepThreads * k2, hf = p >> 9, o16 = p & 511, r = o16 >> 3;
            float x[8];
            unpack8(*reinterpret_cast<const uint4 *>(s.KQ + hf * 2 * kTile + kTile + 16 * o16), x);
            const float f = a.scale * exp_decay(s.gc[r]);
#pragma unroll
            for (int j = 0; j < 8; ++j) x[j] *= f;
            *reinterpret_cast<uint4 *>(uo + kUnitQ + hf * kTile + 16 * o16) = pack8(x);
        }
    }
    // warp-uniform outcome: the tcgen05 loads below are .sync.aligned
    const bool ok_kq = __all_sync(0xffffffffu, !s.abort && mbar_wait(&s.bar_mma, mma_phase, a.wait_ns));
    if (!ok_kq) s.abort = 1;
    mma_phase ^= 1;
    tc_fence_after();
    // ---- M (rows 0-63: K K^T) and P (rows 64-127: Q K^T), one row per thread ----
    if (ok_kq) {
        float v[64];
#pragma unroll
        for (int j = 0; j < 4; ++j) tmem_ld16(tmem_addr(tmem, 32 * warp, 16 * j), v + 16 * j);
        tmem_ld_wait();
        // Decay factor of column i in row r: exp(gc_r - gc_i) for i <= r. The
        // gates are log-decays (g <= 0), so gc does not increase along the
        // chunk and the exponent is never positive: no overflow, and a decay
        // too strong for f32 flushes to zero. Columns past the warp's last row
        // are zero for the whole warp and skipped.
        const int r = tid & 63;            // row of M (warps 0-1) or P (warps 2-3)
        const int rmax = (tid & 32) + 31;  // last row held by this warp
        const float gr = s.gc[r];
        const bool live = r < l;
        const float sr = warp < 2 ? s.beta[r] : a.scale;  // M rows carry beta_r, P rows the output scale
        const int strict = warp < 2 ? 1 : 0;          // M is strictly lower, P includes the diagonal
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const float4 g4 = reinterpret_cast<const float4 *>(s.gc)[q];  // same address in every lane
            const float gq[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) {
                const int i = 4 * q + k2;
                if (i <= rmax) {
                    const bool on = live && i + strict <= r;
                    v[i] = on ? sr * exp_decay(gr - gq[k2]) * v[i] : 0.f;
                } else {
                    v[i] = 0.f;
                }
            }
        }
        if (warp < 2) {
            float4 *row = reinterpret_cast<float4 *>(M + r * kFPitch);
#pragma unroll
            for (int q = 0; q < 16; ++q) row[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q)
                *reinterpret_cast<uint4 *>(uo + kUnitP + sw128_offset(r, q)) = pack8(v + 8 * q);
        }
    }
    tc_fence_before();
    ebar();
    // the Q slots are free now that every warp has copied its share of the
    // scaled Q tile (the barrier above): V_c goes there for U^T, needed only
    // after the solve. Issued before that barrier, the load could overwrite
    // rows a slower warp had still to copy.
    if (tid == 0 && !s.abort) {
        mbar_arrive_expect_tx(&s.bar_v, 2 * kTile);
        for (int hf = 0; hf < 2; ++hf) tma_load_3d(s.KQ + hf * 2 * kTile + kTile, tm_v, 64 * hf, h, ci.start, &s.bar_v);
    }
    if (tid < 64) s.gc[tid] = exp_decay(s.gc[tid]);  // gc -> gamma (read only by the A diag(beta gamma) step)
    // ---- A = (I + M)^-1, 16x16 blocks ----

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
    ebar();
    // off-diagonal blocks by anti-diagonal levels, one warp per block of a
    // level, on warp-level tensor-core MMAs (tf32 operands, f32 accumulate):
    //   level 1: (1,0) (2,1) (3,2);  level 2: (2,0) (3,1);  level 3: (3,0)
    //   T_ij = sum_{k=j}^{i-1} L_ik X_kj,   X_ij = -X_ii T_ij
    // X_ij (i > j) goes to the mirror block (j, i) of the strict upper
    // triangle (zero until now), because later levels still read the
    // original L blocks below the diagonal. No block of a level reads what
    // another block of the same level writes.
    {
        auto blk = [&](int r, int c) { return M + (16 * r) * kFPitch + 16 * c; };
        float *Tw = T + 256 * warp;  // this warp's 16x16 scratch (pitch 16)
#pragma unroll
        for (int lev = 1; lev <= 3; ++lev) {
            if (warp < 4 - lev) {  // warp-uniform: block (warp + lev, warp)
                const int j = warp, i = j + lev;
                float t0[4] = {0.f, 0.f, 0.f, 0.f}, t1[4] = {0.f, 0.f, 0.f, 0.f};
                for (int k = j; k < i; ++k)  // X_kj: the diagonal block in place, else its mirror (j, k)
                    mma_block16(t0, t1, blk(i, k), kFPitch, k == j ? blk(j, j) : blk(j, k), kFPitch);
                store_block16(Tw, 16, t0, t1);
                __syncwarp();
                float x0[4] = {0.f, 0.f, 0.f, 0.f}, x1[4] = {0.f, 0.f, 0.f, 0.f};
                mma_block16(x0, x1, blk(i, i), kFPitch, Tw, 16, /*negate_x=*/true);
                store_block16(blk(j, i), kFPitch, x0, x1);
                __syncwarp();  // the scratch is rewritten at the next level
            }
            ebar();
        }
    }
    // ---- A diag(beta) and A diag(beta gamma) -> bf16 smem operands ----
    // (A is unit lower triangular: the mask j <= i zeroes everything above
    // the diagonal, where the mirror blocks now sit). A diag(beta) overwrites
    // the f32 solve buffer, so every thread reads its pieces first.
    uint8_t *Ab = reinterpret_cast<uint8_t *>(s.MX);
    {
        float xs[4][8];
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
            const int p = tid + kPrepThreads * k2, i = p >> 3, ch = p & 7;
            // block (i/16, ch/2) of A; below the diagonal it sits in the mirror block
            const int bi = i >> 4, bj = ch >> 1;
            const float4 *xr = reinterpret_cast<const float4 *>(
                bj < bi ? M + (16 * bj + (i & 15)) * kFPitch + 16 * bi + 8 * (ch & 1) : M + i * kFPitch + 8 * ch);
            const float4 x0 = xr[0], x1 = xr[1];
            xs[k2][0] = x0.x; xs[k2][1] = x0.y; xs[k2][2] = x0.z; xs[k2][3] = x0.w;
            xs[k2][4] = x1.x; xs[k2][5] = x1.y; xs[k2][6] = x1.z; xs[k2][7] = x1.w;
        }
        ebar();
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
            const int p = tid + kPrepThreads * k2, i = p >> 3, ch = p & 7;
            float y[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int j = 8 * ch + e;
                xs[k2][e] = (j <= i) ? xs[k2][e] * s.beta[j] : 0.f;
                y[e] = xs[k2][e] * s.gc[j];  // gamma_j
            }
            *reinterpret_cast<uint4 *>(Ab + sw128_offset(i, ch)) = pack8(xs[k2]);
            *reinterpret_cast<uint4 *>(s.Ag + sw128_offset(i, ch)) = pack8(y);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    ebar();
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
    ebar();
    if (!s.abort && !mbar_wait(&s.bar_mma, mma_phase, a.wait_ns)) s.abort = 1;
    mma_phase ^= 1;
    tc_fence_after();
    // free now: Ag (the W operand) and the solve buffer past A diag(beta)
    uint8_t *wst1 = reinterpret_cast<uint8_t *>(s.MX) + kTile;
    {
        const int i = 16 * warp + lane;  // M=64 accumulator row (lanes 0-15)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float v[16];
            tmem_ld16(tmem_addr(tmem, 32 * warp, 16 * j), v);
            tmem_ld_wait();
            if (lane < 16) {
                uint8_t *wbh = s.KQ + (j >> 2) * 2 * kTile;  // K slot of d-half j/4 (K_c is done)
                uint8_t *woh = (j >> 2) ? wst1 : s.Ag;        // staging of -gamma_{c-1} W_c for a bulk store
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
    ebar();
    if (tid == 0) {  // whole 8 KiB tiles: one bulk copy each instead of scattered 16-byte stores
        bulk_store(uo + kUnitW, s.Ag, kTile);
        bulk_store(uo + kUnitW + kTile, wst1, kTile);
        bulk_commit_group();
    }
    // ---- U_c^T = V_c^T (A diag(beta))^T : M=128 (e), N=64 (i), K=64 (j),
    //      V tile read as an MN-major A;  K_{c-1} W_c^T : M=64 (t), N=64 (i), K=128
    if (tid == 0 && !s.abort) {
        if (mbar_wait(&s.bar_v, ld_phase, a.wait_ns)) {
            tc_fence_after();
            const uint32_t kq = smem_u32(s.KQ), ab = smem_u32(Ab);
            const uint32_t idu = idesc_bf16_f32(128, 64, true, false);
#pragma unroll
            for (int t = 0; t < 4; ++t)
                mma_bf16(tmem, sdesc_sw128(kq + kTile + 2048 * t, 2 * kTile, 1024), sdesc_sw128(ab + 32 * t, 16, 1024),
                         idu, t > 0);
            if (has_prev) {
                const uint32_t kp = smem_u32(s.Kp);
                const uint32_t idg = idesc_bf16_f32(64, 64, false, false);
#pragma unroll
                for (int t = 0; t < 8; ++t)
                    mma_bf16(tmem + 64, sdesc_sw128(kp + (t >> 2) * kTile + (t & 3) * 32, 16, 1024),
                             sdesc_sw128(kq + (t >> 2) * 2 * kTile + (t & 3) * 32, 16, 1024), idg, t > 0);
            }
            mma_commit(&s.bar_mma);
        } else {
            s.abort = 1;
        }
    }
    ebar();
    const bool ok_u = __all_sync(0xffffffffu, !s.abort && mbar_wait(&s.bar_mma, mma_phase, a.wait_ns));
    if (!ok_u) s.abort = 1;
    mma_phase ^= 1;
    tc_fence_after();
    if (ok_u) {
        // U^T row e = tid (M=128: lane e)
        float v[64];
#pragma unroll
        for (int j = 0; j < 4; ++j) tmem_ld16(tmem_addr(tmem, 32 * warp, 16 * j), v + 16 * j);
        tmem_ld_wait();
        // staged in the V slots (V is done): rows 0-63 and 64-127 are the two
        // 8 KiB halves of the tile, with the same swizzle (it depends on row % 8)
        uint8_t *ust = s.KQ + (tid >> 6) * 2 * kTile + kTile;
#pragma unroll
        for (int q = 0; q < 8; ++q)
            *reinterpret_cast<uint4 *>(ust + sw128_offset(tid & 63, q)) = pack8(v + 8 * q);
        if (has_prev) {
            // row t = 16 warp + lane of -K_{c-1} W_c^T (M=64: lanes 0-15)
#pragma unroll
            for (int j = 0; j < 4; ++j) tmem_ld16(tmem_addr(tmem + 64, 32 * warp, 16 * j), v + 16 * j);
            tmem_ld_wait();
            if (lane < 16) {
                const int t = 16 * warp + lane;
#pragma unroll
                for (int e = 0; e < 64; ++e) v[e] = -v[e];
#pragma unroll
                for (int q = 0; q < 8; ++q)  // staged in the first W slot (the last MMA is done)
                    *reinterpret_cast<uint4 *>(s.KQ + sw128_offset(t, q)) = pack8(v + 8 * q);
            }
        }
    }
    if (!has_prev) {
        for (int p = tid; p < int(kTile / 16); p += kPrepThreads)
            reinterpret_cast<uint4 *>(uo + kUnitG)[p] = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    ebar();
    if (tid == 0) {
        if (ok_u) {
            bulk_store(uo + kUnitU, s.KQ + kTile, kTile);
            bulk_store(uo + kUnitU + kTile, s.KQ + 3 * kTile, kTile);
            if (has_prev) bulk_store(uo + kUnitG, s.KQ, kTile);
            bulk_commit_group();
        }
        bulk_wait_group_all();  // every bulk store has completed before the CTA exits
    }
    if (s.abort && tid == 0) {
        record_status(a.status, GDN_ETIMEOUT);
        mbar_wait(&s.bar_load, ld_phase, 100000000ull);  // bounded drain of the tile copies
        mbar_wait(&s.bar_v, ld_phase, 100000000ull);
        // and of the MMAs this thread issued: the commit tracks every one
        // of them (the engine stops after an abort, so phase 0 is its only use)
        mma_commit(&s.bar_drain);
        mbar_wait(&s.bar_drain, 0, 100000000ull);
    }
    ld_phase ^= 1;
    // publish the unit: the plain stores of every engine thread are ordered
    // before the flag by the barrier and the release store's gpu-scope fence
    // (a sequentially consistent fence on top cost ~2 us here); the bulk
    // copies completed above, the proxy fence orders them before the flag
    tc_fence_before();
    ebar();
    if (tid == 0 && !s.abort) {
        fence_proxy_async_global();
        st_release_gpu(w.ready + unit, 1);
    }
}

// ===========================================================================
// state_walk: one (sequence, v-head) walk on 10 warps
// ===========================================================================
// The walk runs transposed, with dv (e) as the MMA's M dimension so that the
// whole 128-wide state of a head is one M=128 accumulator and the operands the
// math warps produce each step (Sigma = S^T and X = V'^T) are written straight
// into tensor memory as the A operands of the next step's MMAs:
//   (c) [V'^T partial | O_c^T part] = Sigma_c [-gamma_c W_{c+1} ; s Gamma_c Q_c]^T  N=128, K=128
//   (a) [Sigma_{c+1} | V'^T partial] += X'_c [K_c | -K_c W_{c+1}^T]           N=192, K=64
//       with X'_c = X_c diag(d_c) and the Sigma columns preloaded with gamma_c Sigma_c
//   (b) O_c^T part += X_c (s P_c)^T                                          N=64,  K=64
// then V'^T_{c+1} = U^T_{c+1} + partial, and the O columns hold
// O_c^T = s (Sigma_c (Gamma_c Q_c)^T + X_c P_c^T) (s the output scale, folded
// into the prepared Q and P tiles).
constexpr int kMathThreads = 256;   // 8 warps: lane quarter (warp % 4) x column half (warp / 4),
                                    // then a copy warp (one polling thread) and an MMA warp
constexpr int kCopyWarpB = 8, kMmaWarp = 9, kCopyWarpM = 10, kPublishWarp = 11;

// tensor-memory columns (512 allocated)
constexpr uint32_t kTmSig = 0;    // Sigma accumulator f32 [e][k], 128 columns
constexpr uint32_t kTmV = 128;    // V'^T_{c+1} partial, 64 columns
constexpr uint32_t kTmO = 192;    // O_c^T, 64 columns
constexpr uint32_t kTmSA = 320;   // Sigma_c bf16 A operand (K = 128), 64 columns
constexpr uint32_t kTmXA = 384;   // X_c bf16 A operand (K = 64), two buffers of 32 columns
constexpr uint32_t kTmXdA = 448;  // X'_c bf16 A operand, 32 columns

struct BStage {                           // MMA operands of one step
    alignas(1024) uint8_t B1[3 * kTile];  // [K_c (two d-halves) | -K_c W_{c+1}^T], MN-major rows t
    alignas(1024) uint8_t Pc[kTile];      // P_c [r][j], K-major
    alignas(1024) uint8_t B2[4 * kTile];  // per d-half: [-gamma_c W_{c+1} ; s Gamma_c Q_c] rows, K-major
};
struct MStage {                           // what the math warps read in one step
    alignas(1024) uint8_t Ut[2 * kTile];  // U^T_{c+1} [e][i]
    float gbn[128];                       // Gamma_{c+1}, d_{c+1}
    float pad[128];
};
struct StateSmem {
    BStage bs[2];
    MStage ms[2];
    // per math warp, two staging buffers of its 32 x 32 bf16 output block
    // (rows r, 64-byte rows of e) for TMA stores
    alignas(1024) uint8_t Ost[8][2][2048];
    uint64_t fullB[2], emptyB[2], fullM[2], emptyM[2], ready_s, ready_x, mma, mma_o, drain;
    uint32_t tmem;
    int abort;
    int outc[8];  // output gate on: chunks of this walk whose block of math warp w is in memory
};

static_assert(sizeof(BStage) % 1024 == 0 && sizeof(MStage) % 1024 == 0, "stages keep the swizzle alignment");

__device__ __forceinline__ void pack_row(const float *x, uint32_t *r, int n2) {
#pragma unroll
    for (int j = 0; j < n2; ++j) r[j] = pack_bf16x2(x[2 * j], x[2 * j + 1]);
}

// One walk (sequence n, v-head h). Every thread of the CTA calls it (warps
// past the MMA warp only join the barriers); the caller has zeroed the
// shared memory once and holds 512 TMEM columns at `tmem`.
__device__ __forceinline__ void state_walk(const PrefillArgs &a, const TcWs &w, const CUtensorMap *tm_q,
                                           const CUtensorMap *tm_k, const CUtensorMap *tm_o, StateSmem &s,
                                           uint32_t tmem, int n, int h) {
    const int hk = h / a.group;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const SeqInfo si = a.seq_info[n];
    const int nc = si.num_chunks;
    const size_t sbase = (size_t(n) * a.hv + h) * kHeadDim * kHeadDim;

    __syncthreads();  // the previous walk of this CTA is over: barriers may be re-armed
    if (tid == 0) {
        s.abort = 0;
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s.fullB[b], 1);
            mbar_init(&s.emptyB[b], 1);
            mbar_init(&s.fullM[b], 1);
            mbar_init(&s.emptyM[b], kMathThreads / 32);
        }
        mbar_init(&s.ready_s, kMathThreads / 32);
        mbar_init(&s.ready_x, kMathThreads / 32);
        mbar_init(&s.mma, 1);
        mbar_init(&s.mma_o, 1);
        mbar_init(&s.drain, 1);
        for (int i = 0; i < kMathThreads / 32; ++i) s.outc[i] = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp == kCopyWarpB || warp == kCopyWarpM) {
        // ------------------------- copy threads ----------------------------
        // one thread per ring, in warps of their own: the epilogue data of a
        // step is released later than its MMA operands and must not hold back
        // the next operand loads. Both wait in blocking (suspending) waits.
        const bool opnd = warp == kCopyWarpB;
        if (lane == 0 && nc > 0) {
            if (opnd) prefetch_tensormap(tm_k);
            uint64_t *full = opnd ? s.fullB : s.fullM, *empty = opnd ? s.emptyB : s.emptyM;
            // chunks 0 .. known of this walk are written by the prepare engines
            // (their flags acquired, so their stores are visible to the copies)
            int known = -1;
            auto units_ready = [&](int upto) {  // bounded wait for chunks 0 .. upto of this walk
                const uint64_t t0 = globaltimer_ns();
                while (known < upto) {
                    if (ld_acquire_gpu(w.ready + size_t(si.first_chunk + known + 1) * a.hv + h)) {
                        ++known;
                        fence_proxy_async_global();  // the bulk copies read what the flag published
                    } else if (globaltimer_ns() - t0 > a.wait_ns) {
                        return false;
                    } else {
                        __nanosleep(256);
                    }
                }
                return true;
            };
            int last = -1;  // last step whose copies were issued
            for (int c = -1; c < nc && !s.abort; ++c) {
                const int b = (c + 1) & 1, use = (c + 1) >> 1;
                const bool cur = c >= 0, nxt = c + 1 < nc;
                if (!units_ready(min(c + 1, nc - 1)) ||
                    (use > 0 && !mbar_wait(&empty[b], (use - 1) & 1, a.wait_ns))) {
                    s.abort = 1;
                    break;
                }
                if (opnd) {
                    BStage &B = s.bs[b];
                    mbar_arrive_expect_tx(&full[b], (cur ? 5 * kTile : 0) + (nxt ? 3 * kTile : 0));
                    if (cur) {
                        const int start = si.start + kChunk * c;
                        const uint8_t *uc = w.unit + (size_t(si.first_chunk + c) * a.hv + h) * kUnitBytes;
                        for (int hf = 0; hf < 2; ++hf) {
                            tma_load_3d(B.B1 + hf * kTile, tm_k, 64 * hf, hk, start, &full[b]);
                            bulk_load(B.B2 + hf * 2 * kTile + kTile, uc + kUnitQ + hf * kTile, kTile, &full[b]);
                        }
                        bulk_load(B.Pc, uc + kUnitP, kTile, &full[b]);
                    }
                    if (nxt) {
                        const uint8_t *un = w.unit + (size_t(si.first_chunk + c + 1) * a.hv + h) * kUnitBytes;
                        for (int hf = 0; hf < 2; ++hf)
                            bulk_load(B.B2 + hf * 2 * kTile, un + kUnitW + hf * kTile, kTile, &full[b]);
                        bulk_load(B.B1 + 2 * kTile, un + kUnitG, kTile, &full[b]);
                    }
                } else {
                    MStage &M = s.ms[b];
                    mbar_arrive_expect_tx(&full[b], nxt ? 2 * kTile + 512 : 0);
                    if (nxt) {
                        const size_t un = size_t(si.first_chunk + c + 1) * a.hv + h;
                        bulk_load(M.Ut, w.unit + un * kUnitBytes + kUnitU, 2 * kTile, &full[b]);
                        bulk_load(M.gbn, w.gb + un * 128, 512, &full[b]);
                    }
                }
                last = c;
            }
            if (s.abort) {  // bounded drain of copies that may be in flight
                // the last two steps issued (one per stage); with none issued this
                // waits out its 0.1 s bound on a phase that never completes
                for (int c = last; c >= -1 && c >= last - 1; --c)
                    mbar_wait(&full[(c + 1) & 1], ((c + 1) >> 1) & 1, 100000000ull);
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------- MMA issuer ----------------------------
        if (lane == 0 && nc > 0) {
            const uint32_t id_c = idesc_bf16_f32(128, 128, false, false);
            const uint32_t id_a = idesc_bf16_f32(128, 192, false, true);
            const uint32_t id_b = idesc_bf16_f32(128, 64, false, false);
            // the two stages differ by a constant byte offset; a K step adds
            // its byte offset >> 4 to the start-address field (no carry)
            const uint64_t dB1 = sdesc_sw128(smem_u32(s.bs[0].B1), kTile, 1024);
            const uint64_t dPc = sdesc_sw128(smem_u32(s.bs[0].Pc), 16, 1024);
            const uint64_t dB2 = sdesc_sw128(smem_u32(s.bs[0].B2), 16, 1024);
            const uint64_t dstage = uint64_t(sizeof(BStage) >> 4);
            int released[2] = {0, 0};  // operand-release commits issued per stage
            for (int c = -1; c < nc && !s.abort; ++c) {
                const int b = (c + 1) & 1, use = (c + 1) >> 1;
                if (!mbar_wait_spin(&s.ready_s, (c + 1) & 1, a.wait_ns) ||
                    !mbar_wait_spin(&s.fullB[b], use & 1, a.wait_ns)) {
                    s.abort = 1;
                    break;
                }
                tc_fence_after();
                const uint64_t ob = b ? dstage : 0;
#pragma unroll
                for (int t = 0; t < 8; ++t)  // (c) Sigma_c [-gamma_c W_{c+1} ; Q_c]^T
                    mma_bf16_ts(tmem + kTmV, tmem + kTmSA + 8 * t,
                                dB2 + ob + (((t >> 2) * 2 * kTile + (t & 3) * 32) >> 4), id_c, t > 0);
                if (!mbar_wait_spin(&s.ready_x, (c + 1) & 1, a.wait_ns)) {
                    s.abort = 1;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int t = 0; t < 4; ++t)  // (a) X'_c [K_c | -K_c W_{c+1}^T]
                    mma_bf16_ts(tmem + kTmSig, tmem + kTmXdA + 8 * t, dB1 + ob + ((2048 * t) >> 4), id_a, 1);
                mma_commit(&s.mma);
                if (c >= 0) {
                    const uint32_t xa = kTmXA + 32 * ((c + 1) & 1);
#pragma unroll
                    for (int t = 0; t < 4; ++t)  // (b) O_c^T += X_c (s P_c)^T, onto the output part of (c)
                        mma_bf16_ts(tmem + kTmO, tmem + xa + 8 * t, dPc + ob + ((32 * t) >> 4), id_b, 1);
                    mma_commit(&s.mma_o);
                }
                mma_commit(&s.emptyB[b]);
                ++released[b];
            }
            // every MMA this thread issued has completed once the drain
            // commit arrives (after an abort some were issued without a
            // commit of their own): the tensor memory they write is freed
            // when the CTA ends
            mma_commit(&s.drain);
            mbar_wait(&s.drain, 0, 100000000ull);
            // the last arrivals on the operand-release barriers come from MMA
            // completion: wait for them so that nothing lands after the next
            // walk has re-armed the barriers
            for (int b = 0; b < 2; ++b)
                if (released[b] > 0) mbar_wait(&s.emptyB[b], (released[b] - 1) & 1, 100000000ull);
        }
    } else if (warp == kPublishWarp) {
        // ----------------------- output publication -------------------------
        // output gate on: chunks whose 8 blocks are all in memory are counted
        // in the workspace for the gate engines, with one gpu-scope release
        if (a.z && lane == 0 && nc > 0) {
            int published = 0;
            const uint64_t t0 = globaltimer_ns();
            while (published < nc && !*reinterpret_cast<volatile int *>(&s.abort)) {
                int m = nc;
                for (int i = 0; i < kMathThreads / 32; ++i)
                    m = min(m, *reinterpret_cast<volatile int *>(&s.outc[i]));
                if (m > published) {
                    __threadfence_block();
                    fence_proxy_async_global();
                    for (int cc = published; cc < m; ++cc)
                        red_release_add_gpu(a.done + size_t(si.first_chunk + cc) * a.hv + h, kMathThreads / 32);
                    published = m;
                } else if (globaltimer_ns() - t0 > a.wait_ns) {
                    s.abort = 1;
                    break;
                } else {
                    __nanosleep(200);
                }
            }
        }
    } else if (warp < kMathThreads / 32) {
        // --------------------------- math warps ----------------------------
        const int lq = warp & 3, ch = warp >> 2;  // TMEM lane quarter, column half
        const int e = 32 * lq + lane;             // dv index = TMEM lane
        const uint32_t lrow = uint32_t(32 * lq) << 16;
        const int last_len = si.len - kChunk * (nc - 1);  // valid length of the last chunk
        const size_t orow = size_t(a.hv) * kHeadDim;      // output row stride (elements)
        // one of the 8 math warps' blocks of chunk cc is in memory: every
        // lane's plain stores (warp barrier) and the completed store groups
        // (all but the newest when this step issued one) are ordered before
        // the release increment the output-gate engines acquire
        // `newer`: store groups committed after chunk cc's (they may stay
        // pending). Only a CTA-scope counter here: the gpu-scope release (a
        // fence of ~1 us) is the publishing warp's, off the step's chain.
        auto publish_out = [&](int cc, int newer) {
            __syncwarp();
            if (lane == 0) {
                if (newer >= 2) bulk_wait_group<2>();
                else if (newer == 1) bulk_wait_group<1>();
                else bulk_wait_group<0>();
                __threadfence_block();
                *reinterpret_cast<volatile int *>(&s.outc[warp]) = cc + 1;
            }
            __syncwarp();
        };
        bool tma_prev = false;  // the previous step committed a store group
        // state columns k = 64 ch .. 64 ch + 63 of row e: Sigma_-1 = S0^T
        {
            float v[64];
#pragma unroll
            for (int j = 0; j < 64; ++j) v[j] = a.s0 ? a.s0[sbase + size_t(64 * ch + j) * kHeadDim + e] : 0.f;
            if (nc == 0) {  // empty sequence: no steps, the final state is S0
                if (a.final_state) {
#pragma unroll
                    for (int j = 0; j < 64; ++j) a.final_state[sbase + size_t(64 * ch + j) * kHeadDim + e] = v[j];
                }
            } else {
                uint32_t r[32];
                tmem_st32(tmem + lrow + kTmSig + 64 * ch, reinterpret_cast<const uint32_t *>(v));
                tmem_st32(tmem + lrow + kTmSig + 64 * ch + 32, reinterpret_cast<const uint32_t *>(v + 32));
                pack_row(v, r, 32);
                tmem_st32(tmem + lrow + kTmSA + 32 * ch, r);
#pragma unroll
                for (int j = 0; j < 16; ++j) r[j] = 0u;
                tmem_st16(tmem + lrow + kTmXA + 16 * ch, r);  // X_-1 = 0
                tmem_st16(tmem + lrow + kTmXdA + 16 * ch, r);
                tmem_st_wait();
                tc_fence_before();
                warp_arrive(&s.ready_s);
                warp_arrive(&s.ready_x);
            }
        }
        // every branch below is warp-uniform (the tcgen05 loads and stores
        // are .sync.aligned): wait results and the abort flag are combined
        // across the warp before they steer control flow
        for (int c = -1; nc > 0 && c < nc && !__any_sync(0xffffffffu, s.abort); ++c) {
            const int b = (c + 1) & 1, use = (c + 1) >> 1;
            if (!__all_sync(0xffffffffu, mbar_wait_spin(&s.fullM[b], use & 1, a.wait_ns) &&
                                             mbar_wait_spin(&s.mma, (c + 1) & 1, a.wait_ns))) {
                s.abort = 1;
                break;
            }
            tc_fence_after();
            const MStage &M = s.ms[b];
            // O_c (from the output columns, complete once (b) is) is read
            // before the next step's (c) may overwrite those columns
            auto read_o = [&](float *o) {
                if (!__all_sync(0xffffffffu, mbar_wait_spin(&s.mma_o, c & 1, a.wait_ns))) return false;
                tc_fence_after();
                tmem_ld32(tmem + lrow + kTmO + 32 * ch, o);
                tmem_ld_wait();
                return true;
            };
            float o[32], x[32];
            bool ok = true;
            if (c + 1 < nc) {
                // phase 1: Sigma_{c+1} as the bf16 A operand of the next (c), and
                // gamma_{c+1} Sigma_{c+1} back into the accumulator for the next (a),
                // read in two halves of 32 columns. Done while the tensor pipe is
                // idle: TMEM stores slow down MMAs that run beside them. The next (c)
                // overwrites the V'^T partial and output columns, so both are read
                // before it may start; the partial only after the Sigma halves, so
                // that it is not live beside them (loaded first, it made the kernel
                // spill: 116.8 -> 113.5 us at T=4096 without the spills)
                const float gam = M.gbn[63];  // gamma_{c+1}
#pragma unroll
                for (int hq = 0; hq < 2; ++hq) {
                    float v[32];
                    tmem_ld32(tmem + lrow + kTmSig + 64 * ch + 32 * hq, v);
                    tmem_ld_wait();
                    uint32_t r[16];
                    pack_row(v, r, 16);
                    tmem_st16(tmem + lrow + kTmSA + 32 * ch + 16 * hq, r);
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] *= gam;
                    tmem_st32(tmem + lrow + kTmSig + 64 * ch + 32 * hq, reinterpret_cast<const uint32_t *>(v));
                }
                tmem_ld32(tmem + lrow + kTmV + 32 * ch, x);
                if (c >= 0) ok = read_o(o);
                tmem_ld_wait();
                tmem_st_wait();
                tc_fence_before();
                warp_arrive(&s.ready_s);
                // phase 2 (overlaps the next (c)): X_{c+1} = U^T_{c+1} + partial and
                // X' = X diag(d_{c+1})
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float u[8];
                    unpack8(*reinterpret_cast<const uint4 *>(M.Ut + sw128_offset(e, 4 * ch + q)), u);
#pragma unroll
                    for (int j = 0; j < 8; ++j) x[8 * q + j] += u[j];
                }
                uint32_t r[16];
                pack_row(x, r, 16);
                tmem_st16(tmem + lrow + kTmXA + 32 * (c & 1) + 16 * ch, r);  // X_{c+1}: buffer (c+2) & 1
                const float4 *dn = reinterpret_cast<const float4 *>(M.gbn + 64 + 32 * ch);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 d4 = dn[q];
                    x[4 * q] *= d4.x; x[4 * q + 1] *= d4.y; x[4 * q + 2] *= d4.z; x[4 * q + 3] *= d4.w;
                }
                pack_row(x, r, 16);
                tmem_st16(tmem + lrow + kTmXdA + 16 * ch, r);
                tmem_st_wait();
                tc_fence_before();
                warp_arrive(&s.ready_x);
            } else {
                float v[64];
                tmem_ld32(tmem + lrow + kTmSig + 64 * ch, v);
                tmem_ld32(tmem + lrow + kTmSig + 64 * ch + 32, v + 32);
                tmem_ld_wait();
                if (a.final_state) {
#pragma unroll
                    for (int j = 0; j < 64; ++j)
                        a.final_state[sbase + size_t(64 * ch + j) * kHeadDim + e] = v[j];
                }
                if (c >= 0) ok = read_o(o);
            }
            if (!ok) {
                s.abort = 1;
                break;
            }
            bool stored_tma = false;  // this step committed a store group
            if (c >= 0) {
                // O_c rows r = 32 ch + j, column e
                // a 2x2 transpose between lanes e and e^1 on packed pairs: each lane
                // packs rows 2m, 2m+1 of its column, swaps the word with its
                // neighbour, and one byte permute leaves even lanes with row 2m and
                // odd lanes with row 2m+1, in both columns e & ~1 and (e & ~1) + 1
                const int odd = lane & 1;
                const uint32_t sel = odd ? 0x3276u : 0x5410u;
                uint32_t pr[16];
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const uint32_t pk = pack_bf16x2(o[2 * m], o[2 * m + 1]);
                    const uint32_t pt = __shfl_xor_sync(0xffffffffu, pk, 1);
                    pr[m] = __byte_perm(pk, pt, sel);
                }
                const int lc = c == nc - 1 ? last_len : kChunk;
                const int row0 = si.start + kChunk * c + 32 * ch;  // token of the block's first row
                // the TMA store writes all 32 rows unless they run past the tensor's
                // end; rows past a sequence's end inside a packed batch take plain stores
                if (32 * ch + 32 <= lc || si.start + si.len == a.total_tokens) {
                    uint8_t *blk = s.Ost[warp][c & 1];
                    if (lane == 0) bulk_wait_group_read<1>();  // the store from two steps ago has read blk
                    __syncwarp();
#pragma unroll
                    for (int m = 0; m < 16; ++m)
                        *reinterpret_cast<uint32_t *>(blk + (2 * m + odd) * 64 + 4 * (lane >> 1)) = pr[m];
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(tm_o, 32 * lq, h, row0, blk);
                        bulk_commit_group();
                    }
                    stored_tma = true;
                } else {
                    __nv_bfloat16 *obase =
                        static_cast<__nv_bfloat16 *>(a.out) + (size_t(row0 + odd) * a.hv + h) * kHeadDim + (e & ~1);
#pragma unroll
                    for (int m = 0; m < 16; ++m)
                        if (32 * ch + 2 * m + odd < lc)
                            *reinterpret_cast<uint32_t *>(obase + size_t(2 * m) * orow) = pr[m];
                }
            }
            // output gate on: this warp's block of chunk c-2 has landed (its store
            // group, issued two steps ago, completed; waiting on the previous
            // step's group instead held every step up): count it
            if (a.z && c >= 2) publish_out(c - 2, int(stored_tma) + int(tma_prev));
            tma_prev = stored_tma;
            warp_arrive(&s.emptyM[b]);
        }
        if (a.z && !__any_sync(0xffffffffu, s.abort)) {
            if (nc >= 2) publish_out(nc - 2, 0);
            if (nc >= 1) publish_out(nc - 1, 0);
        }
        // the output stores have read their staging buffers (the next walk
        // reuses them, and the CTA may exit); their writes complete with the grid
        if (lane == 0) bulk_wait_group_read<0>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (s.abort && tid == 0) record_status(a.status, GDN_ETIMEOUT);
}

// ===========================================================================
// gate_unit: the output gate of one (chunk, v-head) tile, in place
// ===========================================================================
// y = o / sqrt(mean(o^2) + eps) * weight * silu(z) over each token's 128
// channels (the sgl-qwen3-5-moe page's output_rmsnorm_silu_gate), run by a
// prepare engine after its last unit, once the walk's 8 math warps have each
// counted their block of the chunk as written. Each warp of the engine waits
// for the count itself (bounded), acquires it, and takes rows w, w+4, ...,
// 4 channels per lane.
__device__ __forceinline__ bool gate_unit(const PrefillArgs &a, int c, int h, int etid) {
    const int lane = etid & 31, ew = etid >> 5;
    const int *cnt = a.done + size_t(c) * a.hv + h;
    bool ok = true;
    if (lane == 0) {
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_gpu(cnt) < kMathThreads / 32) {
            if (globaltimer_ns() - t0 > a.wait_ns) {
                ok = false;
                break;
            }
            __nanosleep(500);
        }
    }
    if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
    (void)ld_acquire_gpu(cnt);  // every lane acquires what the walk released
    const ChunkInfo ci = a.chunk_info[c];
    const float4 wt = reinterpret_cast<const float4 *>(a.norm_weight)[lane];
    uint2 *O = static_cast<uint2 *>(a.out);
    const uint2 *Z = static_cast<const uint2 *>(a.z);
    const size_t rstride = size_t(a.hv) * (kHeadDim / 4);  // uint2 (4 bf16) per row of the tensor
    const size_t col = size_t(h) * (kHeadDim / 4) + lane;
    // warp ew takes rows ew, ew + 4, ... (16 of the chunk's 64): all 32 loads
    // are issued before any arithmetic, so a tile costs about one round trip
    constexpr int kRows = kChunk / (kPrepThreads / 32);
    uint2 ov[kRows], zv[kRows];
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
        const int r = min(ew + 4 * j, ci.len - 1);  // rows past the chunk: recomputed, not stored
        const size_t off = size_t(ci.start + r) * rstride + col;
        ov[j] = O[off];
        zv[j] = Z[off];
    }
#pragma unroll
    for (int j4 = 0; j4 < kRows; j4 += 4) {
        float4 x[4], gz[4];
        float ss[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 o0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ov[j4 + j].x));
            const float2 o1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ov[j4 + j].y));
            const float2 z0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&zv[j4 + j].x));
            const float2 z1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&zv[j4 + j].y));
            x[j] = make_float4(o0.x, o0.y, o1.x, o1.y);
            gz[j] = make_float4(wt.x * silu_f(z0.x), wt.y * silu_f(z0.y), wt.z * silu_f(z1.x), wt.w * silu_f(z1.y));
            ss[j] = x[j].x * x[j].x + x[j].y * x[j].y + x[j].z * x[j].z + x[j].w * x[j].w;
        }
#pragma unroll
        for (int m = 16; m; m >>= 1)
#pragma unroll
            for (int j = 0; j < 4; ++j) ss[j] += __shfl_xor_sync(0xffffffffu, ss[j], m);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int r = ew + 4 * (j4 + j);
            if (r >= ci.len) continue;
            const float inv = rsqrtf(ss[j] * (1.f / kHeadDim) + a.norm_eps);
            O[size_t(ci.start + r) * rstride + col] =
                make_uint2(pack_bf16x2(x[j].x * inv * gz[j].x, x[j].y * inv * gz[j].y),
                           pack_bf16x2(x[j].z * inv * gz[j].z, x[j].w * inv * gz[j].w));
        }
    }
    return true;
}

// ===========================================================================
// k_chunk_fused_tc: prepare engines and state walks in one co-resident grid
// ===========================================================================
// One CTA per SM (cooperative launch, so every CTA is resident at once).
// CTAs 0 .. n_state-1 run state walks, one after another in sequence order;
// the others run three prepare engines each, which take the units in
// chunk-major order and never wait on anything but their own copies. A walk
// waits (bounded) on the ready flag of each unit it loads, so the walks run
// while later chunks are still being prepared.
constexpr int kFusedThreads = 384;  // three 4-warp engines, or one walk (8 math + copy + MMA warps)
constexpr int kEngines = kFusedThreads / kPrepThreads;

struct FusedArgs {
    PrefillArgs a;
    TcWs w;
    int n_state;  // CTAs that walk; the rest prepare
};

union FusedSmem {
    PrepSmem prep[kEngines];
    StateSmem state;
};
// dynamic shared memory per block is capped at 227 KiB; one more KiB is
// requested to align the base to 1024 bytes
static_assert(sizeof(FusedSmem) + 1024 <= 227 * 1024, "fused kernel shared memory");
static_assert(sizeof(PrepSmem) % 1024 == 0, "engine slices keep the swizzle alignment");

__global__ void __launch_bounds__(kFusedThreads, 1)
k_chunk_fused_tc(FusedArgs fa, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o) {
    extern __shared__ uint8_t smraw[];
    __shared__ uint32_t tmem_slot;
    FusedSmem &sm = *reinterpret_cast<FusedSmem *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const PrefillArgs &a = fa.a;
    const TcWs &w = fa.w;
    const int nch = *a.n_chunks;
    if (nch < 0) return;  // the chunk table rejected cu_seqlens (uniform over the grid)
    const int tid = threadIdx.x, warp = tid >> 5;
    if (warp == 0) {
        tmem_alloc(&tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    if (int(blockIdx.x) < fa.n_state) {
        StateSmem &s = sm.state;
        // zero once: operand regions a step does not load must hold finite
        // values (their products land in columns that are discarded)
        for (uint32_t o = tid * 16; o < sizeof(StateSmem) - 64; o += kFusedThreads * 16)
            *reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(&s) + o) = make_uint4(0, 0, 0, 0);
        const int walks = a.num_seqs * a.hv;
        for (int wk = blockIdx.x; wk < walks; wk += fa.n_state)
            state_walk(a, w, &tm_q, &tm_k, &tm_o, s, tmem, wk / a.hv, wk % a.hv);
    } else {
        const int e = warp / (kPrepThreads / 32);
        PrepSmem &s = sm.prep[e];
        if ((tid & (kPrepThreads - 1)) == 0) {
            s.abort = 0;
            mbar_init(&s.bar_load, 1);
            mbar_init(&s.bar_v, 1);
            mbar_init(&s.bar_mma, 1);
            mbar_init(&s.bar_drain, 1);
            fence_mbar_init();
        }
        __syncthreads();
        uint32_t ld_phase = 0, mma_phase = 0;
        const int units = nch * a.hv;
        const int nprep = int(gridDim.x) - fa.n_state;
        // engine e of prepare CTA i takes units k * 3 * nprep + e * nprep + i:
        // the first chunks go to engine 0 of every CTA, which starts at once;
        // engines 1 and 2 start 1.5 and 3 us later, so that the engines sharing
        // an SM stay out of step and their load waits overlap the others' work
        if (e > 0) {  // asleep, so as not to take issue slots from engine 0's first units
            const uint64_t t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < uint64_t(e) * 1500ull) __nanosleep(500);
        }
        for (int u = e * nprep + (int(blockIdx.x) - fa.n_state); u < units && !s.abort; u += kEngines * nprep)
            prep_unit(a, w, &tm_q, &tm_k, &tm_v, s, tmem + 128 * e, 1 + e, ld_phase, mma_phase, u / a.hv, u % a.hv);
        // then the output gate of the same units, in chunk order, as the walks
        // finish them (the walks never wait for this)
        if (a.z && !s.abort) {
            const int etid = tid & (kPrepThreads - 1);
            for (int u = e * nprep + (int(blockIdx.x) - fa.n_state); u < units; u += kEngines * nprep) {
                if (!gate_unit(a, u / a.hv, u % a.hv, etid)) {
                    if ((etid & 31) == 0) record_status(a.status, GDN_ETIMEOUT);
                    break;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

size_t prefill_tc_workspace(int max_chunks, int hv) {
    const size_t units = size_t(max_chunks) * hv;
    return al256(units * kUnitBytes) + al256(units * 128 * sizeof(float)) + al256(2 * units * sizeof(int));
}

int *prefill_tc_ready_flags(void *ws_data, int max_chunks, int hv) { return tc_carve(ws_data, max_chunks, hv).ready; }

// CTAs that walk: the split that minimises the larger of the two estimated
// times, with the chunks of a sequence estimated from the mean length (the
// lengths themselves are on the device). Measured at T=4096 and on packed
// batches: ~13 us until the first chunks are prepared, a walk step ~1.32 us,
// ~4 us per walk beyond its steps, a batch of units (one per engine, three
// engines on an SM) ~12 us in the steady state. Walks are dealt round-robin,
// so a walk CTA carries walks / n of them on average (at least one).
static int state_ctas(const PrefillArgs &a, int ctas) {
    const int walks = a.num_seqs * a.hv;
    const double steps = double(a.total_tokens) / (double(kChunk) * (a.num_seqs > 0 ? a.num_seqs : 1)) + 2.0;
    const double units = double(a.max_chunks) * a.hv;
    int best = 1;
    double best_t = 1e300;
    for (int n = 1; n < ctas && n <= walks; ++n) {
        const double per_cta = double(walks) / n;
        const double t_walk = 13.0 + (per_cta > 1.0 ? per_cta : 1.0) * (steps * 1.32 + 4.0);
        const double t_prep = std::ceil(units / (double(ctas - n) * kEngines)) * 12.0;
        const double t = t_walk > t_prep ? t_walk : t_prep;
        if (t < best_t) {
            best_t = t;
            best = n;
        }
    }
    return best;
}

cudaError_t launch_prefill_tc(const PrefillArgs &a, void *ws_data, cudaStream_t s) {
    const TcWs w = tc_carve(ws_data, a.max_chunks, a.hv);
    CUtensorMap tq, tk, tv, to;
    const uint64_t T = uint64_t(a.total_tokens);
    memset(&tq, 0, sizeof(tq));
    memset(&tk, 0, sizeof(tk));
    memset(&tv, 0, sizeof(tv));
    memset(&to, 0, sizeof(to));
    // with no tokens every sequence is empty: the walks only copy S0 to the
    // final state and never touch the (then unset) tensor maps
    if (T > 0 &&
        (!make_tmap_bf16_3d(&tq, a.q, kHeadDim, a.hq, T, kHeadDim * 2, uint64_t(a.hq) * kHeadDim * 2, 64, 1, 64) ||
         !make_tmap_bf16_3d(&tk, a.k, kHeadDim, a.hq, T, kHeadDim * 2, uint64_t(a.hq) * kHeadDim * 2, 64, 1, 64) ||
         !make_tmap_bf16_3d(&tv, a.v, kHeadDim, a.hv, T, kHeadDim * 2, uint64_t(a.hv) * kHeadDim * 2, 64, 1, 64) ||
         !make_tmap_bf16_3d(&to, a.out, kHeadDim, a.hv, T, kHeadDim * 2, uint64_t(a.hv) * kHeadDim * 2, 32, 1, 32,
                            false)))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(FusedSmem) + 1024;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(k_chunk_fused_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))))
        return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) || (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))) return e;
    if (sms < 2) return cudaErrorInvalidConfiguration;
    FusedArgs fa{a, w, state_ctas(a, sms)};
    void *args[] = {&fa, &tq, &tk, &tv, &to};
    {
        LaunchScope scope(GDN_K_CHUNK_FUSED_TC, s);
        e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(k_chunk_fused_tc), dim3(sms),
                                        dim3(kFusedThreads), args, smem, s);
    }
    if (e) return e;
    return cudaGetLastError();
}

}  // namespace gdn
