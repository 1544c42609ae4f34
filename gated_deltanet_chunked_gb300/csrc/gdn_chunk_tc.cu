// Chunk-form prefill on the tensor cores (the GDN_DT_BF16 path), sm_103a.
//
// The Lab3 GDN Prefill page, section "计算过程描述", split into two kernels:
//
// k_chunk_prepare_tc  (grid: chunk x q/k head; chunk-parallel)
//   chunk_gate_cumsum: gc_r = sum_{j<=r} g_j, restarted per chunk
//   chunk_kkt_solve:   K K^T on tcgen05 (shared by the G v-heads of the q/k
//                      head), M_ij = beta_i exp(gc_i - gc_j) (K K^T)_ij for
//                      j < i < l, A = (I + M)^-1 by forward substitution in
//                      f32 (thread j owns column j in registers)
//   writes A diag(beta) as a bf16 64x64 tile already in the 128B-swizzled
//   K-major layout the MMA reads, plus gc and beta of the chunk.
//
// k_chunk_state_output_tc  (grid: 64-column tile of dv x v-head x sequence)
//   walks the chunks of its sequence in order, with the f32 state tile
//   S [128 x 64] held in registers (thread t owns row t):
//   chunk_recompute_w_u: W = (A diag(beta) Gamma) K, U = (A diag(beta)) V
//   chunk_state_h:       V' = U - W S, S <- gamma_l S + K^T (diag(gamma_l /
//                        gamma_i) V')
//   chunk_output_o:      O = scale [Gamma (Q S) + P V'],
//                        P = Lower(Q K^T) masked and scaled by exp(gc_r - gc_i)
//   Seven tcgen05 MMAs per chunk (bf16 operands in shared memory, f32
//   accumulators in tensor memory); q/k/v tiles arrive by TMA, A and the
//   gates by bulk copy, double-buffered one chunk ahead.
//
// Shared-memory operand layouts (all 128-byte swizzled, 1024-byte aligned):
//   [rows][64 bf16] tiles; a 128-wide tile is two 64-wide halves 8 KiB apart
//   (64 rows) so one buffer serves as a K-major operand (rows = M/N) and as
//   an MN-major operand (rows = K) of different MMAs.
// Tensor-memory layout of an M=64 accumulator: row r sits in lane
// 32 (r / 16) + r % 16, so lanes 16..31 of each warp's quarter are unused.
//
// Every wait on an mbarrier is bounded; on timeout the CTA records
// GDN_ETIMEOUT in the status word, stops issuing work, waits (bounded) for
// its outstanding copies, frees its tensor memory and returns.
#include <string.h>

#include "gdn_common.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int kTcThreads = 128;
constexpr int kDvTile = 64;
constexpr uint32_t kTile64 = 64 * 128;  // bytes of a [64][64] bf16 tile
constexpr uint32_t kAPad = 68;          // f32 row pitch of the solve matrices

struct TcWs {
    uint8_t *A;   // [max_chunks][hv][8 KiB]  A diag(beta), bf16, swizzled K-major
    float *gb;    // [max_chunks][hv][128]    gc[0..63], beta[0..63]
};

__host__ __device__ inline size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

TcWs tc_carve(void *base, int max_chunks, int hv) {
    char *p = static_cast<char *>(base);
    const size_t units = size_t(max_chunks) * hv;
    TcWs w;
    w.A = reinterpret_cast<uint8_t *>(p);
    p += al256(units * kTile64);
    w.gb = reinterpret_cast<float *>(p);
    return w;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// writes 8 floats as one 16-byte chunk of bf16
__device__ __forceinline__ void st_chunk_bf16(uint8_t *dst, const float *x) {
    uint4 u;
    u.x = pack_bf16x2(x[0], x[1]);
    u.y = pack_bf16x2(x[2], x[3]);
    u.z = pack_bf16x2(x[4], x[5]);
    u.w = pack_bf16x2(x[6], x[7]);
    *reinterpret_cast<uint4 *>(dst) = u;
}

// row of an M=64 accumulator held by (warp, lane), or -1 for the unused lanes
__device__ __forceinline__ int m64_row(int warp, int lane) { return lane < 16 ? warp * 16 + lane : -1; }

// ===========================================================================
// k_chunk_prepare_tc
// ===========================================================================
struct PrepSmem {
    alignas(1024) uint8_t K[2 * kTile64];  // K tile, two 64-column halves
    float KK[64 * kAPad];                  // K K^T (f32)
    float M[64 * kAPad];                   // masked, gated strict lower part
    alignas(16) uint8_t At[kTile64];       // A diag(beta) bf16 swizzled (staging)
    float gc[64], beta[64], graw[64];
    uint64_t bar_load, bar_mma;
    uint32_t tmem;
    int abort;
};

__global__ void __launch_bounds__(kTcThreads) k_chunk_prepare_tc(PrefillArgs a, TcWs w,
                                                                  const __grid_constant__ CUtensorMap tm_k) {
    extern __shared__ uint8_t smraw[];
    PrepSmem &s = *reinterpret_cast<PrepSmem *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const int c = blockIdx.x, hk = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (c >= *a.n_chunks) return;  // also covers a rejected chunk table (-1)
    const ChunkInfo ci = a.chunk_info[c];
    const int l = ci.len;

    if (tid == 0) {
        s.abort = 0;
        mbar_init(&s.bar_load, 1);
        mbar_init(&s.bar_mma, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&s.bar_load, 2 * kTile64);
        tma_load_3d(s.K, &tm_k, 0, hk, ci.start, &s.bar_load);
        tma_load_3d(s.K + kTile64, &tm_k, 64, hk, ci.start, &s.bar_load);
    }
    if (warp == 0) {
        tmem_alloc(&s.tmem, 64);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem;

    // K K^T (M=64, N=64, K=128): both operands K-major from the K tile
    if (tid == 0) {
        if (mbar_wait(&s.bar_load, 0)) {
            tc_fence_after();
            const uint32_t id = idesc_bf16_f32(64, 64, false, false);
            const uint32_t kb = smem_u32(s.K);
#pragma unroll
            for (int st = 0; st < 8; ++st) {
                const uint32_t off = (st >> 2) * kTile64 + (st & 3) * 32;
                mma_bf16(tmem, sdesc_sw128(kb + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024), id, st > 0);
            }
            mma_commit(&s.bar_mma);
        } else {
            s.abort = 1;
        }
    }
    __syncthreads();
    bool ok = !s.abort;
    if (ok && !mbar_wait(&s.bar_mma, 0)) s.abort = 1;
    __syncthreads();
    ok = !s.abort;
    if (ok) {
        tc_fence_after();
        const int r = m64_row(warp, lane);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float v[16];
            tmem_ld16(tmem_addr(tmem, 32 * warp, 16 * j), v);
            tmem_ld_wait();
            if (r >= 0)
#pragma unroll
                for (int e = 0; e < 16; ++e) s.KK[r * kAPad + 16 * j + e] = v[e];
        }
    }
    tc_fence_before();
    __syncthreads();

    for (int hh = 0; ok && hh < a.group; ++hh) {
        const int h = hk * a.group + hh;
        const size_t unit = size_t(c) * a.hv + h;
        // chunk_gate_cumsum (left-to-right f32 sum, restarted at the chunk)
        if (tid < 64) {
            const bool in = tid < l;
            s.graw[tid] = in ? a.g[size_t(ci.start + tid) * a.hv + h] : 0.f;
            s.beta[tid] = in ? a.beta[size_t(ci.start + tid) * a.hv + h] : 0.f;
        }
        __syncthreads();
        if (tid < 64) {
            float run = 0.f;
            for (int j = 0; j <= tid; ++j) run += s.graw[j];
            s.gc[tid] = run;
            w.gb[unit * 128 + tid] = run;
            w.gb[unit * 128 + 64 + tid] = s.beta[tid];
        }
        __syncthreads();
        // M = StrictLower(B Gamma K K^T Gamma^-1) on the valid block
        for (int e = tid; e < 64 * 64; e += kTcThreads) {
            const int i = e >> 6, j = e & 63;
            float m = 0.f;
            if (j < i && i < l) m = s.beta[i] * __expf(s.gc[i] - s.gc[j]) * s.KK[i * kAPad + j];
            s.M[i * kAPad + j] = m;
        }
        __syncthreads();
        // A = (I + M)^-1: thread j solves column j, keeping it in registers;
        // rows i < j of column j are zero (A is unit lower triangular)
        if (tid < 64) {
            const int j = tid;
            float col[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                float x0 = (i == j) ? 1.f : 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
                const float *Mi = s.M + i * kAPad;
#pragma unroll
                for (int m = 0; m + 3 < i; m += 4) {
                    const float4 mm = *reinterpret_cast<const float4 *>(Mi + m);
                    x0 = fmaf(-mm.x, col[m], x0);
                    x1 = fmaf(-mm.y, col[m + 1], x1);
                    x2 = fmaf(-mm.z, col[m + 2], x2);
                    x3 = fmaf(-mm.w, col[m + 3], x3);
                }
#pragma unroll
                for (int m = i & ~3; m < i; ++m) x0 = fmaf(-Mi[m], col[m], x0);
                col[i] = (j < l && i < l) ? (x0 + x1) + (x2 + x3) : 0.f;
            }
            // A diag(beta): column j scaled by beta_j, into the swizzled tile
            const float bj = s.beta[j];
            const int chunk = j >> 3, sub = j & 7;
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                const __nv_bfloat16 v = __float2bfloat16_rn(col[i] * bj);
                *reinterpret_cast<__nv_bfloat16 *>(s.At + sw128_offset(i, chunk) + 2 * sub) = v;
            }
        }
        __syncthreads();
        uint4 *dst = reinterpret_cast<uint4 *>(w.A + unit * kTile64);
        const uint4 *src = reinterpret_cast<const uint4 *>(s.At);
        for (int e = tid; e < int(kTile64 / 16); e += kTcThreads) dst[e] = src[e];
        __syncthreads();
    }
    if (s.abort && tid == 0) {
        record_status(a.status, GDN_ETIMEOUT);
        mbar_wait(&s.bar_load, 0, 100000000ull);  // bounded drain of the K-tile copy
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 64);
}

// ===========================================================================
// k_chunk_state_output_tc
// ===========================================================================
struct Stage {
    alignas(1024) uint8_t Q[2 * kTile64];
    uint8_t K[2 * kTile64];
    uint8_t V[kTile64];
    uint8_t A[kTile64];
    float gb[128];
};

struct StateSmem {
    Stage st[2];
    alignas(1024) uint8_t Ag[kTile64];    // A diag(beta gamma), K-major [i][j]
    uint8_t W[2 * kTile64];               // W bf16, K-major [i][d]
    uint8_t P[kTile64];                   // masked decayed Q K^T, K-major [r][i]
    uint8_t S[2 * kTile64];               // state bf16 [d][e] (128 rows), MN-major B
    uint8_t Vp[kTile64];                  // V' bf16 [i][e], MN-major B
    uint8_t Vd[kTile64];                  // diag(gamma_l/gamma_i) V' bf16 [i][e]
    uint64_t bar_load[2], bar_mma;
    uint32_t tmem;
    int abort;
};

// tensor-memory columns of the accumulators (512 allocated)
constexpr uint32_t kColW = 0, kColU = 128, kColP = 192, kColWS = 256, kColQS = 320, kColPV = 384, kColKV = 448;
constexpr uint32_t kStageBytes = 2 * kTile64 + 2 * kTile64 + kTile64 + kTile64 + 512;

struct StateArgs {
    PrefillArgs a;
    TcWs w;
};

__device__ __forceinline__ void issue_stage_loads(StateSmem &s, int stage, const PrefillArgs &a, const TcWs &w,
                                                  const CUtensorMap *tq, const CUtensorMap *tk,
                                                  const CUtensorMap *tv, int c, int h, int hk, int e0) {
    const ChunkInfo ci = a.chunk_info[c];
    Stage &st = s.st[stage];
    uint64_t *bar = &s.bar_load[stage];
    const size_t unit = size_t(c) * a.hv + h;
    mbar_arrive_expect_tx(bar, kStageBytes);
    tma_load_3d(st.Q, tq, 0, hk, ci.start, bar);
    tma_load_3d(st.Q + kTile64, tq, 64, hk, ci.start, bar);
    tma_load_3d(st.K, tk, 0, hk, ci.start, bar);
    tma_load_3d(st.K + kTile64, tk, 64, hk, ci.start, bar);
    tma_load_3d(st.V, tv, e0, h, ci.start, bar);
    bulk_load(st.A, w.A + unit * kTile64, kTile64, bar);
    bulk_load(st.gb, w.gb + unit * 128, 512, bar);
}

__global__ void __launch_bounds__(kTcThreads, 1)
k_chunk_state_output_tc(StateArgs sa, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v) {
    extern __shared__ uint8_t smraw[];
    StateSmem &s = *reinterpret_cast<StateSmem *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const PrefillArgs &a = sa.a;
    const TcWs &w = sa.w;
    const int tile = blockIdx.x & 1, n = blockIdx.x >> 1, h = blockIdx.y;
    const int hk = h / a.group, e0 = tile * kDvTile;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (*a.n_chunks < 0) return;  // the chunk table rejected cu_seqlens
    const SeqInfo si = a.seq_info[n];
    const size_t sbase = (size_t(n) * a.hv + h) * kHeadDim * kHeadDim;

    if (tid == 0) {
        s.abort = 0;
        mbar_init(&s.bar_load[0], 1);
        mbar_init(&s.bar_load[1], 1);
        mbar_init(&s.bar_mma, 1);
        fence_mbar_init();
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        if (si.num_chunks > 0) issue_stage_loads(s, 0, a, w, &tm_q, &tm_k, &tm_v, si.first_chunk, h, hk, e0);
    }
    if (warp == 0) {
        tmem_alloc(&s.tmem, 512);
        tmem_relinquish();
    }
    // initial state row d = tid (64 columns of this tile) in registers
    float Sr[64];
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
    // bf16 copy of the state as the MN-major B operand: row d = tid of a
    // [128][64] tile of 128-byte rows
    auto write_state = [&]() {
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) st_chunk_bf16(s.S + sw128_offset(tid, ch), Sr + 8 * ch);
    };
    write_state();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem;
    uint32_t mma_phase = 0;
    const int r64 = m64_row(warp, lane);

    const uint32_t id_w = idesc_bf16_f32(64, 128, false, true);   // A K-major, B MN-major
    const uint32_t id_u = idesc_bf16_f32(64, 64, false, true);
    const uint32_t id_qk = idesc_bf16_f32(64, 64, false, false);  // both K-major
    const uint32_t id_kv = idesc_bf16_f32(128, 64, true, true);   // both MN-major

    for (int cc = 0; cc < si.num_chunks && !s.abort; ++cc) {
        const int c = si.first_chunk + cc;
        const int stg = cc & 1;
        Stage &st = s.st[stg];
        const ChunkInfo ci = a.chunk_info[c];
        const int l = ci.len;
        // prefetch the next chunk into the other stage (its previous user,
        // chunk cc-1, has finished every MMA that read it)
        if (tid == 0 && cc + 1 < si.num_chunks)
            issue_stage_loads(s, stg ^ 1, a, w, &tm_q, &tm_k, &tm_v, c + 1, h, hk, e0);
        if (!mbar_wait(&s.bar_load[stg], (cc >> 1) & 1)) s.abort = 1;
        __syncthreads();
        if (s.abort) break;

        // A diag(beta gamma) = A diag(beta) scaled by gamma_j per column
        for (int e = tid; e < 64 * 8; e += kTcThreads) {
            const int i = e >> 3, ch = e & 7;
            const uint32_t off = sw128_offset(i, ch);
            const uint4 u = *reinterpret_cast<const uint4 *>(st.A + off);
            const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&u);
            float x[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) x[q] = __bfloat162float(b[q]) * __expf(st.gb[8 * ch + q]);
            st_chunk_bf16(s.Ag + off, x);
        }
        fence_proxy_async_smem();
        __syncthreads();

        // MMA group 1: W, U, Q K^T, Q S
        if (tid == 0) {
            tc_fence_after();
            const uint32_t q = smem_u32(st.Q), k = smem_u32(st.K), v = smem_u32(st.V), A = smem_u32(st.A);
            const uint32_t ag = smem_u32(s.Ag), S = smem_u32(s.S);
#pragma unroll
            for (int t = 0; t < 4; ++t)  // W = Ag K : K over chunk positions
                mma_bf16(tmem + kColW, sdesc_sw128(ag + 32 * t, 16, 1024), sdesc_sw128(k + 2048 * t, kTile64, 1024),
                         id_w, t > 0);
#pragma unroll
            for (int t = 0; t < 4; ++t)  // U = A V
                mma_bf16(tmem + kColU, sdesc_sw128(A + 32 * t, 16, 1024), sdesc_sw128(v + 2048 * t, kTile64, 1024),
                         id_u, t > 0);
#pragma unroll
            for (int t = 0; t < 8; ++t) {  // Q K^T and Q S : K over d
                const uint32_t off = (t >> 2) * kTile64 + (t & 3) * 32;
                mma_bf16(tmem + kColP, sdesc_sw128(q + off, 16, 1024), sdesc_sw128(k + off, 16, 1024), id_qk, t > 0);
                mma_bf16(tmem + kColQS, sdesc_sw128(q + off, 16, 1024), sdesc_sw128(S + 2048 * t, kTile64, 1024),
                         id_u, t > 0);
            }
            mma_commit(&s.bar_mma);
        }
        if (!mbar_wait(&s.bar_mma, mma_phase)) s.abort = 1;
        mma_phase ^= 1;
        tc_fence_after();

        // epilogue 1: W -> bf16 operand; P = masked, decayed Q K^T -> bf16
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float v[16];
            tmem_ld16(tmem_addr(tmem, 32 * warp, kColW + 16 * j), v);
            tmem_ld_wait();
            if (r64 >= 0) {
                uint8_t *half = s.W + (j >> 2) * kTile64;
                st_chunk_bf16(half + sw128_offset(r64, (2 * j) & 7), v);
                st_chunk_bf16(half + sw128_offset(r64, (2 * j + 1) & 7), v + 8);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float v[16];
            tmem_ld16(tmem_addr(tmem, 32 * warp, kColP + 16 * j), v);
            tmem_ld_wait();
            if (r64 >= 0) {
                const float gr = st.gb[r64];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int i = 16 * j + e;
                    v[e] = (i <= r64 && r64 < l) ? __expf(gr - st.gb[i]) * v[e] : 0.f;
                }
                st_chunk_bf16(s.P + sw128_offset(r64, 2 * j), v);
                st_chunk_bf16(s.P + sw128_offset(r64, 2 * j + 1), v + 8);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (s.abort) break;

        // MMA group 2: W S
        if (tid == 0) {
            tc_fence_after();
            const uint32_t Wb = smem_u32(s.W), S = smem_u32(s.S);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const uint32_t off = (t >> 2) * kTile64 + (t & 3) * 32;
                mma_bf16(tmem + kColWS, sdesc_sw128(Wb + off, 16, 1024), sdesc_sw128(S + 2048 * t, kTile64, 1024),
                         id_u, t > 0);
            }
            mma_commit(&s.bar_mma);
        }
        if (!mbar_wait(&s.bar_mma, mma_phase)) s.abort = 1;
        mma_phase ^= 1;
        tc_fence_after();

        // epilogue 2: V' = U - W S ; Vd = diag(gamma_l / gamma_i) V'
        {
            const float gl = st.gb[l - 1];
            const float di = (r64 >= 0 && r64 < l) ? __expf(gl - st.gb[r64]) : 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float u[16], ws[16];
                tmem_ld16(tmem_addr(tmem, 32 * warp, kColU + 16 * j), u);
                tmem_ld16(tmem_addr(tmem, 32 * warp, kColWS + 16 * j), ws);
                tmem_ld_wait();
                if (r64 >= 0) {
                    float vp[16], vd[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        vp[e] = u[e] - ws[e];
                        vd[e] = di * vp[e];
                    }
                    st_chunk_bf16(s.Vp + sw128_offset(r64, 2 * j), vp);
                    st_chunk_bf16(s.Vp + sw128_offset(r64, 2 * j + 1), vp + 8);
                    st_chunk_bf16(s.Vd + sw128_offset(r64, 2 * j), vd);
                    st_chunk_bf16(s.Vd + sw128_offset(r64, 2 * j + 1), vd + 8);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (s.abort) break;

        // MMA group 3: P V' and K^T Vd
        if (tid == 0) {
            tc_fence_after();
            const uint32_t P = smem_u32(s.P), vp = smem_u32(s.Vp), vd = smem_u32(s.Vd), k = smem_u32(st.K);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                mma_bf16(tmem + kColPV, sdesc_sw128(P + 32 * t, 16, 1024), sdesc_sw128(vp + 2048 * t, kTile64, 1024),
                         id_u, t > 0);
                mma_bf16(tmem + kColKV, sdesc_sw128(k + 2048 * t, kTile64, 1024),
                         sdesc_sw128(vd + 2048 * t, kTile64, 1024), id_kv, t > 0);
            }
            mma_commit(&s.bar_mma);
        }
        if (!mbar_wait(&s.bar_mma, mma_phase)) s.abort = 1;
        mma_phase ^= 1;
        tc_fence_after();

        // epilogue 3: state update (row d = tid), output rows r < l
        {
            const float gl = __expf(st.gb[l - 1]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float kv[16];
                tmem_ld16(tmem_addr(tmem, 32 * warp, kColKV + 16 * j), kv);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) Sr[16 * j + e] = fmaf(gl, Sr[16 * j + e], kv[e]);
            }
            const float gr = r64 >= 0 ? __expf(st.gb[r64]) : 0.f;
            __nv_bfloat16 *orow =
                r64 >= 0 ? static_cast<__nv_bfloat16 *>(a.out) + (size_t(ci.start + r64) * a.hv + h) * kHeadDim + e0
                         : nullptr;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float qs[16], pv[16];
                tmem_ld16(tmem_addr(tmem, 32 * warp, kColQS + 16 * j), qs);
                tmem_ld16(tmem_addr(tmem, 32 * warp, kColPV + 16 * j), pv);
                tmem_ld_wait();
                if (r64 >= 0 && r64 < l) {
                    float o[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) o[e] = a.scale * fmaf(gr, qs[e], pv[e]);
                    uint4 u0, u1;
                    u0.x = pack_bf16x2(o[0], o[1]);   u0.y = pack_bf16x2(o[2], o[3]);
                    u0.z = pack_bf16x2(o[4], o[5]);   u0.w = pack_bf16x2(o[6], o[7]);
                    u1.x = pack_bf16x2(o[8], o[9]);   u1.y = pack_bf16x2(o[10], o[11]);
                    u1.z = pack_bf16x2(o[12], o[13]); u1.w = pack_bf16x2(o[14], o[15]);
                    reinterpret_cast<uint4 *>(orow + 16 * j)[0] = u0;
                    reinterpret_cast<uint4 *>(orow + 16 * j)[1] = u1;
                }
            }
        }
        tc_fence_before();
        __syncthreads();  // every thread is done reading S (bf16) and TMEM
        write_state();
        fence_proxy_async_smem();
        __syncthreads();
    }

    if (s.abort) {
        if (tid == 0) {
            record_status(a.status, GDN_ETIMEOUT);
            // drain loads that may still be in flight into either stage
            mbar_wait(&s.bar_load[0], 0, 100000000ull);
            mbar_wait(&s.bar_load[1], 0, 100000000ull);
        }
        __syncthreads();
    } else if (a.final_state) {
        float4 *dst = reinterpret_cast<float4 *>(a.final_state + sbase + size_t(tid) * kHeadDim + e0);
#pragma unroll
        for (int q = 0; q < 16; ++q) dst[q] = make_float4(Sr[4 * q], Sr[4 * q + 1], Sr[4 * q + 2], Sr[4 * q + 3]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

size_t prefill_tc_workspace(int max_chunks, int hv) {
    const size_t units = size_t(max_chunks) * hv;
    return al256(units * kTile64) + al256(units * 128 * sizeof(float));
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
        k_chunk_prepare_tc<<<dim3(a.max_chunks, a.hq), kTcThreads, prep_smem, s>>>(a, w, tk);
    }
    if ((e = cudaGetLastError())) return e;
    {
        LaunchScope scope(GDN_K_STATE_OUTPUT_TC, s);
        StateArgs sa{a, w};
        k_chunk_state_output_tc<<<dim3(2 * a.num_seqs, a.hv), kTcThreads, state_smem, s>>>(sa, tq, tk, tv);
    }
    return cudaGetLastError();
}

}  // namespace gdn
