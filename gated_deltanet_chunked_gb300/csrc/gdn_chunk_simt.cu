// Chunk-form prefill with plain f32 SIMT arithmetic (the GDN_DT_F32 path).
//
// Follows the Lab3 GDN Prefill page, section "计算过程描述", step by step:
//   chunk_gate_cumsum + chunk_kkt_solve + chunk_recompute_w_u (k_prep_simt):
//       gc_r = sum_{j<=r} g_j (restarted per chunk),
//       M_ij = beta_i exp(gc_i - gc_j) k_i.k_j (j < i), A = (I + M)^-1,
//       W = A diag(beta gamma) K, U = A diag(beta) V
//   chunk_state_h (k_state_simt), sequential over the chunks of a sequence:
//       R = U - W S_c, S_{c+1} = gamma_l S_c + sum_i exp(gc_l - gc_i) k_i^T R_i
//   chunk_output_o (k_output_simt), parallel over chunks:
//       O_r = scale [gamma_r q_r S_c + sum_{i<=r} exp(gc_r - gc_i)(q_r.k_i) R_i]
// Every sum runs over the valid rows i < l_c only; the exponent of a decay
// ratio is formed only for entries inside the causal mask, so no Gamma^-1 is
// ever materialised. f32 arithmetic throughout keeps max|err|/max|ref| near
// 1e-6, well inside the 1e-4 criterion the decode page uses.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kPad = kHeadDim + 1;  // padded f32 row to spread banks

struct SimtWs {
    float *gc;  // [max_chunks][hv][64]
    float *A;   // [max_chunks][hv][64][64]
    float *W;   // [max_chunks][hv][64][128]
    float *U;   // [max_chunks][hv][64][128]; overwritten by R = U - W S_c
    float *H;   // [max_chunks][hv][128][128] chunk-start states S_c
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

SimtWs carve(void *base, int max_chunks, int hv) {
    char *p = static_cast<char *>(base);
    const size_t units = size_t(max_chunks) * hv;
    SimtWs w;
    w.gc = reinterpret_cast<float *>(p); p += align256(units * kChunk * 4);
    w.A = reinterpret_cast<float *>(p);  p += align256(units * kChunk * kChunk * 4);
    w.W = reinterpret_cast<float *>(p);  p += align256(units * kChunk * kHeadDim * 4);
    w.U = reinterpret_cast<float *>(p);  p += align256(units * kChunk * kHeadDim * 4);
    w.H = reinterpret_cast<float *>(p);
    return w;
}

template <typename T>
__device__ __forceinline__ float ld(const void *p, size_t i) {
    return to_f32<T>(static_cast<const T *>(p)[i]);
}

// ---------------------------------------------------------------------------
// gate prefix sum, KK^T, triangular solve, W and U for one (chunk, v-head)
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads) k_prep_simt(PrefillArgs a, SimtWs w) {
    extern __shared__ float sm[];
    float *Ks = sm;                      // [64][129]
    float *Vs = Ks + kChunk * kPad;      // [64][129]
    float *Ms = Vs + kChunk * kPad;      // [64][65]
    float *As = Ms + kChunk * (kChunk + 1);  // [64][65]
    float *gcs = As + kChunk * (kChunk + 1);  // [64]
    float *bs = gcs + kChunk;            // beta
    float *bgs = bs + kChunk;            // beta * gamma
    const int c = blockIdx.x, h = blockIdx.y, hk = h / a.group, tid = threadIdx.x;
    if (c >= *a.n_chunks) return;
    const ChunkInfo ci = a.chunk_info[c];
    const int l = ci.len;
    const size_t unit = size_t(c) * a.hv + h;

    if (tid < kChunk) bs[tid] = tid < l ? a.beta[size_t(ci.start + tid) * a.hv + h] : 0.f;
    if (tid == 0) {  // chunk_gate_cumsum: prefix sum restarted at the chunk
        float run = 0.f;
        for (int r = 0; r < kChunk; ++r) {
            if (r < l) run += a.g[size_t(ci.start + r) * a.hv + h];
            gcs[r] = run;
        }
    }
    for (int e = tid; e < kChunk * kHeadDim; e += kThreads) {
        const int i = e / kHeadDim, d = e % kHeadDim;
        const bool ok = i < l;
        Ks[i * kPad + d] = ok ? ld<T>(a.k, (size_t(ci.start + i) * a.hq + hk) * kHeadDim + d) : 0.f;
        Vs[i * kPad + d] = ok ? ld<T>(a.v, (size_t(ci.start + i) * a.hv + h) * kHeadDim + d) : 0.f;
    }
    __syncthreads();
    if (tid < kChunk) {
        w.gc[unit * kChunk + tid] = gcs[tid];
        bgs[tid] = bs[tid] * expf(gcs[tid]);
    }
    // M = StrictLower(B Gamma K K^T Gamma^-1), masked before the exponential
    for (int e = tid; e < kChunk * kChunk; e += kThreads) {
        const int i = e / kChunk, j = e % kChunk;
        float m = 0.f;
        if (j < i && i < l) {
            float dot = 0.f;
            for (int d = 0; d < kHeadDim; ++d) dot = fmaf(Ks[i * kPad + d], Ks[j * kPad + d], dot);
            m = bs[i] * expf(gcs[i] - gcs[j]) * dot;
        }
        Ms[i * (kChunk + 1) + j] = m;
    }
    __syncthreads();
    // A = (I + M)^-1 by forward substitution; column j is independent
    if (tid < kChunk) {
        const int j = tid;
        for (int i = 0; i < kChunk; ++i) {
            float x = (i == j) ? 1.f : 0.f;
            if (i > j && i < l)
                for (int m = j; m < i; ++m) x = fmaf(-Ms[i * (kChunk + 1) + m], As[m * (kChunk + 1) + j], x);
            if (j >= l) x = 0.f;
            As[i * (kChunk + 1) + j] = x;
        }
    }
    __syncthreads();
    for (int e = tid; e < kChunk * kChunk; e += kThreads)
        w.A[unit * kChunk * kChunk + e] = As[(e / kChunk) * (kChunk + 1) + e % kChunk];
    // W = A diag(beta gamma) K ; U = A diag(beta) V
    for (int e = tid; e < kChunk * kHeadDim; e += kThreads) {
        const int i = e / kHeadDim, d = e % kHeadDim;
        float wacc = 0.f, uacc = 0.f;
        for (int j = 0; j <= i && j < l; ++j) {
            const float aij = As[i * (kChunk + 1) + j];
            wacc = fmaf(aij * bgs[j], Ks[j * kPad + d], wacc);
            uacc = fmaf(aij * bs[j], Vs[j * kPad + d], uacc);
        }
        w.W[unit * kChunk * kHeadDim + e] = wacc;
        w.U[unit * kChunk * kHeadDim + e] = uacc;
    }
}

// ---------------------------------------------------------------------------
// sequential state pass for one (sequence, v-head, 32-column tile of dv)
// ---------------------------------------------------------------------------
constexpr int kTile = 32;

template <typename T>
__global__ void __launch_bounds__(kThreads) k_state_simt(PrefillArgs a, SimtWs w) {
    __shared__ float Ss[kHeadDim][kTile + 1];
    __shared__ float Rs[kChunk][kTile + 1];
    __shared__ float dec[kChunk];
    __shared__ float gl_s;
    const int n = blockIdx.x, h = blockIdx.y, col0 = blockIdx.z * kTile, hk = h / a.group;
    const int tid = threadIdx.x;
    if (*a.n_chunks < 0) return;  // the chunk table rejected cu_seqlens
    const SeqInfo si = a.seq_info[n];
    const size_t sbase = (size_t(n) * a.hv + h) * kHeadDim * kHeadDim;
    for (int e = tid; e < kHeadDim * kTile; e += kThreads) {
        const int d = e / kTile, j = e % kTile;
        Ss[d][j] = a.s0 ? a.s0[sbase + size_t(d) * kHeadDim + col0 + j] : 0.f;
    }
    __syncthreads();
    for (int cc = 0; cc < si.num_chunks; ++cc) {
        const int c = si.first_chunk + cc;
        const ChunkInfo ci = a.chunk_info[c];
        const int l = ci.len;
        const size_t unit = size_t(c) * a.hv + h;
        const float *gc = w.gc + unit * kChunk;
        if (tid < kChunk) dec[tid] = tid < l ? expf(gc[l - 1] - gc[tid]) : 0.f;
        if (tid == 0) gl_s = expf(gc[l - 1]);
        // keep the chunk-start state for the output kernel
        float *Hc = w.H + unit * kHeadDim * kHeadDim;
        for (int e = tid; e < kHeadDim * kTile; e += kThreads) {
            const int d = e / kTile, j = e % kTile;
            Hc[size_t(d) * kHeadDim + col0 + j] = Ss[d][j];
        }
        // R = U - W S  (rows i < l)
        const float *Wc = w.W + unit * kChunk * kHeadDim;
        float *Uc = w.U + unit * kChunk * kHeadDim;
        for (int e = tid; e < kChunk * kTile; e += kThreads) {
            const int i = e / kTile, j = e % kTile;
            float r = 0.f;
            if (i < l) {
                float acc = 0.f;
                for (int d = 0; d < kHeadDim; ++d) acc = fmaf(Wc[i * kHeadDim + d], Ss[d][j], acc);
                r = Uc[i * kHeadDim + col0 + j] - acc;
            }
            Rs[i][j] = r;
        }
        __syncthreads();
        for (int e = tid; e < kChunk * kTile; e += kThreads) {
            const int i = e / kTile, j = e % kTile;
            Uc[i * kHeadDim + col0 + j] = Rs[i][j];
        }
        // S <- gamma_l S + sum_i exp(gc_l - gc_i) k_i^T R_i
        for (int e = tid; e < kHeadDim * kTile; e += kThreads) {
            const int d = e / kTile, j = e % kTile;
            float acc = 0.f;
            for (int i = 0; i < l; ++i)
                acc = fmaf(dec[i] * ld<T>(a.k, (size_t(ci.start + i) * a.hq + hk) * kHeadDim + d), Rs[i][j], acc);
            Ss[d][j] = fmaf(gl_s, Ss[d][j], acc);
        }
        __syncthreads();
    }
    if (a.final_state)
        for (int e = tid; e < kHeadDim * kTile; e += kThreads) {
            const int d = e / kTile, j = e % kTile;
            a.final_state[sbase + size_t(d) * kHeadDim + col0 + j] = Ss[d][j];
        }
}

// ---------------------------------------------------------------------------
// output of one (chunk, v-head): O = scale [Gamma Q S_c + P R]
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads) k_output_simt(PrefillArgs a, SimtWs w) {
    extern __shared__ float sm[];
    float *Qs = sm;                          // [64][129]
    float *Ks = Qs + kChunk * kPad;          // [64][129]
    float *Ps = Ks + kChunk * kPad;          // [64][65]
    float *gcs = Ps + kChunk * (kChunk + 1);  // [64]
    const int c = blockIdx.x, h = blockIdx.y, hk = h / a.group, tid = threadIdx.x;
    if (c >= *a.n_chunks) return;
    const ChunkInfo ci = a.chunk_info[c];
    const int l = ci.len;
    const size_t unit = size_t(c) * a.hv + h;
    if (tid < kChunk) gcs[tid] = w.gc[unit * kChunk + tid];
    for (int e = tid; e < kChunk * kHeadDim; e += kThreads) {
        const int i = e / kHeadDim, d = e % kHeadDim;
        const bool ok = i < l;
        const size_t row = (size_t(ci.start + i) * a.hq + hk) * kHeadDim + d;
        Qs[i * kPad + d] = ok ? ld<T>(a.q, row) : 0.f;
        Ks[i * kPad + d] = ok ? ld<T>(a.k, row) : 0.f;
    }
    __syncthreads();
    // P = Gamma Lower(Q K^T) Gamma^-1 on the valid block (diagonal included)
    for (int e = tid; e < kChunk * kChunk; e += kThreads) {
        const int r = e / kChunk, i = e % kChunk;
        float p = 0.f;
        if (i <= r && r < l) {
            float dot = 0.f;
            for (int d = 0; d < kHeadDim; ++d) dot = fmaf(Qs[r * kPad + d], Ks[i * kPad + d], dot);
            p = expf(gcs[r] - gcs[i]) * dot;
        }
        Ps[r * (kChunk + 1) + i] = p;
    }
    __syncthreads();
    const float *Hc = w.H + unit * kHeadDim * kHeadDim;
    const float *Rc = w.U + unit * kChunk * kHeadDim;
    for (int e = tid; e < kChunk * kHeadDim; e += kThreads) {
        const int r = e / kHeadDim, j = e % kHeadDim;
        if (r >= l) continue;
        float inter = 0.f, intra = 0.f;
        for (int d = 0; d < kHeadDim; ++d) inter = fmaf(Qs[r * kPad + d], Hc[d * kHeadDim + j], inter);
        for (int i = 0; i <= r; ++i) intra = fmaf(Ps[r * (kChunk + 1) + i], Rc[i * kHeadDim + j], intra);
        const float o = a.scale * fmaf(expf(gcs[r]), inter, intra);
        static_cast<T *>(a.out)[(size_t(ci.start + r) * a.hv + h) * kHeadDim + j] = from_f32<T>(o);
    }
}

template <typename T>
cudaError_t launch_all(const PrefillArgs &a, void *ws, cudaStream_t s) {
    const SimtWs w = carve(ws, a.max_chunks, a.hv);
    const size_t prep_smem = (2 * kChunk * kPad + 2 * kChunk * (kChunk + 1) + 3 * kChunk) * sizeof(float);
    const size_t out_smem = (2 * kChunk * kPad + kChunk * (kChunk + 1) + kChunk) * sizeof(float);
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(k_prep_simt<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(prep_smem))))
        return e;
    if ((e = cudaFuncSetAttribute(k_output_simt<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(out_smem))))
        return e;
    if (a.max_chunks > 0) {
        LaunchScope scope(GDN_K_PREP_SIMT, s);
        k_prep_simt<T><<<dim3(a.max_chunks, a.hv), kThreads, prep_smem, s>>>(a, w);
    }
    if ((e = cudaGetLastError())) return e;
    {
        LaunchScope scope(GDN_K_STATE_SIMT, s);
        k_state_simt<T><<<dim3(a.num_seqs, a.hv, kHeadDim / kTile), kThreads, 0, s>>>(a, w);
    }
    if ((e = cudaGetLastError())) return e;
    if (a.max_chunks > 0) {
        LaunchScope scope(GDN_K_OUTPUT_SIMT, s);
        k_output_simt<T><<<dim3(a.max_chunks, a.hv), kThreads, out_smem, s>>>(a, w);
    }
    if ((e = cudaGetLastError())) return e;
    return cudaSuccess;
}

}  // namespace

size_t prefill_simt_workspace(int max_chunks, int hv) {
    const size_t units = size_t(max_chunks) * hv;
    return align256(units * kChunk * 4) + align256(units * kChunk * kChunk * 4) +
           2 * align256(units * kChunk * kHeadDim * 4) + align256(units * kHeadDim * kHeadDim * 4);
}

cudaError_t launch_prefill_simt(const PrefillArgs &a, void *ws_data, cudaStream_t s) {
    return launch_all<float>(a, ws_data, s);
}

}  // namespace gdn
