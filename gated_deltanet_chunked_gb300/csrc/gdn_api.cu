// C ABI of libgdn.so: argument checks, workspace carving and dispatch.
//
// Every entry point validates all of its arguments before the first launch
// and returns a gdn_status; nothing is enqueued on failure. There is one
// compute path per io dtype (f32: SIMT kernels; bf16: tensor-core kernels)
// and no host-side fallback of any kind.
#include <atomic>
#include <mutex>

#include "gdn_common.cuh"
#include "tma_host.cuh"

namespace gdn {
namespace {

__device__ int g_status_word;  // device status word (first device-side error)

constexpr unsigned long long kDefaultWaitNs = 2000000000ull;
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};  // limit of the prefill kernels' bounded waits

constexpr int kMaxDevices = 64;
int *g_status_ptr[kMaxDevices];
unsigned long long g_status_ctx[kMaxDevices];  // context id the cached address belongs to
std::mutex g_status_mu;

// Device address of the status word for the current device, looked up once
// per device and context (cudaGetSymbolAddress needs that device current;
// the context id catches a cudaDeviceReset, after which the module and its
// variables are loaded anew).
int *status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_status_mu);
    unsigned long long ctx = 0;
    const bool have_ctx = current_context_id(&ctx);
    if (!g_status_ptr[dev] || !have_ctx || g_status_ctx[dev] != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int *>(p);
        // the symbol lookup made the context current if it was not yet
        g_status_ctx[dev] = (have_ctx || current_context_id(&ctx)) ? ctx : 0;
    }
    return g_status_ptr[dev];
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Checks shared by prefill and decode. Returns GDN_OK or the error code.
// `allowed_flags`: the gdn_problem.flags bits the entry point accepts.
int check_common(const gdn_problem *p, uint32_t allowed_flags = 0) {
    if (!p) return GDN_EINVAL;
    if (p->hq <= 0 || p->hv <= 0 || p->dk <= 0 || p->dv <= 0) return GDN_EINVAL;
    if (p->hv % p->hq != 0) return GDN_EINVAL;
    if (p->io_dtype != GDN_DT_F32 && p->io_dtype != GDN_DT_BF16) return GDN_EINVAL;
    if (p->num_seqs < 0 || p->total_tokens < 0) return GDN_EINVAL;
    if (p->dk != kHeadDim || p->dv != kHeadDim) return GDN_EUNSUPPORTED;
    if (p->flags & ~allowed_flags) return GDN_EUNSUPPORTED;
    return GDN_OK;
}

int check_prefill_shape(const gdn_problem *p, bool packed) {
    int st = check_common(p);
    if (st) return st;
    if (p->num_seqs < 1) return GDN_EINVAL;
    if (!packed) {
        if (p->batch < 1 || p->seqlen < 0 || p->num_seqs != p->batch) return GDN_EINVAL;
        if (int64_t(p->batch) * p->seqlen != p->total_tokens) return GDN_EINVAL;
    }
    // token-row products must stay addressable with 64-bit offsets and the
    // chunk count must fit the int32 chunk table
    if (int64_t(p->total_tokens) / kChunk + p->num_seqs > (int64_t(1) << 30)) return GDN_EINVAL;
    // the per-(chunk, head) flags and counters are indexed with int
    if ((int64_t(p->total_tokens) / kChunk + p->num_seqs) * p->hv * 2 >= (int64_t(1) << 31)) return GDN_EINVAL;
    return GDN_OK;
}

int max_chunks_of(const gdn_problem *p) { return p->total_tokens / kChunk + p->num_seqs; }

// Workspace layout: [n_chunks | seq_info | chunk_info | kernel data].
struct WsLayout {
    size_t seq_off, chunk_off, data_off, data_bytes, total;
};

WsLayout ws_layout(const gdn_problem *p) {
    WsLayout l;
    const int mc = max_chunks_of(p);
    l.seq_off = 256;
    l.chunk_off = l.seq_off + align256(sizeof(SeqInfo) * size_t(p->num_seqs));
    l.data_off = l.chunk_off + align256(sizeof(ChunkInfo) * size_t(mc));
    l.data_bytes = p->io_dtype == GDN_DT_BF16 ? prefill_tc_workspace(mc, p->hv) : prefill_simt_workspace(mc, p->hv);
    l.total = l.data_off + l.data_bytes;
    return l;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ECUDA; }

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

int gdn_version(void) { return 102; }

const char *gdn_status_string(int status) {
    switch (status) {
        case GDN_OK: return "GDN_OK";
        case GDN_EINVAL: return "GDN_EINVAL: invalid argument (pointer, shape, size or alignment)";
        case GDN_EUNSUPPORTED: return "GDN_EUNSUPPORTED: valid but unsupported (dk/dv must be 128, flags 0)";
        case GDN_ECUDA: return "GDN_ECUDA: a CUDA runtime call or kernel launch failed";
        case GDN_ETIMEOUT: return "GDN_ETIMEOUT: a bounded device-side wait gave up";
        case GDN_EDEVICE_INPUT: return "GDN_EDEVICE_INPUT: device-side input check failed (cu_seqlens or slot index)";
        case GDN_ETOOBIG:
            return "GDN_ETOOBIG: workspace need exceeds the fixed no-alloc scratch (GDN_NOALLOC_SCRATCH_BYTES)";
        default: return "unknown gdn_status";
    }
}

size_t gdn_chunk_fwd_workspace_size(const gdn_problem *p) {
    // the size depends only on total_tokens, num_seqs and hv, so the packed
    // checks (a superset of nothing layout-specific) are the right ones here
    if (check_prefill_shape(p, /*packed=*/true) != GDN_OK) return 0;
    return ws_layout(p).total;
}

}  // extern "C"

namespace gdn {
namespace {

// The output gate of gdn_chunk_fwd_gated (null z: none).
struct OutGate {
    const void *z;
    const float *weight;
    float eps;
};

int chunk_fwd(const gdn_problem *p, const void *q, const void *k, const void *v, const float *g, const float *beta,
              float scale, const float *initial_state, const int32_t *cu_seqlens, const OutGate &gate, void *out,
              float *final_state, void *workspace, size_t workspace_bytes, void *stream) {
    const bool packed = cu_seqlens != nullptr;
    int st = check_prefill_shape(p, packed);
    if (st) return st;
    if (p->total_tokens > 0) {
        if (!q || !k || !v || !g || !beta || !out) return GDN_EINVAL;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) || !aligned16(out))
            return GDN_EINVAL;
    }
    if ((initial_state && !aligned16(initial_state)) || (final_state && !aligned16(final_state)) ||
        (cu_seqlens && !aligned16(cu_seqlens)))
        return GDN_EINVAL;
    const WsLayout L = ws_layout(p);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < L.total)
        return GDN_EINVAL;
    int *status = status_ptr();
    if (!status) return GDN_ECUDA;

    char *ws = static_cast<char *>(workspace);
    PrefillArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
    a.s0 = initial_state; a.final_state = final_state; a.out = out; a.scale = scale;
    a.hq = p->hq; a.hv = p->hv; a.group = p->hv / p->hq;
    a.num_seqs = p->num_seqs; a.total_tokens = p->total_tokens;
    a.dense_batch = packed ? 0 : p->batch;
    a.dense_seqlen = packed ? 0 : p->seqlen;
    a.cu = cu_seqlens;
    a.max_chunks = max_chunks_of(p);
    a.n_chunks = reinterpret_cast<int *>(ws);
    a.seq_info = reinterpret_cast<SeqInfo *>(ws + L.seq_off);
    a.chunk_info = reinterpret_cast<ChunkInfo *>(ws + L.chunk_off);
    a.status = status;
    a.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    if (p->io_dtype == GDN_DT_BF16) {
        a.ready = prefill_tc_ready_flags(ws + L.data_off, a.max_chunks, a.hv);
        a.done = a.ready + size_t(a.max_chunks) * a.hv;  // output counters follow the ready flags
        a.ready_count = 2 * a.max_chunks * a.hv;
    }
    if (gate.z) {
        if (p->total_tokens > 0 && (!aligned16(gate.z) || !gate.weight || !aligned16(gate.weight))) return GDN_EINVAL;
        if (!(gate.eps >= 0.f)) return GDN_EINVAL;
        a.z = gate.z;
        a.norm_weight = gate.weight;
        a.norm_eps = gate.eps;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = cuda_status(launch_chunk_table(a, s)))) return st;
    if (p->io_dtype == GDN_DT_BF16) return cuda_status(launch_prefill_tc(a, ws + L.data_off, s));
    if ((st = cuda_status(launch_prefill_simt(a, ws + L.data_off, s)))) return st;
    if (!gate.z) return GDN_OK;
    return cuda_status(launch_gated_rmsnorm(out, gate.z, gate.weight, gate.eps, out,
                                            (long long)p->total_tokens * p->hv, p->io_dtype, status, s));
}

}  // namespace
}  // namespace gdn

extern "C" {

int gdn_chunk_fwd(const gdn_problem *p, const void *q, const void *k, const void *v, const float *g,
                  const float *beta, float scale, const float *initial_state, const int32_t *cu_seqlens,
                  void *out, float *final_state, void *workspace, size_t workspace_bytes, void *stream) {
    return gdn::chunk_fwd(p, q, k, v, g, beta, scale, initial_state, cu_seqlens, gdn::OutGate{nullptr, nullptr, 0.f},
                          out, final_state, workspace, workspace_bytes, stream);
}

int gdn_chunk_fwd_gated(const gdn_problem *p, const void *q, const void *k, const void *v, const float *g,
                        const float *beta, float scale, const float *initial_state, const int32_t *cu_seqlens,
                        const void *z, const float *norm_weight, float norm_eps, void *out, float *final_state,
                        void *workspace, size_t workspace_bytes, void *stream) {
    if (!z) return GDN_EINVAL;
    return gdn::chunk_fwd(p, q, k, v, g, beta, scale, initial_state, cu_seqlens,
                          gdn::OutGate{z, norm_weight, norm_eps}, out, final_state, workspace, workspace_bytes,
                          stream);
}

constexpr uint32_t kDecodeFlags = GDN_FLAG_BETA_BF16 | GDN_FLAG_STATE_BF16;

int gdn_recurrent_step(const gdn_problem *p, const void *q, const void *k, const void *v, const float *g,
                       const float *beta, float scale, void *state, const int32_t *state_indices, void *out,
                       void *stream) {
    int st = check_common(p, kDecodeFlags);
    if (st) return st;
    if (p->total_tokens != p->num_seqs) return GDN_EINVAL;
    if (p->num_state_slots < 0 || (!state_indices && p->num_state_slots < p->num_seqs)) return GDN_EINVAL;
    if (p->num_seqs > 0) {
        if (!q || !k || !v || !g || !beta || !out || !state) return GDN_EINVAL;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) ||
            !aligned16(out) || !aligned16(state) || (state_indices && !aligned16(state_indices)))
            return GDN_EINVAL;
    }
    if (int64_t(p->num_seqs) * p->hv >= (int64_t(1) << 31)) return GDN_EINVAL;
    int *status = status_ptr();
    if (!status) return GDN_ECUDA;
    return cuda_status(launch_recurrent_step(*p, q, k, v, g, beta, nullptr, scale, state, state_indices, out,
                                             status, static_cast<cudaStream_t>(stream)));
}

int gdn_recurrent_step_gated(const gdn_problem *p, const void *q, const void *k, const void *v, const float *a,
                             const float *b, const float *A_log, const float *dt_bias, float scale, void *state,
                             const int32_t *state_indices, const void *z, const float *norm_weight,
                             float norm_eps, void *out, void *stream) {
    int st = check_common(p, kDecodeFlags);
    if (st) return st;
    if (p->total_tokens != p->num_seqs) return GDN_EINVAL;
    if (p->num_state_slots < 0 || (!state_indices && p->num_state_slots < p->num_seqs)) return GDN_EINVAL;
    if (p->num_seqs > 0) {
        if (!q || !k || !v || !a || !b || !A_log || !dt_bias || !out || !state) return GDN_EINVAL;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(state) ||
            (state_indices && !aligned16(state_indices)))
            return GDN_EINVAL;
        if (!aligned4(a) || !aligned4(b) || !aligned4(A_log) || !aligned4(dt_bias)) return GDN_EINVAL;
        if (z && (!norm_weight || !aligned16(z) || !aligned16(norm_weight))) return GDN_EINVAL;
    }
    if (z && !(norm_eps >= 0.f)) return GDN_EINVAL;
    if (int64_t(p->num_seqs) * p->hv >= (int64_t(1) << 31)) return GDN_EINVAL;
    int *status = status_ptr();
    if (!status) return GDN_ECUDA;
    const DecodeFront front{a, b, A_log, dt_bias, z, z ? norm_weight : nullptr, norm_eps};
    return cuda_status(launch_recurrent_step(*p, q, k, v, nullptr, nullptr, &front, scale, state, state_indices,
                                             out, status, static_cast<cudaStream_t>(stream)));
}

int gdn_gated_rmsnorm(const gdn_problem *p, const void *o, const void *z, const float *weight, float eps, void *y,
                      void *stream) {
    if (!p || p->hv <= 0 || p->total_tokens < 0) return GDN_EINVAL;
    if (p->io_dtype != GDN_DT_F32 && p->io_dtype != GDN_DT_BF16) return GDN_EINVAL;
    if (p->dv != kHeadDim) return p->dv > 0 ? GDN_EUNSUPPORTED : GDN_EINVAL;
    if (!(eps >= 0.f)) return GDN_EINVAL;
    const long long rows = (long long)p->total_tokens * p->hv;
    if (rows > 0) {
        if (!o || !z || !weight || !y) return GDN_EINVAL;
        if (!aligned16(o) || !aligned16(z) || !aligned16(weight) || !aligned16(y)) return GDN_EINVAL;
    }
    int *status = status_ptr();
    if (!status) return GDN_ECUDA;
    return cuda_status(launch_gated_rmsnorm(o, z, weight, eps, y, rows, p->io_dtype, status,
                                            static_cast<cudaStream_t>(stream)));
}

int gdn_causal_conv1d_silu(const gdn_problem *p, const void *x, const float *weight, const float *bias,
                           void *conv_state, const int32_t *state_indices, const int32_t *cu_seqlens, int norm_qk,
                           void *q, void *k, void *v, void *stream) {
    int st = check_common(p);
    if (st) return st;
    if (p->num_seqs < 1 || p->num_state_slots < 0) return GDN_EINVAL;
    if (!cu_seqlens && p->num_seqs != 1) return GDN_EINVAL;
    if (conv_state && !state_indices && p->num_state_slots < p->num_seqs) return GDN_EINVAL;
    // token offsets stay in int (a tile start plus its length), channel blocks in grid.y
    if (int64_t(p->total_tokens) + 64 >= (int64_t(1) << 31) || (2 * p->hq + p->hv) > 65535 * 8) return GDN_EINVAL;
    if (!weight || !aligned16(weight) || (bias && !aligned16(bias))) return GDN_EINVAL;
    if ((conv_state && !aligned16(conv_state)) || (state_indices && !aligned4(state_indices)) ||
        (cu_seqlens && !aligned4(cu_seqlens)))
        return GDN_EINVAL;
    if (p->total_tokens > 0) {
        if (!x || !q || !k || !v) return GDN_EINVAL;
        if (!aligned16(x) || !aligned16(q) || !aligned16(k) || !aligned16(v)) return GDN_EINVAL;
    }
    int *status = status_ptr();
    if (!status) return GDN_ECUDA;
    return cuda_status(launch_conv1d_silu(*p, x, weight, bias, conv_state, state_indices, cu_seqlens, norm_qk, q, k,
                                          v, status, static_cast<cudaStream_t>(stream)));
}

int gdn_causal_conv1d_silu_step(const gdn_problem *p, const void *x, const float *weight, const float *bias,
                                void *conv_state, const int32_t *state_indices, int norm_qk, void *q, void *k,
                                void *v, void *stream) {
    int st = check_common(p);
    if (st) return st;
    if (p->num_seqs < 0 || p->total_tokens != p->num_seqs || p->num_state_slots < 0) return GDN_EINVAL;
    if (conv_state && !state_indices && p->num_state_slots < p->num_seqs) return GDN_EINVAL;
    if ((2 * p->hq + p->hv) > 65535 * 8) return GDN_EINVAL;
    if (!weight || !aligned16(weight) || (bias && !aligned16(bias))) return GDN_EINVAL;
    if ((conv_state && !aligned16(conv_state)) || (state_indices && !aligned4(state_indices))) return GDN_EINVAL;
    if (p->num_seqs > 0) {
        if (!x || !q || !k || !v) return GDN_EINVAL;
        if (!aligned16(x) || !aligned16(q) || !aligned16(k) || !aligned16(v)) return GDN_EINVAL;
    }
    int *status = status_ptr();
    if (!status) return GDN_ECUDA;
    return cuda_status(launch_conv1d_step(*p, x, weight, bias, conv_state, state_indices, norm_qk, q, k, v, status,
                                          static_cast<cudaStream_t>(stream)));
}

int gdn_gating(const gdn_problem *p, const float *a, const float *b, const float *A_log, const float *dt_bias,
               float *g, float *beta, void *stream) {
    if (!p || p->hv <= 0 || p->total_tokens < 0) return GDN_EINVAL;
    const long long n = (long long)p->total_tokens * p->hv;
    if (n > 0) {
        if (!a || !b || !A_log || !dt_bias || !g || !beta) return GDN_EINVAL;
        if (!aligned4(a) || !aligned4(b) || !aligned4(A_log) || !aligned4(dt_bias) || !aligned4(g) ||
            !aligned4(beta))
            return GDN_EINVAL;
    }
    return cuda_status(launch_gating(a, b, A_log, dt_bias, g, beta, n, p->hv, static_cast<cudaStream_t>(stream)));
}

int gdn_read_device_status(void *stream, int clear) {
    int *status = status_ptr();
    if (!status) return GDN_ECUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int host = 0;
    if (cudaMemcpyAsync(&host, status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return GDN_ECUDA;
    if (clear && cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess) return GDN_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ECUDA;
    return host;
}

int gdn_get_device_status(void *stream) { return gdn_read_device_status(stream, 1); }

int gdn_set_wait_limit_ns(unsigned long long ns) {
    g_wait_ns.store(ns ? ns : kDefaultWaitNs, std::memory_order_relaxed);
    return GDN_OK;
}

}  // extern "C"
