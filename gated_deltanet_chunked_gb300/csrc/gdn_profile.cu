// Launch accounting and optional per-kernel CUDA-event timing.
//
// Every kernel launch of the library goes through a LaunchScope, which
// counts it (always) and, while gdn_profile_enable(1) is in force, brackets
// it with a pair of CUDA events recorded on the launching stream. The events
// are read back by gdn_profile_collect, which is how a benchmark obtains the
// live duration of each kernel over its timed region.
#include <mutex>
#include <vector>

#include "gdn_common.cuh"

namespace gdn {
namespace {

struct Pending {
    int kernel;
    cudaEvent_t start, stop;
};

std::mutex g_mu;
bool g_enabled = false;
long long g_launches[GDN_K_COUNT];
double g_ms[GDN_K_COUNT];
long long g_timed[GDN_K_COUNT];
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_free;

cudaEvent_t take_event() {
    if (!g_free.empty()) {
        cudaEvent_t e = g_free.back();
        g_free.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

const char *const kNames[GDN_K_COUNT] = {
    "chunk_table", "prep_simt", "state_simt", "output_simt", "recurrent_step",
    "chunk_fused_tc", "recurrent_step_gated", "gated_rmsnorm", "conv1d_silu", "gating", "conv1d_step",
};

}  // namespace

LaunchScope::LaunchScope(int kernel, cudaStream_t s) : kernel_(kernel), stream_(s), start_(nullptr) {
    std::lock_guard<std::mutex> lk(g_mu);
    ++g_launches[kernel];
    if (g_enabled) {
        start_ = take_event();
        if (start_) cudaEventRecord(start_, s);
    }
}

LaunchScope::~LaunchScope() {
    if (!start_) return;
    std::lock_guard<std::mutex> lk(g_mu);
    cudaEvent_t stop = take_event();
    if (!stop) return;
    cudaEventRecord(stop, stream_);
    g_pending.push_back(Pending{kernel_, start_, stop});
}

}  // namespace gdn

using namespace gdn;

extern "C" {

int gdn_profile_enable(int enable) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_enabled = enable != 0;
    return GDN_OK;
}

const char *gdn_kernel_name(int kernel) {
    return (kernel >= 0 && kernel < GDN_K_COUNT) ? kNames[kernel] : "unknown";
}

int gdn_profile_collect(long long *launches, double *ms, long long *timed, int count, int reset) {
    std::lock_guard<std::mutex> lk(g_mu);
    int st = GDN_OK;
    for (const Pending &p : g_pending) {
        float t = 0.f;
        if (cudaEventSynchronize(p.stop) != cudaSuccess || cudaEventElapsedTime(&t, p.start, p.stop) != cudaSuccess)
            st = GDN_ECUDA;
        else {
            g_ms[p.kernel] += t;
            ++g_timed[p.kernel];
        }
        g_free.push_back(p.start);
        g_free.push_back(p.stop);
    }
    g_pending.clear();
    for (int i = 0; i < count && i < GDN_K_COUNT; ++i) {
        if (launches) launches[i] = g_launches[i];
        if (ms) ms[i] = g_ms[i];
        if (timed) timed[i] = g_timed[i];
    }
    if (reset)
        for (int i = 0; i < GDN_K_COUNT; ++i) g_launches[i] = g_timed[i] = 0, g_ms[i] = 0.0;
    return st;
}

}  // extern "C"
