// Chunk table: splits every sequence into 64-token chunks on the device.
//
// The Lab3 GDN Prefill page ("计算过程描述") gives a sequence of length L
// ceil(L / 64) chunks, the last of valid length l_c = min(64, L - 64c). For
// packed sequences each one starts its own chunk grid at its cu_seqlens
// offset, so a chunk never straddles two sequences. cu_seqlens lives on the
// device, so it is checked and scanned here rather than on the host.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kTableThreads = 1024;

__device__ __forceinline__ int seq_begin(const PrefillArgs &a, int n) {
    return a.cu ? a.cu[n] : n * a.dense_seqlen;
}

__global__ void __launch_bounds__(kTableThreads) k_chunk_table(PrefillArgs a) {
    __shared__ int wsum[kTableThreads / 32];
    __shared__ int bad;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int N = a.num_seqs;
    if (tid == 0) bad = 0;
    for (int i = tid; i < a.ready_count; i += kTableThreads) a.ready[i] = 0;
    __syncthreads();
    // 1) per-thread contiguous range of sequences: validate the offsets (start
    //    at 0, non-decreasing, end at total_tokens) and count their chunks
    const int per = (N + kTableThreads - 1) / kTableThreads;
    const int n0 = min(N, tid * per), n1 = min(N, n0 + per);
    int local = 0;
    if (n0 < n1) {
        int b = seq_begin(a, n0);
        if (a.cu && n0 == 0 && b != 0) bad = 1;
        for (int n = n0; n < n1; ++n) {
            const int e = seq_begin(a, n + 1);
            if (e < b) bad = 1;
            local += (e - b + kChunk - 1) / kChunk;
            b = e;
        }
        if (a.cu && n1 == N && b != a.total_tokens) bad = 1;
    }
    // 2) exclusive scan of the counts: within each warp by shuffles, then over warps
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) wsum[wid] = incl;
    __syncthreads();
    if (bad) {  // uniform: read after the barrier
        if (tid == 0) {
            record_status(a.status, GDN_EDEVICE_INPUT);
            *a.n_chunks = -1;  // every later kernel of this call returns at once
        }
        for (int n = tid; n < N; n += kTableThreads) a.seq_info[n] = SeqInfo{0, 0, 0, 0};
        return;
    }
    if (wid == 0) {
        int x = lane < kTableThreads / 32 ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += t;
        }
        if (lane < kTableThreads / 32) wsum[lane] = x;  // inclusive over warps
    }
    __syncthreads();
    int first = (wid > 0 ? wsum[wid - 1] : 0) + incl - local;
    const int total = wsum[kTableThreads / 32 - 1];
    if (tid == 0) *a.n_chunks = min(total, a.max_chunks);
    // 3) sequence records
    for (int n = n0; n < n1; ++n) {
        const int b = seq_begin(a, n), L = seq_begin(a, n + 1) - b;
        const int nc = (L + kChunk - 1) / kChunk;
        a.seq_info[n] = SeqInfo{first, nc, b, L};
        first += nc;
    }
    __syncthreads();  // the records are visible to the whole block
    // 4) chunk records, one per thread: the sequence of global chunk c is the
    //    last one whose first chunk is <= c (an empty sequence shares its
    //    first-chunk index with the next non-empty one, or lies past the end)
    const int nch = min(total, a.max_chunks);
    for (int c = tid; c < nch; c += kTableThreads) {
        int lo = 0, hi = N - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.seq_info[mid].first_chunk <= c) lo = mid; else hi = mid - 1;
        }
        const SeqInfo si = a.seq_info[lo];
        const int k = c - si.first_chunk;
        a.chunk_info[c] = ChunkInfo{lo, si.start + k * kChunk, min(kChunk, si.len - k * kChunk), k};
    }
}

}  // namespace

cudaError_t launch_chunk_table(const PrefillArgs &a, cudaStream_t s) {
    {
        LaunchScope scope(GDN_K_CHUNK_TABLE, s);
        k_chunk_table<<<1, kTableThreads, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace gdn
