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
    __shared__ int part[kTableThreads];
    __shared__ int bad;
    const int tid = threadIdx.x;
    const int N = a.num_seqs;
    if (tid == 0) bad = 0;
    for (int i = tid; i < a.ready_count; i += kTableThreads) a.ready[i] = 0;
    __syncthreads();
    // 1) validate offsets: start at 0, non-decreasing, end at total_tokens
    if (a.cu) {
        if (tid == 0 && (a.cu[0] != 0 || a.cu[N] != a.total_tokens)) bad = 1;
        for (int n = tid; n < N; n += kTableThreads)
            if (a.cu[n + 1] < a.cu[n]) bad = 1;
    }
    __syncthreads();
    if (bad) {
        if (tid == 0) {
            record_status(a.status, GDN_EDEVICE_INPUT);
            *a.n_chunks = -1;  // every later kernel of this call returns at once
        }
        for (int n = tid; n < N; n += kTableThreads) a.seq_info[n] = SeqInfo{0, 0, 0, 0};
        return;
    }
    // 2) exclusive scan of per-sequence chunk counts (contiguous ranges per thread)
    const int per = (N + kTableThreads - 1) / kTableThreads;
    const int n0 = min(N, tid * per), n1 = min(N, n0 + per);
    int local = 0;
    for (int n = n0; n < n1; ++n) local += (seq_begin(a, n + 1) - seq_begin(a, n) + kChunk - 1) / kChunk;
    part[tid] = local;
    __syncthreads();
    for (int off = 1; off < kTableThreads; off <<= 1) {
        int v = (tid >= off) ? part[tid - off] : 0;
        __syncthreads();
        part[tid] += v;
        __syncthreads();
    }
    int first = part[tid] - local;
    if (tid == kTableThreads - 1) *a.n_chunks = min(part[tid], a.max_chunks);
    // 3) write the sequence and chunk records
    for (int n = n0; n < n1; ++n) {
        const int b = seq_begin(a, n), L = seq_begin(a, n + 1) - b;
        const int nc = (L + kChunk - 1) / kChunk;
        a.seq_info[n] = SeqInfo{first, nc, b, L};
        for (int c = 0; c < nc; ++c) {
            if (first + c < a.max_chunks)
                a.chunk_info[first + c] = ChunkInfo{n, b + c * kChunk, min(kChunk, L - c * kChunk), c};
        }
        first += nc;
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
