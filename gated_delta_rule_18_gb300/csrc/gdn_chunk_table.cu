// gdn_chunk_table.cu -- varlen chunk list for the bf16 path.
//
// chunk_table_kernel checks cu_seqlens on the device (0 = c_0 <= c_1 <= ...
// <= c_n = T; a violation sets the workspace error word and marks the call
// invalid so every later kernel of the call skips its work) and lists every
// 64-token chunk as (sequence, chunk index) with each sequence's first global
// chunk. Chunks never cross a sequence boundary (hyper-parallel
// coverage_diff page: per-sequence chunk counts ceil(len / BT),
// `chunk_indices` / `chunk_offsets`).
#include "gdn_common.cuh"

namespace gdn {
namespace {

// ------------------------------------------------------------- table ------

__global__ void __launch_bounds__(1024) chunk_table_kernel(const int32_t *__restrict__ cu,
                                                           int n_seq, int T, int *n_chunks,
                                                           int2 *tab, int *seq_chunk0,
                                                           int *err) {
    __shared__ int bad;
    __shared__ int wsum[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) bad = (cu[0] != 0 || cu[n_seq] != T) ? 1 : 0;
    __syncthreads();
    for (int s = tid; s < n_seq; s += blockDim.x)
        if (cu[s + 1] < cu[s]) bad = 1;
    __syncthreads();
    // (the host clears the word on the stream before a call's first kernel)
    if (tid == 0 && bad) atomicOr(err, 1);
    if (bad) {
        if (tid == 0) *n_chunks = -1;
        return;
    }
    const int per = (n_seq + blockDim.x - 1) / blockDim.x;
    const int lo = min(n_seq, tid * per), hi = min(n_seq, lo + per);
    int local = 0;
    for (int s = lo; s < hi; ++s) local += (cu[s + 1] - cu[s] + kChunk - 1) / kChunk;
    // block-wide exclusive scan of `local`
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int x = (lane < (int)(blockDim.x >> 5)) ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        wsum[lane] = x;  // inclusive over warps
    }
    __syncthreads();
    const int excl = incl - local + (warp > 0 ? wsum[warp - 1] : 0);
    int run = excl;
    for (int s = lo; s < hi; ++s) {
        seq_chunk0[s] = run;
        const int nc = (cu[s + 1] - cu[s] + kChunk - 1) / kChunk;
        for (int c = 0; c < nc; ++c) tab[run + c] = make_int2(s, c);
        run += nc;
    }
    if (tid == (int)blockDim.x - 1) *n_chunks = excl + local;
}

// ------------------------------------------------------------- state ------

}  // namespace

cudaError_t launch_chunk_table(const FwdParams &p, cudaStream_t st) {
    chunk_table_kernel<<<1, 1024, 0, st>>>(p.cu_seqlens, p.n_seq, p.T, p.n_chunks, p.chunk_tab,
                                           p.seq_chunk0, p.err);
    return cudaGetLastError();
}

}  // namespace gdn
