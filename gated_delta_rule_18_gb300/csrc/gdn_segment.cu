// gdn_segment.cu -- the serial step of segment-parallel state passing on one
// GPU.
//
// The state recurrence over one piece of a sequence is affine in the state
// that enters it: h_out = M h_in + E, with E the piece's state from h_in = 0
// (`state_ext`) and M = prod_c (diag(e^{G_last,c}) - kg_c^T w_c) its
// transition (hyper-parallel coverage_diff page,
// `kda_state_summary_forward_from_prepared`, which packs [state_ext |
// transition] as one state with V + K columns, and the chunk transition
// `diagonal - interaction`). The pages pass these summaries between the
// ranks of a context-parallel group; here the pieces are segments of one
// sequence on one GPU: the state kernel forms every segment's (E, M) in
// parallel, this kernel runs the short chain
//     h_in[0] = h0,   h_in[s+1] = M_s h_in[s] + E_s
// and the state kernel then re-runs every segment from its h_in, again in
// parallel, producing the outputs.
//
// One CTA per (sequence x head, 8-column tile: many CTAs for the few
// sequence-heads this path serves); each thread keeps 4 rows of one column, the tile and M_s^T (stored transposed by the summary
// pass, so a thread's four rows are one 16-byte load) sit in shared memory,
// and M_{s+1}^T is copied in (cp.async) while step s computes.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kCT = 8;           // state columns per CTA
constexpr int kThreads = 256;    // thread: rows 4 rb .. 4 rb + 3, column cp

struct CombineSmem {
    float mt[2][kKP * kKP];      // M_s^T and M_{s+1}^T, [a][r] (double buffer)
    float s[kKP * kCT];          // the state tile h_in[s], [a][column]
};

// M_s^T (K x K, rows contiguous) into buffer `buf` by 16-byte async copies
__device__ __forceinline__ void stage_mt(const SegParams &p, CombineSmem &sm, int buf, int s, int64_t bh) {
    // thread t copies 16-byte piece t % 32 of rows t / 32, t / 32 + 8, ...
    const int K = p.K, c = (threadIdx.x & 31) * 4;
    const float *Mt = p.sum_tr + ((int64_t)s * p.n_bh + bh) * K * K;
    if (c < K)
        for (int a = threadIdx.x >> 5; a < K; a += kThreads / 32)
            cp_async16(sm.mt[buf] + a * kKP + c, Mt + (int64_t)a * K + c, 16);
    cp_async_commit();
}

__global__ void __launch_bounds__(kThreads) seg_combine_kernel(const SegParams p) {
    extern __shared__ __align__(16) unsigned char smraw[];
    CombineSmem &sm = *reinterpret_cast<CombineSmem *>(smraw);
    const int tid = threadIdx.x;
    const int64_t bh = blockIdx.x;
    const int j0 = blockIdx.y * kCT;
    const int K = p.K, Vt = p.Vt;
    const int rb = tid >> 3, cp = tid & 7;
    const int r0 = 4 * rb, jc = j0 + cp;  // this thread's rows r0 .. r0+3 and column jc
    // rows K .. 127 of M^T's columns are never copied: zero them once
    if (K < kKP)
        for (int e = tid; e < 2 * kKP * kKP; e += kThreads)
            if (e % kKP >= K) (&sm.mt[0][0])[e] = 0.f;
    __syncthreads();
    if (p.n_seg > 1) stage_mt(p, sm, 0, 0, bh);
    float acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = r0 + i;
        acc[i] = (p.h0 && r < K && jc < Vt) ? p.h0[(bh * K + r) * Vt + jc] : 0.f;
    }
    for (int s = 0;; ++s) {
        // h_in[s]: to global and to the shared tile
        if (jc < Vt) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (r0 + i < K) p.h_in[(((int64_t)s * p.n_bh + bh) * K + r0 + i) * Vt + jc] = acc[i];
        }
        if (s + 1 >= p.n_seg) break;
#pragma unroll
        for (int i = 0; i < 4; ++i) sm.s[(r0 + i) * kCT + cp] = acc[i];
        // M_{s+1}^T streams in while step s computes
        const bool next = s + 2 < p.n_seg;
        if (next) stage_mt(p, sm, (s + 1) & 1, s + 1, bh);
        float e[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = r0 + i;
            e[i] = (r < K && jc < Vt) ? p.sum_ext[(((int64_t)s * p.n_bh + bh) * K + r) * Vt + jc] : 0.f;
        }
        if (next) cp_async_wait<1>();
        else cp_async_wait<0>();
        __syncthreads();  // M_s^T and the tile are complete
        const float *mt = sm.mt[s & 1];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = 0.f;
#pragma unroll 8
        for (int a = 0; a < K; ++a) {
            const float4 m4 = *reinterpret_cast<const float4 *>(mt + a * kKP + r0);
            const float sv = sm.s[a * kCT + cp];
            acc[0] = fmaf(m4.x, sv, acc[0]);
            acc[1] = fmaf(m4.y, sv, acc[1]);
            acc[2] = fmaf(m4.z, sv, acc[2]);
            acc[3] = fmaf(m4.w, sv, acc[3]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] += e[i];
        __syncthreads();  // the tile and buffer s & 1 are rewritten next
    }
}

}  // namespace

cudaError_t launch_seg_combine(const SegParams &p, cudaStream_t st) {
    const int bytes = (int)sizeof(CombineSmem);
    cudaError_t e = cudaFuncSetAttribute(seg_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    seg_combine_kernel<<<dim3(p.n_bh, (p.Vt + kCT - 1) / kCT), kThreads, bytes, st>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
