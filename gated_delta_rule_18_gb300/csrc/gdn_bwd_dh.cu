// gdn_bwd_dh.cu -- the serial part of the backward: the state gradient walked
// back over the chunks (hyper-parallel coverage_diff page,
// `chunk_gated_delta_rule_bwd_dhu`: dh accumulates q do^T and - w dv each
// chunk and is decayed by the chunk's e^{g_last}; dv gains k dh).
//
// The forward per chunk (state h entering it, G the in-chunk cumulative gate):
//   v_new = u - w h,   o = qg h + P v_new,   h' = e^{G_C} h + kg^T v_new
// with qg = e^{G} q, kg = e^{G_C - G} k. For the loss gradient dh' at the
// chunk's end and do of its outputs, reverse mode gives
//   dv_new = P^T do + kg dh'                   (the chunk's dL/dv_new)
//   dh     = e^{G_C} dh' + qg^T do - w^T dv_new (dL/dh, handed to chunk c-1)
// One CTA (8 warps) per (sequence, head, 64-column value tile) walks the
// chunks last to first; dh (128 keys x 64 columns, fp32) lives in the warps'
// mma accumulators, warp w holding keys 16w .. 16w+15. The chunk operands
// (the forward's P, qg, kg, w images and decay, and the do tile) are copied
// with cp.async one chunk ahead into row-major tiles. Per chunk it stores
// dh' and dv_new (bf16) for the chunk-parallel gradient kernels.
#include "gdn_mma.cuh"

namespace gdn {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kThreads = 256;
constexpr int kLK = kKP + 8;  // row stride of a 128-column tile
constexpr int kL6 = 64 + 8;   // row stride of a 64-column tile

struct DhStage {
    bf16 p[kChunk * kL6];    // P [i][j]
    bf16 qg[kChunk * kLK];   // qg [i][d]
    bf16 kd[kChunk * kLK];   // kg [i][d]
    bf16 w[kChunk * kLK];    // w [i][d]
    bf16 dout[kChunk * kL6]; // do [i][col]
    float dec[kKP];
};
struct DhSmem {
    DhStage st[2];
    bf16 dh[kKP * kL6];      // dh' [d][col] (B operand)
    bf16 dvn[kChunk * kL6];  // -dv_new [i][col] (B operand)
};

__global__ void __launch_bounds__(kThreads, 1) bwd_dh_kernel(const BwdParams p) {
    extern __shared__ __align__(16) unsigned char smraw[];
    DhSmem &sm = *reinterpret_cast<DhSmem *>(smraw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, t4 = lane & 3;
    const int s = blockIdx.x / p.H, hh = blockIdx.x % p.H;
    const int v0 = blockIdx.y * 64;
    const int K = p.K, V = p.V, T = p.T;
    const int nts = (T + kChunk - 1) / kChunk;
    const bf16 *dout = (const bf16 *)p.dout;

    auto stage = [&](int c) {
        DhStage &S = sm.st[c & 1];
        const int64_t gch = (int64_t)hh * p.max_chunks + (int64_t)s * nts + c;
        const int pos0 = c * kChunk, Lc = min(kChunk, T - pos0);
        for (int e = tid; e < kChunk * 8; e += kThreads) {  // P and do: 64 rows x 8 pieces
            const int i = e >> 3, j8 = (e & 7) * 8;
            cp_async16(S.p + i * kL6 + j8, p.p_img + gch * kImgP + img_p_off(i, j8), 16);
            const int col = v0 + j8;
            const bool in = i < Lc && col < V;
            const int tq = in ? q_token(p.reverse, T, pos0 + i) : 0;
            const bf16 *src = in ? dout + s * p.do_sb + (int64_t)tq * p.do_st + hh * p.do_sh + col : dout;
            cp_async16(S.dout + i * kL6 + j8, src, in ? 16 : 0);
        }
        for (int e = tid; e < kChunk * 16; e += kThreads) {  // qg, kg, w: 64 rows x 16 pieces
            const int i = e >> 4, d8 = (e & 15) * 8;
            cp_async16(S.qg + i * kLK + d8, p.qg_img + gch * kImgW + img_w_off(i, d8), 16);
            cp_async16(S.kd + i * kLK + d8, p.kg_img + gch * kImgW + img_kt_off(i, d8), 16);
            cp_async16(S.w + i * kLK + d8, p.w_img + gch * kImgW + img_w_off(i, d8), 16);
        }
        if (tid < kKP / 4) cp_async16(S.dec + 4 * tid, p.dec + gch * kKP + 4 * tid, 16);
        cp_async_commit();
    };

    // dh' at the sequence end: dh_final (or 0); warp w holds keys 16w..16w+15
    float acc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int r = 16 * warp + g8 + 8 * (e >> 1), col = v0 + 8 * n + 2 * t4 + (e & 1);
            acc[n][e] = (p.dh_final && r < K && col < V) ? p.dh_final[(((int64_t)s * p.H + hh) * K + r) * V + col]
                                                         : 0.f;
        }
    if (nts > 0) stage(nts - 1);
    for (int c = nts - 1; c >= 0; --c) {
        const DhStage &S = sm.st[c & 1];
        if (c > 0) {
            stage(c - 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        // dh' to the B-operand tile and to its snapshot
        const int64_t gch = (int64_t)hh * p.max_chunks + (int64_t)s * nts + c;
        bf16 *snap = p.dh_snap + gch * K * V;
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int r = 16 * warp + g8 + 8 * hf, cl = 8 * n + 2 * t4;
                const uint32_t pk = pack_bf16(acc[n][2 * hf], acc[n][2 * hf + 1]);
                *reinterpret_cast<uint32_t *>(sm.dh + r * kL6 + cl) = pk;
                if (r < K && v0 + cl < V) *reinterpret_cast<uint32_t *>(snap + (int64_t)r * V + v0 + cl) = pk;
            }
        __syncthreads();
        // dv_new = P^T do + kg dh'  (64 tokens x 64 columns; warp: 16 rows x 32 columns)
        {
            float a2[4][4];
            acc_zero(a2);
            const int m0 = 16 * (warp & 3), n0 = 32 * (warp >> 2);
            warp_gemm(a2, Tile{S.p, kL6}, true, Tile{S.dout, kL6}, true, m0, n0, kChunk, lane);
            warp_gemm(a2, Tile{S.kd, kLK}, false, Tile{sm.dh, kL6}, true, m0, n0, kKP, lane);
            bf16 *vsnap = p.dvn_snap + gch * kChunk * V;
#pragma unroll
            for (int n = 0; n < 4; ++n)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int i = m0 + g8 + 8 * hf, cl = n0 + 8 * n + 2 * t4;
                    const float x0 = a2[n][2 * hf], x1 = a2[n][2 * hf + 1];
                    *reinterpret_cast<uint32_t *>(sm.dvn + i * kL6 + cl) = pack_bf16(-x0, -x1);
                    if (v0 + cl < V) *reinterpret_cast<uint32_t *>(vsnap + (int64_t)i * V + v0 + cl) = pack_bf16(x0, x1);
                }
        }
        __syncthreads();
        // dh = e^{G_C} dh' + qg^T do - w^T dv_new
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const float d = S.dec[16 * warp + g8 + 8 * hf];
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                acc[n][2 * hf] *= d;
                acc[n][2 * hf + 1] *= d;
            }
        }
        warp_gemm(acc, Tile{S.qg, kLK}, true, Tile{S.dout, kL6}, true, 16 * warp, 0, kChunk, lane);
        warp_gemm(acc, Tile{S.w, kLK}, true, Tile{sm.dvn, kL6}, true, 16 * warp, 0, kChunk, lane);
        __syncthreads();  // stage c & 1, dh and dvn are rewritten next
    }
    if (p.dh0) {
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = 16 * warp + g8 + 8 * (e >> 1), col = v0 + 8 * n + 2 * t4 + (e & 1);
                if (r < K && col < V) p.dh0[(((int64_t)s * p.H + hh) * K + r) * V + col] = acc[n][e];
            }
    }
}

}  // namespace

cudaError_t launch_bwd_dh(const BwdParams &p, cudaStream_t st) {
    const int bytes = (int)sizeof(DhSmem);
    cudaError_t e = cudaFuncSetAttribute(bwd_dh_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    bwd_dh_kernel<<<dim3(p.B * p.H, (p.V + 63) / 64), kThreads, bytes, st>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
