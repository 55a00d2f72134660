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
// mma accumulators, warp w holding keys 16w .. 16w+15. The forward's P, qg,
// kg and w images and decay arrive one chunk ahead by one bulk async copy
// each onto an mbarrier and are read by ldmatrix in their stored (core
// block) layout; the do tile comes by cp.async. Per chunk the kernel stores
// dh' and dv_new (bf16, 16-byte stores from shared memory) for the
// chunk-parallel gradient kernels. Every wait is bounded (about 0.5 s); a
// wait that gives up marks the error word and the CTA leaves after its
// copies in flight have landed (again bounded).
#include "gdn_mma.cuh"

namespace gdn {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kThreads = 256;
constexpr int kL6 = 64 + 8;  // row stride of a 64-column tile
constexpr uint32_t kStageBytes = kImgP + 3 * kImgW + kDecB;

struct DhStage {
    unsigned char p[kImgP];   // P image
    unsigned char qg[kImgW];  // qg image
    unsigned char kd[kImgW];  // kg^T image
    unsigned char w[kImgW];   // w image
    float dec[kKP];
    bf16 dout[kChunk * kL6];  // do [i][col]
};
struct DhSmem {
    DhStage st[2];
    bf16 dh[kKP * kL6];       // dh' [d][col] (B operand)
    bf16 dvn[kChunk * kL6];   // -dv_new [i][col] (B operand)
};

__global__ void __launch_bounds__(kThreads, 1) bwd_dh_kernel(const BwdParams p) {
    extern __shared__ __align__(128) unsigned char smraw[];
    DhSmem &sm = *reinterpret_cast<DhSmem *>(smraw);
    __shared__ __align__(8) uint64_t bars[2];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, t4 = lane & 3;
    const int s = blockIdx.x / p.H, hh = blockIdx.x % p.H;
    const int v0 = blockIdx.y * 64;
    const int K = p.K, V = p.V;
    if (p.cu_seqlens && *p.n_chunks < 0) return;  // a bad cu_seqlens: nothing was recomputed
    // the sequence: its tokens at flat rows b * T + tstart + t, its chunks at
    // global chunk slots c0 .. c0 + nts - 1
    const int b = p.cu_seqlens ? 0 : s, tstart = p.cu_seqlens ? p.cu_seqlens[s] : 0;
    const int T = p.cu_seqlens ? p.cu_seqlens[s + 1] - tstart : p.T;
    const int nts = (T + kChunk - 1) / kChunk;
    const int c0 = p.cu_seqlens ? p.seq_chunk0[s] : s * nts;
    const bf16 *dout = (const bf16 *)p.dout;
    const uint32_t bar[2] = {smem_u32(&bars[0]), smem_u32(&bars[1])};
    if (tid == 0) {
        mbar_init(bar[0], 1);
        mbar_init(bar[1], 1);
        fence_mbar_init();
    }
    __syncthreads();

    // step `it` handles chunk nts - 1 - it in stage it & 1
    auto gch_of = [&](int it) { return (int64_t)hh * p.max_chunks + c0 + (nts - 1 - it); };
    auto stage = [&](int it) {
        DhStage &S = sm.st[it & 1];
        const int c = nts - 1 - it;
        const int64_t gch = gch_of(it);
        if (tid == 0) {
            fence_async_smem();  // earlier generic reads of this stage come first
            arrive_expect_tx(bar[it & 1], kStageBytes);
            bulk_g2s(smem_u32(S.p), p.p_img + gch * kImgP, kImgP, bar[it & 1]);
            bulk_g2s(smem_u32(S.qg), p.qg_img + gch * kImgW, kImgW, bar[it & 1]);
            bulk_g2s(smem_u32(S.kd), p.kg_img + gch * kImgW, kImgW, bar[it & 1]);
            bulk_g2s(smem_u32(S.w), p.w_img + gch * kImgW, kImgW, bar[it & 1]);
            bulk_g2s(smem_u32(S.dec), p.dec + gch * kKP, kDecB, bar[it & 1]);
        }
        const int pos0 = c * kChunk, Lc = min(kChunk, T - pos0);
        for (int e = tid; e < kChunk * 8; e += kThreads) {  // do: 64 rows x 8 pieces
            const int i = e >> 3, c8 = (e & 7) * 8, col = v0 + c8;
            const bool in = i < Lc && col < (p.den_col >= 0 ? p.den_col : V);
            const int tq = in ? q_token(p.reverse, T, pos0 + i) : 0;
            const bf16 *src = in ? dout + b * p.do_sb + (int64_t)(tstart + tq) * p.do_st + hh * p.do_sh + col : dout;
            cp_async16(S.dout + i * kL6 + c8, src, in ? 16 : 0);
        }
        cp_async_commit();
    };

    // dh' at the sequence end: dh_final (or 0); warp w holds keys 16w..16w+15
    float acc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int r = 16 * warp + g8 + 8 * (e >> 1), col = v0 + 8 * n + 2 * t4 + (e & 1);
            acc[n][e] = (p.dh_final && r < K && col < V)
                            ? p.dh_final[(((int64_t)s * p.H + hh) * K + r) * p.vfull + col]
                            : 0.f;
        }
    if (nts > 0) stage(0);
    bool ok = true;
    int it = 0;
    for (; it < nts; ++it) {
        DhStage &S = sm.st[it & 1];
        if (it + 1 < nts) {
            stage(it + 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        ok = wait_bar(bar[it & 1], (it >> 1) & 1, nullptr);
        // the denominator's column of the do tile: dden (the barrier below
        // precedes its readers)
        if (p.den_col >= v0 && p.den_col < v0 + 64 && tid < kChunk) {
            const int c = nts - 1 - it, pos0 = c * kChunk, Lc = min(kChunk, T - pos0);
            float dd = 0.f;
            if (tid < Lc) dd = p.dden[((int64_t)b * p.H + hh) * p.T + tstart + q_token(p.reverse, T, pos0 + tid)];
            S.dout[tid * kL6 + (p.den_col - v0)] = __float2bfloat16_rn(dd);
        }
        // dh' to the B-operand tile
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
                *reinterpret_cast<uint32_t *>(sm.dh + (16 * warp + g8 + 8 * hf) * kL6 + 8 * n + 2 * t4) =
                    pack_bf16(acc[n][2 * hf], acc[n][2 * hf + 1]);
        if (__syncthreads_or(!ok)) break;
        const int64_t gch = gch_of(it);
        {  // its snapshot, 16-byte pieces
            bf16 *snap = p.dh_snap + gch * K * p.snap_ld + v0;
            for (int e = tid; e < kKP * 8; e += kThreads) {
                const int r = e >> 3, c8 = (e & 7) * 8;
                if (r < K && v0 + c8 < V)
                    *reinterpret_cast<uint4 *>(snap + (int64_t)r * p.snap_ld + c8) =
                        *reinterpret_cast<const uint4 *>(sm.dh + r * kL6 + c8);
            }
        }
        // dv_new = P^T do + kg dh'  (64 tokens x 64 columns; warp: 16 rows x 32 columns)
        {
            float a2[4][4];
            acc_zero(a2);
            const int m0 = 16 * (warp & 3), n0 = 32 * (warp >> 2);
            const Tile tdo{S.dout, kL6}, tdh{sm.dh, kL6};
#pragma unroll
            for (int k0 = 0; k0 < kChunk; k0 += 16) {  // P^T: stored [i][j], read transposed
                uint32_t a[4];
                ldsm_x4_t(a, S.p + img_p_off(k0 + (lane & 7) + ((lane >> 4) << 3), m0 + ((lane >> 3) & 1) * 8));
#pragma unroll
                for (int np = 0; np < 2; ++np) {
                    uint32_t b[4];
                    frag_b2(b, tdo, true, n0 + 16 * np, k0, lane);
                    mma_bf16(a2[2 * np], a, b[0], b[1]);
                    mma_bf16(a2[2 * np + 1], a, b[2], b[3]);
                }
            }
#pragma unroll
            for (int k0 = 0; k0 < kKP; k0 += 16) {  // kg: [j][d] pieces of the kg^T image
                uint32_t a[4];
                ldsm_x4(a, S.kd + img_kt_off(m0 + (lane & 15), k0 + (lane >> 4) * 8));
#pragma unroll
                for (int np = 0; np < 2; ++np) {
                    uint32_t b[4];
                    frag_b2(b, tdh, true, n0 + 16 * np, k0, lane);
                    mma_bf16(a2[2 * np], a, b[0], b[1]);
                    mma_bf16(a2[2 * np + 1], a, b[2], b[3]);
                }
            }
#pragma unroll
            for (int n = 0; n < 4; ++n)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
                    *reinterpret_cast<uint32_t *>(sm.dvn + (m0 + g8 + 8 * hf) * kL6 + n0 + 8 * n + 2 * t4) =
                        pack_bf16(-a2[n][2 * hf], -a2[n][2 * hf + 1]);
        }
        __syncthreads();
        {  // dv_new's snapshot (the tile holds -dv_new: flip the sign bits)
            bf16 *vsnap = p.dvn_snap + gch * kChunk * p.snap_ld + v0;
            for (int e = tid; e < kChunk * 8; e += kThreads) {
                const int i = e >> 3, c8 = (e & 7) * 8;
                if (v0 + c8 < V) {
                    uint4 u = *reinterpret_cast<const uint4 *>(sm.dvn + i * kL6 + c8);
                    u.x ^= 0x80008000u, u.y ^= 0x80008000u, u.z ^= 0x80008000u, u.w ^= 0x80008000u;
                    *reinterpret_cast<uint4 *>(vsnap + (int64_t)i * p.snap_ld + c8) = u;
                }
            }
        }
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
        {
            const Tile tdo{S.dout, kL6}, tdv{sm.dvn, kL6};
            const int m0 = 16 * warp;
#pragma unroll
            for (int k0 = 0; k0 < kChunk; k0 += 16) {  // qg^T and w^T: stored [i][d], read transposed
                uint32_t aq[4], aw[4];
                ldsm_x4_t(aq, S.qg + img_w_off(k0 + (lane & 7) + ((lane >> 4) << 3), m0 + ((lane >> 3) & 1) * 8));
                ldsm_x4_t(aw, S.w + img_w_off(k0 + (lane & 7) + ((lane >> 4) << 3), m0 + ((lane >> 3) & 1) * 8));
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    uint32_t b[4], bv[4];
                    frag_b2(b, tdo, true, 16 * np, k0, lane);
                    frag_b2(bv, tdv, true, 16 * np, k0, lane);
                    mma_bf16(acc[2 * np], aq, b[0], b[1]);
                    mma_bf16(acc[2 * np + 1], aq, b[2], b[3]);
                    mma_bf16(acc[2 * np], aw, bv[0], bv[1]);
                    mma_bf16(acc[2 * np + 1], aw, bv[2], bv[3]);
                }
            }
        }
        __syncthreads();  // stage it & 1, dh and dvn are rewritten next
    }
    if (!ok) {
        // a copy wait gave up: record it, let the copies in flight land, leave
        if (tid == 0) atomicOr(p.err, kDevErrTimeout);
        cp_async_wait<0>();
        wait_bar(bar[it & 1], (it >> 1) & 1, nullptr);
        if (it + 1 < nts) wait_bar(bar[(it + 1) & 1], ((it + 1) >> 1) & 1, nullptr);
        return;
    }
    if (p.dh0) {
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = 16 * warp + g8 + 8 * (e >> 1), col = v0 + 8 * n + 2 * t4 + (e & 1);
                if (r < K && col < V) p.dh0[(((int64_t)s * p.H + hh) * K + r) * p.vfull + col] = acc[n][e];
            }
    }
}

}  // namespace

cudaError_t launch_bwd_dh(const BwdParams &p, cudaStream_t st) {
    const int bytes = (int)sizeof(DhSmem);
    cudaError_t e = cudaFuncSetAttribute(bwd_dh_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    bwd_dh_kernel<<<dim3(p.n_seq * p.H, (p.V + 63) / 64), kThreads, bytes, st>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
