// gdn_chunk_bf16.cu -- the bf16 tensor-core path (fp32 accumulate, fp32
// state) of the chunked gated delta rule runs in three launches; this file
// holds the first and the last:
//
//  1. chunk_table_kernel (varlen only): checks cu_seqlens on the device and
//     lists every 64-token chunk as (sequence, chunk) -- chunks never cross a
//     sequence boundary (hyper-parallel coverage_diff page: per-sequence
//     chunk counts ceil(len / BT), `chunk_indices` / `chunk_offsets`).
//  2. the intra-chunk kernel (gdn_intra_bf16.cu), one CTA per (chunk, head),
//     writes w, u, P, qg, kg and the chunk decay to the workspace.
//  3. state_bf16_kernel: one CTA per (sequence, head, 64-column value tile),
//     serial over the sequence's chunks, state h (K x 64, fp32) in registers:
//        v_new = u - w h
//        o     = qg h + P v_new
//        h    <- dec . h + kg^T v_new
//     (coverage_diff page, `chunk_gated_delta_rule_fwd_kernel_h_blockdim64`:
//     b_v = u - w h, h *= exp(g_last), h += k^T v_new; the output uses the
//     state at chunk start plus the in-chunk term, and reads the state after
//     each token's own write, as the SANA `fused_gdn.py` page's Pass 2 does.)
//     The next chunk's tiles stream in with cp.async while this one computes.
//
// Contractions use mma.sync m16n8k16 bf16 with fp32 accumulators, fed by
// ldmatrix from padded (bank-conflict-free) shared-memory tiles.
#include "gdn_common.cuh"

namespace gdn {
namespace {

using bf16 = __nv_bfloat16;

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
    if (tid == 0) *err = bad ? 1 : 0;  // the word describes this call only
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

constexpr int kStateThreads = 128;
constexpr int kBV = 64;     // value columns per CTA
constexpr int kUS = kBV + 8;
constexpr int kPS = kChunk + 8;

template <int KP>
struct StateLayout {
    static constexpr int KS = KP + 8;
    // one pipeline stage: w, qg, kg (64 x KS), u (64 x kUS), P (64 x kPS) bf16; dec KP fp32
    static constexpr size_t w = 0;
    static constexpr size_t qg = w + 2 * kChunk * KS;
    static constexpr size_t kg = qg + 2 * kChunk * KS;
    static constexpr size_t u = kg + 2 * kChunk * KS;
    static constexpr size_t pm = u + 2 * kChunk * kUS;
    static constexpr size_t dec = pm + 2 * kChunk * kPS;
    static constexpr size_t stage = dec + 4 * KP;
    static constexpr size_t h = 2 * stage;             // bf16 KP x kUS
    static constexpr size_t vn = h + 2 * KP * kUS;     // bf16 64 x kUS
    static constexpr size_t bytes = vn + 2 * kChunk * kUS;
};

template <int KP>
__global__ void __launch_bounds__(kStateThreads) state_bf16_kernel(const FwdParams p) {
    using Lay = StateLayout<KP>;
    constexpr int KS = Lay::KS;
    constexpr int MT = KP / 64;   // 16-row key tiles per warp
    constexpr int RW = KP / 4;    // key rows per warp
    extern __shared__ __align__(16) unsigned char smraw[];
    bf16 *sH = reinterpret_cast<bf16 *>(smraw + Lay::h);
    bf16 *sVn = reinterpret_cast<bf16 *>(smraw + Lay::vn);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, t4 = lane & 3;
    const int H = p.H, K = p.K, V = p.V;
    const int s = blockIdx.x / H, hh = blockIdx.x % H;
    const int v0 = blockIdx.y * kBV;
    if (!p.cu_seqlens && blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) *p.err = 0;
    if (p.cu_seqlens && *p.n_chunks < 0) return;
    SeqInfo si;
    if (!seq_info(p, s, si)) return;
    const int nchunks = (si.len + kChunk - 1) / kChunk;
    const int gc0 = p.cu_seqlens ? p.seq_chunk0[s] : s * ((p.T + kChunk - 1) / kChunk);

    float hf[MT][8][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = warp * RW + mt * 16 + g8 + 8 * (e >> 1);
                const int col = v0 + 8 * n + 2 * t4 + (e & 1);
                hf[mt][n][e] = (p.h0 && r < K && col < V)
                                   ? p.h0[(((int64_t)s * H + hh) * K + r) * V + col]
                                   : 0.f;
            }

    auto prefetch = [&](int c, int st) {
        unsigned char *base = smraw + st * Lay::stage;
        bf16 *dW = reinterpret_cast<bf16 *>(base + Lay::w);
        bf16 *dQ = reinterpret_cast<bf16 *>(base + Lay::qg);
        bf16 *dK = reinterpret_cast<bf16 *>(base + Lay::kg);
        bf16 *dU = reinterpret_cast<bf16 *>(base + Lay::u);
        bf16 *dP = reinterpret_cast<bf16 *>(base + Lay::pm);
        float *dD = reinterpret_cast<float *>(base + Lay::dec);
        const int Lc = min(kChunk, si.len - c * kChunk);
        const int64_t hrow = (int64_t)hh * p.rows + si.row0 + c * kChunk;
        const bf16 *gw = p.w + hrow * KP, *gq = p.qg + hrow * KP, *gk = p.kg + hrow * KP;
        for (int e = tid; e < kChunk * (KP / 8); e += kStateThreads) {
            const int i = e / (KP / 8), d = (e % (KP / 8)) * 8;
            const bool ok = i < Lc;
            const int64_t off = ok ? (int64_t)i * KP + d : 0;
            const int n = ok ? 16 : 0;
            cp_async16(dW + i * KS + d, gw + off, n);
            cp_async16(dQ + i * KS + d, gq + off, n);
            cp_async16(dK + i * KS + d, gk + off, n);
        }
        const bf16 *gu = p.u + hrow * p.UW;
        const bf16 *gp = p.aqk + hrow * kChunk;
        for (int e = tid; e < kChunk * 8; e += kStateThreads) {
            const int i = e >> 3, m = (e & 7) * 8;
            const bool oku = i < Lc && v0 + m < p.UW;
            cp_async16(dU + i * kUS + m, gu + (oku ? (int64_t)i * p.UW + v0 + m : 0), oku ? 16 : 0);
            const bool okp = i < Lc;
            cp_async16(dP + i * kPS + m, gp + (okp ? (int64_t)i * kChunk + m : 0), okp ? 16 : 0);
        }
        const float *gd = p.dec + ((int64_t)hh * p.max_chunks + gc0 + c) * KP;
        for (int e = tid; e < KP / 4; e += kStateThreads) cp_async16(dD + 4 * e, gd + 4 * e, 16);
        cp_async_commit();
    };

    if (nchunks > 0) prefetch(0, 0);
    for (int c = 0; c < nchunks; ++c) {
        const int st = c & 1;
        if (c + 1 < nchunks) {
            prefetch(c + 1, st ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        unsigned char *base = smraw + st * Lay::stage;
        const bf16 *sW = reinterpret_cast<const bf16 *>(base + Lay::w);
        const bf16 *sQg = reinterpret_cast<const bf16 *>(base + Lay::qg);
        const bf16 *sKg = reinterpret_cast<const bf16 *>(base + Lay::kg);
        const bf16 *sU = reinterpret_cast<const bf16 *>(base + Lay::u);
        const bf16 *sP = reinterpret_cast<const bf16 *>(base + Lay::pm);
        const float *sDec = reinterpret_cast<const float *>(base + Lay::dec);
        const int pos0 = c * kChunk;
        const int Lc = min(kChunk, si.len - pos0);

        // 1. state to shared memory as the bf16 MMA operand
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int n = 0; n < 8; ++n)
#pragma unroll
                for (int hfi = 0; hfi < 2; ++hfi) {
                    const int r = warp * RW + mt * 16 + g8 + 8 * hfi;
                    *reinterpret_cast<uint32_t *>(sH + r * kUS + 8 * n + 2 * t4) =
                        pack_bf16(hf[mt][n][2 * hfi], hf[mt][n][2 * hfi + 1]);
                }
        __syncthreads();

        // 2. w h and qg h for token rows 16*warp .. +15
        float aw[8][4], ao[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) aw[n][e] = ao[n][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KP / 16; ++kk) {
            uint32_t a1[4], a2[4];
            ldsm_x4(a1, sW + (16 * warp + (lane & 15)) * KS + 16 * kk + (lane >> 4) * 8);
            ldsm_x4(a2, sQg + (16 * warp + (lane & 15)) * KS + 16 * kk + (lane >> 4) * 8);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t b[4];
                ldsm_x4_t(b, sH + (16 * kk + (lane & 15)) * kUS + 16 * np + (lane >> 4) * 8);
                mma_bf16(aw[2 * np], a1, b[0], b[1]);
                mma_bf16(aw[2 * np + 1], a1, b[2], b[3]);
                mma_bf16(ao[2 * np], a2, b[0], b[1]);
                mma_bf16(ao[2 * np + 1], a2, b[2], b[3]);
            }
        }
        // v_new = u - w h
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int hfi = 0; hfi < 2; ++hfi) {
                const int i = 16 * warp + g8 + 8 * hfi;
                const int col = 8 * n + 2 * t4;
                const float2 uu = __bfloat1622float2(
                    *reinterpret_cast<const __nv_bfloat162 *>(sU + i * kUS + col));
                *reinterpret_cast<uint32_t *>(sVn + i * kUS + col) =
                    pack_bf16(uu.x - aw[n][2 * hfi], uu.y - aw[n][2 * hfi + 1]);
            }
        __syncthreads();

        // 3. o = qg h + P v_new (P lower triangular: column blocks 0..warp)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            if (kk <= warp) {
                uint32_t a[4];
                ldsm_x4(a, sP + (16 * warp + (lane & 15)) * kPS + 16 * kk + (lane >> 4) * 8);
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    uint32_t b[4];
                    ldsm_x4_t(b, sVn + (16 * kk + (lane & 15)) * kUS + 16 * np + (lane >> 4) * 8);
                    mma_bf16(ao[2 * np], a, b[0], b[1]);
                    mma_bf16(ao[2 * np + 1], a, b[2], b[3]);
                }
            }
        }
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const int cb = v0 + 8 * n;
#pragma unroll
            for (int hfi = 0; hfi < 2; ++hfi) {
                const int i = 16 * warp + g8 + 8 * hfi;
                if (i >= Lc) continue;
                const int tq = q_token(p.reverse, si.len, pos0 + i);
                const float o0 = ao[n][2 * hfi], o1 = ao[n][2 * hfi + 1];
                if (cb + 8 <= V) {
                    const int64_t off = si.b * p.o_sb + (int64_t)(si.tstart + tq) * p.o_st +
                                        hh * p.o_sh + cb + 2 * t4;
                    if (p.out_f32) {
                        float2 *op = reinterpret_cast<float2 *>((float *)p.out + off);
                        float2 x = make_float2(o0, o1);
                        if (p.accumulate) {
                            const float2 y = *op;
                            x.x += y.x;
                            x.y += y.y;
                        }
                        *op = x;
                    } else {
                        __nv_bfloat162 *op = reinterpret_cast<__nv_bfloat162 *>((bf16 *)p.out + off);
                        float2 x = make_float2(o0, o1);
                        if (p.accumulate) {
                            const float2 y = __bfloat1622float2(*op);
                            x.x += y.x;
                            x.y += y.y;
                        }
                        *op = __floats2bfloat162_rn(x.x, x.y);
                    }
                } else if (p.has_den && cb == V && t4 == 0) {
                    float *dp = p.den + ((int64_t)si.b * H + hh) * p.T + si.tstart + tq;
                    *dp = p.accumulate ? *dp + o0 : o0;
                }
            }
        }

        // 4. h <- dec . h + kg^T v_new
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int r = warp * RW + mt * 16 + g8;
            const float d0 = sDec[r], d1 = sDec[r + 8];
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                hf[mt][n][0] *= d0;
                hf[mt][n][1] *= d0;
                hf[mt][n][2] *= d1;
                hf[mt][n][3] *= d1;
            }
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            uint32_t b[4][4];
#pragma unroll
            for (int np = 0; np < 4; ++np)
                ldsm_x4_t(b[np], sVn + (16 * kk + (lane & 15)) * kUS + 16 * np + (lane >> 4) * 8);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                uint32_t a[4];
                const int m0 = warp * RW + mt * 16;
                ldsm_x4_t(a, sKg + (16 * kk + (lane & 7) + ((lane >> 4) << 3)) * KS + m0 +
                                 ((lane >> 3) & 1) * 8);
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    mma_bf16(hf[mt][2 * np], a, b[np][0], b[np][1]);
                    mma_bf16(hf[mt][2 * np + 1], a, b[np][2], b[np][3]);
                }
            }
        }
        __syncthreads();
    }

    if (p.h_final) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int n = 0; n < 8; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = warp * RW + mt * 16 + g8 + 8 * (e >> 1);
                    const int col = v0 + 8 * n + 2 * t4 + (e & 1);
                    if (r < K && col < V)
                        p.h_final[(((int64_t)s * H + hh) * K + r) * V + col] = hf[mt][n][e];
                }
    }
}

template <int KP>
cudaError_t launch_state_t(const FwdParams &p, cudaStream_t st) {
    using Lay = StateLayout<KP>;
    auto kern = state_bf16_kernel<KP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Lay::bytes);
    if (e != cudaSuccess) return e;
    dim3 grid(p.n_seq * p.H, (p.Vt + kBV - 1) / kBV);
    kern<<<grid, kStateThreads, Lay::bytes, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_table(const FwdParams &p, cudaStream_t st) {
    chunk_table_kernel<<<1, 1024, 0, st>>>(p.cu_seqlens, p.n_seq, p.T, p.n_chunks, p.chunk_tab,
                                           p.seq_chunk0, p.err);
    return cudaGetLastError();
}

cudaError_t launch_state_bf16(const FwdParams &p, int KP, cudaStream_t st) {
    if (KP == 64) return launch_state_t<64>(p, st);
    return launch_state_t<128>(p, st);
}

}  // namespace gdn
