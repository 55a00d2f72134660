// gdn_chunk_bf16.cu -- the bf16 tensor-core path (fp32 accumulate, fp32
// state) of the chunked gated delta rule, in three launches:
//
//  1. chunk_table_kernel (varlen only): checks cu_seqlens on the device and
//     lists every 64-token chunk as (sequence, chunk) -- chunks never cross a
//     sequence boundary (hyper-parallel coverage_diff page: per-sequence
//     chunk counts ceil(len / BT), `chunk_indices` / `chunk_offsets`).
//  2. intra_bf16_kernel: one CTA per (chunk, head), parallel over all chunks.
//     From the chunk's q, k, v, beta and gates it builds
//        A   = strictly_lower(diag(beta) (K K^T . Gamma))
//        T   = (I + A)^{-1}            (blocked forward substitution, fp32)
//        w   = T (beta e^{G} . K),  u = T (beta . V)
//        P   = lower_incl(Q K^T . Gamma)      (intra-chunk output matrix)
//        qg  = e^{G} . Q,  kg = e^{G_last - G} . K,  dec = e^{G_last}
//     and stores them (bf16; dec fp32) in the workspace, head-major.
//     Gamma_ij = e^{G_i - G_j} (per key for the gk gate). This is the intra
//     step whose outputs the hyper-parallel coverage_diff page consumes
//     (`chunk_kda_fwd_intra` returning w, u, kg, Aqk, Akk); its body is not on
//     the pages and is derived here from the token recurrence.
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

// ------------------------------------------------------------- intra ------

constexpr int kIntraThreads = 128;
constexpr int kAS = 68;  // fp32 row stride of A / T
constexpr int kTS = 72;  // bf16 row stride of T (MMA operand)

template <int KP, bool PERKEY>
struct IntraLayout {
    static constexpr int KS = KP + 8;
    static constexpr size_t q = 0;
    static constexpr size_t k = q + 2 * kChunk * KS;
    static constexpr size_t gates = k + 2 * kChunk * KS;
    static constexpr size_t beta = gates + 4 * (PERKEY ? kChunk * KP : kChunk);
    static constexpr size_t a = beta + 4 * kChunk;
    static constexpr size_t t = a + 4 * kChunk * kAS;
    static constexpr size_t tb = t + 4 * kChunk * kAS;
    static constexpr size_t scratch = tb + 2 * kChunk * kTS;
    static size_t scratch_bytes(int VP) {
        size_t s1 = PERKEY ? (size_t)3 * 2 * kChunk * KS : 0;
        size_t s2 = (size_t)2 * kChunk * (VP + 8);
        size_t s3 = (size_t)4 * 4 * 16 * 17;
        size_t m = s1 > s2 ? s1 : s2;
        return m > s3 ? m : s3;
    }
    static size_t bytes(int VP) { return scratch + scratch_bytes(VP); }
};

__device__ __forceinline__ void unpack8(const uint4 &u, float *f) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}
__device__ __forceinline__ uint4 pack8(const float *f) {
    uint4 u;
    u.x = pack_bf16(f[0], f[1]);
    u.y = pack_bf16(f[2], f[3]);
    u.z = pack_bf16(f[4], f[5]);
    u.w = pack_bf16(f[6], f[7]);
    return u;
}

template <int KP, bool PERKEY>
__global__ void __launch_bounds__(kIntraThreads) intra_bf16_kernel(const FwdParams p, int VP) {
    using Lay = IntraLayout<KP, PERKEY>;
    constexpr int KS = Lay::KS;
    constexpr int VPR = KP / 8;  // 16-byte vectors per q/k row
    extern __shared__ __align__(16) unsigned char smraw[];
    bf16 *sQ = reinterpret_cast<bf16 *>(smraw + Lay::q);
    bf16 *sK = reinterpret_cast<bf16 *>(smraw + Lay::k);
    float *sG = reinterpret_cast<float *>(smraw + Lay::gates);  // [64] or [64][KP]
    float *sBeta = reinterpret_cast<float *>(smraw + Lay::beta);
    float *sA = reinterpret_cast<float *>(smraw + Lay::a);
    float *sT = reinterpret_cast<float *>(smraw + Lay::t);
    bf16 *sTb = reinterpret_cast<bf16 *>(smraw + Lay::tb);
    unsigned char *sScr = smraw + Lay::scratch;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, t4 = lane & 3;
    const int gid = blockIdx.x, hh = blockIdx.y;
    int s, c;
    if (p.cu_seqlens) {
        if (gid >= *p.n_chunks) return;
        const int2 e = p.chunk_tab[gid];
        s = e.x;
        c = e.y;
    } else {
        const int nts = (p.T + kChunk - 1) / kChunk;
        s = gid / nts;
        c = gid - s * nts;
        if (s >= p.n_seq) return;
    }
    SeqInfo si;
    if (!seq_info(p, s, si)) return;
    const int pos0 = c * kChunk;
    const int Lc = min(kChunk, si.len - pos0);
    if (Lc <= 0) return;
    const int K = p.K, H = p.H, V = p.V;
    const int64_t rowL = si.row0 + pos0;  // first intermediate row of the chunk
    const int64_t hrow = (int64_t)hh * p.rows + rowL;
    const bf16 *q = (const bf16 *)p.q, *k = (const bf16 *)p.k, *v = (const bf16 *)p.v;

    // ---- 1. load q, k rows (zero padded to KP), beta and gates
    for (int e = tid; e < kChunk * VPR; e += kIntraThreads) {
        const int i = e / VPR, d = (e % VPR) * 8;
        uint4 zq = make_uint4(0, 0, 0, 0), zk = zq;
        if (i < Lc && d < K) {
            const int tq = q_token(p.reverse, si.len, pos0 + i);
            const int tk = kv_token(p.reverse, si.len, pos0 + i);
            zq = *reinterpret_cast<const uint4 *>(q + si.b * p.qk_sb +
                                                  (int64_t)(si.tstart + tq) * p.qk_st +
                                                  hh * p.qk_sh + d);
            if (tk >= 0)
                zk = *reinterpret_cast<const uint4 *>(k + si.b * p.qk_sb +
                                                      (int64_t)(si.tstart + tk) * p.qk_st +
                                                      hh * p.qk_sh + d);
        }
        *reinterpret_cast<uint4 *>(sQ + i * KS + d) = zq;
        *reinterpret_cast<uint4 *>(sK + i * KS + d) = zk;
    }
    if (PERKEY) {
        for (int e = tid; e < kChunk * KP; e += kIntraThreads) {
            const int i = e / KP, d = e % KP;
            float x = 0.f;
            if (i < Lc && d < K) {
                const int tk = kv_token(p.reverse, si.len, pos0 + i);
                if (tk >= 0)
                    x = fmaxf(p.gk[((si.row0 + tk) * H + hh) * (int64_t)K + d],
                              kLogGateMinPerKeyTC);
            }
            sG[i * KP + d] = x;
        }
    }
    if (tid < kChunk) {
        const int i = tid;
        float b = 0.f, gg = 0.f;
        if (i < Lc) {
            const int tk = kv_token(p.reverse, si.len, pos0 + i);
            if (tk >= 0) {
                b = p.beta[(si.row0 + tk) * H + hh];
                if (!PERKEY) gg = fmaxf(p.g[(si.row0 + tk) * H + hh], kLogGateMin);
            }
        }
        sBeta[i] = b;
        if (!PERKEY) sG[i] = gg;
    }
    __syncthreads();

    // ---- 2. optional L2 normalisation of q and k rows; in-chunk gate cumsum
    if (p.l2norm) {
        for (int r = warp; r < 2 * kChunk; r += kIntraThreads / 32) {
            bf16 *row = (r < kChunk) ? (sQ + r * KS) : (sK + (r - kChunk) * KS);
            float2 f[KP / 64];
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < KP / 64; ++j) {
                f[j] = __bfloat1622float2(
                    *reinterpret_cast<const __nv_bfloat162 *>(row + 2 * lane + 64 * j));
                ss += f[j].x * f[j].x + f[j].y * f[j].y;
            }
            ss = warp_sum(ss);
            const float inv = rsqrtf(ss + 1e-6f);
#pragma unroll
            for (int j = 0; j < KP / 64; ++j)
                *reinterpret_cast<__nv_bfloat162 *>(row + 2 * lane + 64 * j) =
                    __floats2bfloat162_rn(f[j].x * inv, f[j].y * inv);
        }
    }
    if (PERKEY) {
        for (int d = tid; d < KP; d += kIntraThreads) {
            float acc = 0.f;
            for (int i = 0; i < kChunk; ++i) {
                acc += sG[i * KP + d];
                sG[i * KP + d] = acc;
            }
        }
    } else if (warp == 0) {
        const float a0 = sG[2 * lane], a1 = sG[2 * lane + 1];
        float incl = a0 + a1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const float excl = incl - (a0 + a1);
        sG[2 * lane] = excl + a0;
        sG[2 * lane + 1] = incl;
    }
    __syncthreads();

    // P rows of this chunk (64 columns) go straight to global memory; A
    // (strictly lower, beta-scaled) stays in shared memory. Column blocks
    // right of the diagonal block are never written nor read.
    bf16 *gP = p.aqk + hrow * kChunk;

    // ---- 3. A and P
    if (!PERKEY) {
        float ak[8][4], ap[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) ak[n][e] = ap[n][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KP / 16; ++kk) {
            uint32_t aK[4], aQ[4];
            ldsm_x4(aK, sK + (16 * warp + (lane & 15)) * KS + kk * 16 + (lane >> 4) * 8);
            ldsm_x4(aQ, sQ + (16 * warp + (lane & 15)) * KS + kk * 16 + (lane >> 4) * 8);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                if (np <= warp) {
                    uint32_t b[4];
                    ldsm_x4(b, sK + (16 * np + (lane & 7) + ((lane >> 4) << 3)) * KS + kk * 16 +
                                   ((lane >> 3) & 1) * 8);
                    mma_bf16(ak[2 * np], aK, b[0], b[1]);
                    mma_bf16(ak[2 * np + 1], aK, b[2], b[3]);
                    mma_bf16(ap[2 * np], aQ, b[0], b[1]);
                    mma_bf16(ap[2 * np + 1], aQ, b[2], b[3]);
                }
            }
        }
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            if (n < 2 * (warp + 1)) {
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int i = 16 * warp + g8 + 8 * hf;
                    const int j = 8 * n + 2 * t4;
                    float pv[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int jj = j + e;
                        const float gam = (jj <= i) ? __expf(sG[i] - sG[jj]) : 0.f;
                        if (jj < i) sA[i * kAS + jj] = sBeta[i] * ak[n][2 * hf + e] * gam;
                        pv[e] = ap[n][2 * hf + e] * gam;
                    }
                    if (i < Lc)
                        *reinterpret_cast<uint32_t *>(gP + (int64_t)i * kChunk + j) =
                            pack_bf16(pv[0], pv[1]);
                }
            }
        }
    } else {
        // Per-key gate: Gamma_ij = e^{G_i - G_j} per key channel. For column
        // block J split it about the block's middle row r = 16J + 8:
        //   left  x_i . e^{G_i - G_r}   (rows i >= 16J)
        //   right k_j . e^{G_r - G_j}   (rows j of block J)
        // Each factor spans at most 8 tokens of decay, so with the -10 floor
        // it stays below e^80; entries with j > i are discarded, not used.
        bf16 *sR = reinterpret_cast<bf16 *>(sScr);
        bf16 *sLq = sR + kChunk * KS;
        bf16 *sLk = sLq + kChunk * KS;
        for (int e = tid; e < kChunk * KP; e += kIntraThreads) {
            const int i = e / KP, d = e % KP, r = (i & ~15) + 8;
            const float f = __expf(sG[r * KP + d] - sG[i * KP + d]);
            sR[i * KS + d] = __float2bfloat16_rn(bf16_to_f(sK[i * KS + d]) * f);
        }
        for (int J = 0; J < 4; ++J) {
            __syncthreads();
            const int r0 = 16 * J, r = r0 + 8;
            for (int e = tid; e < (kChunk - r0) * KP; e += kIntraThreads) {
                const int i = r0 + e / KP, d = e % KP;
                const float f = __expf(sG[i * KP + d] - sG[r * KP + d]);
                sLq[i * KS + d] = __float2bfloat16_rn(bf16_to_f(sQ[i * KS + d]) * f);
                sLk[i * KS + d] = __float2bfloat16_rn(bf16_to_f(sK[i * KS + d]) * f);
            }
            __syncthreads();
            if (warp >= J) {
                float ak[2][4], ap[2][4];
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) ak[n][e] = ap[n][e] = 0.f;
#pragma unroll
                for (int kk = 0; kk < KP / 16; ++kk) {
                    uint32_t aK[4], aQ[4], b[4];
                    ldsm_x4(aK, sLk + (16 * warp + (lane & 15)) * KS + kk * 16 + (lane >> 4) * 8);
                    ldsm_x4(aQ, sLq + (16 * warp + (lane & 15)) * KS + kk * 16 + (lane >> 4) * 8);
                    ldsm_x4(b, sR + (r0 + (lane & 7) + ((lane >> 4) << 3)) * KS + kk * 16 +
                                   ((lane >> 3) & 1) * 8);
                    mma_bf16(ak[0], aK, b[0], b[1]);
                    mma_bf16(ak[1], aK, b[2], b[3]);
                    mma_bf16(ap[0], aQ, b[0], b[1]);
                    mma_bf16(ap[1], aQ, b[2], b[3]);
                }
#pragma unroll
                for (int n = 0; n < 2; ++n) {
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int i = 16 * warp + g8 + 8 * hf;
                        const int j = r0 + 8 * n + 2 * t4;
                        float pv[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int jj = j + e;
                            if (jj < i) sA[i * kAS + jj] = sBeta[i] * ak[n][2 * hf + e];
                            pv[e] = (jj <= i) ? ap[n][2 * hf + e] : 0.f;
                        }
                        if (i < Lc)
                            *reinterpret_cast<uint32_t *>(gP + (int64_t)i * kChunk + j) =
                                pack_bf16(pv[0], pv[1]);
                    }
                }
            }
        }
    }
    __syncthreads();

    // ---- 4. T = (I + A)^{-1}, A strictly lower: blocked forward substitution
    {   // 4a. diagonal 16x16 blocks, one warp each, lane = column
        const int I = warp;
        if (lane < 16) {
            const int cc = lane;
            for (int r = 0; r < 16; ++r) {
                const int i = 16 * I + r;
                float val;
                if (r < cc) {
                    val = 0.f;
                } else if (r == cc) {
                    val = 1.f;
                } else {
                    float acc = 0.f;
                    for (int j = cc; j < r; ++j)
                        acc = fmaf(sA[i * kAS + 16 * I + j], sT[(16 * I + j) * kAS + 16 * I + cc],
                                   acc);
                    val = -acc;
                }
                sT[i * kAS + 16 * I + cc] = val;
            }
        }
    }
    __syncthreads();
    {   // 4b. off-diagonal blocks, one block diagonal at a time:
        //     T_IJ = -T_II * sum_{M=J}^{I-1} A_IM T_MJ
        float *sX = reinterpret_cast<float *>(sScr) + warp * 16 * 17;
        for (int dd = 1; dd < 4; ++dd) {
            const int I = warp, J = warp - dd;
            if (J >= 0) {
#pragma unroll 1
                for (int m = 0; m < 8; ++m) {
                    const int e = lane + 32 * m, r = e >> 4, cc = e & 15;
                    float acc = 0.f;
                    for (int M = J; M < I; ++M)
#pragma unroll 4
                        for (int j = 0; j < 16; ++j)
                            acc = fmaf(sA[(16 * I + r) * kAS + 16 * M + j],
                                       sT[(16 * M + j) * kAS + 16 * J + cc], acc);
                    sX[r * 17 + cc] = acc;
                }
                __syncwarp();
#pragma unroll 1
                for (int m = 0; m < 8; ++m) {
                    const int e = lane + 32 * m, r = e >> 4, cc = e & 15;
                    float acc = 0.f;
                    for (int j = 0; j <= r; ++j)
                        acc = fmaf(sT[(16 * I + r) * kAS + 16 * I + j], sX[j * 17 + cc], acc);
                    sT[(16 * I + r) * kAS + 16 * J + cc] = -acc;
                }
                __syncwarp();
            }
            __syncthreads();
        }
    }
    for (int e = tid; e < kChunk * kChunk; e += kIntraThreads) {
        const int i = e >> 6, j = e & 63;
        sTb[i * kTS + j] = __float2bfloat16_rn(j <= i ? sT[i * kAS + j] : 0.f);
    }

    // ---- 5a. qg, kg, dec to global; w operand (beta e^G k) in place in sK;
    //          beta-scaled value tile (+ ones column) into scratch
    const int last = Lc - 1;
    bf16 *gQg = p.qg + hrow * KP;
    bf16 *gKg = p.kg + hrow * KP;
    for (int e = tid; e < kChunk * VPR; e += kIntraThreads) {
        const int i = e / VPR, d0 = (e % VPR) * 8;
        float fq[8], fk[8], fw[8];
        unpack8(*reinterpret_cast<const uint4 *>(sQ + i * KS + d0), fq);
        unpack8(*reinterpret_cast<const uint4 *>(sK + i * KS + d0), fk);
        const float b = sBeta[i];
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            float eg, el;
            if (PERKEY) {
                const float Gi = sG[i * KP + d0 + x];
                eg = __expf(Gi);
                el = __expf(sG[last * KP + d0 + x] - Gi);
            } else {
                eg = __expf(sG[i]);
                el = __expf(sG[last] - sG[i]);
            }
            fw[x] = b * eg * fk[x];
            fq[x] *= eg;
            fk[x] *= el;
        }
        if (i < Lc) {
            *reinterpret_cast<uint4 *>(gQg + (int64_t)i * KP + d0) = pack8(fq);
            *reinterpret_cast<uint4 *>(gKg + (int64_t)i * KP + d0) = pack8(fk);
        }
        *reinterpret_cast<uint4 *>(sK + i * KS + d0) = pack8(fw);
    }
    for (int d = tid; d < KP; d += kIntraThreads)
        p.dec[((int64_t)hh * p.max_chunks + gid) * KP + d] =
            PERKEY ? __expf(sG[last * KP + d]) : __expf(sG[last]);
    bf16 *sVb = reinterpret_cast<bf16 *>(sScr);
    const int VSb = VP + 8;
    const int VPRv = VP / 8;
    for (int e = tid; e < kChunk * VPRv; e += kIntraThreads) {
        const int i = e / VPRv, c0 = (e % VPRv) * 8;
        float f[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) f[x] = 0.f;
        if (i < Lc) {
            const int tk = kv_token(p.reverse, si.len, pos0 + i);
            if (tk >= 0) {
                if (c0 + 8 <= V) {
                    unpack8(*reinterpret_cast<const uint4 *>(
                                v + si.b * p.v_sb + (int64_t)(si.tstart + tk) * p.v_st +
                                hh * p.v_sh + c0),
                            f);
                } else if (p.has_den && c0 == V) {
                    f[0] = 1.f;
                }
                const float b = sBeta[i];
#pragma unroll
                for (int x = 0; x < 8; ++x) f[x] *= b;
            }
        }
        *reinterpret_cast<uint4 *>(sVb + i * VSb + c0) = pack8(f);
    }
    __syncthreads();

    // ---- 5b. w = T (beta e^G K), u = T (beta V); T is lower triangular so
    //          row block `warp` only needs column blocks 0..warp.
    auto tri_gemm = [&](const bf16 *sB, int ldb, int ncols, bf16 *gdst, int ldd, int ncols_out) {
        for (int ng = 0; ng < ncols; ng += 64) {
            float acc[8][4];
#pragma unroll
            for (int n = 0; n < 8; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                if (kk <= warp) {
                    uint32_t a[4];
                    ldsm_x4(a, sTb + (16 * warp + (lane & 15)) * kTS + 16 * kk + (lane >> 4) * 8);
#pragma unroll
                    for (int np = 0; np < 4; ++np) {
                        uint32_t b[4];
                        ldsm_x4_t(b, sB + (16 * kk + (lane & 15)) * ldb + ng + 16 * np +
                                         (lane >> 4) * 8);
                        mma_bf16(acc[2 * np], a, b[0], b[1]);
                        mma_bf16(acc[2 * np + 1], a, b[2], b[3]);
                    }
                }
            }
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                const int col = ng + 8 * n + 2 * t4;
                if (col < ncols_out) {
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int i = 16 * warp + g8 + 8 * hf;
                        if (i < Lc)
                            *reinterpret_cast<uint32_t *>(gdst + (int64_t)i * ldd + col) =
                                pack_bf16(acc[n][2 * hf], acc[n][2 * hf + 1]);
                    }
                }
            }
        }
    };
    tri_gemm(sK, KS, KP, p.w + hrow * KP, KP, KP);
    tri_gemm(sVb, VSb, VP, p.u + hrow * p.UW, p.UW, p.UW);
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

template <int KP, bool PERKEY>
cudaError_t launch_intra_t(const FwdParams &p, cudaStream_t st) {
    using Lay = IntraLayout<KP, PERKEY>;
    const int VP = (p.Vt + 63) / 64 * 64;
    const size_t bytes = Lay::bytes(VP);
    auto kern = intra_bf16_kernel<KP, PERKEY>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    dim3 grid(p.max_chunks, p.H);
    kern<<<grid, kIntraThreads, bytes, st>>>(p, VP);
    return cudaGetLastError();
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

cudaError_t launch_intra_bf16(const FwdParams &p, int KP, int perkey, cudaStream_t st) {
    if (p.max_chunks == 0) return cudaSuccess;
    if (KP == 64) return perkey ? launch_intra_t<64, true>(p, st) : launch_intra_t<64, false>(p, st);
    return perkey ? launch_intra_t<128, true>(p, st) : launch_intra_t<128, false>(p, st);
}

cudaError_t launch_state_bf16(const FwdParams &p, int KP, cudaStream_t st) {
    if (KP == 64) return launch_state_t<64>(p, st);
    return launch_state_t<128>(p, st);
}

}  // namespace gdn
