// gdn_intra_bf16.cu -- intra-chunk WY kernel of the bf16 tensor-core path.
//
// One CTA (4 warps) per (64-token chunk, head), all chunks in parallel. From
// the chunk's raw q, k, v, beta and log gates it produces, in the workspace:
//   w  = T (beta e^{G} . k^)      u = T (beta . V)          (T = (I + A)^{-1})
//   P  = lower_incl(q^ k^T . Gamma)                      (intra-chunk output)
//   qg = e^{G} . q^,  kg = e^{G_last - G} . k^,  dec = e^{G_last}
// with A = strictly_lower(diag(beta) (k^ k^T . Gamma)), Gamma_ij = e^{G_i-G_j}
// (per key channel for gk), and q^, k^ the L2-normalised rows (when asked).
// The hyper-parallel coverage_diff page consumes these factors
// (`chunk_kda_fwd_intra` returns w, u, kg, Aqk, Akk) but does not show how
// they are built; this construction is derived from the token recurrence
// (SANA `fused_gdn.py` page, `_fused_gdn_kernel` Pass 1).
//
// Steps:
//  1. cp.async every tile (q, k, v rows -- remapped for the reverse scan --
//     and the gk tile); scalars (beta, g) load meanwhile.
//  2. Row norms r = 1/sqrt(|x|^2 + 1e-6) as per-row scalars (the tiles stay
//     raw); in-chunk cumulative gates.
//  3. K K^T and Q K^T on tensor cores (mma.sync bf16 -> fp32), scaled by the
//     norms, beta and Gamma: A's diagonal 16x16 blocks in fp32, its other
//     blocks in bf16, P straight to its global image.
//  4. Each warp inverts one diagonal block, T_II = (I + A_II)^{-1}, by
//     forward substitution in registers (lane = column).
//  5. (I + A) W = X is solved by block forward substitution,
//     W_I = T_II (X_I - sum_{M<I} A_IM W_M), for X = [beta e^G k^ | beta V].
//     Every warp owns 64-column slices of W, so the four block steps need no
//     block-wide barrier; W overwrites X in shared memory.
//  6. 16-byte stores of w and u.
// Every output is written as a per-chunk image in the shared-memory operand
// layout the state kernel's tensor-core MMAs read (gdn_common.cuh), all 64
// rows included (zeros past the chunk's end), so the state kernel stages each
// one with a single bulk copy.
#include "gdn_common.cuh"

namespace gdn {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kThreads = 128;
constexpr int kAbS = 72;  // bf16 row stride of A (MMA operand) and of warp scratch
constexpr int kAdS = 17;  // fp32 row stride of A's diagonal blocks
constexpr int kTdS = 24;  // bf16 row stride of T's diagonal blocks

template <bool PERKEY>
struct Lay {
    static constexpr int KP = kKP;
    static constexpr int KS = KP + 8;
    static constexpr size_t q = 0;
    static constexpr size_t k = q + 2 * kChunk * KS;
    static constexpr size_t gates = k + 2 * kChunk * KS;
    static constexpr size_t beta = gates + 4 * (PERKEY ? kChunk * KP : kChunk);
    static constexpr size_t rq = beta + 4 * kChunk;
    static constexpr size_t rk = rq + 4 * kChunk;
    static constexpr size_t ab = rk + 4 * kChunk;
    static constexpr size_t ad = ab + 2 * kChunk * kAbS;
    static constexpr size_t td = ad + 4 * 4 * 16 * kAdS;
    static constexpr size_t v = td + 2 * 4 * 16 * kTdS;
    // the value tile shares its space with the per-key operand scratch
    static size_t v_bytes(int VP) {
        const size_t a = (size_t)2 * kChunk * (VP + 8);
        const size_t b = PERKEY ? (size_t)3 * 2 * kChunk * KS : 0;
        return a > b ? a : b;
    }
    static size_t bytes(int VP) { return v + v_bytes(VP); }
};

__device__ __forceinline__ void unpack8(const uint4 &u, float *f) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(h[i]);
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
__device__ __forceinline__ float2 ld_bf2(const bf16 *p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
}

template <bool PERKEY>
__global__ void __launch_bounds__(kThreads) intra_kernel(const FwdParams p, int VP) {
    using L = Lay<PERKEY>;
    constexpr int KP = kKP;
    constexpr int KS = L::KS;
    constexpr int VPR = KP / 8;  // 16-byte vectors per q/k row
    extern __shared__ __align__(16) unsigned char sm[];
    bf16 *sQ = reinterpret_cast<bf16 *>(sm + L::q);
    bf16 *sK = reinterpret_cast<bf16 *>(sm + L::k);
    float *sG = reinterpret_cast<float *>(sm + L::gates);  // [64] or [64][KP]
    float *sB = reinterpret_cast<float *>(sm + L::beta);
    float *sRq = reinterpret_cast<float *>(sm + L::rq);
    float *sRk = reinterpret_cast<float *>(sm + L::rk);
    bf16 *sAb = reinterpret_cast<bf16 *>(sm + L::ab);
    float *sAd = reinterpret_cast<float *>(sm + L::ad);
    bf16 *sTd = reinterpret_cast<bf16 *>(sm + L::td);
    bf16 *sV = reinterpret_cast<bf16 *>(sm + L::v);
    const int VS = VP + 8;

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
    const size_t gch = (size_t)hh * p.max_chunks + gid;  // this chunk's image slot
    const bf16 *q = (const bf16 *)p.q, *k = (const bf16 *)p.k, *v = (const bf16 *)p.v;
    const int64_t qk_base = si.b * p.qk_sb + hh * p.qk_sh;
    const int64_t v_base = si.b * p.v_sb + hh * p.v_sh;

    // ---- 1. asynchronous tile loads (zero fill outside the chunk / K / V)
    for (int e = tid; e < kChunk * VPR; e += kThreads) {
        const int i = e / VPR, d = (e % VPR) * 8;
        const int tq = i < Lc ? q_token(p.reverse, si.len, pos0 + i) : -1;
        const int tk = i < Lc ? kv_token(p.reverse, si.len, pos0 + i) : -1;
        const bool okq = tq >= 0 && d < K, okk = tk >= 0 && d < K;
        cp_async16(sQ + i * KS + d, okq ? (const void *)(q + qk_base + (int64_t)(si.tstart + tq) * p.qk_st + d) : (const void *)q,
                   okq ? 16 : 0);
        cp_async16(sK + i * KS + d, okk ? (const void *)(k + qk_base + (int64_t)(si.tstart + tk) * p.qk_st + d) : (const void *)k,
                   okk ? 16 : 0);
    }
    if (PERKEY) {
        for (int e = tid; e < kChunk * (KP / 4); e += kThreads) {
            const int i = e / (KP / 4), d = (e % (KP / 4)) * 4;
            const int tk = i < Lc ? kv_token(p.reverse, si.len, pos0 + i) : -1;
            const bool ok = tk >= 0 && d < K;
            cp_async16(sG + i * KP + d,
                       ok ? (const void *)(p.gk + ((si.row0 + tk) * H + hh) * (int64_t)K + d) : (const void *)p.gk,
                       ok ? 16 : 0);
        }
    }
    auto load_v = [&]() {
        const int VPRv = VP / 8;
        for (int e = tid; e < kChunk * VPRv; e += kThreads) {
            const int i = e / VPRv, c0 = (e % VPRv) * 8;
            const int tk = i < Lc ? kv_token(p.reverse, si.len, pos0 + i) : -1;
            const bool ok = tk >= 0 && c0 + 8 <= V;
            cp_async16(sV + i * VS + c0,
                       ok ? (const void *)(v + v_base + (int64_t)(si.tstart + tk) * p.v_st + c0) : (const void *)v,
                       ok ? 16 : 0);
        }
    };
    if (!PERKEY) load_v();
    cp_async_commit();
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
        sB[i] = b;
        if (!PERKEY) sG[i] = gg;
    }
    cp_async_wait<0>();
    __syncthreads();

    // ---- 2. row norms (as scalars) and in-chunk cumulative gates
    {
        const int r = tid & 63;
        const bf16 *row = (tid < 64 ? sQ : sK) + r * KS;
        float ss = 0.f;
#pragma unroll
        for (int d = 0; d < KP; d += 8) {
            float f[8];
            unpack8(*reinterpret_cast<const uint4 *>(row + d), f);
#pragma unroll
            for (int x = 0; x < 8; ++x) ss = fmaf(f[x], f[x], ss);
        }
        (tid < 64 ? sRq : sRk)[r] = p.l2norm ? rsqrtf(ss + 1e-6f) : 1.f;
    }
    if (PERKEY) {
        for (int d = tid; d < KP; d += kThreads) {
            float acc = 0.f;
#pragma unroll 8
            for (int i = 0; i < kChunk; ++i) {
                acc += fmaxf(sG[i * KP + d], kLogGateMinPerKeyTC);
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
        sG[2 * lane] = incl - a1;
        sG[2 * lane + 1] = incl;
    }
    __syncthreads();

    // ---- 3. A (strictly lower, beta-scaled) and P (lower incl. diagonal)
    unsigned char *gP = p.p_img + gch * kImgP;
    auto put_p = [&](int i, int j, float v0f, float v1f) {
        *reinterpret_cast<uint32_t *>(gP + img_p_off(i, j)) = pack_bf16(v0f, v1f);
    };
    // store one A entry: diagonal block -> fp32, below -> bf16 operand
    auto put_a = [&](int i, int j, float a) {
        const int I = i >> 4;
        if (j >= 16 * I)
            sAd[(I * 16 + (i & 15)) * kAdS + (j & 15)] = a;
        else
            sAb[i * kAbS + j] = __float2bfloat16_rn(a);
    };
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
                    const float Gi = sG[i], bi = sB[i], rki = sRk[i], rqi = sRq[i];
                    float pv[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int jj = j + e;
                        const float gam = (jj <= i) ? __expf(Gi - sG[jj]) * sRk[jj] : 0.f;
                        if (jj < i) put_a(i, jj, bi * rki * ak[n][2 * hf + e] * gam);
                        pv[e] = rqi * ap[n][2 * hf + e] * gam;
                    }
                    put_p(i, j, pv[0], pv[1]);
                }
            } else {  // right of the diagonal block: the image must hold zeros
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) put_p(16 * warp + g8 + 8 * hf, 8 * n + 2 * t4, 0.f, 0.f);
            }
        }
    } else {
        // Per-key gate: for column block J split e^{G_i - G_j} about the
        // block's middle row r = 16J + 8: left x_i^ . e^{G_i - G_r} (rows
        // i >= 16J), right k_j^ . e^{G_r - G_j} (rows of block J). Each factor
        // spans at most 8 tokens of decay, so with the -10 floor it stays
        // below e^80; entries with j > i are discarded, never used.
        bf16 *sR = sV;
        bf16 *sLq = sR + kChunk * KS;
        bf16 *sLk = sLq + kChunk * KS;
        for (int e = tid; e < kChunk * KP; e += kThreads) {
            const int i = e / KP, d = e % KP, r = (i & ~15) + 8;
            const float f = __expf(sG[r * KP + d] - sG[i * KP + d]) * sRk[i];
            sR[i * KS + d] = __float2bfloat16_rn(__bfloat162float(sK[i * KS + d]) * f);
        }
        for (int J = 0; J < 4; ++J) {
            __syncthreads();
            const int r0 = 16 * J, r = r0 + 8;
            for (int e = tid; e < (kChunk - r0) * KP; e += kThreads) {
                const int i = r0 + e / KP, d = e % KP;
                const float f = __expf(sG[i * KP + d] - sG[r * KP + d]);
                sLq[i * KS + d] = __float2bfloat16_rn(__bfloat162float(sQ[i * KS + d]) * f * sRq[i]);
                sLk[i * KS + d] = __float2bfloat16_rn(__bfloat162float(sK[i * KS + d]) * f * sRk[i]);
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
                            if (jj < i) put_a(i, jj, sB[i] * ak[n][2 * hf + e]);
                            pv[e] = (jj <= i) ? ap[n][2 * hf + e] : 0.f;
                        }
                        put_p(i, j, pv[0], pv[1]);
                    }
                }
            } else {  // column block right of this warp's diagonal: zeros
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) put_p(16 * warp + g8 + 8 * hf, r0 + 8 * n + 2 * t4, 0.f, 0.f);
            }
        }
    }
    __syncthreads();
    if (PERKEY) {  // the operand scratch is free: bring in the value tile now
        load_v();
        cp_async_commit();
    }

    // ---- 4. T_II = (I + A_II)^{-1} for the diagonal block of this warp;
    //         lane c < 16 holds column c: t = e_c, t_r = -sum_{j<r} A_rj t_j
    {
        const int I = warp, cc = lane & 15;
        const float *Ad = sAd + I * 16 * kAdS;
        float t[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) t[r] = (r == cc) ? 1.f : 0.f;
#pragma unroll
        for (int r = 1; r < 16; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < r; ++j) acc = fmaf(Ad[r * kAdS + j], t[j], acc);
            if (r > cc) t[r] = -acc;
        }
        if (lane < 16) {
#pragma unroll
            for (int r = 0; r < 16; ++r) sTd[(I * 16 + r) * kTdS + cc] = __float2bfloat16_rn(t[r]);
        }
    }

    //         qg, kg and the chunk decay to global
    const int last = Lc - 1;
    unsigned char *gQg = p.qg_img + gch * kImgW;
    unsigned char *gKg = p.kg_img + gch * kImgW;
    for (int e = tid; e < kChunk * VPR; e += kThreads) {
        const int i = e / VPR, d0 = (e % VPR) * 8;
        float fq[8], fk[8];
        unpack8(*reinterpret_cast<const uint4 *>(sQ + i * KS + d0), fq);
        unpack8(*reinterpret_cast<const uint4 *>(sK + i * KS + d0), fk);
        const float rq = sRq[i], rk = sRk[i];
        if (PERKEY) {
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                const float Gi = sG[i * KP + d0 + x];
                fq[x] *= __expf(Gi) * rq;
                fk[x] *= __expf(sG[last * KP + d0 + x] - Gi) * rk;
            }
        } else {
            const float eq = __expf(sG[i]) * rq, ek = __expf(sG[last] - sG[i]) * rk;
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                fq[x] *= eq;
                fk[x] *= ek;
            }
        }
        *reinterpret_cast<uint4 *>(gQg + img_w_off(i, d0)) = pack8(fq);
        *reinterpret_cast<uint4 *>(gKg + img_kt_off(i, d0)) = pack8(fk);
    }
    for (int d = tid; d < KP; d += kThreads)
        p.dec[gch * KP + d] =
            PERKEY ? __expf(sG[last * KP + d]) : __expf(sG[last]);
    if (PERKEY) cp_async_wait<0>();
    __syncthreads();

    // ---- 5. W_I = T_II (X_I - sum_{M<I} A_IM W_M), per 64-column slice
    bf16 *scratch = sQ + warp * 16 * kAbS;  // q tile is no longer needed
    const int nsw = KP / 64, nsu = VP / 64;
    for (int sl = warp; sl < nsw + nsu; sl += kThreads / 32) {
        const bool isw = sl < nsw;
        bf16 *tile = isw ? sK : sV;
        const int ts = isw ? KS : VS;
        const int c0 = isw ? 64 * sl : 64 * (sl - nsw);
#pragma unroll 1
        for (int I = 0; I < 4; ++I) {
            float acc[8][4];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int i = 16 * I + g8 + 8 * hf;
                const float bi = sB[i];
                const float srow = isw ? (PERKEY ? bi * sRk[i] : bi * sRk[i] * __expf(sG[i])) : bi;
#pragma unroll
                for (int n = 0; n < 8; ++n) {
                    const int col = c0 + 8 * n + 2 * t4;
                    float2 x = ld_bf2(tile + i * ts + col);
                    if (!isw && p.has_den) {
                        if (col == V) x.x = 1.f;
                        if (col + 1 == V) x.y = 1.f;
                    }
                    float s0 = srow, s1 = srow;
                    if (isw && PERKEY) {
                        s0 *= __expf(sG[i * KP + col]);
                        s1 *= __expf(sG[i * KP + col + 1]);
                    }
                    acc[n][2 * hf] = x.x * s0;
                    acc[n][2 * hf + 1] = x.y * s1;
                }
            }
#pragma unroll
            for (int M = 0; M < 3; ++M) {
                if (M < I) {
                    uint32_t a[4];
                    ldsm_x4(a, sAb + (16 * I + (lane & 15)) * kAbS + 16 * M + (lane >> 4) * 8);
#pragma unroll
                    for (int x = 0; x < 4; ++x) a[x] ^= 0x80008000u;  // -A
#pragma unroll
                    for (int np = 0; np < 4; ++np) {
                        uint32_t b[4];
                        ldsm_x4_t(b, tile + (16 * M + (lane & 15)) * ts + c0 + 16 * np + (lane >> 4) * 8);
                        mma_bf16(acc[2 * np], a, b[0], b[1]);
                        mma_bf16(acc[2 * np + 1], a, b[2], b[3]);
                    }
                }
            }
#pragma unroll
            for (int n = 0; n < 8; ++n)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
                    *reinterpret_cast<uint32_t *>(scratch + (g8 + 8 * hf) * kAbS + 8 * n + 2 * t4) =
                        pack_bf16(acc[n][2 * hf], acc[n][2 * hf + 1]);
            __syncwarp();
            float wa[8][4];
#pragma unroll
            for (int n = 0; n < 8; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) wa[n][e] = 0.f;
            uint32_t a[4];
            ldsm_x4(a, sTd + (16 * I + (lane & 15)) * kTdS + (lane >> 4) * 8);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t b[4];
                ldsm_x4_t(b, scratch + (lane & 15) * kAbS + 16 * np + (lane >> 4) * 8);
                mma_bf16(wa[2 * np], a, b[0], b[1]);
                mma_bf16(wa[2 * np + 1], a, b[2], b[3]);
            }
#pragma unroll
            for (int n = 0; n < 8; ++n)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
                    *reinterpret_cast<uint32_t *>(tile + (16 * I + g8 + 8 * hf) * ts + c0 + 8 * n + 2 * t4) =
                        pack_bf16(wa[n][2 * hf], wa[n][2 * hf + 1]);
            __syncwarp();
        }
    }
    __syncthreads();

    // ---- 6. w and u images (all 64 rows; rows past the chunk are zero)
    unsigned char *gW = p.w_img + gch * kImgW;
    for (int e = tid; e < kChunk * VPR; e += kThreads) {
        const int i = e / VPR, d = (e % VPR) * 8;
        *reinterpret_cast<uint4 *>(gW + img_w_off(i, d)) = *reinterpret_cast<const uint4 *>(sK + i * KS + d);
    }
    unsigned char *gU = p.u_img + gch * p.n_vt * kImgU;
    const int VPRv = VP / 8;
    for (int e = tid; e < kChunk * VPRv; e += kThreads) {
        const int i = e / VPRv, c = (e % VPRv) * 8;
        *reinterpret_cast<uint4 *>(gU + (c >> 6) * kImgU + i * (kUS * 2) + (c & 63) * 2) =
            *reinterpret_cast<const uint4 *>(sV + i * VS + c);
    }
}

template <bool PERKEY>
cudaError_t launch_t(const FwdParams &p, cudaStream_t st) {
    using L = Lay<PERKEY>;
    const int VP = p.n_vt * 64;
    const size_t bytes = L::bytes(VP);
    auto kern = intra_kernel<PERKEY>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    dim3 grid(p.max_chunks, p.H);
    kern<<<grid, kThreads, bytes, st>>>(p, VP);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_intra_bf16(const FwdParams &p, int perkey, cudaStream_t st) {
    if (p.max_chunks == 0) return cudaSuccess;
    return perkey ? launch_t<true>(p, st) : launch_t<false>(p, st);
}

}  // namespace gdn
