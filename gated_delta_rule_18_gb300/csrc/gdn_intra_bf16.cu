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
//  1. One bulk async copy per q / k row (and gk row), remapped for the
//     reverse scan, counted on an mbarrier; rows with no token are zeroed.
//  2. K K^T and Q K^T on tensor cores (mma.sync bf16 -> fp32). Scalar gate:
//     the squared row norms come from the diagonals of K K^T and of an extra
//     Q Q^T diagonal block, and the in-chunk gate cumsum runs meanwhile.
//     Per-key gate: norms and per-channel cumsums first, then the split
//     products (below).
//  3. Scaling by the norms, beta and Gamma: A's diagonal 16x16 blocks in fp32,
//     its six blocks below the diagonal in bf16, P straight to its image.
//  4. qg / kg images and the chunk decay. The value tile is then copied in
//     (scalar gate: into the q tile's space, now free) while each warp
//     inverts one diagonal block, T_II = (I + A_II)^{-1}, by forward
//     substitution in registers (lane = column).
//  5. (I + A) W = X is solved by block forward substitution,
//     W_I = T_II (X_I - sum_{M<I} A_IM W_M), for X = [beta e^G k^ | beta V].
//     The row scales of X are folded into T's columns and B_IM = -T_II A_IM
//     is formed once per block, so W_I = T_II diag(s_I) X~_I + sum B_IM W_M
//     with X~ the raw tile. Every warp owns 64-column slices of W, writes each
//     solved W_I over X~_I in shared memory (the operand of later blocks) and
//     straight to its global image; the solve needs no block-wide barrier.
// Every output is written as a per-chunk image in the shared-memory operand
// layout the state kernel's tensor-core MMAs read (gdn_common.cuh), all 64
// rows included (zeros past the chunk's end), so the state kernel stages each
// one with a single bulk copy.
//
// Every wait on a copy is bounded (about 0.5 s); a wait that gives up sets
// GDN_DEVERR_TIMEOUT in the error word and the CTA leaves after a second
// bounded wait for its copies in flight.
#include "gdn_common.cuh"

namespace gdn {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kThreads = 128;
constexpr int kBS = 24;   // bf16 row stride of a 16x16 block (A below the diagonal, T)
constexpr int kTSet = 4 * 16 * kBS;  // one set of T's four diagonal blocks
constexpr int kAdS = 17;  // fp32 row stride of A's diagonal blocks

// Shared memory. The scalar-gate kernel copies the value tile into the q
// tile's space once qg is written; the per-key kernel keeps it apart (its
// space first holds the two split operands of step 2) and puts T's blocks
// over its gate tile, so that two per-key CTAs fit on an SM.
template <bool PERKEY>
struct Lay {
    static constexpr int KP = kKP;
    static constexpr int KS = KP + 8;
    static constexpr size_t tile = (size_t)2 * kChunk * KS;
    static constexpr size_t k = 0;
    static constexpr size_t gates = k + tile;
    static constexpr size_t beta = gates + 4 * (PERKEY ? kChunk * KP : kChunk);
    static constexpr size_t rq = beta + 4 * kChunk;
    static constexpr size_t rk = rq + 4 * kChunk;
    static constexpr size_t ab = rk + 4 * kChunk;
    static constexpr size_t ad = ab + 2 * 6 * 16 * kBS;
    // per key, T's blocks take the gate tile's space once the gates are used up
    static constexpr size_t td = PERKEY ? gates : ad + 4 * 4 * 16 * kAdS;
    static constexpr size_t q = PERKEY ? ad + 4 * 4 * 16 * kAdS : td + 3 * 2 * kTSet;
    static size_t vtile(int VP) { return (size_t)2 * kChunk * (VP + 8); }
    static constexpr size_t v = PERKEY ? q + tile : q;
    static size_t bytes(int VP) {
        if (PERKEY) {
            const size_t a = vtile(VP), b = 2 * tile;
            return q + tile + (a > b ? a : b);
        }
        const size_t a = vtile(VP);
        return q + (a > tile ? a : tile);
    }
};

// index of A's block (I, M), M < I, among the six below the diagonal
__device__ __forceinline__ int blk(int I, int M) { return I * (I - 1) / 2 + M; }

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
constexpr float kLog2e = 1.4426950408889634f;
// 2^x (the per-key gates are kept in base 2)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ void ld8f(const float *p, float *f) {  // 16-byte aligned
    const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
    f[0] = a.x, f[1] = a.y, f[2] = a.z, f[3] = a.w, f[4] = b.x, f[5] = b.y, f[6] = b.z, f[7] = b.w;
}
__device__ __forceinline__ void zero_row(bf16 *row, int from, int to) {  // 8-aligned bounds
    for (int d = from; d < to; d += 8) *reinterpret_cast<uint4 *>(row + d) = make_uint4(0, 0, 0, 0);
}
// a bounded wait for a copy barrier; on time-out the error word is marked and
// the copies in flight get a second bounded window before the caller leaves
__device__ __forceinline__ bool wait_copies(uint32_t bar, int *err) {
    if (wait_bar(bar, 0, nullptr)) return true;
    atomicOr(err, kDevErrTimeout);
    wait_bar(bar, 0, nullptr);
    return false;
}

// STALL: the instantiation with the stall testing aid (launched only while it
// is on, so that the working kernel carries none of its code)
template <bool PERKEY, bool STALL>
__global__ void __launch_bounds__(PERKEY ? 2 * kThreads : kThreads, PERKEY ? 2 : 4)
    intra_kernel(const FwdParams p, int VP) {
    using L = Lay<PERKEY>;
    // the per-key kernel runs 8 warps: warps 0-3 own the 16-row blocks of the
    // products, all 8 share the elementwise passes and the solve's slices
    constexpr int NT = PERKEY ? 2 * kThreads : kThreads;
    constexpr int KP = kKP;
    constexpr int KS = L::KS;
    constexpr int VPR = KP / 8;  // 16-byte vectors per q/k row
    extern __shared__ __align__(16) unsigned char sm[];
    __shared__ __align__(8) uint64_t bar_qk, bar_v;
    bf16 *sQ = reinterpret_cast<bf16 *>(sm + L::q);
    bf16 *sK = reinterpret_cast<bf16 *>(sm + L::k);
    float *sG = reinterpret_cast<float *>(sm + L::gates);  // [64] or [64][KP]
    float *sB = reinterpret_cast<float *>(sm + L::beta);
    float *sRq = reinterpret_cast<float *>(sm + L::rq);
    float *sRk = reinterpret_cast<float *>(sm + L::rk);
    bf16 *sAb = reinterpret_cast<bf16 *>(sm + L::ab);
    float *sAd = reinterpret_cast<float *>(sm + L::ad);
    bf16 *sTd = reinterpret_cast<bf16 *>(sm + L::td);  // T_II, then T_II diag(s_w), T_II diag(beta)
    bf16 *sV = reinterpret_cast<bf16 *>(sm + L::v);
    const int VS = VP + 8;
    const uint32_t b_qk = smem_u32(&bar_qk), b_v = smem_u32(&bar_v);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, t4 = lane & 3;
    // heads vary fastest across the grid, so CTAs resident together read the
    // same tokens of all heads (whole DRAM pages) rather than one head's rows
    const int hh = blockIdx.x % p.H, gid = blockIdx.x / p.H;
    if (STALL && stall_test(p.stall_cta, p.stall_us, p.err)) return;
    int s, c, slot;  // slot: the chunk's image index within the head
    if (p.cu_seqlens) {
        if (gid >= *p.n_chunks) return;
        const int2 e = p.chunk_tab[gid];
        s = e.x;
        c = e.y;
        slot = gid;
    } else {
        // chunks in descending order over the grid, sequences next: the last
        // CTAs write every sequence's first chunks, which the state pass
        // reads first, so those images are still in L2 when it starts
        const int nts = (p.T + kChunk - 1) / kChunk;
        const int cr = gid / p.n_seq;
        s = gid - cr * p.n_seq;
        c = nts - 1 - cr;
        if (c < 0) return;
        slot = s * nts + c;
    }
    SeqInfo si;
    if (!seq_info(p, s, si)) return;
    const int pos0 = c * kChunk;
    const int Lc = min(kChunk, si.len - pos0);
    if (Lc <= 0) return;
    const int K = p.K, H = p.H, V = p.V;
    const size_t gch = (size_t)hh * p.max_chunks + slot;
    const bf16 *q = (const bf16 *)p.q, *k = (const bf16 *)p.k, *v = (const bf16 *)p.v;
    const int64_t qk_base = si.b * p.qk_sb + hh * p.qk_sh;
    const int64_t v_base = si.b * p.v_sb + hh * p.v_sh;

    if (tid == 0) {
        mbar_init(b_qk, kChunk);
        mbar_init(b_v, kChunk);
        fence_mbar_init();
    }
    __syncthreads();

    // ---- 1. row copies: thread i < 64 owns row i (its token, beta, gate)
    int tk_row = -1;
    if (tid < kChunk) {
        const int i = tid;
        const int tq = i < Lc ? q_token(p.reverse, si.len, pos0 + i) : -1;
        const int tk = i < Lc ? kv_token(p.reverse, si.len, pos0 + i) : -1;
        tk_row = tk;
        const uint32_t rowb = (uint32_t)K * 2;
        uint32_t bytes = (tq >= 0 ? rowb : 0) + (tk >= 0 ? rowb : 0);
        if (PERKEY && tk >= 0) bytes += (uint32_t)K * 4;
        arrive_expect_tx(b_qk, bytes);
        if (tq >= 0) bulk_g2s(smem_u32(sQ + i * KS), q + qk_base + (int64_t)(si.tstart + tq) * p.qk_st, rowb, b_qk);
        else zero_row(sQ + i * KS, 0, K);
        if (tk >= 0) {
            bulk_g2s(smem_u32(sK + i * KS), k + qk_base + (int64_t)(si.tstart + tk) * p.qk_st, rowb, b_qk);
            if (PERKEY) bulk_g2s(smem_u32(sG + i * KP), p.gk + ((si.row0 + tk) * H + hh) * (int64_t)K, K * 4, b_qk);
        } else {
            zero_row(sK + i * KS, 0, K);
            if (PERKEY)
                for (int d = 0; d < K; d += 4) *reinterpret_cast<float4 *>(sG + i * KP + d) = make_float4(0, 0, 0, 0);
        }
        if (K < KP) {  // padding keys
            zero_row(sQ + i * KS, K, KP);
            zero_row(sK + i * KS, K, KP);
            if (PERKEY)
                for (int d = K; d < KP; d += 4) *reinterpret_cast<float4 *>(sG + i * KP + d) = make_float4(0, 0, 0, 0);
        }
        float b = 0.f, gg = 0.f;
        if (tk >= 0) {
            b = p.beta[(si.row0 + tk) * H + hh];
            if (!PERKEY) gg = fmaxf(p.g[(si.row0 + tk) * H + hh], kLogGateMin);
        }
        sB[i] = b;
        if (!PERKEY) sG[i] = gg;
    }
    const bool copied = wait_copies(b_qk, p.err);
    if (__syncthreads_or(!copied)) return;

    // ---- 2./3. A (strictly lower, beta-scaled) and P (lower incl. diagonal)
    unsigned char *gP = p.p_img + gch * kImgP;
    auto put_p = [&](int i, int j, float v0f, float v1f) {
        *reinterpret_cast<uint32_t *>(gP + img_p_off(i, j)) = pack_bf16(v0f, v1f);
    };
    // store one A entry: diagonal block -> fp32, below -> bf16 operand block
    auto put_a = [&](int i, int j, float a) {
        const int I = i >> 4, M = j >> 4;
        if (M == I)
            sAd[(I * 16 + (i & 15)) * kAdS + (j & 15)] = a;
        else
            sAb[(blk(I, M) * 16 + (i & 15)) * kBS + (j & 15)] = __float2bfloat16_rn(a);
    };
    if (!PERKEY) {
        if (warp == 0) {  // in-chunk cumulative gates (exclusive of nothing: G_i includes g_i)
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
        float ak[8][4], ap[8][4], aq[2][4];
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) ak[n][e] = ap[n][e] = 0.f;
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) aq[n][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KP / 16; ++kk) {
            uint32_t aK[4], aQ[4];
            ldsm_x4(aK, sK + (16 * warp + (lane & 15)) * KS + kk * 16 + (lane >> 4) * 8);
            ldsm_x4(aQ, sQ + (16 * warp + (lane & 15)) * KS + kk * 16 + (lane >> 4) * 8);
            const int brow = (lane & 7) + ((lane >> 4) << 3), bcol = kk * 16 + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                if (np <= warp) {
                    uint32_t b[4];
                    ldsm_x4(b, sK + (16 * np + brow) * KS + bcol);
                    mma_bf16(ak[2 * np], aK, b[0], b[1]);
                    mma_bf16(ak[2 * np + 1], aK, b[2], b[3]);
                    mma_bf16(ap[2 * np], aQ, b[0], b[1]);
                    mma_bf16(ap[2 * np + 1], aQ, b[2], b[3]);
                }
            }
            uint32_t bq[4];  // Q Q^T, diagonal block only (the q norms)
            ldsm_x4(bq, sQ + (16 * warp + brow) * KS + bcol);
            mma_bf16(aq[0], aQ, bq[0], bq[1]);
            mma_bf16(aq[1], aQ, bq[2], bq[3]);
        }
        // row i = 16 warp + g8 + 8 hf sits on the diagonal in lane t4 = g8/2,
        // element 2 hf + (g8 & 1) of column group 2 warp + hf
        if (t4 == (g8 >> 1)) {
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                if (np == warp) {
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int i = 16 * warp + g8 + 8 * hf;
                        const float kk2 = (g8 & 1) ? ak[2 * np + hf][2 * hf + 1] : ak[2 * np + hf][2 * hf];
                        const float qq2 = (g8 & 1) ? aq[hf][2 * hf + 1] : aq[hf][2 * hf];
                        sRk[i] = p.l2norm ? rsqrtf(kk2 + 1e-6f) : 1.f;
                        sRq[i] = p.l2norm ? rsqrtf(qq2 + 1e-6f) : 1.f;
                    }
                }
            }
        }
        __syncthreads();
        // every scale factor first, then the stores (shared loads cannot be
        // moved across stores the compiler must assume may alias them)
        float Gi[2], ai[2], rqi[2];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int i = 16 * warp + g8 + 8 * hf;
            Gi[hf] = sG[i];
            ai[hf] = sB[i] * sRk[i];
            rqi[hf] = sRq[i];
        }
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            if (n < 2 * (warp + 1)) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int jj = 8 * n + 2 * t4 + e;
                    const float Gj = sG[jj], rkj = sRk[jj];
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int i = 16 * warp + g8 + 8 * hf;
                        const float gam = (jj <= i) ? __expf(Gi[hf] - Gj) * rkj : 0.f;
                        ak[n][2 * hf + e] = (jj < i) ? ai[hf] * ak[n][2 * hf + e] * gam : 0.f;
                        ap[n][2 * hf + e] = rqi[hf] * ap[n][2 * hf + e] * gam;
                    }
                }
            }
        }
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const bool on = n < 2 * (warp + 1);  // else right of the diagonal block: zeros
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int i = 16 * warp + g8 + 8 * hf, j = 8 * n + 2 * t4;
                put_p(i, j, on ? ap[n][2 * hf] : 0.f, on ? ap[n][2 * hf + 1] : 0.f);
                if (on) {
                    if ((n >> 1) == warp) {  // diagonal block, fp32 (entries j >= i are zero, unread)
                        float *d = sAd + (16 * warp + (i & 15)) * kAdS + (j & 15);
                        d[0] = ak[n][2 * hf];
                        d[1] = ak[n][2 * hf + 1];
                    } else {
                        *reinterpret_cast<uint32_t *>(sAb + (blk(warp, n >> 1) * 16 + (i & 15)) * kBS + (j & 15)) =
                            pack_bf16(ak[n][2 * hf], ak[n][2 * hf + 1]);
                    }
                }
            }
        }
    } else {
        // row norms as scalars (the tiles stay raw) on the upper 128 threads,
        // alongside the channel cumsums on the lower 128
        static_assert(!PERKEY || NT >= 2 * kChunk + KP, "norms and cumsums on separate threads");
        if (tid >= NT - 2 * kChunk) {
            const int t2 = tid - (NT - 2 * kChunk), r = t2 & 63;
            const bf16 *row = (t2 < 64 ? sQ : sK) + r * KS;
            float ss = 0.f;
#pragma unroll
            for (int d = 0; d < KP; d += 8) {
                float f[8];
                unpack8(*reinterpret_cast<const uint4 *>(row + d), f);
#pragma unroll
                for (int x = 0; x < 8; ++x) ss = fmaf(f[x], f[x], ss);
            }
            (t2 < 64 ? sRq : sRk)[r] = p.l2norm ? rsqrtf(ss + 1e-6f) : 1.f;
        }
        if (tid < KP) {  // per-channel cumsums: thread d keeps its channel's 64 gates in registers
            static_assert(kThreads == KP, "one thread per key channel");
            const int d = tid;
            float a[kChunk];
#pragma unroll
            for (int i = 0; i < kChunk; ++i) a[i] = fmaxf(sG[i * KP + d], kLogGateMinPerKeyTC);
#pragma unroll
            for (int i = 1; i < kChunk; ++i) a[i] += a[i - 1];
            // kept in base 2 (G log2 e): every factor below is then one ex2
#pragma unroll
            for (int i = 0; i < kChunk; ++i) sG[i * KP + d] = a[i] * kLog2e;
        }
        // Per-key gate: for column block J split e^{G_i - G_j} about the
        // block's middle row r = 16J + 8: left x_i^ . e^{G_i - G_r} (rows
        // i >= 16J), right k_j^ . e^{G_r - G_j} (rows of block J). Each factor
        // spans at most 8 tokens of decay, so with the -10 floor it stays
        // below e^80; entries with j > i are discarded, never used. Eight
        // channels per step (16-byte loads and stores).
        bf16 *sR = sV;                // right factors, all 64 rows
        bf16 *sL = sR + kChunk * KS;  // left factors of keys, then of queries
        __syncthreads();
        for (int e = tid; e < kChunk * (KP / 8); e += NT) {
            const int i = e / (KP / 8), d = (e % (KP / 8)) * 8, r = (i & ~15) + 8;
            float gi[8], gr[8], kx[8], o[8];
            ld8f(sG + i * KP + d, gi);
            ld8f(sG + r * KP + d, gr);
            unpack8(*reinterpret_cast<const uint4 *>(sK + i * KS + d), kx);
            const float rk = sRk[i];
#pragma unroll
            for (int x = 0; x < 8; ++x) o[x] = kx[x] * (ex2(gr[x] - gi[x]) * rk);
            *reinterpret_cast<uint4 *>(sR + i * KS + d) = pack8(o);
        }
        for (int J = 0; J < 4; ++J) {
            const int r0 = 16 * J, r = r0 + 8;
            float ak[2][4], ap[2][4];
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) ak[n][e] = ap[n][e] = 0.f;
            // this thread's items: (64 - r0) rows x 16 eight-channel groups
            // over the block, at most kItems each; the factors e^{G_i - G_r}
            // of the key pass stay in registers for the query pass
            constexpr int kItems = kChunk * (KP / 8) / NT;
            const int n_items = (kChunk - r0) * (KP / 8);
            float fct[kItems][8];
            // a thread's items all sit in one eight-channel group (NT is a
            // multiple of KP / 8), so the reference row's gates load once
            static_assert(NT % (KP / 8) == 0, "fixed channel group per thread");
            float gr[8];
            ld8f(sG + r * KP + (tid % (KP / 8)) * 8, gr);
#pragma unroll
            for (int pass = 0; pass < 2; ++pass) {  // 0: keys (A), 1: queries (P)
                __syncthreads();  // the previous product has read sL
                const bf16 *src = pass ? sQ : sK;
                const float *rs = pass ? sRq : sRk;
#pragma unroll
                for (int u = 0; u < kItems; ++u) {
                    const int e = tid + u * NT;
                    if (e >= n_items) break;
                    const int i = r0 + e / (KP / 8), d = (e % (KP / 8)) * 8;
                    if (pass == 0) {
                        float gi[8];
                        ld8f(sG + i * KP + d, gi);
#pragma unroll
                        for (int x = 0; x < 8; ++x) fct[u][x] = ex2(gi[x] - gr[x]);
                    }
                    float xx[8], o[8];
                    unpack8(*reinterpret_cast<const uint4 *>(src + i * KS + d), xx);
                    const float rr = rs[i];
#pragma unroll
                    for (int x = 0; x < 8; ++x) o[x] = xx[x] * fct[u][x] * rr;
                    *reinterpret_cast<uint4 *>(sL + i * KS + d) = pack8(o);
                }
                __syncthreads();
                if (warp < 4 && warp >= J) {
#pragma unroll
                    for (int kk = 0; kk < KP / 16; ++kk) {
                        uint32_t aL[4], b[4];
                        ldsm_x4(aL, sL + (16 * warp + (lane & 15)) * KS + kk * 16 + (lane >> 4) * 8);
                        ldsm_x4(b, sR + (r0 + (lane & 7) + ((lane >> 4) << 3)) * KS + kk * 16 +
                                       ((lane >> 3) & 1) * 8);
                        float(&acc)[2][4] = pass ? ap : ak;
                        mma_bf16(acc[0], aL, b[0], b[1]);
                        mma_bf16(acc[1], aL, b[2], b[3]);
                    }
                }
            }
            if (warp < 4 && warp >= J) {
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
            } else if (warp < 4) {  // column block right of this warp's diagonal: zeros
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) put_p(16 * warp + g8 + 8 * hf, r0 + 8 * n + 2 * t4, 0.f, 0.f);
            }
        }
    }
    __syncthreads();

    // ---- 4. qg, kg and the chunk decay to global
    const int last = Lc - 1;
    unsigned char *gQg = p.qg_img + gch * kImgW;
    unsigned char *gKg = p.kg_img + gch * kImgW;
    constexpr int kQgBatch = 4;  // items loaded before any is stored
    static_assert((kChunk * VPR) % (kQgBatch * NT) == 0, "qg batches");
    static_assert(VPR == 16, "item map below assumes 16 eight-key vectors per row");
    // item e -> (row i, keys d0 .. d0+7): the 32 items of a warp instruction
    // are 8 consecutive rows x 4 consecutive 8-key blocks, so each warp store
    // fills whole 128-byte lines of both images (512 contiguous bytes of qg)
    auto item_row = [](int e) { return (((e >> 5) & 7) << 3) + (e & 7); };
    auto item_key = [](int e) { return ((((e >> 5) >> 3) << 2) + ((e & 31) >> 3)) * 8; };
    for (int e0 = tid; e0 < kChunk * VPR; e0 += kQgBatch * NT) {
        uint4 xq[kQgBatch], xk[kQgBatch];
        float sq[kQgBatch], sk[kQgBatch], gi[kQgBatch];
#pragma unroll
        for (int u = 0; u < kQgBatch; ++u) {
            const int e = e0 + u * NT, i = item_row(e), d0 = item_key(e);
            xq[u] = *reinterpret_cast<const uint4 *>(sQ + i * KS + d0);
            xk[u] = *reinterpret_cast<const uint4 *>(sK + i * KS + d0);
            sq[u] = sRq[i];
            sk[u] = sRk[i];
            gi[u] = PERKEY ? 0.f : sG[i];
        }
        const float glast = PERKEY ? 0.f : sG[last];
#pragma unroll
        for (int u = 0; u < kQgBatch; ++u) {
            const int e = e0 + u * NT, i = item_row(e), d0 = item_key(e);
            float fq[8], fk[8];
            unpack8(xq[u], fq);
            unpack8(xk[u], fk);
            if (PERKEY) {
                float fx[8], gi8[8], gl8[8];
                ld8f(sG + i * KP + d0, gi8);
                ld8f(sG + last * KP + d0, gl8);
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    const float eg = ex2(gi8[x]);
                    fx[x] = fk[x] * eg;  // e^{G} . k (raw k: the norm goes into T's columns)
                    fq[x] *= eg * sq[u];
                    fk[x] *= ex2(gl8[x] - gi8[x]) * sk[u];
                }
                *reinterpret_cast<uint4 *>(sK + i * KS + d0) = pack8(fx);
            } else {
                const float eq = __expf(gi[u]) * sq[u], ek = __expf(glast - gi[u]) * sk[u];
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    fq[x] *= eq;
                    fk[x] *= ek;
                }
            }
            *reinterpret_cast<uint4 *>(gQg + img_w_off(i, d0)) = pack8(fq);
            *reinterpret_cast<uint4 *>(gKg + img_kt_off(i, d0)) = pack8(fk);
        }
    }
    for (int d = tid; d < KP; d += NT)
        p.dec[gch * KP + d] = PERKEY ? ex2(sG[last * KP + d]) : __expf(sG[last]);
    fence_async_smem();  // these generic accesses come before the copies that reuse the space
    __syncthreads();     // the q tile (scalar gate) and the split operands (per key) are free

    //         the value tile, one bulk copy per row, into the freed space
    if (tid < kChunk) {
        const int i = tid;
        const uint32_t rowb = (uint32_t)V * 2;
        arrive_expect_tx(b_v, tk_row >= 0 ? rowb : 0);
        if (tk_row >= 0)
            bulk_g2s(smem_u32(sV + i * VS), v + v_base + (int64_t)(si.tstart + tk_row) * p.v_st, rowb, b_v);
        else
            zero_row(sV + i * VS, 0, V);
        if (V < VP) zero_row(sV + i * VS, V, VP);
        if (p.has_den) sV[i * VS + V] = __float2bfloat16_rn(1.f);  // the denominator's ones column
    }

    //         T_II = (I + A_II)^{-1} for the diagonal block of this warp;
    //         lane c < 16 holds column c: t = e_c, t_r = -sum_{j<r} A_rj t_j
    if (warp < 4) {
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
        if (lane < 16) {  // T_II and its column-scaled copies for the w and u right-hand sides
            const int j = 16 * I + cc;
            const float bj = sB[j];
            const float sw = PERKEY ? bj * sRk[j] : bj * sRk[j] * __expf(sG[j]);
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const int o = (I * 16 + r) * kBS + cc;
                sTd[o] = __float2bfloat16_rn(t[r]);
                sTd[kTSet + o] = __float2bfloat16_rn(t[r] * sw);
                sTd[2 * kTSet + o] = __float2bfloat16_rn(t[r] * bj);
            }
        }
        __syncwarp();
        //     B_IM = -T_II A_IM for the blocks left of this warp's diagonal
        //     block, in place of A_IM
        if (I > 0) {
            uint32_t a[4];
            ldsm_x4(a, sTd + (16 * I + (lane & 15)) * kBS + (lane >> 4) * 8);
#pragma unroll
            for (int x = 0; x < 4; ++x) a[x] ^= 0x80008000u;  // -T_II
            for (int M = 0; M < I; ++M) {
                bf16 *blkp = sAb + blk(I, M) * 16 * kBS;
                uint32_t b[4];
                ldsm_x4_t(b, blkp + (lane & 15) * kBS + (lane >> 4) * 8);
                float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
                mma_bf16(c0, a, b[0], b[1]);
                mma_bf16(c1, a, b[2], b[3]);
                __syncwarp();  // every lane has read A_IM before it is overwritten
                *reinterpret_cast<uint32_t *>(blkp + g8 * kBS + 2 * t4) = pack_bf16(c0[0], c0[1]);
                *reinterpret_cast<uint32_t *>(blkp + (g8 + 8) * kBS + 2 * t4) = pack_bf16(c0[2], c0[3]);
                *reinterpret_cast<uint32_t *>(blkp + g8 * kBS + 8 + 2 * t4) = pack_bf16(c1[0], c1[1]);
                *reinterpret_cast<uint32_t *>(blkp + (g8 + 8) * kBS + 8 + 2 * t4) = pack_bf16(c1[2], c1[3]);
            }
        }
    }
    __syncthreads();

    // ---- 5. W_I = T_II diag(s_I) X~_I + sum_{M<I} B_IM W_M per 64-column
    //         slice, straight to the w / u images. X = diag(s) X~ with X~ the
    //         tile in shared memory (k, or e^{G} . k per key; V) and s the row
    //         scales, folded into T's columns.
    unsigned char *gW = p.w_img + gch * kImgW;
    unsigned char *gU = p.u_img + gch * p.n_vt * kImgU;
    const int nsw = KP / 64, nsu = VP / 64;
    bool v_ready = false;
    for (int sl = warp; sl < nsw + nsu; sl += NT / 32) {
        const bool isw = sl < nsw;
        if (!isw && !v_ready) {
            if (!wait_copies(b_v, p.err)) return;
            v_ready = true;
        }
        bf16 *tile = isw ? sK : sV;  // rows of X~_I, then of W_I once solved
        const bf16 *sTs = sTd + (isw ? kTSet : 2 * kTSet);
        const int ts = isw ? KS : VS;
        const int c0 = isw ? 64 * sl : 64 * (sl - nsw);
#pragma unroll
        for (int I = 0; I < 4; ++I) {
            float wa[8][4];
#pragma unroll
            for (int n = 0; n < 8; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) wa[n][e] = 0.f;
#pragma unroll
            for (int M = 0; M < I; ++M) {
                uint32_t a[4];
                ldsm_x4(a, sAb + (blk(I, M) * 16 + (lane & 15)) * kBS + (lane >> 4) * 8);
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    uint32_t b[4];
                    ldsm_x4_t(b, tile + (16 * M + (lane & 15)) * ts + c0 + 16 * np + (lane >> 4) * 8);
                    mma_bf16(wa[2 * np], a, b[0], b[1]);
                    mma_bf16(wa[2 * np + 1], a, b[2], b[3]);
                }
            }
            {
                uint32_t a[4];
                ldsm_x4(a, sTs + (16 * I + (lane & 15)) * kBS + (lane >> 4) * 8);
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    uint32_t b[4];
                    ldsm_x4_t(b, tile + (16 * I + (lane & 15)) * ts + c0 + 16 * np + (lane >> 4) * 8);
                    mma_bf16(wa[2 * np], a, b[0], b[1]);
                    mma_bf16(wa[2 * np + 1], a, b[2], b[3]);
                }
            }
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                const uint32_t lo = pack_bf16(wa[n][0], wa[n][1]), hi = pack_bf16(wa[n][2], wa[n][3]);
                const int i = 16 * I + g8, cl = 8 * n + 2 * t4;
                if (isw) {
                    *reinterpret_cast<uint32_t *>(gW + img_w_off(i, c0 + cl)) = lo;
                    *reinterpret_cast<uint32_t *>(gW + img_w_off(i + 8, c0 + cl)) = hi;
                } else {
                    unsigned char *u = gU + (c0 >> 6) * kImgU;
                    *reinterpret_cast<uint32_t *>(u + img_u_off(i, cl)) = lo;
                    *reinterpret_cast<uint32_t *>(u + img_u_off(i + 8, cl)) = hi;
                }
                if (I < 3) {
                    *reinterpret_cast<uint32_t *>(tile + i * ts + c0 + cl) = lo;
                    *reinterpret_cast<uint32_t *>(tile + (i + 8) * ts + c0 + cl) = hi;
                }
            }
            __syncwarp();
        }
    }
    // (every value-tile copy was waited for by the warp owning a u slice, so
    // none outlives the CTA)
}

template <bool PERKEY>
cudaError_t launch_t(const FwdParams &p, cudaStream_t st) {
    using L = Lay<PERKEY>;
    const int VP = p.n_vt * 64;
    const size_t bytes = L::bytes(VP);
    auto kern = p.stall_cta >= 0 ? intra_kernel<PERKEY, true> : intra_kernel<PERKEY, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    // the whole shared-memory carveout, so that 4 (scalar) / 2 (per-key) CTAs fit per SM
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)p.max_chunks * (unsigned)p.H);
    kern<<<grid, PERKEY ? 2 * kThreads : kThreads, bytes, st>>>(p, VP);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_intra_bf16(const FwdParams &p, int perkey, cudaStream_t st) {
    if (p.max_chunks == 0) return cudaSuccess;
    return perkey ? launch_t<true>(p, st) : launch_t<false>(p, st);
}

}  // namespace gdn
