// gdn_chunk_f32_split.cu -- the fp32 path for problems too small to fill the
// GPU with the fused kernel's (sequence, head, 32-column tile) CTAs: the
// chunk-parallel part and the chunk-serial part in two kernels, as in the
// bf16 path, so that the serial chain per chunk is three small products.
//
//   f32_prep    one CTA per (64-token chunk, head), all chunks at once:
//               A, P, T_II (as in the fused kernel), then by block forward
//               substitution w = (I + A)^{-1} (beta e^{G} . k^) and
//               u = (I + A)^{-1} (beta . V) in 32-column tiles, qg = e^{G} . q^,
//               kg = e^{G_last - G} . k^, dec = e^{G_last}; fp32 images.
//   f32_serial  one CTA per (sequence, head, 32-column tile), chunk by chunk:
//               v_new = u - w h,  o = qg h + P v_new,  h = dec . h + kg^T v_new.
// The same chunked WY form as the fused kernel (SANA `fused_gdn.py` page,
// `_fused_gdn_kernel`; hyper-parallel coverage_diff page,
// `chunk_gated_delta_rule_fwd_kernel_h_blockdim64`), IEEE fp32 throughout.
// The images live in the workspace (indexed [head][global chunk], rows in
// chunk order): w, qg, kg 64 x KP, P 64 x 64, u 64 x VP32, dec KP floats.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kT = 256;   // threads per prep CTA
constexpr int kTS = 512;  // threads per serial CTA: two halves splitting each reduction
constexpr int kBV = 32;  // value columns per tile of the serial pass
constexpr int kBW = 128;  // right-hand-side columns per substitution pass of the prep
constexpr int kAS = kChunk + 1, kWS = kBW + 1;
constexpr int kVS = kBV + 4;  // 16-byte aligned rows of h and v_new: a thread's 4 columns in one load

// ---------------------------------------------------------------- prep ----
template <int KP, bool PERKEY>
struct PrepSmem {
    static constexpr int QS = KP + 1;
    static constexpr int q = 0;
    static constexpr int k = q + kChunk * QS;
    static constexpr int gk = k + kChunk * QS;
    static constexpr int g = gk + (PERKEY ? kChunk * QS : 0);
    static constexpr int beta = g + kChunk;
    static constexpr int a = beta + kChunk;
    static constexpr int t = a + kChunk * kAS;
    static constexpr int pm = t + kChunk * kAS;
    static constexpr int x = pm + kChunk * kAS;
    static constexpr int r = x + kChunk * kWS;
    static constexpr int total = r + kChunk * kWS;
    static constexpr size_t bytes = sizeof(float) * total;
};

template <int KP, bool PERKEY>
__global__ void __launch_bounds__(kT) f32_prep_kernel(const FwdParams p, int vp32) {
    using L = PrepSmem<KP, PERKEY>;
    constexpr int QS = L::QS;
    extern __shared__ float sm[];
    float *sQ = sm + L::q, *sK = sm + L::k, *sGk = sm + L::gk, *sG = sm + L::g, *sB = sm + L::beta;
    float *sA = sm + L::a, *sT = sm + L::t, *sP = sm + L::pm, *sX = sm + L::x, *sR = sm + L::r;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hh = blockIdx.x % p.H, gid = blockIdx.x / p.H;
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
    const int pos0 = c * kChunk, Lc = min(kChunk, si.len - pos0);
    if (Lc <= 0) return;
    const int K = p.K, V = p.V, H = p.H;
    const size_t gch = (size_t)hh * p.max_chunks + gid;
    const float *q = (const float *)p.q, *k = (const float *)p.k, *v = (const float *)p.v;

    // ---- q, k (zero padded), per-key gates, beta, scalar gates
    // (every load of a thread issued before its stores)
    constexpr int KV4 = KP / 4, NQ = kChunk * KV4 / kT;
    {
        float4 xq[NQ], xk[NQ], xg[NQ];
#pragma unroll
        for (int u = 0; u < NQ; ++u) {
            const int e = tid + u * kT, i = e / KV4, d = (e % KV4) * 4;
            xq[u] = xk[u] = xg[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < Lc && d < K) {
                const int tq = q_token(p.reverse, si.len, pos0 + i), tk = kv_token(p.reverse, si.len, pos0 + i);
                xq[u] = __ldg(reinterpret_cast<const float4 *>(q + si.b * p.qk_sb + (int64_t)(si.tstart + tq) * p.qk_st +
                                                               hh * p.qk_sh + d));
                if (tk >= 0) {
                    xk[u] = __ldg(reinterpret_cast<const float4 *>(k + si.b * p.qk_sb +
                                                                   (int64_t)(si.tstart + tk) * p.qk_st + hh * p.qk_sh + d));
                    if (PERKEY)
                        xg[u] = __ldg(reinterpret_cast<const float4 *>(p.gk + ((si.row0 + tk) * H + hh) * (int64_t)K + d));
                }
            }
        }
#pragma unroll
        for (int u = 0; u < NQ; ++u) {
            const int e = tid + u * kT, i = e / KV4, d = (e % KV4) * 4;
            const float qa[4] = {xq[u].x, xq[u].y, xq[u].z, xq[u].w}, ka[4] = {xk[u].x, xk[u].y, xk[u].z, xk[u].w};
            const float ga[4] = {xg[u].x, xg[u].y, xg[u].z, xg[u].w};
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                sQ[i * QS + d + x] = qa[x];
                sK[i * QS + d + x] = ka[x];
                if (PERKEY) sGk[i * QS + d + x] = (i < Lc && d < K) ? fmaxf(ga[x], kLogGateMin) : 0.f;
            }
        }
    }
    if (tid < kChunk) {
        float b = 0.f, gg = 0.f;
        if (tid < Lc) {
            const int tk = kv_token(p.reverse, si.len, pos0 + tid);
            if (tk >= 0) {
                b = p.beta[(si.row0 + tk) * H + hh];
                if (!PERKEY) gg = fmaxf(p.g[(si.row0 + tk) * H + hh], kLogGateMin);
            }
        }
        sB[tid] = b;
        sG[tid] = gg;
    }
    __syncthreads();
    // ---- L2 normalisation (two threads per row), in-chunk gate cumsums
    if (p.l2norm) {
        const int row = tid >> 1, half = tid & 1;
        float *rp = (row < kChunk) ? (sQ + row * QS) : (sK + (row - kChunk) * QS);
        float s0 = 0.f, s1 = 0.f;
        for (int d = half; d < KP; d += 4) {
            s0 = fmaf(rp[d], rp[d], s0);
            if (d + 2 < KP) s1 = fmaf(rp[d + 2], rp[d + 2], s1);
        }
        float ss = s0 + s1;
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        const float inv = rsqrtf(ss + 1e-6f);
        for (int d = half; d < KP; d += 2) rp[d] *= inv;
    }
    if (PERKEY) {
        for (int d = tid; d < KP; d += kT) {
            float acc = 0.f;
            for (int i = 0; i < kChunk; ++i) {
                acc += sGk[i * QS + d];
                sGk[i * QS + d] = acc;
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
    // ---- A (strictly lower, beta-scaled) and P (lower incl. diagonal);
    // scalar gate: a 4 x 4 block of (i, j) per thread
    if constexpr (!PERKEY) {
        const int bi = tid >> 4, bj = tid & 15;
        float sa[4][4], sp[4][4];
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int y = 0; y < 4; ++y) sa[x][y] = sp[x][y] = 0.f;
        if (bj <= bi) {
#pragma unroll 4
            for (int d = 0; d < KP; ++d) {
                float ki[4], qi[4], kj[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    ki[x] = sK[(4 * bi + x) * QS + d];
                    qi[x] = sQ[(4 * bi + x) * QS + d];
                    kj[x] = sK[(4 * bj + x) * QS + d];
                }
#pragma unroll
                for (int x = 0; x < 4; ++x)
#pragma unroll
                    for (int y = 0; y < 4; ++y) {
                        sa[x][y] = fmaf(ki[x], kj[y], sa[x][y]);
                        sp[x][y] = fmaf(qi[x], kj[y], sp[x][y]);
                    }
            }
        }
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int y = 0; y < 4; ++y) {
                const int i = 4 * bi + x, j = 4 * bj + y;
                float a = 0.f, pm = 0.f;
                if (j <= i) {
                    const float gam = __expf(sG[i] - sG[j]);
                    pm = sp[x][y] * gam;
                    if (j < i) a = sB[i] * (sa[x][y] * gam);
                }
                sA[i * kAS + j] = a;
                sP[i * kAS + j] = pm;
            }
    } else
    for (int e = tid; e < kChunk * kChunk; e += kT) {
        const int i = e / kChunk, j = e % kChunk;
        float a = 0.f, pm = 0.f;
        if (j <= i) {
            float sa = 0.f, sp = 0.f;
            if (PERKEY) {
                for (int d = 0; d < KP; ++d) {
                    const float kj = sK[j * QS + d] * __expf(sGk[i * QS + d] - sGk[j * QS + d]);
                    sa = fmaf(sK[i * QS + d], kj, sa);
                    sp = fmaf(sQ[i * QS + d], kj, sp);
                }
            } else {
                for (int d = 0; d < KP; ++d) {
                    sa = fmaf(sK[i * QS + d], sK[j * QS + d], sa);
                    sp = fmaf(sQ[i * QS + d], sK[j * QS + d], sp);
                }
                const float gam = __expf(sG[i] - sG[j]);
                sa *= gam;
                sp *= gam;
            }
            pm = sp;
            if (j < i) a = sB[i] * sa;
        }
        sA[i * kAS + j] = a;
        sP[i * kAS + j] = pm;
    }
    __syncthreads();
    // ---- diagonal blocks T_II = (I + A_II)^{-1}: one warp per block, lane = column
    if (warp < 4 && lane < 16) {
        const int o = 16 * warp;
        float t[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = (r == lane) ? 1.f : 0.f;
#pragma unroll
            for (int j = 0; j < r; ++j) acc = fmaf(-sA[(o + r) * kAS + o + j], t[j], acc);
            t[r] = acc;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) sT[(o + r) * kAS + o + lane] = t[r];
    }
    // ---- P, qg, kg and the chunk decay to their images
    const int last = Lc - 1;
    float *gP = reinterpret_cast<float *>(p.p_img) + gch * kChunk * kChunk;
    float *gQg = reinterpret_cast<float *>(p.qg_img) + gch * kChunk * KP;
    float *gKg = reinterpret_cast<float *>(p.kg_img) + gch * kChunk * KP;
    for (int e = tid; e < kChunk * kChunk; e += kT) gP[e] = sP[(e / kChunk) * kAS + e % kChunk];
    for (int e = tid; e < kChunk * KP; e += kT) {
        const int i = e / KP, d = e % KP;
        const float gi = PERKEY ? sGk[i * QS + d] : sG[i], gl = PERKEY ? sGk[last * QS + d] : sG[last];
        gQg[e] = __expf(gi) * sQ[i * QS + d];
        gKg[e] = __expf(gl - gi) * sK[i * QS + d];
    }
    for (int d = tid; d < KP; d += kT) p.dec[gch * KP + d] = __expf(PERKEY ? sGk[last * QS + d] : sG[last]);
    __syncthreads();  // T's diagonal blocks are complete

    // ---- w and u by block forward substitution, kBW right-hand-side columns
    // at a time: R_I = T_II (X_I - sum_{M<I} A_IM R_M) for X = [beta e^{G} .
    // k^ | beta . V] (the value part with the denominator's ones column)
    const int nx = KP + vp32;
    float *gW = reinterpret_cast<float *>(p.w_img) + gch * kChunk * KP;
    float *gU = reinterpret_cast<float *>(p.u_img) + gch * kChunk * vp32;
    for (int c0 = 0; c0 < nx; c0 += kBW) {
        const int nc = min(kBW, nx - c0);
        // 4 columns per item (KP, vp32, V and kBW are multiples of 4... V of 8)
        constexpr int NI = kChunk * (kBW / 4) / kT;
        float4 xv[NI];
#pragma unroll
        for (int u = 0; u < NI; ++u) {  // the value loads first
            const int e = tid + u * kT, i = e / (kBW / 4), n = (e % (kBW / 4)) * 4, gc = c0 + n, col = gc - KP;
            xv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (n < nc && gc >= KP && i < Lc && col < V) {
                const int tk = kv_token(p.reverse, si.len, pos0 + i);
                if (tk >= 0)
                    xv[u] = __ldg(reinterpret_cast<const float4 *>(
                        v + si.b * p.v_sb + (int64_t)(si.tstart + tk) * p.v_st + hh * p.v_sh + col));
            }
        }
#pragma unroll
        for (int u = 0; u < NI; ++u) {
            const int e = tid + u * kT, i = e / (kBW / 4), n = (e % (kBW / 4)) * 4;
            const float va[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const int gc = c0 + n + x, col = gc - KP;
                float xx = 0.f;
                if (n + x < nc) {
                    if (gc < KP) xx = sB[i] * __expf(PERKEY ? sGk[i * QS + gc] : sG[i]) * sK[i * QS + gc];
                    else if (col < V) xx = sB[i] * va[x];
                    else if (p.has_den && col == V && i < Lc && kv_token(p.reverse, si.len, pos0 + i) >= 0) xx = sB[i];
                }
                sX[i * kWS + n + x] = xx;
            }
        }
        __syncthreads();
        for (int I = 0; I < 4; ++I) {
            const int o = 16 * I;
            if (I > 0) {
                for (int e = tid; e < 16 * kBW; e += kT) {
                    const int i = o + e / kBW, n = e % kBW;
                    float a4[4] = {0.f, 0.f, 0.f, 0.f};
                    for (int j = 0; j < o; j += 4) {
#pragma unroll
                        for (int u = 0; u < 4; ++u) a4[u] = fmaf(sA[i * kAS + j + u], sR[(j + u) * kWS + n], a4[u]);
                    }
                    sX[i * kWS + n] -= (a4[0] + a4[1]) + (a4[2] + a4[3]);
                }
                __syncthreads();
            }
            for (int e = tid; e < 16 * kBW; e += kT) {
                const int i = o + e / kBW, n = e % kBW;
                float a4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < 16; ++j) a4[j & 3] = fmaf(sT[i * kAS + o + j], sX[(o + j) * kWS + n], a4[j & 3]);
                sR[i * kWS + n] = (a4[0] + a4[1]) + (a4[2] + a4[3]);
            }
            __syncthreads();
        }
        for (int e = tid; e < kChunk * kBW; e += kT) {
            const int i = e / kBW, n = e % kBW, gc = c0 + n;
            if (n >= nc) continue;
            if (gc < KP) gW[i * KP + gc] = sR[i * kWS + n];
            else gU[i * vp32 + gc - KP] = sR[i * kWS + n];
        }
        __syncthreads();  // sX and sR are rewritten by the next group
    }
}

// -------------------------------------------------------------- serial ----
static_assert(PrepSmem<128, true>::bytes <= 227 * 1024, "prep shared memory");
// one chunk's operands (16-byte aligned rows, filled by asynchronous copies),
// twice over where that fits (64 keys), so that chunk c+1's arrive while
// chunk c computes; with 128 keys one buffer, refilled after each chunk
template <int KP>
struct SerSmem {
    static constexpr int QS = KP + 4, PS = kChunk + 4, US = kBV + 4;
    static constexpr int w = 0;
    static constexpr int qg = w + kChunk * QS;
    static constexpr int kg = qg + kChunk * QS;
    static constexpr int pm = kg + kChunk * QS;
    static constexpr int u = pm + kChunk * PS;
    static constexpr int dec = u + kChunk * US;
    static constexpr int buf = dec + KP;  // floats per operand buffer
    static constexpr int NB = KP == 64 ? 2 : 1;
    static constexpr int vn = NB * buf;
    static constexpr int h = vn + kChunk * kVS;
    static constexpr int part = h + KP * kVS;  // the upper half's partial sums
    static constexpr int total = part + KP * kVS;
    static constexpr size_t bytes = sizeof(float) * total;
};
static_assert(SerSmem<64>::bytes <= 227 * 1024 && SerSmem<128>::bytes <= 227 * 1024, "serial shared memory");

template <int KP>
__global__ void __launch_bounds__(kTS) f32_serial_kernel(const FwdParams p, int vp32) {
    using L = SerSmem<KP>;
    constexpr int QS = L::QS, PS = L::PS, US = L::US;
    extern __shared__ __align__(16) float sm[];
    float *sVn = sm + L::vn, *sH = sm + L::h;
    const int tid = threadIdx.x;
    const int s = blockIdx.x / p.H, hh = blockIdx.x % p.H;
    const int v0 = blockIdx.y * kBV;
    const int K = p.K, V = p.V, H = p.H;
    if (p.cu_seqlens && *p.n_chunks < 0) return;  // cu_seqlens rejected on the device
    SeqInfo si;
    if (!seq_info(p, s, si)) return;
    const int nchunks = (si.len + kChunk - 1) / kChunk;
    const int gc0 = p.cu_seqlens ? p.seq_chunk0[s] : s * ((p.T + kChunk - 1) / kChunk);

    for (int e = tid; e < KP * kBV; e += kTS) {  // state tile h[d][n]
        const int d = e / kBV, n = e % kBV, col = v0 + n;
        sH[d * kVS + n] = (p.h0 && d < K && col < p.Vt) ? p.h0[(((int64_t)s * H + hh) * K + d) * p.Vt + col] : 0.f;
    }
    // 2 rows x 4 columns per thread for the 64 x 32 products, KP/32 key rows
    // x 4 columns for the state update; the two halves of the CTA (hf) take
    // two halves of each reduction, the upper one handing its partial sums
    // over through sPart
    const int hf = tid >> 8, lt = tid & 255;
    const int nq = lt & 7, ig = lt >> 3, dg = lt >> 3;
    constexpr int RD = KP / 32;
    float *sPart = sm + L::part;
    // chunk c's operands into buffer c % NB: 16-byte asynchronous copies
    auto fetch = [&](int c) {
        float *bs = sm + (c % L::NB) * L::buf;
        const size_t gch = (size_t)hh * p.max_chunks + gc0 + c;
        const float *gW = reinterpret_cast<const float *>(p.w_img) + gch * kChunk * KP;
        const float *gQg = reinterpret_cast<const float *>(p.qg_img) + gch * kChunk * KP;
        const float *gKg = reinterpret_cast<const float *>(p.kg_img) + gch * kChunk * KP;
        const float *gP = reinterpret_cast<const float *>(p.p_img) + gch * kChunk * kChunk;
        const float *gU = reinterpret_cast<const float *>(p.u_img) + gch * kChunk * vp32 + v0;
        for (int e = tid; e < kChunk * KP / 4; e += kTS) {
            const int i = e / (KP / 4), d = (e % (KP / 4)) * 4;
            cp_async16(bs + L::w + i * QS + d, gW + i * KP + d, 16);
            cp_async16(bs + L::qg + i * QS + d, gQg + i * KP + d, 16);
            cp_async16(bs + L::kg + i * QS + d, gKg + i * KP + d, 16);
        }
        for (int e = tid; e < kChunk * kChunk / 4; e += kTS) {
            const int i = e / (kChunk / 4), j = (e % (kChunk / 4)) * 4;
            cp_async16(bs + L::pm + i * PS + j, gP + i * kChunk + j, 16);
        }
        for (int e = tid; e < kChunk * kBV / 4; e += kTS) {
            const int i = e / (kBV / 4), n = (e % (kBV / 4)) * 4;
            cp_async16(bs + L::u + i * US + n, gU + i * vp32 + n, 16);
        }
        for (int e = tid; e < KP / 4; e += kTS) cp_async16(bs + L::dec + 4 * e, p.dec + gch * KP + 4 * e, 16);
    };
    if (nchunks > 0) fetch(0);
    cp_async_commit();
    for (int c = 0; c < nchunks; ++c) {
        const int pos0 = c * kChunk, Lc = min(kChunk, si.len - pos0);
        // two buffers: chunk c+1's copies go out now (their buffer's last
        // reader, chunk c-1, finished before the sync that closed it)
        if (L::NB == 2 && c + 1 < nchunks) fetch(c + 1);
        cp_async_commit();
        // chunk c's operands landed: every group but chunk c+1's (two
        // buffers); every group (one buffer: chunk c's copies, issued at the
        // end of the previous iteration, are in the group just committed)
        if (L::NB == 2) cp_async_wait<1>();
        else cp_async_wait<0>();
        __syncthreads();
        const float *bs = sm + (c % L::NB) * L::buf;
        const float *sW = bs + L::w, *sQG = bs + L::qg, *sKG = bs + L::kg, *sP = bs + L::pm;
        const float *sU = bs + L::u, *sDec = bs + L::dec;
        // ---- v_new = u - w h: keys [hf KP/2, (hf+1) KP/2) per half
        {
            float acc[2][4];
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) acc[r][c4] = 0.f;
            const int d0 = hf * (KP / 2);
#pragma unroll 16
            for (int d = d0; d < d0 + KP / 2; ++d) {
                const float4 h4 = *reinterpret_cast<const float4 *>(sH + d * kVS + 4 * nq);
                const float hv[4] = {h4.x, h4.y, h4.z, h4.w};
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float wv = sW[(ig + 32 * r) * QS + d];
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) acc[r][c4] = fmaf(wv, hv[c4], acc[r][c4]);
                }
            }
            if (hf)
#pragma unroll
                for (int r = 0; r < 2; ++r)
                    *reinterpret_cast<float4 *>(sPart + (ig + 32 * r) * kVS + 4 * nq) =
                        make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
            __syncthreads();
            if (!hf)
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int i = ig + 32 * r;
                    const float4 o4 = *reinterpret_cast<const float4 *>(sPart + i * kVS + 4 * nq);
                    const float oa[4] = {o4.x, o4.y, o4.z, o4.w};
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const int n = 4 * nq + c4;
                        sVn[i * kVS + n] = sU[i * US + n] - (acc[r][c4] + oa[c4]);
                    }
                }
        }
        __syncthreads();
        // ---- o = qg h (lower half) + P v_new (upper half; P is zero right of
        // the diagonal)
        {
            float acc[2][4];
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) acc[r][c4] = 0.f;
            if (!hf) {
#pragma unroll 16
                for (int d = 0; d < KP; ++d) {
                    const float4 h4 = *reinterpret_cast<const float4 *>(sH + d * kVS + 4 * nq);
                    const float hv[4] = {h4.x, h4.y, h4.z, h4.w};
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const float qv = sQG[(ig + 32 * r) * QS + d];
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) acc[r][c4] = fmaf(qv, hv[c4], acc[r][c4]);
                    }
                }
            } else {
#pragma unroll 16
                for (int j = 0; j < kChunk; ++j) {
                    const float4 v4 = *reinterpret_cast<const float4 *>(sVn + j * kVS + 4 * nq);
                    const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const float pj = sP[(ig + 32 * r) * PS + j];
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) acc[r][c4] = fmaf(pj, vv[c4], acc[r][c4]);
                    }
                }
#pragma unroll
                for (int r = 0; r < 2; ++r)
                    *reinterpret_cast<float4 *>(sPart + (ig + 32 * r) * kVS + 4 * nq) =
                        make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
            }
            __syncthreads();
            if (!hf) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int i = ig + 32 * r;
                    if (i >= Lc) continue;
                    const float4 o4 = *reinterpret_cast<const float4 *>(sPart + i * kVS + 4 * nq);
                    const float oa[4] = {o4.x, o4.y, o4.z, o4.w};
                    const int tq = q_token(p.reverse, si.len, pos0 + i);
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const int col = v0 + 4 * nq + c4;
                        const float val = acc[r][c4] + oa[c4];
                        if (col < V) {
                            const int64_t off = si.b * p.o_sb + (int64_t)(si.tstart + tq) * p.o_st + hh * p.o_sh + col;
                            if (p.out_f32) {
                                float *o = (float *)p.out + off;
                                *o = p.accumulate ? *o + val : val;
                            } else {
                                __nv_bfloat16 *o = (__nv_bfloat16 *)p.out + off;
                                *o = __float2bfloat16_rn(p.accumulate ? __bfloat162float(*o) + val : val);
                            }
                        } else if (p.has_den && col == V) {
                            float *o = p.den + ((int64_t)si.b * H + hh) * p.T + si.tstart + tq;
                            *o = p.accumulate ? *o + val : val;
                        }
                    }
                }
            }
        }
        __syncthreads();  // sPart is rewritten below
        // ---- h = dec . h + kg^T v_new: tokens [32 hf, 32 hf + 32) per half
        {
            float acc[RD][4];
#pragma unroll
            for (int r = 0; r < RD; ++r) {
                const float dd = hf ? 0.f : sDec[dg + 32 * r];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) acc[r][c4] = hf ? 0.f : dd * sH[(dg + 32 * r) * kVS + 4 * nq + c4];
            }
            const int i0 = 32 * hf, i1 = min(Lc, i0 + 32);
#pragma unroll 8
            for (int i = i0; i < i1; ++i) {
                const float4 v4 = *reinterpret_cast<const float4 *>(sVn + i * kVS + 4 * nq);
                const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
                for (int r = 0; r < RD; ++r) {
                    const float kf = sKG[i * QS + dg + 32 * r];
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) acc[r][c4] = fmaf(kf, vv[c4], acc[r][c4]);
                }
            }
            if (hf)
#pragma unroll
                for (int r = 0; r < RD; ++r)
                    *reinterpret_cast<float4 *>(sPart + (dg + 32 * r) * kVS + 4 * nq) =
                        make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
            __syncthreads();  // the partials are in, and every read of h is done
            if (!hf)
#pragma unroll
                for (int r = 0; r < RD; ++r) {
                    const float4 o4 = *reinterpret_cast<const float4 *>(sPart + (dg + 32 * r) * kVS + 4 * nq);
                    *reinterpret_cast<float4 *>(sH + (dg + 32 * r) * kVS + 4 * nq) =
                        make_float4(acc[r][0] + o4.x, acc[r][1] + o4.y, acc[r][2] + o4.z, acc[r][3] + o4.w);
                }
        }
        __syncthreads();  // this buffer is refilled and v_new rewritten next
        if (L::NB == 1 && c + 1 < nchunks) fetch(c + 1);
    }
    cp_async_wait<0>();
    __syncthreads();
    if (p.h_final) {
        for (int e = tid; e < KP * kBV; e += kTS) {
            const int d = e / kBV, n = e % kBV, col = v0 + n;
            if (d < K && col < p.Vt) p.h_final[(((int64_t)s * H + hh) * K + d) * p.Vt + col] = sH[d * kVS + n];
        }
    }
}

template <int KP, bool PERKEY>
cudaError_t launch_prep_t(const FwdParams &p, cudaStream_t st) {
    using L = PrepSmem<KP, PERKEY>;
    auto kern = f32_prep_kernel<KP, PERKEY>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::bytes);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)p.max_chunks * (unsigned)p.H, kT, L::bytes, st>>>(p, f32_vp32(p.Vt));
    return cudaGetLastError();
}

template <int KP>
cudaError_t launch_serial_t(const FwdParams &p, cudaStream_t st) {
    using L = SerSmem<KP>;
    auto kern = f32_serial_kernel<KP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::bytes);
    if (e != cudaSuccess) return e;
    dim3 grid(p.n_seq * p.H, (p.Vt + kBV - 1) / kBV);
    kern<<<grid, kTS, L::bytes, st>>>(p, f32_vp32(p.Vt));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_f32_prep(const FwdParams &p, int KP, int perkey, cudaStream_t st) {
    if (p.max_chunks == 0) return cudaSuccess;
    if (KP == 64) return perkey ? launch_prep_t<64, true>(p, st) : launch_prep_t<64, false>(p, st);
    return perkey ? launch_prep_t<128, true>(p, st) : launch_prep_t<128, false>(p, st);
}

cudaError_t launch_f32_serial(const FwdParams &p, int KP, cudaStream_t st) {
    return KP == 64 ? launch_serial_t<64>(p, st) : launch_serial_t<128>(p, st);
}

}  // namespace gdn
