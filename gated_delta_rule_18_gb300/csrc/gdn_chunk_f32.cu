// gdn_chunk_f32.cu -- the fp32 path: one fused CUDA-core kernel per
// (sequence, head, 32-column value tile) that walks the sequence chunk by
// chunk with IEEE fp32 products throughout (no tensor cores, no TF32).
//
// Per chunk of L <= 64 tokens (logical positions; the reverse scan remaps
// rows, see gdn_common.cuh), with G the in-chunk cumulative log gate
// (per key for gk) and h the state entering the chunk:
//   A_ij = beta_i sum_d k_id k_jd e^{G_id - G_jd}      (j < i)
//   T    = (I + A)^{-1}                               forward substitution
//   Y    = beta . (V - (e^{G} . K) h)
//   v_new = T Y                                        (= u - w h)
//   o    = (e^{G} . Q) h + P v_new,  P_ij = sum_d q_id k_jd e^{G_id - G_jd} (j <= i)
//   h   <- e^{G_last} . h + (e^{G_last - G} . K)^T v_new
// This is the chunked WY form of the token recurrence of the SANA
// `fused_gdn.py` page (`_fused_gdn_kernel`); v_new = u - w h and the
// h update follow the hyper-parallel coverage_diff page
// (`chunk_gated_delta_rule_fwd_kernel_h_blockdim64`), with the state kept in
// shared memory for the whole sequence. Per-key gate factors are evaluated
// element by element (exp of differences of cumulative gates, all <= 0), so
// nothing overflows for any gate magnitude.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kBVf = 32;  // value columns per CTA
constexpr int kThreadsF = 256;

template <int KP, bool PERKEY>
struct F32Smem {
    static constexpr int QS = KP + 1;    // row stride of q/k/gk tiles
    static constexpr int VS = kBVf + 1;  // row stride of value tiles
    static constexpr int AS = kChunk + 1;
    static constexpr int q = 0;
    static constexpr int k = q + kChunk * QS;
    static constexpr int gk = k + kChunk * QS;
    static constexpr int g = gk + (PERKEY ? kChunk * QS : 0);
    static constexpr int beta = g + kChunk;
    static constexpr int h = beta + kChunk;
    static constexpr int v = h + KP * VS;
    static constexpr int x = v + kChunk * VS;
    static constexpr int a = x + kChunk * VS;
    static constexpr int t = a + kChunk * AS;
    static constexpr int pm = t + kChunk * AS;
    static constexpr int total = pm + kChunk * AS;  // floats
    static constexpr size_t bytes = sizeof(float) * total;
};

template <int KP, bool PERKEY>
__global__ void __launch_bounds__(kThreadsF) fused_f32_kernel(const FwdParams p) {
    using L = F32Smem<KP, PERKEY>;
    extern __shared__ float sm[];
    float *sQ = sm + L::q, *sK = sm + L::k, *sGk = sm + L::gk, *sG = sm + L::g;
    float *sB = sm + L::beta, *sH = sm + L::h, *sV = sm + L::v, *sX = sm + L::x;
    float *sA = sm + L::a, *sT = sm + L::t, *sP = sm + L::pm;
    constexpr int QS = L::QS, VS = L::VS, AS = L::AS;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int s = blockIdx.x / p.H, hh = blockIdx.x % p.H;
    const int v0 = blockIdx.y * kBVf;
    const int K = p.K, V = p.V, H = p.H;
    if (p.cu_seqlens && *p.n_chunks < 0) return;  // cu_seqlens rejected on the device
    SeqInfo si;
    if (!seq_info(p, s, si)) return;
    const float *q = (const float *)p.q, *k = (const float *)p.k, *v = (const float *)p.v;

    // state tile h[d][n], d < KP, n < 32 (value column v0 + n)
    for (int e = tid; e < KP * kBVf; e += kThreadsF) {
        const int d = e / kBVf, n = e % kBVf, col = v0 + n;
        float x = 0.f;
        if (p.h0 && d < K && col < p.Vt) x = p.h0[(((int64_t)s * H + hh) * K + d) * p.Vt + col];
        sH[d * VS + n] = x;
    }

    const int nchunks = (si.len + kChunk - 1) / kChunk;
    for (int c = 0; c < nchunks; ++c) {
        const int pos0 = c * kChunk;
        const int Lc = min(kChunk, si.len - pos0);
        __syncthreads();  // previous chunk fully consumed
        // ---- load q, k (zero padded), v, beta, gates: 16-byte pieces, every
        // load of a thread issued before its stores
        constexpr int KV4 = KP / 4, NQ = kChunk * KV4 / kThreadsF;
        {
            float4 xq[NQ], xk[NQ], xg[NQ];
#pragma unroll
            for (int u = 0; u < NQ; ++u) {
                const int e = tid + u * kThreadsF, i = e / KV4, d = (e % KV4) * 4;
                xq[u] = xk[u] = xg[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (i < Lc && d < K) {
                    const int tq = q_token(p.reverse, si.len, pos0 + i);
                    const int tk = kv_token(p.reverse, si.len, pos0 + i);
                    xq[u] = __ldg(reinterpret_cast<const float4 *>(
                        q + si.b * p.qk_sb + (int64_t)(si.tstart + tq) * p.qk_st + hh * p.qk_sh + d));
                    if (tk >= 0) {
                        xk[u] = __ldg(reinterpret_cast<const float4 *>(
                            k + si.b * p.qk_sb + (int64_t)(si.tstart + tk) * p.qk_st + hh * p.qk_sh + d));
                        if (PERKEY)
                            xg[u] = __ldg(reinterpret_cast<const float4 *>(
                                p.gk + ((si.row0 + tk) * H + hh) * (int64_t)K + d));
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < NQ; ++u) {
                const int e = tid + u * kThreadsF, i = e / KV4, d = (e % KV4) * 4;
                const float qa[4] = {xq[u].x, xq[u].y, xq[u].z, xq[u].w};
                const float ka[4] = {xk[u].x, xk[u].y, xk[u].z, xk[u].w};
                const float ga[4] = {xg[u].x, xg[u].y, xg[u].z, xg[u].w};
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    sQ[i * QS + d + x] = qa[x];
                    sK[i * QS + d + x] = ka[x];
                    if (PERKEY) sGk[i * QS + d + x] = (i < Lc && d < K) ? fmaxf(ga[x], kLogGateMin) : 0.f;
                }
            }
        }
        {
            constexpr int NV = kChunk * (kBVf / 4) / kThreadsF;
            float4 xv[NV];
#pragma unroll
            for (int u = 0; u < NV; ++u) {
                const int e = tid + u * kThreadsF, i = e / (kBVf / 4), n = (e % (kBVf / 4)) * 4, col = v0 + n;
                xv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (i < Lc) {
                    const int tk = kv_token(p.reverse, si.len, pos0 + i);
                    if (tk >= 0) {
                        if (col < V)  // V is a multiple of 8: a group is wholly inside or at V
                            xv[u] = __ldg(reinterpret_cast<const float4 *>(
                                v + si.b * p.v_sb + (int64_t)(si.tstart + tk) * p.v_st + hh * p.v_sh + col));
                        else if (p.has_den && col == V)
                            xv[u].x = 1.f;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < NV; ++u) {
                const int e = tid + u * kThreadsF, i = e / (kBVf / 4), n = (e % (kBVf / 4)) * 4;
                sV[i * VS + n] = xv[u].x;
                sV[i * VS + n + 1] = xv[u].y;
                sV[i * VS + n + 2] = xv[u].z;
                sV[i * VS + n + 3] = xv[u].w;
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
            sB[i] = b;
            sG[i] = gg;
        }
        __syncthreads();
        // ---- optional L2 normalisation of q and k rows; gate cumsums
        if (p.l2norm) {  // two threads per row (128 rows: q then k), then the scaling
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
            for (int d = tid; d < KP; d += kThreadsF) {
                float acc = 0.f;
                for (int i = 0; i < kChunk; ++i) {
                    acc += sGk[i * QS + d];
                    sGk[i * QS + d] = acc;
                }
            }
        } else if (warp == 0) {  // scan over the chunk, two gates per lane
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
        // ---- A (strict lower, beta-scaled) and P (lower incl. diagonal);
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
                    sA[i * AS + j] = a;
                    sP[i * AS + j] = pm;
                }
        } else
        for (int e = tid; e < kChunk * kChunk; e += kThreadsF) {
            const int i = e / kChunk, j = e % kChunk;
            float a = 0.f, pm = 0.f;
            if (j <= i) {
                float sa = 0.f, sp = 0.f;
                if (PERKEY) {
                    for (int d = 0; d < KP; ++d) {
                        const float gam = __expf(sGk[i * QS + d] - sGk[j * QS + d]);
                        const float kj = sK[j * QS + d] * gam;
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
            sA[i * AS + j] = a;
            sP[i * AS + j] = pm;
        }
        __syncthreads();
        // ---- diagonal blocks T_II = (I + A_II)^{-1}, 16 x 16: one warp per
        // block, lane = column, forward substitution in registers
        if (warp < 4 && lane < 16) {
            const int o = 16 * warp;
            float t[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc = (r == lane) ? 1.f : 0.f;
#pragma unroll
                for (int j = 0; j < r; ++j) acc = fmaf(-sA[(o + r) * AS + o + j], t[j], acc);
                t[r] = acc;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) sT[(o + r) * AS + o + lane] = t[r];
        }
        // ---- Y = beta (V - (e^G . K) h) into sX; scalar gate: 2 rows x 4
        // columns per thread (rows ig, ig + 32; columns 4 nq .. 4 nq + 3)
        const int nq = tid & 7, ig = tid >> 3;
        if constexpr (!PERKEY) {
            float acc[2][4];
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) acc[r][c4] = 0.f;
#pragma unroll 4
            for (int d = 0; d < KP; ++d) {
                float hv[4];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) hv[c4] = sH[d * VS + 4 * nq + c4];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float kv = sK[(ig + 32 * r) * QS + d];
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) acc[r][c4] = fmaf(kv, hv[c4], acc[r][c4]);
                }
            }
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int i = ig + 32 * r;
                const float eg = __expf(sG[i]);
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
                    sX[i * VS + 4 * nq + c4] = sB[i] * (sV[i * VS + 4 * nq + c4] - acc[r][c4] * eg);
            }
        } else
        for (int e = tid; e < kChunk * kBVf; e += kThreadsF) {
            const int i = e / kBVf, n = e % kBVf;
            float acc = 0.f;
            if (PERKEY) {
                for (int d = 0; d < KP; ++d)
                    acc = fmaf(sK[i * QS + d] * __expf(sGk[i * QS + d]), sH[d * VS + n], acc);
            } else {
                for (int d = 0; d < KP; ++d) acc = fmaf(sK[i * QS + d], sH[d * VS + n], acc);
                acc *= __expf(sG[i]);
            }
            sX[i * VS + n] = sB[i] * (sV[i * VS + n] - acc);
        }
        __syncthreads();
        // ---- v_new = (I + A)^{-1} Y into sV by block forward substitution,
        // v_new_I = T_II (Y_I - sum_{M<I} A_IM v_new_M), four 16-row blocks
        for (int I = 0; I < 4; ++I) {
            const int o = 16 * I;
            if (I > 0) {
                for (int e = tid; e < 16 * kBVf; e += kThreadsF) {
                    const int i = o + e / kBVf, n = e % kBVf;
                    float a4[4] = {0.f, 0.f, 0.f, 0.f};  // independent partial sums
                    for (int j = 0; j < o; j += 4) {
#pragma unroll
                        for (int u = 0; u < 4; ++u) a4[u] = fmaf(sA[i * AS + j + u], sV[(j + u) * VS + n], a4[u]);
                    }
                    sX[i * VS + n] -= (a4[0] + a4[1]) + (a4[2] + a4[3]);
                }
                __syncthreads();
            }
            for (int e = tid; e < 16 * kBVf; e += kThreadsF) {
                const int i = o + e / kBVf, n = e % kBVf;
                float a4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < 16; ++j) a4[j & 3] = fmaf(sT[i * AS + o + j], sX[(o + j) * VS + n], a4[j & 3]);
                sV[i * VS + n] = (a4[0] + a4[1]) + (a4[2] + a4[3]);
            }
            __syncthreads();
        }
        // ---- o = (e^G . Q) h + P v_new; scalar gate: 2 rows x 4 columns per
        // thread as for Y (P is zero right of the diagonal)
        if constexpr (!PERKEY) {
            float acc[2][4], pv[2][4];
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) acc[r][c4] = pv[r][c4] = 0.f;
#pragma unroll 4
            for (int d = 0; d < KP; ++d) {
                float hv[4];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) hv[c4] = sH[d * VS + 4 * nq + c4];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float qv = sQ[(ig + 32 * r) * QS + d];
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) acc[r][c4] = fmaf(qv, hv[c4], acc[r][c4]);
                }
            }
#pragma unroll 4
            for (int j = 0; j < kChunk; ++j) {
                float vv[4];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) vv[c4] = sV[j * VS + 4 * nq + c4];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float pj = sP[(ig + 32 * r) * AS + j];
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) pv[r][c4] = fmaf(pj, vv[c4], pv[r][c4]);
                }
            }
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int i = ig + 32 * r;
                if (i >= Lc) continue;
                const float eg = __expf(sG[i]);
                const int tq = q_token(p.reverse, si.len, pos0 + i);
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const int col = v0 + 4 * nq + c4;
                    const float val = acc[r][c4] * eg + pv[r][c4];
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
        } else
        for (int e = tid; e < kChunk * kBVf; e += kThreadsF) {
            const int i = e / kBVf, n = e % kBVf, col = v0 + n;
            if (i >= Lc) continue;
            float acc = 0.f;
            if (PERKEY) {
                for (int d = 0; d < KP; ++d)
                    acc = fmaf(sQ[i * QS + d] * __expf(sGk[i * QS + d]), sH[d * VS + n], acc);
            } else {
                for (int d = 0; d < KP; ++d) acc = fmaf(sQ[i * QS + d], sH[d * VS + n], acc);
                acc *= __expf(sG[i]);
            }
            for (int j = 0; j <= i; ++j) acc = fmaf(sP[i * AS + j], sV[j * VS + n], acc);
            const int tq = q_token(p.reverse, si.len, pos0 + i);
            if (col < V) {
                const int64_t off =
                    si.b * p.o_sb + (int64_t)(si.tstart + tq) * p.o_st + hh * p.o_sh + col;
                if (p.out_f32) {
                    float *o = (float *)p.out + off;
                    *o = p.accumulate ? *o + acc : acc;
                } else {
                    __nv_bfloat16 *o = (__nv_bfloat16 *)p.out + off;
                    *o = __float2bfloat16_rn(p.accumulate ? __bfloat162float(*o) + acc : acc);
                }
            } else if (p.has_den && col == V) {
                float *o = p.den + ((int64_t)si.b * H + hh) * p.T + si.tstart + tq;
                *o = p.accumulate ? *o + acc : acc;
            }
        }
        __syncthreads();
        // ---- h <- e^{G_last} h + (e^{G_last - G} . K)^T v_new (scalar gate:
        // beta is no longer needed, its slots take the row factors)
        const int last = Lc - 1;
        if (!PERKEY) {
            if (tid < kChunk) sB[tid] = __expf(sG[last] - sG[tid]);
            __syncthreads();
        }
        if constexpr (!PERKEY) {  // KP / 32 key rows x 4 columns per thread
            constexpr int RD = KP / 32;
            const int dg = tid >> 3;
            const float el = __expf(sG[last]);
            float acc[RD][4];
#pragma unroll
            for (int r = 0; r < RD; ++r)
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) acc[r][c4] = el * sH[(dg + 32 * r) * VS + 4 * nq + c4];
#pragma unroll 4
            for (int i = 0; i < Lc; ++i) {
                const float f = sB[i];
                float vv[4];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) vv[c4] = sV[i * VS + 4 * nq + c4];
#pragma unroll
                for (int r = 0; r < RD; ++r) {
                    const float kf = sK[i * QS + dg + 32 * r] * f;
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) acc[r][c4] = fmaf(kf, vv[c4], acc[r][c4]);
                }
            }
            __syncthreads();  // every thread has read its h block before any is rewritten
#pragma unroll
            for (int r = 0; r < RD; ++r)
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) sH[(dg + 32 * r) * VS + 4 * nq + c4] = acc[r][c4];
        } else
        for (int e = tid; e < KP * kBVf; e += kThreadsF) {
            const int d = e / kBVf, n = e % kBVf;
            float acc;
            if (PERKEY) {
                const float gl = sGk[last * QS + d];
                acc = __expf(gl) * sH[d * VS + n];
                for (int i = 0; i < Lc; ++i)
                    acc = fmaf(sK[i * QS + d] * __expf(gl - sGk[i * QS + d]), sV[i * VS + n], acc);
            } else {
                acc = __expf(sG[last]) * sH[d * VS + n];
                for (int i = 0; i < Lc; ++i) acc = fmaf(sK[i * QS + d] * sB[i], sV[i * VS + n], acc);
            }
            sH[d * VS + n] = acc;
        }
    }
    __syncthreads();
    if (p.h_final) {
        for (int e = tid; e < KP * kBVf; e += kThreadsF) {
            const int d = e / kBVf, n = e % kBVf, col = v0 + n;
            if (d < K && col < p.Vt)
                p.h_final[(((int64_t)s * H + hh) * K + d) * p.Vt + col] = sH[d * VS + n];
        }
    }
}

template <int KP, bool PERKEY>
cudaError_t launch_f32_t(const FwdParams &p, cudaStream_t st) {
    using L = F32Smem<KP, PERKEY>;
    auto kern = fused_f32_kernel<KP, PERKEY>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L::bytes);
    if (e != cudaSuccess) return e;
    dim3 grid(p.n_seq * p.H, (p.Vt + kBVf - 1) / kBVf);
    kern<<<grid, kThreadsF, L::bytes, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fused_f32(const FwdParams &p, int KP, int perkey, cudaStream_t st) {
    if (KP == 64) return perkey ? launch_f32_t<64, true>(p, st) : launch_f32_t<64, false>(p, st);
    return perkey ? launch_f32_t<128, true>(p, st) : launch_f32_t<128, false>(p, st);
}

}  // namespace gdn
