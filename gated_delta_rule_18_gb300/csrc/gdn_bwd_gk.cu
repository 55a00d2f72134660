// gdn_bwd_gk.cu -- the chunk-parallel part of the backward with per-key
// gates (hyper-parallel coverage_diff page, `chunk_gated_delta_rule_bwd_dhu`
// and its chunk gradient kernels under USE_GK: the decay scales the state's
// key rows). The serial dh pass is shared with the scalar gate: it reads the
// forward's images (qg, kg^T, w, P and the per-key decay), which already
// carry the gates.
//
// Forward per chunk, with G_i the in-chunk cumulative (floored) per-key log
// gate of row i, a K-vector, and x^ the normalised rows:
//   Gam[X, Y]_ij = sum_d X_id Y_jd e^{G_id - G_jd}
//   A   = strictly_lower(diag(beta) Gam[K^, K^]),  T = (I + A)^{-1}
//   w   = T diag(beta) (e^{G} . K^),  u = T diag(beta) V,  v_new = u - w h
//   P   = lower_incl(Gam[Q^, K^]),  o = (e^{G} . Q^) h + P v_new
//   h'  = diag(e^{G_C}) h + (e^{G_C - G} . K^)^T v_new
// Reverse mode with dv_new = dL/dv_new and dh' from the dh pass:
//   dP = lower_incl(do v_new^T), dQp = do h^T, dKc = v_new dh'^T,
//   dw = -dv_new h^T, dB_w = T^T dw, dB_u = T^T dv_new,
//   dA = -strictly_lower(T^T (dw X_w^T + dv_new (beta . V)^T) T^T),
//   M_A = dA . beta_row.
// A gated product Gam[X, Y] with upstream M passes
//   left_i  = sum_j M_ij (Y_j . e^{G_i - G_j})   to X_i, and X_i . left_i to dG_i,
//   right_j = sum_i M_ij (X_i . e^{G_i - G_j})   to Y_j, and -Y_j . right_j to dG_j,
// and a scaled row x_i . e^{c G_i} passes e^{c G_i} . dx_i to x_i and
// c (x_i e^{c G_i}) . dx_i to dG_i. So
//   dq^ = e^{G} . dQp + left(dP; K^)
//   dk^ = right(dP; Q^) + e^{G_C - G} . dKc + left(M_A; K^) + right(M_A; K^)
//         + beta e^{G} . dB_w
//   dG  = the terms above, plus e^{G_C} . rowsum(dh' . h) and
//         sum_i (e^{G_C - G_i} . k^_i) . dKc_i at the chunk's last row,
//   dgk_i = sum_{j >= i in the chunk} dG_j (0 where the forward floored gk),
// then through the L2 normalisation.
//
// Range of the exponentials: e^{G_i - G_j} is formed as
// e^{G_i - G_r} e^{G_r - G_j} about the middle row r of j's (left) or i's
// (right) 16-row block, as the forward's intra-chunk kernel does; with gk
// floored at -10 per token each factor stays below e^80 where it is used,
// and the factor that scales a block's rows outside the triangle is never
// applied. The operand factor goes into a bf16 copy of the tile, the other
// scales the fp32 product.
//
// Two kernels as for the scalar gate: bwd_dq_gk forms dq, the P part of dk
// (into the workspace) and its share of dG (64 x K, into the workspace);
// bwd_dk_gk forms dk, dv, dbeta and dgk. Products on mma.sync (bf16
// operands, fp32 accumulate), 8 warps per CTA.
#include "gdn_bwd_common.cuh"

namespace gdn {
namespace {

// row stride of the fp32 gate tile: the fragment epilogues read it as float2
// pairs at 8 rows x 4 column pairs, conflict-free at this stride
constexpr int kGS = kKP + 8;

// G at (row i, keys d, d + 1), d even
__device__ __forceinline__ float2 g2(const float *G, int i, int d) {
    return *reinterpret_cast<const float2 *>(G + i * kGS + d);
}
// G at (row i, keys d .. d + 7), d a multiple of 8
__device__ __forceinline__ void g8v(const float *G, int i, int d, float *f) {
    const float4 a = *reinterpret_cast<const float4 *>(G + i * kGS + d);
    const float4 b = *reinterpret_cast<const float4 *>(G + i * kGS + d + 4);
    f[0] = a.x, f[1] = a.y, f[2] = a.z, f[3] = a.w, f[4] = b.x, f[5] = b.y, f[6] = b.z, f[7] = b.w;
}

// the raw per-key log gates of the kv rows into G (fp32, row stride kGS),
// by 16-byte async copies in the caller's commit group: keys 64 hf .. 64 hf
// + 63 (256 bytes a row) per half; rows without a token and keys >= K are
// zero-filled
__device__ __forceinline__ void gates_gk_load(const BwdParams &p, const ChunkCtx &x, float *G) {
    const int K = p.K;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        const int k0 = 64 * hf;
        load_rows(reinterpret_cast<bf16 *>(G + k0), 2 * kGS, kChunk, 2 * max(0, min(64, K - k0)),
                  [&](int i) -> const bf16 * {
                      const int tk = i < x.Lc ? kv_token(p.reverse, x.len, x.pos0 + i) : -1;
                      return tk < 0 ? nullptr
                                    : reinterpret_cast<const bf16 *>(p.gk + ((x.row0 + tk) * p.H + x.hh) * K + k0);
                  });
    }
}
// once those copies have landed (and a barrier): the floor of the forward,
// then the in-chunk cumulative sums, one key per thread; ends with a barrier
__device__ __forceinline__ void gates_gk_cumsum(float *G) {
    if (threadIdx.x < kKP) {
        float run = 0.f;
        for (int i = 0; i < kChunk; ++i) {
            run += fmaxf(G[i * kGS + threadIdx.x], kLogGateMinPerKeyTC);  // zero rows stay 0
            G[i * kGS + threadIdx.x] = run;
        }
    }
    __syncthreads();
}

// Items of a 64 x kKP per-key tile by thread: key d = tid % kKP, rows
// tid / kKP + (kThreads / kKP) u for u < kTileItems. Loops over them are
// unrolled with every global load issued before the first use, so a
// thread's loads are in flight together.
constexpr int kRowStep = kThreads / kKP;
constexpr int kTileItems = kChunk / kRowStep;
static_assert(kThreads % kKP == 0, "whole rows of keys per pass");

// scr row j = Y_j . e^{c (G_j - G_r(j))}, r(j) the middle row of j's 16-row
// block (c = -1: the left product's operand, c = +1: the right's); columns
// from kq on are zero (fragments read all 128)
__device__ __forceinline__ void scaled_rows(bf16 *scr, const bf16 *Y, const float *G, int kq, float c) {
    constexpr int n8 = kKP / 8;
    for (int e = threadIdx.x; e < kChunk * n8; e += kThreads) {
        const int j = e / n8, d = (e % n8) * 8, r = (j & ~15) + 8;
        if (d >= kq) {
            *reinterpret_cast<uint4 *>(scr + j * kLK + d) = make_uint4(0, 0, 0, 0);
            continue;
        }
        uint4 u = *reinterpret_cast<const uint4 *>(Y + j * kLK + d);
        __nv_bfloat162 *h2 = reinterpret_cast<__nv_bfloat162 *>(&u);
        float gj[8], gr[8];
        g8v(G, j, d, gj);
        g8v(G, r, d, gr);
#pragma unroll
        for (int x2 = 0; x2 < 4; ++x2) {
            const float2 f = __bfloat1622float2(h2[x2]);
            const float e0 = __expf(c * (gj[2 * x2] - gr[2 * x2]));
            const float e1 = __expf(c * (gj[2 * x2 + 1] - gr[2 * x2 + 1]));
            h2[x2] = __floats2bfloat162_rn(f.x * e0, f.y * e1);
        }
        *reinterpret_cast<uint4 *>(scr + j * kLK + d) = u;
    }
}

// out += left(M; Y) for this warp's fragment (rows m0 .. m0+15, keys nk0 ..
// nk0+63): out_id = sum_j M_ij Y_jd e^{G_id - G_jd}. M: 64 x 64 bf16 (row
// stride kL6), zero outside its triangle (j <= i). scr: a 64 x kLK bf16
// scratch tile. Every thread calls it (barriers inside).
__device__ __forceinline__ void gated_left(float (&out)[8][4], const bf16 *M, const bf16 *Y, const float *G,
                                           bf16 *scr, int kq, int m0, int nk0) {
    const int lane = threadIdx.x & 31, g8 = lane >> 2, t4 = lane & 3;
    scaled_rows(scr, Y, G, kq, -1.f);  // Y_j e^{G_r - G_j}
    __syncthreads();
    if (nk0 < kq) {
        for (int J = 0; 16 * J <= m0; ++J) {  // column blocks that reach this warp's rows
            float c[8][4];
            acc_zero(c);
            warp_gemm(c, Tile{M + 16 * J, kL6}, false, Tile{scr + 16 * J * kLK, kLK}, true, m0, nk0, 16, lane);
            const int r = 16 * J + 8;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                const int d = nk0 + 8 * n + 2 * t4;
                const float2 gr = g2(G, r, d);
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const float2 gi = g2(G, m0 + g8 + 8 * hf, d);
                    out[n][2 * hf] = fmaf(c[n][2 * hf], __expf(gi.x - gr.x), out[n][2 * hf]);
                    out[n][2 * hf + 1] = fmaf(c[n][2 * hf + 1], __expf(gi.y - gr.y), out[n][2 * hf + 1]);
                }
            }
        }
    }
    __syncthreads();
}

// out += right(M; X) for this warp's fragment (rows m0.. are j): out_jd =
// sum_i M_ij X_id e^{G_id - G_jd}, M as for gated_left.
__device__ __forceinline__ void gated_right(float (&out)[8][4], const bf16 *M, const bf16 *X, const float *G,
                                            bf16 *scr, int kq, int m0, int nk0) {
    const int lane = threadIdx.x & 31, g8 = lane >> 2, t4 = lane & 3;
    scaled_rows(scr, X, G, kq, 1.f);  // X_i e^{G_i - G_r}
    __syncthreads();
    if (nk0 < kq) {
        for (int I = m0 / 16; I < 4; ++I) {  // row blocks of M at or below this warp's rows
            float c[8][4];
            acc_zero(c);
            warp_gemm(c, Tile{M + 16 * I * kL6, kL6}, true, Tile{scr + 16 * I * kLK, kLK}, true, m0, nk0, 16, lane);
            const int r = 16 * I + 8;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                const int d = nk0 + 8 * n + 2 * t4;
                const float2 gr = g2(G, r, d);
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const float2 gj = g2(G, m0 + g8 + 8 * hf, d);
                    out[n][2 * hf] = fmaf(c[n][2 * hf], __expf(gr.x - gj.x), out[n][2 * hf]);
                    out[n][2 * hf + 1] = fmaf(c[n][2 * hf + 1], __expf(gr.y - gj.y), out[n][2 * hf + 1]);
                }
            }
        }
    }
    __syncthreads();
}

// value of a bf16 tile at this warp's fragment element (row, key)
__device__ __forceinline__ float tile_at(const bf16 *t, int row, int col) {
    return __bfloat162float(t[row * kLK + col]);
}

// row sums of x . y over this warp's fragment, added into dst[row]
__device__ __forceinline__ void frag_rowdot_add(const float (&x)[8][4], const bf16 *t, int m0, int nk0, float *dst) {
    const int lane = threadIdx.x & 31, g8 = lane >> 2, t4 = lane & 3;
    float part[2] = {0.f, 0.f};
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int hf = e >> 1, i = m0 + g8 + 8 * hf, d = nk0 + 8 * n + 2 * t4 + (e & 1);
            part[hf] += x[n][e] * tile_at(t, i, d);
        }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        float v = part[hf];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        if (t4 == 0 && v != 0.f) atomicAdd(dst + m0 + g8 + 8 * hf, v);
    }
}

// column sums of x over this warp's fragment rows, stored into dst[key]
// (one writer per key and warp: sums stay in a fixed order)
__device__ __forceinline__ void frag_colsum_store(const float (&x)[8][4], int nk0, float *dst) {
    const int lane = threadIdx.x & 31, g8 = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            float v = x[n][b] + x[n][2 + b];
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            if (g8 == 0) dst[nk0 + 8 * n + 2 * t4 + b] = v;
        }
}

// row sums of a warp's fragment reduced over its four t4 lanes and stored
// into dst[row] (one writer per row and warp)
__device__ __forceinline__ void rowsum_store(float (&part)[2], int m0, float *dst) {
    const int lane = threadIdx.x & 31, g8 = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        float v = part[hf];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        if (t4 == 0) dst[m0 + g8 + 8 * hf] = v;
    }
}

// ------------------------------------------------------------------ dq ---
struct GkDqSmem {
    bf16 q[kChunk * kLK], k[kChunk * kLK], dout[kChunk * kLK], vn[kChunk * kLK];
    bf16 h[kKP * kLK];
    bf16 mp[kChunk * kL6];   // dP, lower including the diagonal
    bf16 scr[kChunk * kLK];  // the gated products' scaled operand
    float G[kChunk * kGS];
    float rq[kChunk], rk[kChunk], row[kChunk];
};

__global__ void __launch_bounds__(kThreads, 1) bwd_dq_gk_kernel(const BwdParams p) {
    extern __shared__ __align__(16) unsigned char smraw[];
    GkDqSmem &sm = *reinterpret_cast<GkDqSmem *>(smraw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, t4 = lane & 3;
    const ChunkCtx x = chunk_ctx(p);
    if (x.s < 0) return;
    const int K = p.K, V = p.V, kq = round16(K), kv = round16(V);
    const bf16 *q = (const bf16 *)p.q, *k = (const bf16 *)p.k, *dout = (const bf16 *)p.dout;
    auto kv_row = [&](int i) { return i < x.Lc ? kv_token(p.reverse, x.len, x.pos0 + i) : -1; };

    load_rows(sm.q, kLK, kChunk, K, [&](int i) -> const bf16 * {
        if (i >= x.Lc) return nullptr;
        return q + x.b * p.qk_sb + (int64_t)(x.tstart + q_token(p.reverse, x.len, x.pos0 + i)) * p.qk_st +
               x.hh * p.qk_sh;
    });
    load_rows(sm.k, kLK, kChunk, K, [&](int i) -> const bf16 * {
        const int tk = kv_row(i);
        return tk < 0 ? nullptr : k + x.b * p.qk_sb + (int64_t)(x.tstart + tk) * p.qk_st + x.hh * p.qk_sh;
    });
    gates_gk_load(p, x, sm.G);
    cp_async_commit();
    load_rows(sm.dout, kLK, kChunk, value_cols(p), [&](int i) -> const bf16 * {
        if (i >= x.Lc) return nullptr;
        return dout + x.b * p.do_sb + (int64_t)(x.tstart + q_token(p.reverse, x.len, x.pos0 + i)) * p.do_st +
               x.hh * p.do_sh;
    });
    load_rows(sm.vn, kLK, kChunk, V, [&](int i) -> const bf16 * {
        return p.vn_snap + (x.gch * kChunk + i) * p.snap_ld;
    });
    load_rows(sm.h, kLK, kKP, V, [&](int r) -> const bf16 * {
        return r < K ? p.h_snap + (x.gch * K + r) * p.snap_ld : nullptr;
    });
    cp_async_commit();
    if (tid < kChunk) sm.row[tid] = 0.f;
    cp_async_wait<1>();
    __syncthreads();
    gates_gk_cumsum(sm.G);
    norm_rows(sm.q, kLK, kq, sm.rq, p.l2norm);
    norm_rows(sm.k, kLK, kq, sm.rk, p.l2norm);
    cp_async_wait<0>();
    __syncthreads();
    fill_den_dout(p, x, sm.dout, kLK);
    __syncthreads();

    const int m0 = 16 * (warp & 3), n0 = 32 * (warp >> 2), nk0 = 64 * (warp >> 2);
    {  // dP = lower_incl(do v_new^T)
        float dp[4][4];
        acc_zero(dp);
        warp_gemm(dp, Tile{sm.dout, kLK}, false, Tile{sm.vn, kLK}, false, m0, n0, kv, lane);
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int i = m0 + g8 + 8 * hf, j = n0 + 8 * n + 2 * t4;
                const bool on0 = j <= i && i < x.Lc, on1 = j + 1 <= i && i < x.Lc;
                *reinterpret_cast<uint32_t *>(sm.mp + i * kL6 + j) =
                    pack_bf16(on0 ? dp[n][2 * hf] : 0.f, on1 ? dp[n][2 * hf + 1] : 0.f);
            }
    }
    __syncthreads();
    float dq[8][4], dG[8][4];
    acc_zero(dq);
    acc_zero(dG);
    if (nk0 < kq) {  // e^{G} . (do h^T), and its dG term (e^{G} q^) . dQp
        warp_gemm(dq, Tile{sm.dout, kLK}, false, Tile{sm.h, kLK}, false, m0, nk0, kv, lane);
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int i = m0 + g8 + 8 * hf, d = nk0 + 8 * n + 2 * t4;
                const float2 gi = g2(sm.G, i, d);
                dq[n][2 * hf] *= __expf(gi.x);
                dq[n][2 * hf + 1] *= __expf(gi.y);
                dG[n][2 * hf] = dq[n][2 * hf] * tile_at(sm.q, i, d);
                dG[n][2 * hf + 1] = dq[n][2 * hf + 1] * tile_at(sm.q, i, d + 1);
            }
    }
    {  // left(dP; K^)
        float L[8][4];
        acc_zero(L);
        gated_left(L, sm.mp, sm.k, sm.G, sm.scr, kq, m0, nk0);
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = m0 + g8 + 8 * (e >> 1), d = nk0 + 8 * n + 2 * t4 + (e & 1);
                dq[n][e] += L[n][e];
                dG[n][e] = fmaf(tile_at(sm.q, i, d), L[n][e], dG[n][e]);
            }
    }
    // through the normalisation: dq = (dq^ - q^ (q^ . dq^)) / |q|
    if (nk0 < kq) frag_rowdot_add(dq, sm.q, m0, nk0, sm.row);
    // an earlier value range's dq, read before any store so that the loads
    // do not wait one after another behind the stores
    float2 prev[2][8];
    acc_rows_load(prev, p, x, p.dq, m0 + g8, nk0, nk0 < kq, [&](int i) {
        return i < x.Lc ? q_token(p.reverse, x.len, x.pos0 + i) : -1;
    });
    __syncthreads();
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        const int i = m0 + g8 + 8 * hf;
        if (i >= x.Lc || nk0 >= kq) continue;
        const int tq = q_token(p.reverse, x.len, x.pos0 + i);
        float *dst = p.dq + ((x.row0 + tq) * p.H + x.hh) * K;
        const float r = sm.rq[i], dot = sm.row[i];
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const int d = nk0 + 8 * n + 2 * t4;
            if (d >= K) continue;
            float2 o;
            o.x = p.l2norm ? r * (dq[n][2 * hf] - tile_at(sm.q, i, d) * dot) : dq[n][2 * hf];
            o.y = p.l2norm ? r * (dq[n][2 * hf + 1] - tile_at(sm.q, i, d + 1) * dot) : dq[n][2 * hf + 1];
            if (p.acc) o.x += prev[hf][n].x, o.y += prev[hf][n].y;
            *reinterpret_cast<float2 *>(dst + d) = o;
        }
    }
    {  // right(dP; Q^): the P part of dk^ (workspace), and -k^ . right to dG
        float R[8][4];
        acc_zero(R);
        gated_right(R, sm.mp, sm.q, sm.G, sm.scr, kq, m0, nk0);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int j = m0 + g8 + 8 * hf;
            const int tk = kv_row(j);
#pragma unroll
            for (int n = 0; n < 8; ++n)
#pragma unroll
                for (int b = 0; b < 2; ++b)
                    dG[n][2 * hf + b] = fmaf(-tile_at(sm.k, j, nk0 + 8 * n + 2 * t4 + b), R[n][2 * hf + b],
                                             dG[n][2 * hf + b]);
            if (tk < 0 || nk0 >= kq) continue;
            float *dst = p.dk_part + ((x.row0 + tk) * p.H + x.hh) * K;
            float *gdst = p.dg_part + ((x.row0 + tk) * p.H + x.hh) * K;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                const int d = nk0 + 8 * n + 2 * t4;
                if (d >= K) continue;
                *reinterpret_cast<float2 *>(dst + d) = make_float2(R[n][2 * hf], R[n][2 * hf + 1]);
                *reinterpret_cast<float2 *>(gdst + d) = make_float2(dG[n][2 * hf], dG[n][2 * hf + 1]);
            }
        }
    }
}

// ------------------------------------------------------------------ dk ---
struct GkDkP1 {  // until the products with h and dh' are done
    bf16 vn[kChunk * kLK];
    bf16 h[kKP * kLK];
    bf16 dh[kKP * kLK];
};
struct GkDkP2 {  // afterwards
    bf16 tb[kChunk * kL6], y[kChunk * kL6], z[kChunk * kL6], ms[kChunk * kL6];
    bf16 xw[kChunk * kLK];   // K^ . e^{G - G_r} while Gam[K^, K^] is formed, then X_w
    bf16 scr[kChunk * kLK];
    float dGs[kChunk * kKP];  // dG, for the suffix sums
};
struct GkDkSmem {
    bf16 k[kChunk * kLK], v[kChunk * kLK], dvn[kChunk * kLK], dw[kChunk * kLK];
    union {
        GkDkP1 a;
        GkDkP2 b;
    } u;
    float G[kChunk * kGS];
    float kkg[kChunk * kPS];  // Gam[K^, K^], strictly lower
    float beta[kChunk], rk[kChunk], row[kChunk];
    // dbeta's and the last row's dG pieces, one slot per contributing warp,
    // summed in a fixed order (runs are bit-reproducible)
    float dBp[6][kChunk];  // dA . Gam (2 column halves), X_w (2), u (2)
    float gcp[5][kKP];     // the decay's term, then e^{G_C - G} k^ . dKc per row block
};

__global__ void __launch_bounds__(kThreads, 1) bwd_dk_gk_kernel(const BwdParams p) {
    extern __shared__ __align__(16) unsigned char smraw[];
    GkDkSmem &sm = *reinterpret_cast<GkDkSmem *>(smraw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, t4 = lane & 3;
    const ChunkCtx x = chunk_ctx(p);
    if (x.s < 0) return;
    const int K = p.K, V = p.V, kq = round16(K), kv = round16(V);
    const bf16 *k = (const bf16 *)p.k, *v = (const bf16 *)p.v;
    auto kv_row = [&](int i) { return i < x.Lc ? kv_token(p.reverse, x.len, x.pos0 + i) : -1; };

    load_rows(sm.k, kLK, kChunk, K, [&](int i) -> const bf16 * {
        const int tk = kv_row(i);
        return tk < 0 ? nullptr : k + x.b * p.qk_sb + (int64_t)(x.tstart + tk) * p.qk_st + x.hh * p.qk_sh;
    });
    gates_gk_load(p, x, sm.G);
    cp_async_commit();
    load_rows(sm.v, kLK, kChunk, value_cols(p), [&](int i) -> const bf16 * {
        const int tk = kv_row(i);
        return tk < 0 ? nullptr : v + x.b * p.v_sb + (int64_t)(x.tstart + tk) * p.v_st + x.hh * p.v_sh;
    });
    load_rows(sm.dvn, kLK, kChunk, V, [&](int i) -> const bf16 * {
        return p.dvn_snap + (x.gch * kChunk + i) * p.snap_ld;
    });
    load_rows(sm.u.a.vn, kLK, kChunk, V, [&](int i) -> const bf16 * {
        return p.vn_snap + (x.gch * kChunk + i) * p.snap_ld;
    });
    load_rows(sm.u.a.h, kLK, kKP, V, [&](int r) -> const bf16 * {
        return r < K ? p.h_snap + (x.gch * K + r) * p.snap_ld : nullptr;
    });
    load_rows(sm.u.a.dh, kLK, kKP, V, [&](int r) -> const bf16 * {
        return r < K ? p.dh_snap + (x.gch * K + r) * p.snap_ld : nullptr;
    });
    cp_async_commit();
    if (tid < kChunk) {
        const int tk = kv_row(tid);
        sm.beta[tid] = tk >= 0 ? p.beta[(x.row0 + tk) * p.H + x.hh] : 0.f;
        sm.row[tid] = 0.f;
#pragma unroll
        for (int x6 = 0; x6 < 6; ++x6) sm.dBp[x6][tid] = 0.f;
    }
    if (tid < kKP)
#pragma unroll
        for (int x5 = 0; x5 < 5; ++x5) sm.gcp[x5][tid] = 0.f;
    cp_async_wait<1>();
    __syncthreads();
    gates_gk_cumsum(sm.G);
    norm_rows(sm.k, kLK, kq, sm.rk, p.l2norm);
    cp_async_wait<0>();
    __syncthreads();
    fill_den_v(p, x, sm.v, kLK);
    __syncthreads();
    const int last = x.Lc - 1;
    const int m0 = 16 * (warp & 3), n0 = 32 * (warp >> 2), nk0 = 64 * (warp >> 2);

    // the state decay's term at the last row: e^{G_C} . rowsum(dh' . h)
    for (int d = tid; d < K; d += kThreads) {
        float acc = 0.f;
        for (int c8 = 0; c8 < kv; c8 += 8) {
            const uint4 ua = *reinterpret_cast<const uint4 *>(sm.u.a.h + d * kLK + c8);
            const uint4 ub = *reinterpret_cast<const uint4 *>(sm.u.a.dh + d * kLK + c8);
            const __nv_bfloat162 *a2 = reinterpret_cast<const __nv_bfloat162 *>(&ua);
            const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&ub);
#pragma unroll
            for (int x2 = 0; x2 < 4; ++x2) {
                const float2 a = __bfloat1622float2(a2[x2]), b = __bfloat1622float2(b2[x2]);
                acc = fmaf(a.x, b.x, fmaf(a.y, b.y, acc));
            }
        }
        sm.gcp[0][d] = acc * __expf(sm.G[last * kGS + d]);
    }
    float dk[8][4], dG[8][4];
    acc_zero(dk);
    acc_zero(dG);
    if (nk0 < kq) {  // dKc = v_new dh'^T: dk^ += e^{G_C - G} . dKc; dG -= Kc . dKc; last row += colsum
        float c[8][4];
        acc_zero(c);
        warp_gemm(c, Tile{sm.u.a.vn, kLK}, false, Tile{sm.u.a.dh, kLK}, false, m0, nk0, kv, lane);
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const int d0 = nk0 + 8 * n + 2 * t4;
            const float2 gl = g2(sm.G, last, d0);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int i = m0 + g8 + 8 * hf;
                const float2 gi = g2(sm.G, i, d0);
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    const int e = 2 * hf + b;
                    const float f = i < x.Lc ? __expf((b ? gl.y : gl.x) - (b ? gi.y : gi.x)) : 0.f;
                    dk[n][e] = f * c[n][e];
                    c[n][e] = f * tile_at(sm.k, i, d0 + b) * c[n][e];  // Kc . dKc
                    dG[n][e] = -c[n][e];
                }
            }
        }
        frag_colsum_store(c, nk0, sm.gcp[1 + (warp & 3)]);
    }
    if (nk0 < kq) {  // dw = -(dv_new h^T)
        float dw[8][4];
        acc_zero(dw);
        warp_gemm(dw, Tile{sm.dvn, kLK}, false, Tile{sm.u.a.h, kLK}, false, m0, nk0, kv, lane);
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
                *reinterpret_cast<uint32_t *>(sm.dw + (m0 + g8 + 8 * hf) * kLK + nk0 + 8 * n + 2 * t4) =
                    pack_bf16(-dw[n][2 * hf], -dw[n][2 * hf + 1]);
    } else if (nk0 < kKP) {  // keys past K: zero columns of the tile
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
                *reinterpret_cast<uint32_t *>(sm.dw + (m0 + g8 + 8 * hf) * kLK + nk0 + 8 * n + 2 * t4) = 0u;
    }
    __syncthreads();  // v_new, h, dh' are done with: their space takes T and the rest

    // Gam[K^, K^], strictly lower: column block J is
    // (K^ . e^{G - G_r}) (K^_J . e^{G_r - G_J})^T over the rows i >= 16 J
    scaled_rows(sm.u.b.scr, sm.k, sm.G, kq, -1.f);
    for (int J = 0; J < 4; ++J) {
        const int r = 16 * J + 8, n8 = kq / 8;
        for (int e = tid; e < kChunk * n8; e += kThreads) {
            const int i = e / n8, d = (e % n8) * 8;
            uint4 u = make_uint4(0, 0, 0, 0);
            if (i >= 16 * J) {
                u = *reinterpret_cast<const uint4 *>(sm.k + i * kLK + d);
                __nv_bfloat162 *h2 = reinterpret_cast<__nv_bfloat162 *>(&u);
                float gi[8], gr[8];
                g8v(sm.G, i, d, gi);
                g8v(sm.G, r, d, gr);
#pragma unroll
                for (int x2 = 0; x2 < 4; ++x2) {
                    const float2 f = __bfloat1622float2(h2[x2]);
                    h2[x2] = __floats2bfloat162_rn(f.x * __expf(gi[2 * x2] - gr[2 * x2]),
                                                   f.y * __expf(gi[2 * x2 + 1] - gr[2 * x2 + 1]));
                }
            }
            *reinterpret_cast<uint4 *>(sm.u.b.xw + i * kLK + d) = u;
        }
        __syncthreads();
        if (warp < 4 && warp >= J) {  // rows 16 warp .. 16 warp + 15, columns 16 J .. 16 J + 15
            float c2[2][4];
            acc_zero(c2);
            warp_gemm(c2, Tile{sm.u.b.xw, kLK}, false, Tile{sm.u.b.scr, kLK}, false, 16 * warp, 16 * J, kq, lane);
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = 16 * warp + g8 + 8 * (e >> 1), j = 16 * J + 8 * n + 2 * t4 + (e & 1);
                    sm.kkg[i * kPS + j] = (j < i && i < x.Lc) ? c2[n][e] : 0.f;
                }
        }
        __syncthreads();
    }
    // T = (I + A)^{-1}, A_ij = beta_i Gam_ij (i > j); A and the solve's
    // B_IM take the Y and Z tiles' space until those are formed
    const Tile tT{sm.u.b.tb, kL6};
    solve_t(sm.kkg, sm.beta, sm.u.b.tb, sm.u.b.y, sm.u.b.z);
    // X_w = beta e^{G} . K^
    for (int e = tid; e < kChunk * (kKP / 8); e += kThreads) {
        const int i = e >> 4, d = (e & 15) * 8;
        uint4 u = *reinterpret_cast<const uint4 *>(sm.k + i * kLK + d);
        __nv_bfloat162 *h2 = reinterpret_cast<__nv_bfloat162 *>(&u);
        float gi[8];
        g8v(sm.G, i, d, gi);
        const float bi = sm.beta[i];
#pragma unroll
        for (int x2 = 0; x2 < 4; ++x2) {
            const float2 kk = __bfloat1622float2(h2[x2]);
            h2[x2] = __floats2bfloat162_rn(bi * __expf(gi[2 * x2]) * kk.x, bi * __expf(gi[2 * x2 + 1]) * kk.y);
        }
        *reinterpret_cast<uint4 *>(sm.u.b.xw + i * kLK + d) = u;
    }
    __syncthreads();
    {  // Y = dv_new (beta . V)^T + dw X_w^T
        float y[4][4];
        acc_zero(y);
        warp_gemm(y, Tile{sm.dvn, kLK}, false, Tile{sm.v, kLK}, false, m0, n0, kv, lane);
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) y[n][e] *= sm.beta[n0 + 8 * n + 2 * t4 + (e & 1)];
        warp_gemm(y, Tile{sm.dw, kLK}, false, Tile{sm.u.b.xw, kLK}, false, m0, n0, kq, lane);
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
                *reinterpret_cast<uint32_t *>(sm.u.b.y + (m0 + g8 + 8 * hf) * kL6 + n0 + 8 * n + 2 * t4) =
                    pack_bf16(y[n][2 * hf], y[n][2 * hf + 1]);
    }
    __syncthreads();
    {  // Z = Y T^T
        float z[4][4];
        acc_zero(z);
        warp_gemm(z, Tile{sm.u.b.y, kL6}, false, tT, false, m0, n0, kChunk, lane);
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
                *reinterpret_cast<uint32_t *>(sm.u.b.z + (m0 + g8 + 8 * hf) * kL6 + n0 + 8 * n + 2 * t4) =
                    pack_bf16(z[n][2 * hf], z[n][2 * hf + 1]);
    }
    __syncthreads();
    {  // dA = -T^T Z (strictly lower): dbeta, and M_A = dA . beta_row
        float a[4][4];
        acc_zero(a);
        warp_gemm(a, tT, true, Tile{sm.u.b.z, kL6}, true, m0, n0, kChunk, lane);
        float pb[2] = {0.f, 0.f};
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int i = m0 + g8 + 8 * hf, j = n0 + 8 * n + 2 * t4;
                float ma[2];
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    ma[b] = 0.f;
                    if (j + b < i && i < x.Lc) {
                        const float da = -a[n][2 * hf + b];
                        pb[hf] += da * sm.kkg[i * kPS + j + b];
                        ma[b] = da * sm.beta[i];
                    }
                }
                *reinterpret_cast<uint32_t *>(sm.u.b.ms + i * kL6 + j) = pack_bf16(ma[0], ma[1]);
            }
        rowsum_store(pb, m0, sm.dBp[warp >> 2]);
    }
    __syncthreads();
    {  // left(M_A; K^) and right(M_A; K^): dk^ += both, dG += k^ . (left - right)
        float lr[8][4];
        acc_zero(lr);
        gated_left(lr, sm.u.b.ms, sm.k, sm.G, sm.u.b.scr, kq, m0, nk0);
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = m0 + g8 + 8 * (e >> 1), d = nk0 + 8 * n + 2 * t4 + (e & 1);
                dk[n][e] += lr[n][e];
                dG[n][e] = fmaf(tile_at(sm.k, i, d), lr[n][e], dG[n][e]);
            }
        acc_zero(lr);
        gated_right(lr, sm.u.b.ms, sm.k, sm.G, sm.u.b.scr, kq, m0, nk0);
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = m0 + g8 + 8 * (e >> 1), d = nk0 + 8 * n + 2 * t4 + (e & 1);
                dk[n][e] += lr[n][e];
                dG[n][e] = fmaf(-tile_at(sm.k, i, d), lr[n][e], dG[n][e]);
            }
    }
    if (nk0 < kq) {  // beta e^{G} . (T^T dw): dk^, dbeta and dG (Kp = e^{G} . k^)
        float bw[8][4];
        acc_zero(bw);
        warp_gemm(bw, tT, true, Tile{sm.dw, kLK}, true, m0, nk0, kChunk, lane);
        float part[2] = {0.f, 0.f};
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int i = m0 + g8 + 8 * hf, d0 = nk0 + 8 * n + 2 * t4;
                const float2 gi = g2(sm.G, i, d0);
                const float bi = sm.beta[i];
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    const int e = 2 * hf + b;
                    const float eg = __expf(b ? gi.y : gi.x);
                    const float kp = eg * tile_at(sm.k, i, d0 + b);
                    part[hf] += bw[n][e] * kp;
                    dk[n][e] = fmaf(bi * eg, bw[n][e], dk[n][e]);
                    dG[n][e] = fmaf(bi * kp, bw[n][e], dG[n][e]);
                }
            }
        rowsum_store(part, m0, sm.dBp[2 + (warp >> 2)]);
    }
    // plus bwd_dq_gk's right(dP; Q^), then through the normalisation
    if (nk0 < kq) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int i = m0 + g8 + 8 * hf;
            const int tk = kv_row(i);
            const float *src = tk >= 0 ? p.dk_part + ((x.row0 + tk) * p.H + x.hh) * K : nullptr;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                const int d = nk0 + 8 * n + 2 * t4;
                if (src && d < K) {
                    const float2 a = *reinterpret_cast<const float2 *>(src + d);
                    dk[n][2 * hf] += a.x;
                    dk[n][2 * hf + 1] += a.y;
                }
            }
        }
        frag_rowdot_add(dk, sm.k, m0, nk0, sm.row);
    }
    if (nk0 < kv) {  // dB_u = T^T dv_new: dv and the beta term of u (value columns nk0 ..)
        float bu[8][4];
        acc_zero(bu);
        warp_gemm(bu, tT, true, Tile{sm.dvn, kLK}, true, m0, nk0, kChunk, lane);
        float part[2] = {0.f, 0.f};
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int i = m0 + g8 + 8 * hf;
            const int tk = kv_row(i);
            float *dst = tk >= 0 ? p.dv + ((x.row0 + tk) * p.H + x.hh) * p.dv_ld : nullptr;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                const int c = nk0 + 8 * n + 2 * t4;
                part[hf] += bu[n][2 * hf] * tile_at(sm.v, i, c) + bu[n][2 * hf + 1] * tile_at(sm.v, i, c + 1);
                if (dst && c < value_cols(p))
                    *reinterpret_cast<float2 *>(dst + c) =
                        make_float2(sm.beta[i] * bu[n][2 * hf], sm.beta[i] * bu[n][2 * hf + 1]);
            }
        }
        rowsum_store(part, m0, sm.dBp[4 + (warp >> 2)]);
    }
    // this warp's dG rows into shared memory (keys past K and rows past the
    // chunk stay 0), bwd_dq_gk's share and the last row's terms added there
    for (int e = tid; e < kChunk * kKP; e += kThreads) sm.u.b.dGs[e] = 0.f;
    __syncthreads();
    if (nk0 < kq) {
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = m0 + g8 + 8 * (e >> 1), d = nk0 + 8 * n + 2 * t4 + (e & 1);
                if (i < x.Lc && d < K) sm.u.b.dGs[i * kKP + d] = dG[n][e];
            }
    }
    __syncthreads();
    // dk out (an earlier value range's dk read first, as for dq)
    {
        float2 prev[2][8];
        acc_rows_load(prev, p, x, p.dk, m0 + g8, nk0, nk0 < kq, kv_row);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int i = m0 + g8 + 8 * hf;
            const int tk = kv_row(i);
            if (tk < 0 || nk0 >= kq) continue;
            float *dst = p.dk + ((x.row0 + tk) * p.H + x.hh) * K;
            const float r = sm.rk[i], dot = sm.row[i];
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                const int d = nk0 + 8 * n + 2 * t4;
                if (d >= K) continue;
                float2 o;
                o.x = p.l2norm ? r * (dk[n][2 * hf] - tile_at(sm.k, i, d) * dot) : dk[n][2 * hf];
                o.y = p.l2norm ? r * (dk[n][2 * hf + 1] - tile_at(sm.k, i, d + 1) * dot) : dk[n][2 * hf + 1];
                if (p.acc) o.x += prev[hf][n].x, o.y += prev[hf][n].y;
                *reinterpret_cast<float2 *>(dst + d) = o;
            }
        }
    }
    // the reverse scan never reads token 0's key and value: zero gradients
    if (p.reverse && x.c == 0) {
        const int64_t row = x.row0 * p.H + x.hh;
        for (int e = tid; e < K; e += kThreads) p.dk[row * K + e] = p.dg[row * K + e] = 0.f;
        for (int e = tid; e < value_cols(p); e += kThreads) p.dv[row * p.dv_ld + e] = 0.f;
        if (tid == 0) p.dbeta[row] = 0.f;
    }
    // dbeta, and dgk = suffix sums of dG within the chunk, one key per thread
    if (tid < kChunk) {
        const int tk = kv_row(tid);
        if (tk >= 0) {
            const int64_t row = (x.row0 + tk) * p.H + x.hh;
            float db = 0.f;
#pragma unroll
            for (int x6 = 0; x6 < 6; ++x6) db += sm.dBp[x6][tid];
            p.dbeta[row] = p.acc ? p.dbeta[row] + db : db;
        }
    }
    // (1) every term of dG_i: bwd_dq_gk's share and the last row's terms;
    // whether the forward floored gk there (its derivative is then 0). The
    // global loads are coalesced over keys and independent of one another.
    unsigned char *floored = reinterpret_cast<unsigned char *>(sm.u.b.scr);  // [64][kKP]
    const int dk0 = tid % kKP, ir = tid / kKP;
    {
        float part[kTileItems], graw[kTileItems];
#pragma unroll
        for (int u = 0; u < kTileItems; ++u) {
            const int i = ir + kRowStep * u, tk = kv_row(i);
            part[u] = graw[u] = 0.f;
            if (tk >= 0 && dk0 < K) {
                const int64_t row = ((x.row0 + tk) * p.H + x.hh) * K + dk0;
                part[u] = p.dg_part[row];
                graw[u] = p.gk[row];
            }
        }
#pragma unroll
        for (int u = 0; u < kTileItems; ++u) {
            const int i = ir + kRowStep * u, tk = kv_row(i);
            if (i >= x.Lc || dk0 >= K) continue;
            float t = sm.u.b.dGs[i * kKP + dk0] + part[u];
            if (i == last)
#pragma unroll
                for (int x5 = 0; x5 < 5; ++x5) t += sm.gcp[x5][dk0];
            sm.u.b.dGs[i * kKP + dk0] = t;
            floored[i * kKP + dk0] = tk >= 0 && graw[u] < kLogGateMinPerKeyTC;
        }
    }
    __syncthreads();
    // (2) suffix sums within the chunk, one key per thread, in shared memory
    for (int d = tid; d < K; d += kThreads) {
        float run = 0.f;
        for (int i = x.Lc - 1; i >= 0; --i) {
            run += sm.u.b.dGs[i * kKP + d];
            sm.u.b.dGs[i * kKP + d] = floored[i * kKP + d] ? 0.f : run;
        }
    }
    __syncthreads();
    // (3) the stores (a later value range adds to the earlier ranges' sums)
    {
        float prev[kTileItems];
#pragma unroll
        for (int u = 0; u < kTileItems; ++u) {
            const int i = ir + kRowStep * u, tk = kv_row(i);
            prev[u] = (p.acc && tk >= 0 && dk0 < K) ? p.dg[((x.row0 + tk) * p.H + x.hh) * K + dk0] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kTileItems; ++u) {
            const int i = ir + kRowStep * u, tk = kv_row(i);
            if (tk < 0 || dk0 >= K) continue;
            p.dg[((x.row0 + tk) * p.H + x.hh) * K + dk0] = prev[u] + sm.u.b.dGs[i * kKP + dk0];
        }
    }
}

template <class Kern>
cudaError_t launch_gk(Kern kern, int bytes, const BwdParams &p, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    kern<<<p.max_chunks * p.H, kThreads, bytes, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq_gk(const BwdParams &p, cudaStream_t st) {
    return launch_gk(bwd_dq_gk_kernel, (int)sizeof(GkDqSmem), p, st);
}
cudaError_t launch_bwd_dk_gk(const BwdParams &p, cudaStream_t st) {
    return launch_gk(bwd_dk_gk_kernel, (int)sizeof(GkDkSmem), p, st);
}

}  // namespace gdn
