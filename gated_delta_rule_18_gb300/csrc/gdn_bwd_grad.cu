// gdn_bwd_grad.cu -- the chunk-parallel part of the backward: per (64-token
// chunk, head), the input gradients from the chunk's inputs, the state h
// entering it, the state gradient dh' at its end and dL/dv_new (the forward
// snapshots and the dh pass).
//
// Forward per chunk (G the in-chunk cumulative log gate, Gamma_ij =
// e^{G_i - G_j}, q^ / k^ the normalised rows, S = K^ K^T):
//   A   = strictly_lower(diag(beta) (S . Gamma)),  T = (I + A)^{-1}
//   w   = T diag(beta e^{G}) K^,   u = T diag(beta) V,   v_new = u - w h
//   P   = lower_incl(Q^ K^T . Gamma),  o = diag(e^{G}) Q^ h + P v_new
//   h'  = e^{G_C} h + (diag(e^{G_C - G}) K^)^T v_new
// (the WY form of the token rule of the SANA `fused_gdn.py` page; w, u,
// v_new and the h update as on the hyper-parallel coverage_diff page, whose
// backward kernels `chunk_bwd_dqkwg` and `prepare_wy_repr_bwd` split the same
// reverse-mode derivative). With dv_new = dL/dv_new and dh', reverse mode:
//   dP  = lower_incl(do v_new^T),   M_P = dP . Gamma
//   dq^ = e^{G} . (do h^T) + M_P K^
//   dw  = -dv_new h^T,   dB_w = T^T dw,   dB_u = T^T dv_new
//   dA  = -strictly_lower(T^T (dw (beta e^G . K^)^T + dv_new (beta . V)^T) T^T)
//   M_A = dA . Gamma . beta_row,   dS = M_A + M_A^T
//   dk^ = M_P^T Q^ + e^{G_C - G} . (v_new dh'^T) + beta e^{G} . dB_w + dS K^
//   dv  = beta . dB_u
//   dbeta_i = sum_c dB_u v + e^{G_i} sum_d dB_w k^ + sum_j dA_ij (S . Gamma)_ij
//   dG_i   = terms of P, A, qg, kg, B_w and, at the last token, of e^{G_C}
//   dg_i   = sum_{j >= i} dG_j (G is the running sum of g),
// then through the L2 normalisation: dx = (dx^ - x^ (x^ . dx^)) / |x|.
//
// Two kernels share the work (each within the shared-memory budget):
//   bwd_dq  dq, the P and qg parts of dG, and M_P^T Q^ (stored into dk as a
//           partial sum)
//   bwd_dk  dk (adding that partial), dv, dbeta, dg (adding bwd_dq's dG).
// Products run on mma.sync (bf16 operands, fp32 accumulate); T = (I + A)^{-1}
// is formed by blocks (fp32 diagonal inverses, bf16 block products). 8 warps
// per CTA for bwd_dq, 16 for bwd_dk (4 row blocks x 4 column groups).
#include "gdn_bwd_common.cuh"

namespace gdn {
namespace {

// in-chunk cumulative (floored) log gates of the kv rows, and beta
__device__ __forceinline__ void gates(const BwdParams &p, const ChunkCtx &x, float *sG, float *sB, float *graw) {
    const int tid = threadIdx.x;
    if (tid < kChunk) {
        const int tk = tid < x.Lc ? kv_token(p.reverse, x.len, x.pos0 + tid) : -1;
        const int64_t row = (x.row0 + tk) * p.H + x.hh;
        const float g = tk >= 0 ? p.g[row] : 0.f;
        graw[tid] = g;
        sG[tid] = tk >= 0 ? fmaxf(g, kLogGateMin) : 0.f;
        if (sB) sB[tid] = tk >= 0 ? p.beta[row] : 0.f;
    }
    __syncthreads();
    if (tid < 32) {
        const float a0 = sG[2 * tid], a1 = sG[2 * tid + 1];
        float incl = a0 + a1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, o);
            if (tid >= o) incl += y;
        }
        sG[2 * tid] = incl - a1;
        sG[2 * tid + 1] = incl;
    }
    __syncthreads();
}

// ------------------------------------------------------------------ dq ---
struct DqSmem {
    bf16 q[kChunk * kLK], k[kChunk * kLK], dout[kChunk * kLK], vn[kChunk * kLK];
    bf16 h[kKP * kLK];  // (M_P takes the v_new tile's space once dP is formed)
    float G[kChunk], graw[kChunk], rq[kChunk], rk[kChunk], row[kChunk];
    // dG's pieces, one slot per contributing warp (summed in a fixed order):
    // P's row sums by column half, its column sums by row block, qg's by key half
    float dGs[8][kChunk];
};

__global__ void __launch_bounds__(kThreads, 2) bwd_dq_kernel(const BwdParams p) {
    extern __shared__ __align__(16) unsigned char smraw[];
    DqSmem &sm = *reinterpret_cast<DqSmem *>(smraw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, t4 = lane & 3;
    const ChunkCtx x = chunk_ctx(p);
    if (x.s < 0) return;
    const int K = p.K, V = p.V, kq = round16(K), kv = round16(V);
    const bf16 *q = (const bf16 *)p.q, *k = (const bf16 *)p.k, *dout = (const bf16 *)p.dout;

    load_rows(sm.q, kLK, kChunk, K, [&](int i) -> const bf16 * {
        if (i >= x.Lc) return nullptr;
        return q + x.b * p.qk_sb + (int64_t)(x.tstart + q_token(p.reverse, x.len, x.pos0 + i)) * p.qk_st +
               x.hh * p.qk_sh;
    });
    load_rows(sm.k, kLK, kChunk, K, [&](int i) -> const bf16 * {
        const int tk = i < x.Lc ? kv_token(p.reverse, x.len, x.pos0 + i) : -1;
        if (tk < 0) return nullptr;
        return k + x.b * p.qk_sb + (int64_t)(x.tstart + tk) * p.qk_st + x.hh * p.qk_sh;
    });
    cp_async_commit();  // q and k first: the norms and Q K^T start while the rest lands
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
    for (int e = tid; e < 8 * kChunk; e += kThreads) (&sm.dGs[0][0])[e] = 0.f;
    if (tid < kChunk) sm.row[tid] = 0.f;
    gates(p, x, sm.G, nullptr, sm.graw);
    cp_async_wait<1>();
    __syncthreads();
    norm_rows(sm.q, kLK, kq, sm.rq, p.l2norm);
    norm_rows(sm.k, kLK, kq, sm.rk, p.l2norm);
    __syncthreads();

    // P (kept in registers) and dP = do v_new^T on the same fragments
    const int m0 = 16 * (warp & 3), n0 = 32 * (warp >> 2);
    {
        float sp[4][4], dp[4][4];
        acc_zero(sp);
        acc_zero(dp);
        warp_gemm(sp, Tile{sm.q, kLK}, false, Tile{sm.k, kLK}, false, m0, n0, kq, lane);
        cp_async_wait<0>();
        __syncthreads();
        fill_den_dout(p, x, sm.dout, kLK);
        __syncthreads();
        warp_gemm(dp, Tile{sm.dout, kLK}, false, Tile{sm.vn, kLK}, false, m0, n0, kv, lane);
        __syncthreads();  // v_new is read out everywhere: M_P takes its space
        float ct[4][4];  // dP_ij P_ij: d/dG_i of P_ij is P_ij, d/dG_j is -P_ij
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int i = m0 + g8 + 8 * hf;
                float mpv[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int j = n0 + 8 * n + 2 * t4 + e;
                    const bool on = j <= i && i < x.Lc;
                    const float gam = on ? __expf(sm.G[i] - sm.G[j]) : 0.f;
                    const float P = gam * sp[n][2 * hf + e], dP = on ? dp[n][2 * hf + e] : 0.f;
                    mpv[e] = dP * gam;
                    ct[n][2 * hf + e] = dP * P;
                }
                *reinterpret_cast<uint32_t *>(sm.vn + i * kL6 + n0 + 8 * n + 2 * t4) = pack_bf16(mpv[0], mpv[1]);
            }
        rowcol_store(ct, m0, n0, sm.dGs[warp >> 2], sm.dGs[2 + (warp & 3)], -1.f);
    }
    __syncthreads();

    // dq^ = e^{G} . (do h^T) + M_P K^   (64 x 128; warp: 16 rows x 64 keys)
    const int nk0 = 64 * (warp >> 2);
    // e^{G_i} of this thread's two fragment rows
    const float egr[2] = {__expf(sm.G[m0 + g8]), __expf(sm.G[m0 + g8 + 8])};
    float dq[8][4];
    {
        acc_zero(dq);
        warp_gemm(dq, Tile{sm.dout, kLK}, false, Tile{sm.h, kLK}, false, m0, nk0, kv, lane);
        float part[2] = {0.f, 0.f};
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int hf = e >> 1, i = m0 + g8 + 8 * hf, d = nk0 + 8 * n + 2 * t4 + (e & 1);
                const float eg = egr[hf];
                // dG_i of qg = e^{G_i} q^_i: sum_d dqg_id qg_id
                part[hf] += dq[n][e] * eg * __bfloat162float(sm.q[i * kLK + d]);
                dq[n][e] *= eg;
            }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float v = part[hf];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            if (t4 == 0) sm.dGs[6 + (warp >> 2)][m0 + g8 + 8 * hf] = m0 + g8 + 8 * hf < x.Lc ? v : 0.f;
        }
        warp_gemm(dq, Tile{sm.vn, kL6}, false, Tile{sm.k, kLK}, true, m0, nk0, kChunk, lane);
    }
    // through the normalisation: dq = (dq^ - q^ (q^ . dq^)) / |q|
    {
        float part[2] = {0.f, 0.f};
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int hf = e >> 1, i = m0 + g8 + 8 * hf, d = nk0 + 8 * n + 2 * t4 + (e & 1);
                part[hf] += dq[n][e] * __bfloat162float(sm.q[i * kLK + d]);
            }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float v = part[hf];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            if (t4 == 0) atomicAdd(&sm.row[m0 + g8 + 8 * hf], v);
        }
    }
    // an earlier value range's dq, read before any store (the loads then overlap)
    float2 prev[2][8];
    acc_rows_load(prev, p, x, p.dq, m0 + g8, nk0, true, [&](int i) {
        return i < x.Lc ? q_token(p.reverse, x.len, x.pos0 + i) : -1;
    });
    __syncthreads();
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        const int i = m0 + g8 + 8 * hf;
        if (i >= x.Lc) continue;
        const int tq = q_token(p.reverse, x.len, x.pos0 + i);
        float *dst = p.dq + ((x.row0 + tq) * p.H + x.hh) * K;
        const float r = sm.rq[i], dot = sm.row[i];
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const int d = nk0 + 8 * n + 2 * t4;
            if (d >= K) continue;
            float2 o;
            o.x = p.l2norm ? r * (dq[n][2 * hf] - __bfloat162float(sm.q[i * kLK + d]) * dot) : dq[n][2 * hf];
            o.y = p.l2norm ? r * (dq[n][2 * hf + 1] - __bfloat162float(sm.q[i * kLK + d + 1]) * dot)
                           : dq[n][2 * hf + 1];
            if (p.acc) o.x += prev[hf][n].x, o.y += prev[hf][n].y;
            *reinterpret_cast<float2 *>(dst + d) = o;
        }
    }
    // M_P^T Q^: bwd_dk adds it into dk^
    {
        float pk[8][4];
        acc_zero(pk);
        warp_gemm(pk, Tile{sm.vn, kL6}, true, Tile{sm.q, kLK}, true, m0, nk0, kChunk, lane);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int j = m0 + g8 + 8 * hf;
            const int tk = j < x.Lc ? kv_token(p.reverse, x.len, x.pos0 + j) : -1;
            if (tk < 0) continue;
            float *dst = p.dk_part + ((x.row0 + tk) * p.H + x.hh) * K;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                const int d = nk0 + 8 * n + 2 * t4;
                if (d < K) *reinterpret_cast<float2 *>(dst + d) = make_float2(pk[n][2 * hf], pk[n][2 * hf + 1]);
            }
        }
    }
    __syncthreads();
    if (tid < x.Lc) {  // this kernel's share of dG, at the kv rows (bwd_dk adds the rest)
        const int tk = kv_token(p.reverse, x.len, x.pos0 + tid);
        float dGv = 0.f;
#pragma unroll
        for (int x8 = 0; x8 < 8; ++x8) dGv += sm.dGs[x8][tid];
        if (tk >= 0) p.dg_part[(x.row0 + tk) * p.H + x.hh] = dGv;
    }
}

// ------------------------------------------------------------------ dk ---
struct DkP1 {  // until the products with h and dh' are done
    bf16 vn[kChunk * kLK];
    bf16 h[kKP * kLK];
    bf16 dh[kKP * kLK];
};
struct DkP2 {  // afterwards
    bf16 tb[kChunk * kL6];
    bf16 xw[kChunk * kLK];
    bf16 y[kChunk * kL6];
    bf16 z[kChunk * kL6];
    bf16 ms[kChunk * kL6];
};
// NW warps: 4 row blocks of 16 times NQ = NW / 4 column groups
template <int NW>
struct DkSmem {
    static constexpr int NQ = NW / 4;
    bf16 k[kChunk * kLK], v[kChunk * kLK], dvn[kChunk * kLK], dw[kChunk * kLK];
    union {
        DkP1 a;
        DkP2 b;
    } u;
    float kkg[kChunk * kPS];  // (K^ K^T . Gamma), strictly lower
    float G[kChunk], graw[kChunk], beta[kChunk], rk[kChunk];
    // dG's, dbeta's and dG_C's pieces, one slot per contributing warp (summed in
    // a fixed order): dG: kg (by column group), A's rows (column group), A's
    // columns (row block), X_w (column group); dbeta: A, X_w, u (column
    // group); dG_C: the decay per warp, kg per column group and row; the
    // normalisation's row dot dk^ . k^ per column group
    float dGs[3 * NQ + 4][kChunk], dBs[3 * NQ][kChunk], gck[NQ][kChunk], gcs[NW], rowp[NQ][kChunk];
};

template <int NW>
__global__ void __launch_bounds__(NW * 32, 1) bwd_dk_kernel(const BwdParams p) {
    constexpr int NT = NW * 32, NQ = NW / 4;
    constexpr int F64 = 8 / NQ, FK = 16 / NQ;  // 8-column fragments per warp: 64- and 128-wide outputs
    extern __shared__ __align__(16) unsigned char smraw[];
    DkSmem<NW> &sm = *reinterpret_cast<DkSmem<NW> *>(smraw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, hq = warp >> 2;
    const int g8 = lane >> 2, t4 = lane & 3;
    const ChunkCtx x = chunk_ctx(p);
    if (x.s < 0) return;
    const int K = p.K, V = p.V, kq = round16(K), kv = round16(V);
    const bf16 *k = (const bf16 *)p.k, *v = (const bf16 *)p.v;
    auto kv_row = [&](int i) { return i < x.Lc ? kv_token(p.reverse, x.len, x.pos0 + i) : -1; };

    load_rows<NT>(sm.k, kLK, kChunk, K, [&](int i) -> const bf16 * {
        const int tk = kv_row(i);
        return tk < 0 ? nullptr : k + x.b * p.qk_sb + (int64_t)(x.tstart + tk) * p.qk_st + x.hh * p.qk_sh;
    });
    cp_async_commit();  // k first: the norms and K K^T start while the rest lands
    load_rows<NT>(sm.v, kLK, kChunk, value_cols(p), [&](int i) -> const bf16 * {
        const int tk = kv_row(i);
        return tk < 0 ? nullptr : v + x.b * p.v_sb + (int64_t)(x.tstart + tk) * p.v_st + x.hh * p.v_sh;
    });
    load_rows<NT>(sm.dvn, kLK, kChunk, V, [&](int i) -> const bf16 * {
        return p.dvn_snap + (x.gch * kChunk + i) * p.snap_ld;
    });
    load_rows<NT>(sm.u.a.vn, kLK, kChunk, V, [&](int i) -> const bf16 * {
        return p.vn_snap + (x.gch * kChunk + i) * p.snap_ld;
    });
    load_rows<NT>(sm.u.a.h, kLK, kKP, V, [&](int r) -> const bf16 * {
        return r < K ? p.h_snap + (x.gch * K + r) * p.snap_ld : nullptr;
    });
    load_rows<NT>(sm.u.a.dh, kLK, kKP, V, [&](int r) -> const bf16 * {
        return r < K ? p.dh_snap + (x.gch * K + r) * p.snap_ld : nullptr;
    });
    cp_async_commit();
    const int m0 = 16 * (warp & 3), n0 = (64 / NQ) * hq, nk0 = (128 / NQ) * hq;
    // bwd_dq's M_P^T Q^ for this thread's dk fragment, loaded now (added at the end)
    float2 pdk[2][FK];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        const int tk = kv_row(m0 + g8 + 8 * hf);
        const float *src = tk >= 0 ? p.dk_part + ((x.row0 + tk) * p.H + x.hh) * K : nullptr;
#pragma unroll
        for (int n = 0; n < FK; ++n) {
            const int d = nk0 + 8 * n + 2 * t4;
            pdk[hf][n] = (src && d < K) ? *reinterpret_cast<const float2 *>(src + d) : make_float2(0.f, 0.f);
        }
    }
    for (int e = tid; e < (3 * NQ + 4) * kChunk; e += NT) (&sm.dGs[0][0])[e] = 0.f;
    for (int e = tid; e < 3 * NQ * kChunk; e += NT) (&sm.dBs[0][0])[e] = 0.f;
    for (int e = tid; e < NQ * kChunk; e += NT) (&sm.gck[0][0])[e] = (&sm.rowp[0][0])[e] = 0.f;
    gates(p, x, sm.G, sm.beta, sm.graw);
    cp_async_wait<1>();
    __syncthreads();
    norm_rows<NT>(sm.k, kLK, kq, sm.rk, p.l2norm);
    const int last = x.Lc - 1;
    const float GC = sm.G[last];
    __syncthreads();
    // S . Gamma, strictly lower
    {
        float sk[F64][4];
        acc_zero(sk);
        warp_gemm(sk, Tile{sm.k, kLK}, false, Tile{sm.k, kLK}, false, m0, n0, kq, lane);
#pragma unroll
        for (int n = 0; n < F64; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = m0 + g8 + 8 * (e >> 1), j = n0 + 8 * n + 2 * t4 + (e & 1);
                sm.kkg[i * kPS + j] = (j < i && i < x.Lc) ? __expf(sm.G[i] - sm.G[j]) * sk[n][e] : 0.f;
            }
    }
    cp_async_wait<0>();
    __syncthreads();
    fill_den_v(p, x, sm.v, kLK);
    // (the barrier after the decay term below precedes the value tile's readers)
    // e^{G_C} h . dh'  (dG_C of the state decay), 8 columns per step
    {
        float acc = 0.f;
        for (int e = tid; e < K * (kv / 8); e += NT) {
            const int r = e / (kv / 8), c8 = (e % (kv / 8)) * 8;
            const uint4 ua = *reinterpret_cast<const uint4 *>(sm.u.a.h + r * kLK + c8);
            const uint4 ub = *reinterpret_cast<const uint4 *>(sm.u.a.dh + r * kLK + c8);
            const __nv_bfloat162 *a2 = reinterpret_cast<const __nv_bfloat162 *>(&ua);
            const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&ub);
#pragma unroll
            for (int x2 = 0; x2 < 4; ++x2) {
                const float2 a = __bfloat1622float2(a2[x2]), b = __bfloat1622float2(b2[x2]);
                acc = fmaf(a.x, b.x, fmaf(a.y, b.y, acc));
            }
        }
        acc = warp_sum(acc);
        if (lane == 0) sm.gcs[warp] = acc * __expf(GC);
    }
    __syncthreads();

    // factors of this thread's two fragment rows: e^{G_i}, e^{G_C - G_i} (0
    // past the chunk's end)
    float egr[2], ecr[2];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        const int i = m0 + g8 + 8 * hf;
        egr[hf] = __expf(sm.G[i]);
        ecr[hf] = i < x.Lc ? __expf(GC - sm.G[i]) : 0.f;
    }
    // dk^ starts with the kg term: e^{G_C - G} . (v_new dh'^T)
    float dk[FK][4];
    {
        acc_zero(dk);
        warp_gemm(dk, Tile{sm.u.a.vn, kLK}, false, Tile{sm.u.a.dh, kLK}, false, m0, nk0, kv, lane);
        float part[2] = {0.f, 0.f};
#pragma unroll
        for (int n = 0; n < FK; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int hf = e >> 1, i = m0 + g8 + 8 * hf, d = nk0 + 8 * n + 2 * t4 + (e & 1);
                const float f = ecr[hf];
                dk[n][e] *= f;
                part[hf] += dk[n][e] * __bfloat162float(sm.k[i * kLK + d]);
            }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float s = part[hf];
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            if (t4 == 0) {  // kg_i = e^{G_C - G_i} k^_i
                sm.dGs[hq][m0 + g8 + 8 * hf] = -s;
                sm.gck[hq][m0 + g8 + 8 * hf] = s;
            }
        }
    }
    // dw = -v_new' ... = -(dv_new h^T)
    {
        float dw[FK][4];
        acc_zero(dw);
        warp_gemm(dw, Tile{sm.dvn, kLK}, false, Tile{sm.u.a.h, kLK}, false, m0, nk0, kv, lane);
#pragma unroll
        for (int n = 0; n < FK; ++n)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
                *reinterpret_cast<uint32_t *>(sm.dw + (m0 + g8 + 8 * hf) * kLK + nk0 + 8 * n + 2 * t4) =
                    pack_bf16(-dw[n][2 * hf], -dw[n][2 * hf + 1]);
    }
    __syncthreads();  // v_new, h, dh' are done with: their space takes T and the rest

    // T = (I + A)^{-1}, A_ij = beta_i (S . Gamma)_ij (i > j); A and the
    // solve's B_IM take the Y and Z tiles' space until those are formed
    bf16 *sTb = sm.u.b.tb;
    solve_t<NT>(sm.kkg, sm.beta, sTb, sm.u.b.y, sm.u.b.z);
    // X_w = beta e^{G} . K^
    for (int e = tid; e < kChunk * (kKP / 8); e += NT) {
        const int i = e >> 4, d = (e & 15) * 8;
        const float f = sm.beta[i] * __expf(sm.G[i]);
        uint4 u = *reinterpret_cast<const uint4 *>(sm.k + i * kLK + d);
        __nv_bfloat162 *h2 = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
        for (int x2 = 0; x2 < 4; ++x2) {
            const float2 kk = __bfloat1622float2(h2[x2]);
            h2[x2] = __floats2bfloat162_rn(f * kk.x, f * kk.y);
        }
        *reinterpret_cast<uint4 *>(sm.u.b.xw + i * kLK + d) = u;
    }
    __syncthreads();
    const Tile tT{sm.u.b.tb, kL6};
    // Y = dv_new (beta . V)^T + dw X_w^T
    {
        float y[F64][4];
        acc_zero(y);
        warp_gemm(y, Tile{sm.dvn, kLK}, false, Tile{sm.v, kLK}, false, m0, n0, kv, lane);
#pragma unroll
        for (int n = 0; n < F64; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) y[n][e] *= sm.beta[n0 + 8 * n + 2 * t4 + (e & 1)];
        warp_gemm(y, Tile{sm.dw, kLK}, false, Tile{sm.u.b.xw, kLK}, false, m0, n0, kq, lane);
#pragma unroll
        for (int n = 0; n < F64; ++n)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
                *reinterpret_cast<uint32_t *>(sm.u.b.y + (m0 + g8 + 8 * hf) * kL6 + n0 + 8 * n + 2 * t4) =
                    pack_bf16(y[n][2 * hf], y[n][2 * hf + 1]);
    }
    __syncthreads();
    // Z = Y T^T
    {
        float z[F64][4];
        acc_zero(z);
        warp_gemm(z, Tile{sm.u.b.y, kL6}, false, tT, false, m0, n0, kChunk, lane);
#pragma unroll
        for (int n = 0; n < F64; ++n)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
                *reinterpret_cast<uint32_t *>(sm.u.b.z + (m0 + g8 + 8 * hf) * kL6 + n0 + 8 * n + 2 * t4) =
                    pack_bf16(z[n][2 * hf], z[n][2 * hf + 1]);
    }
    __syncthreads();
    // dA = -T^T Z (strictly lower): dbeta, dG, and dS = M_A + M_A^T
    {
        float a[F64][4];
        acc_zero(a);
        warp_gemm(a, tT, true, Tile{sm.u.b.z, kL6}, true, m0, n0, kChunk, lane);
        float pb[2] = {0.f, 0.f};
        float ct[F64][4];  // dA_ij A_ij: d/dG_i of A_ij is A_ij, d/dG_j is -A_ij
#pragma unroll
        for (int n = 0; n < F64; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int hf = e >> 1, i = m0 + g8 + 8 * hf, j = n0 + 8 * n + 2 * t4 + (e & 1);
                float ms = 0.f;
                ct[n][e] = 0.f;
                if (j < i && i < x.Lc) {
                    const float da = -a[n][e], kk = sm.kkg[i * kPS + j];
                    pb[hf] += da * kk;
                    ct[n][e] = da * sm.beta[i] * kk;
                    ms = da * sm.beta[i] * __expf(sm.G[i] - sm.G[j]);
                }
                if (j <= i) {  // (i, j) and its mirror; the diagonal stays 0
                    sm.u.b.ms[i * kL6 + j] = __float2bfloat16_rn(ms);
                    sm.u.b.ms[j * kL6 + i] = __float2bfloat16_rn(ms);
                }
            }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float s = pb[hf];
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            if (t4 == 0) sm.dBs[hq][m0 + g8 + 8 * hf] = s;
        }
        rowcol_store(ct, m0, n0, sm.dGs[NQ + hq], sm.dGs[2 * NQ + (warp & 3)], -1.f);
    }
    __syncthreads();
    // dk^ += dS K^ + beta e^{G} . (T^T dw)
    warp_gemm(dk, Tile{sm.u.b.ms, kL6}, false, Tile{sm.k, kLK}, true, m0, nk0, kChunk, lane);
    {
        float bw[FK][4];
        acc_zero(bw);
        warp_gemm(bw, tT, true, Tile{sm.dw, kLK}, true, m0, nk0, kChunk, lane);
        float part[2] = {0.f, 0.f};
#pragma unroll
        for (int n = 0; n < FK; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int hf = e >> 1, i = m0 + g8 + 8 * hf, d = nk0 + 8 * n + 2 * t4 + (e & 1);
                part[hf] += bw[n][e] * __bfloat162float(sm.k[i * kLK + d]);
                dk[n][e] = fmaf(sm.beta[i] * egr[hf], bw[n][e], dk[n][e]);
            }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float s = part[hf];
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            const int i = m0 + g8 + 8 * hf;
            if (t4 == 0) {
                sm.dBs[NQ + hq][i] = i < x.Lc ? egr[hf] * s : 0.f;
                sm.dGs[2 * NQ + 4 + hq][i] = i < x.Lc ? sm.beta[i] * egr[hf] * s : 0.f;
            }
        }
    }
    // plus bwd_dq's M_P^T Q^, then through the normalisation
    {
        float part[2] = {0.f, 0.f};
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int i = m0 + g8 + 8 * hf;
#pragma unroll
            for (int n = 0; n < FK; ++n) {
                const int d = nk0 + 8 * n + 2 * t4;
                dk[n][2 * hf] += pdk[hf][n].x;
                dk[n][2 * hf + 1] += pdk[hf][n].y;
                part[hf] += dk[n][2 * hf] * __bfloat162float(sm.k[i * kLK + d]) +
                            dk[n][2 * hf + 1] * __bfloat162float(sm.k[i * kLK + d + 1]);
            }
        }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float s = part[hf];
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            if (t4 == 0) sm.rowp[hq][m0 + g8 + 8 * hf] = s;
        }
    }
    // dB_u = T^T dv_new: dv and the beta term of u
    {
        float bu[FK][4];
        acc_zero(bu);
        warp_gemm(bu, tT, true, Tile{sm.dvn, kLK}, true, m0, nk0, kChunk, lane);
        float part[2] = {0.f, 0.f};
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int i = m0 + g8 + 8 * hf;
            const int tk = kv_row(i);
            float *dst = tk >= 0 ? p.dv + ((x.row0 + tk) * p.H + x.hh) * p.dv_ld : nullptr;
#pragma unroll
            for (int n = 0; n < FK; ++n) {
                const int c = nk0 + 8 * n + 2 * t4;
                part[hf] += bu[n][2 * hf] * __bfloat162float(sm.v[i * kLK + c]) +
                            bu[n][2 * hf + 1] * __bfloat162float(sm.v[i * kLK + c + 1]);
                if (dst && c < value_cols(p))
                    *reinterpret_cast<float2 *>(dst + c) =
                        make_float2(sm.beta[i] * bu[n][2 * hf], sm.beta[i] * bu[n][2 * hf + 1]);
            }
        }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float s = part[hf];
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            if (t4 == 0) sm.dBs[2 * NQ + hq][m0 + g8 + 8 * hf] = s;
        }
    }
    __syncthreads();
    // dk out (an earlier value range's dk read first, as for dq)
    float2 prev[2][FK];
    acc_rows_load(prev, p, x, p.dk, m0 + g8, nk0, true, kv_row);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        const int i = m0 + g8 + 8 * hf;
        const int tk = kv_row(i);
        if (tk < 0) continue;
        float *dst = p.dk + ((x.row0 + tk) * p.H + x.hh) * K;
        float dot = 0.f;
#pragma unroll
        for (int q = 0; q < NQ; ++q) dot += sm.rowp[q][i];
        const float r = sm.rk[i];
#pragma unroll
        for (int n = 0; n < FK; ++n) {
            const int d = nk0 + 8 * n + 2 * t4;
            if (d >= K) continue;
            float2 o;
            o.x = p.l2norm ? r * (dk[n][2 * hf] - __bfloat162float(sm.k[i * kLK + d]) * dot) : dk[n][2 * hf];
            o.y = p.l2norm ? r * (dk[n][2 * hf + 1] - __bfloat162float(sm.k[i * kLK + d + 1]) * dot)
                           : dk[n][2 * hf + 1];
            if (p.acc) o.x += prev[hf][n].x, o.y += prev[hf][n].y;
            *reinterpret_cast<float2 *>(dst + d) = o;
        }
    }
    // the reverse scan never reads token 0's key and value: zero gradients
    if (p.reverse && x.c == 0) {
        const int64_t row = x.row0 * p.H + x.hh;
        for (int e = tid; e < K; e += NT) p.dk[row * K + e] = 0.f;
        for (int e = tid; e < value_cols(p); e += NT) p.dv[row * p.dv_ld + e] = 0.f;
        if (tid == 0) p.dbeta[row] = p.dg[row] = 0.f;
    }
    // dbeta, and dg = suffix sums of dG within the chunk (G is the running sum of g)
    if (warp == 0) {
        float d0 = 0.f, d1 = 0.f;
        const int i0 = 2 * lane, i1 = 2 * lane + 1;
        const int t0 = kv_row(i0), t1 = kv_row(i1);
        float dG0 = 0.f, dG1 = 0.f, dB0 = 0.f, dB1 = 0.f;
#pragma unroll
        for (int sl = 0; sl < 3 * NQ + 4; ++sl) dG0 += sm.dGs[sl][i0], dG1 += sm.dGs[sl][i1];
#pragma unroll
        for (int sl = 0; sl < 3 * NQ; ++sl) dB0 += sm.dBs[sl][i0], dB1 += sm.dBs[sl][i1];
        // dG_C: the decay's pieces and the kg terms of every row (a fixed reduction tree)
        float gl = lane < NW ? sm.gcs[lane] : 0.f;
#pragma unroll
        for (int q = 0; q < NQ; ++q) gl += sm.gck[q][i0] + sm.gck[q][i1];
        const float gc = warp_sum(gl);
        const int64_t row0 = (x.row0 + t0) * p.H + x.hh, row1 = (x.row0 + t1) * p.H + x.hh;
        if (t0 >= 0) d0 = dG0 + p.dg_part[row0];
        if (t1 >= 0) d1 = dG1 + p.dg_part[row1];
        // a later value range adds to the earlier ranges' sums: read them
        // here, before the stores below
        float pg0 = 0.f, pb0 = 0.f, pg1 = 0.f, pb1 = 0.f;
        if (p.acc && t0 >= 0) pg0 = p.dg[row0], pb0 = p.dbeta[row0];
        if (p.acc && t1 >= 0) pg1 = p.dg[row1], pb1 = p.dbeta[row1];
        if (i0 == last) d0 += gc;
        if (i1 == last) d1 += gc;
        // suffix sum over lanes of the pair sums
        float incl = d0 + d1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_down_sync(0xffffffffu, incl, o);
            if (lane + o < 32) incl += y;
        }
        const float s1 = incl - d0, s0 = incl;  // dg at i1 and at i0
        if (t0 >= 0) {
            const float dg0 = sm.graw[i0] < kLogGateMin ? 0.f : s0;
            p.dg[row0] = p.acc ? pg0 + dg0 : dg0;
            p.dbeta[row0] = p.acc ? pb0 + dB0 : dB0;
        }
        if (t1 >= 0) {
            const float dg1 = sm.graw[i1] < kLogGateMin ? 0.f : s1;
            p.dg[row1] = p.acc ? pg1 + dg1 : dg1;
            p.dbeta[row1] = p.acc ? pb1 + dB1 : dB1;
        }
    }
}

template <class Kern>
cudaError_t launch_grid(Kern kern, int bytes, const BwdParams &p, cudaStream_t st, int threads = kThreads) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    kern<<<p.max_chunks * p.H, threads, bytes, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq(const BwdParams &p, cudaStream_t st) {
    // two CTAs per SM: ask for the whole shared-memory carveout
    cudaError_t e = cudaFuncSetAttribute(bwd_dq_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    return launch_grid(bwd_dq_kernel, (int)sizeof(DqSmem), p, st);
}
cudaError_t launch_bwd_dk(const BwdParams &p, cudaStream_t st) {
    // 16 warps: half the fragment work per warp of an 8-warp CTA, at one CTA
    // per SM either way (shared memory)
    return launch_grid(bwd_dk_kernel<16>, (int)sizeof(DkSmem<16>), p, st, 16 * 32);
}

}  // namespace gdn
