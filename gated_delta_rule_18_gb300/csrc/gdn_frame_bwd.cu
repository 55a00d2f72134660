// gdn_frame_bwd.cu -- gradients of the frame-causal rule (SANA `fused_gdn.py`
// page, `_fused_gdn_bwd_kernel`; SANA `fused_cam_gdn.py` page,
// `_cam_scan_bwd_kernel`), for q, k as the forward takes them (prepared).
//
// Forward per frame f (S tokens, keys K_f, values X_f = [V_f | 1], betas,
// log decay g_f): P_f = e^{g_f} S_prev, S_f = A_f P_f + B_f with
// A_f = I - K_f^T diag(beta) K_f (symmetric), B_f = K_f^T diag(beta) X_f, and
// the frame's outputs O_f = Q_f R_f read a state R_f: the causal direction
// reads S_f itself, the reverse reads the state built from the later frames
// (frame f's write then yields the state frame f-1 reads). In the order the
// writes happen, each write is followed by the frame that reads its result.
// With Lam = dL/d(state after a write) and [dO | dden] the upstream gradient
// of [O | den]:
//   Lam(write of f) = Q_r^T [dO | dden]_r + e^{g_n} A_n Lam(write of n)
// where r reads the write's result and n is the next write (dh_final after
// the causal direction's last), and per token t of the written frame, with
// u_t = Lam^T k_t and the prediction error e_t = x_t - P_f^T k_t:
//   dv_t = beta_t u_t,  dbeta_t = u_t . e_t,
//   dk_t = beta_t (Lam e_t - P_f u_t)  (P_f = e^{g_f} S_prev, as predicted from),
//   dg_f = e^{g_f} sum(A_f Lam . S_prev),  dS_prev = e^{g_f} A_f Lam (dh0),
// and per token of the reading frame dq_t = R_f [do_t | dden_t].
// Three kernels (frame_xt once, the other two per direction):
//   frame_xt      per (sequence x head, frame): C_f = Q_f^T [dO_f | dden_f]
//                 over the frame's chunks on tensor cores (mma.sync); both
//                 directions read it
//   frame_lam     per (sequence x head, 32-column tile): the fp32 chain of
//                 Lam over the writes in reverse order, A_f applied from
//                 shared memory (copied in one step ahead); the dg_f parts
//                 of its tile; dh0
//   frame_tokgrad per (sequence x head, 1 to 4 chunks of one frame): U = K
//                 Lam, E = X - K P, dv, dbeta, dk = beta (E Lam^T - U P^T),
//                 dq = [dO | dden] R^T on tensor cores, and dg_frame from
//                 the parts
// The two directions of a bidirectional pass run one after the other, the
// second adding into the first's outputs (reductions for the per-token
// gradients).
#include "gdn_frame_bwd.cuh"
#include "gdn_mma.cuh"

namespace gdn {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kThreads = 256;
constexpr int kKS = kKP + 8;  // bf16 row stride of 128-column tiles

// ------------------------------------------------------------------ xt ---
struct XtStage {
    bf16 q[kChunk * kKS];  // [token][key]
    bf16 x[kChunk * kKS];  // [token][column]: dO, then dden in column V
};
struct XtSmem {
    XtStage st[2];
};

// Two CTAs per SM (at most 128 registers a thread): a grid of (sequence x
// head, frame) CTAs, 256 on the video shape, is then resident in one wave.
__global__ void __launch_bounds__(kThreads, 2) frame_xt_kernel(const FrameBwdParams p) {
    extern __shared__ __align__(16) unsigned char smraw[];
    XtSmem &sm = *reinterpret_cast<XtSmem *>(smraw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g8 = lane >> 2, t4 = lane & 3;
    const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H, f = blockIdx.y;
    const int K = p.K, V = p.V, Vs = p.Vs;
    const int nch = p.frame / kChunk;
    const bf16 *q = (const bf16 *)p.q, *dout = (const bf16 *)p.dout;
    auto stage = [&](int c) {
        XtStage &S = sm.st[c & 1];
        const int64_t t0 = (int64_t)f * p.frame + (int64_t)c * kChunk;
        for (int e = tid; e < kChunk * (kKP / 8); e += kThreads) {
            const int i = e >> 4, c8 = (e & 15) * 8;
            const int64_t t = t0 + i;
            const bool inq = c8 < K, inx = c8 < V;
            cp_async16(S.q + i * kKS + c8, inq ? q + b * p.qk_sb + t * p.qk_st + h * p.qk_sh + c8 : q, inq ? 16 : 0);
            cp_async16(S.x + i * kKS + c8, inx ? dout + b * p.do_sb + t * p.do_st + h * p.do_sh + c8 : dout,
                       inx ? 16 : 0);
        }
        cp_async_commit();
    };
    float c[2][8][4];
    acc_zero(c[0]);
    acc_zero(c[1]);
    const int n0 = 64 * (warp >> 2);
    stage(0);
    for (int ci = 0; ci < nch; ++ci) {
        if (ci + 1 < nch) {
            stage(ci + 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        XtStage &S = sm.st[ci & 1];
        if (p.dden && tid < kChunk) {  // the ones column's upstream gradient (zero copies landed there)
            const int64_t t = (int64_t)f * p.frame + (int64_t)ci * kChunk + tid;
            S.x[tid * kKS + V] = __float2bfloat16_rn(p.dden[((int64_t)b * p.H + h) * p.T + t]);
        }
        __syncthreads();
        if (n0 < Vs)
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
                warp_gemm(c[mt], Tile{S.q, kKS}, true, Tile{S.x, kKS}, true, 32 * (warp & 3) + 16 * mt, n0, kChunk,
                          lane);
        __syncthreads();  // this stage is refilled next
    }
    if (n0 >= Vs) return;
    float *dst = p.cmat + ((int64_t)bh * p.F + f) * K * Vs;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int r = 32 * (warp & 3) + 16 * mt + g8 + 8 * hf, col = n0 + 8 * n + 2 * t4;
                if (r < K && col < Vs)
                    *reinterpret_cast<float2 *>(dst + (int64_t)r * Vs + col) =
                        make_float2(c[mt][n][2 * hf], c[mt][n][2 * hf + 1]);
            }
}

// ----------------------------------------------------------------- lam ---
// The writes of direction d in the order they happen: step c writes frame
// w(c); the frame that reads its result is r(c).
__device__ __forceinline__ int write_frame(int d, int F, int c) { return d == 0 ? c : F - 1 - c; }
__device__ __forceinline__ int read_frame(int d, int F, int c) { return d == 0 ? c : F - 2 - c; }

struct LamSmem {
    float a[2][kKP * kKP];          // A_f of this step and of the next
    float s[kKP * kFrameBwdCT];     // Lam tile, [key][column]
    float red[kThreads / 32];
};
__device__ __forceinline__ void lam_stage_a(const FrameBwdParams &p, LamSmem &sm, int buf, int64_t fi) {
    const int K = p.K, c = (threadIdx.x & 31) * 4;
    const float *A = p.amat + fi * K * K;
    if (c < K)
        for (int r = threadIdx.x >> 5; r < K; r += 8)
            cp_async16(sm.a[buf] + r * kKP + c, A + (int64_t)r * K + c, 16);
    cp_async_commit();
}
// the state frame w's write starts from (K x Vt fp32 at row stride ld), or
// null for the zero state
__device__ __forceinline__ const float *pre_state(const FrameBwdParams &p, int64_t bh, int w, int &ld) {
    ld = p.Vs;
    if (p.direction == 1) return p.sread + ((int64_t)bh * p.F + w) * p.K * p.Vs;
    if (w > 0) return p.sread + ((int64_t)bh * p.F + w - 1) * p.K * p.Vs;
    ld = p.Vt;
    return p.h0 ? p.h0 + bh * p.K * p.Vt : nullptr;
}

__global__ void __launch_bounds__(kThreads, 1) frame_lam_kernel(const FrameBwdParams p) {
    extern __shared__ __align__(16) unsigned char smraw[];
    LamSmem &sm = *reinterpret_cast<LamSmem *>(smraw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
    const int tile = blockIdx.y, j0 = tile * kFrameBwdCT, ntile = gridDim.y;
    const int K = p.K, Vt = p.Vt, Vs = p.Vs, F = p.F, d = p.direction;
    const int r0 = 4 * (tid >> 3), c0 = 4 * (tid & 7);
    const int nsteps = d == 0 ? F : F - 1;
    if (K < kKP)  // columns K .. 127 of A_f are never copied
        for (int e = tid; e < 2 * kKP * kKP; e += kThreads)
            if (e % kKP >= K) (&sm.a[0][0])[e] = 0.f;
    __syncthreads();
    float carry[4][4];
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int r = r0 + x, j = j0 + c0 + c;
            carry[x][c] = (d == 0 && p.dh_final && r < K && j < Vt) ? p.dh_final[(bh * K + r) * (int64_t)Vt + j] : 0.f;
        }
    if (nsteps > 0) lam_stage_a(p, sm, (nsteps - 1) & 1, (int64_t)bh * F + write_frame(d, F, nsteps - 1));
    for (int cs = nsteps - 1; cs >= 0; --cs) {
        const int w = write_frame(d, F, cs), rf = read_frame(d, F, cs);
        // Lam = C_r + carry, to the workspace and the shared tile (every C
        // value is loaded before the first store: a load after a store to
        // Lam could not be moved above it, and each would wait its own
        // round trip)
        const float *C = p.cmat + ((int64_t)bh * F + rf) * K * Vs;
        float *L = p.lam + ((int64_t)bh * F + w) * K * Vs;
        float cin[4][4];
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int r = r0 + x, j = j0 + c0 + c;
                cin[x][c] = (r < K && j < Vs) ? C[(int64_t)r * Vs + j] : 0.f;
            }
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const int r = r0 + x;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int j = j0 + c0 + c;
                carry[x][c] += cin[x][c];
                if (r < K && j < Vs) L[(int64_t)r * Vs + j] = carry[x][c];
            }
            *reinterpret_cast<float4 *>(sm.s + r * kFrameBwdCT + c0) =
                make_float4(carry[x][0], carry[x][1], carry[x][2], carry[x][3]);
        }
        const bool next = cs > 0;
        if (next) lam_stage_a(p, sm, (cs - 1) & 1, (int64_t)bh * F + write_frame(d, F, cs - 1));
        if (next) cp_async_wait<1>();
        else cp_async_wait<0>();
        __syncthreads();  // A_w and the tile are complete
        const float *A = sm.a[cs & 1];
        float m[4][4];
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int c = 0; c < 4; ++c) m[x][c] = 0.f;
#pragma unroll 8
        for (int a = 0; a < K; ++a) {  // M = A_w Lam (A_w symmetric: row a holds column a)
            const float4 a4 = *reinterpret_cast<const float4 *>(A + a * kKP + r0);
            const float4 s4 = *reinterpret_cast<const float4 *>(sm.s + a * kFrameBwdCT + c0);
            const float av[4] = {a4.x, a4.y, a4.z, a4.w}, sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int c = 0; c < 4; ++c) m[x][c] = fmaf(av[x], sv[c], m[x][c]);
        }
        // dg_w's part of this tile: e^{g_w} sum(M . S_prev), then carry = e^{g_w} M
        const float dec = __expf(fmaxf(p.g_frame[((int64_t)b * F + w) * p.H + h], kLogGateMin));
        int ld = 0;
        const float *pre = pre_state(p, bh, w, ld);
        float part = 0.f;
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int r = r0 + x, j = j0 + c0 + c;
                if (pre && r < K && j < Vt) part = fmaf(m[x][c], pre[(int64_t)r * ld + j], part);
                carry[x][c] = dec * m[x][c];
            }
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) sm.red[warp] = part;
        __syncthreads();  // (also: the tile and this A buffer are rewritten next)
        if (tid == 0) {
            float s = 0.f;
            for (int x = 0; x < kThreads / 32; ++x) s += sm.red[x];
            p.dgp[((int64_t)bh * F + w) * ntile + tile] = dec * s;
        }
    }
    if (d == 0 && p.dh0) {  // dL/dh0 = e^{g_0} A_0 Lam(write of frame 0)
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int r = r0 + x, j = j0 + c0 + c;
                if (r < K && j < Vt) p.dh0[(bh * K + r) * (int64_t)Vt + j] = nsteps > 0 ? carry[x][c] : 0.f;
            }
    }
}

// ------------------------------------------------------------- tokgrad ---
struct TokSmem {
    bf16 lam[kKP * kKS], pre[kKP * kKS], rd[kKP * kKS];  // [key][column]
    bf16 k[kChunk * kKS];  // [token][key]
    bf16 x[kChunk * kKS];  // [token][column]: [dO | dden]
    bf16 e[kChunk * kKS];  // [token][column]: [v | 1], then E = X - K P
    bf16 u[kChunk * kKS];  // U = K Lam
    float beta[kChunk];
    float dbp[2][kChunk];  // dbeta per column half (summed in order)
};
// fp32 (K x Vt-or-more, row stride ld) state -> bf16 [key][column] tile,
// zero past K rows and Vt columns (or everywhere for a null state). A
// thread's 16 reads go out in batches of kStBatch before their shared-memory
// stores, so their latencies overlap instead of adding up.
constexpr int kStPer = kKP * (kKP / 4) / kThreads;  // float4 groups per thread
constexpr int kStBatch = 8;
static_assert(kStPer % kStBatch == 0, "state tile batches");
__device__ __forceinline__ void state_tile(bf16 *dst, const float *src, int ld, int K, int Vt) {
    const bool vec = (ld & 3) == 0;
#pragma unroll
    for (int b0 = 0; b0 < kStPer; b0 += kStBatch) {
        float v[kStBatch][4];
#pragma unroll
        for (int u = 0; u < kStBatch; ++u) {
            const int e = threadIdx.x + (b0 + u) * kThreads;
            const int r = e / (kKP / 4), c = (e % (kKP / 4)) * 4;
            v[u][0] = v[u][1] = v[u][2] = v[u][3] = 0.f;
            if (src && r < K) {
                if (vec && c + 4 <= Vt) {
                    const float4 f4 = *reinterpret_cast<const float4 *>(src + (int64_t)r * ld + c);
                    v[u][0] = f4.x, v[u][1] = f4.y, v[u][2] = f4.z, v[u][3] = f4.w;
                } else {
#pragma unroll
                    for (int x = 0; x < 4; ++x)
                        if (c + x < Vt) v[u][x] = src[(int64_t)r * ld + c + x];
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kStBatch; ++u) {
            const int e = threadIdx.x + (b0 + u) * kThreads;
            const int r = e / (kKP / 4), c = (e % (kKP / 4)) * 4;
            *reinterpret_cast<uint2 *>(dst + r * kKS + c) =
                make_uint2(pack_bf16(v[u][0], v[u][1]), pack_bf16(v[u][2], v[u][3]));
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) frame_tokgrad_kernel(const FrameBwdParams p) {
    extern __shared__ __align__(16) unsigned char smraw[];
    TokSmem &sm = *reinterpret_cast<TokSmem *>(smraw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, t4 = lane & 3;
    const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
    const int K = p.K, V = p.V, Vt = p.Vt, Vs = p.Vs, F = p.F, d = p.direction;
    const int kq = (K + 15) & ~15, kv = (Vt + 15) & ~15;
    // this CTA's tok_group chunks, all in frame f: the frame's states are
    // converted once
    const int64_t tg0 = (int64_t)blockIdx.y * p.tok_group * kChunk;
    const int f = (int)(tg0 / p.frame);
    const bool wr = d == 0 || f >= 1;  // the reverse never writes frame 0
    const bf16 *k = (const bf16 *)p.k, *v = (const bf16 *)p.v, *dout = (const bf16 *)p.dout;
    int ld = 0;
    const float *pre = wr ? pre_state(p, bh, f, ld) : nullptr;
    state_tile(sm.rd, p.sread + ((int64_t)bh * F + f) * K * Vs, Vs, K, Vt);
    state_tile(sm.lam, wr ? p.lam + ((int64_t)bh * F + f) * K * Vs : nullptr, Vs, K, Vt);
    state_tile(sm.pre, pre, ld, K, Vt);
    // the frame predicts from the decayed state P = e^{g_f} S_prev
    const float dec = __expf(fmaxf(p.g_frame[((int64_t)b * F + f) * p.H + h], kLogGateMin));
    for (int gi = 0; gi < p.tok_group; ++gi) {
    const int64_t t0 = tg0 + (int64_t)gi * kChunk;
    for (int e = tid; e < kChunk * (kKP / 8); e += kThreads) {
        const int i = e >> 4, c8 = (e & 15) * 8;
        const int64_t t = t0 + i;
        const bool ink = c8 < K, inv = c8 < V;
        cp_async16(sm.k + i * kKS + c8, ink ? k + b * p.qk_sb + t * p.qk_st + h * p.qk_sh + c8 : k, ink ? 16 : 0);
        cp_async16(sm.e + i * kKS + c8, inv ? v + b * p.v_sb + t * p.v_st + h * p.v_sh + c8 : v, inv ? 16 : 0);
        cp_async16(sm.x + i * kKS + c8, inv ? dout + b * p.do_sb + t * p.do_st + h * p.do_sh + c8 : dout,
                   inv ? 16 : 0);
    }
    cp_async_commit();
    if (tid < kChunk) sm.beta[tid] = p.beta[((int64_t)b * p.T + t0 + tid) * p.H + h];
    cp_async_wait<0>();
    __syncthreads();
    if (p.dden && tid < kChunk) {  // the ones column: x = 1 in the value tile, dden in the gradient tile
        sm.e[tid * kKS + V] = __float2bfloat16_rn(1.f);
        sm.x[tid * kKS + V] = __float2bfloat16_rn(p.dden[((int64_t)b * p.H + h) * p.T + t0 + tid]);
    }
    __syncthreads();
    const int m0 = 16 * (warp & 3), n0 = 64 * (warp >> 2);
    if (wr) {
        float uf[8][4], kp[8][4];
        acc_zero(uf);
        acc_zero(kp);
        if (n0 < kv) {
            warp_gemm(uf, Tile{sm.k, kKS}, false, Tile{sm.lam, kKS}, true, m0, n0, kq, lane);
            warp_gemm(kp, Tile{sm.k, kKS}, false, Tile{sm.pre, kKS}, true, m0, n0, kq, lane);
        }
        // E = X - K P, dbeta = rowsum(U . E), dv = beta U; E and U to the tiles
        float pb[2] = {0.f, 0.f};
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int i = m0 + g8 + 8 * hf, c = n0 + 8 * n + 2 * t4;
                const float2 xv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(sm.e + i * kKS + c));
                const float e0 = c < Vt ? xv.x - dec * kp[n][2 * hf] : 0.f;
                const float e1 = c + 1 < Vt ? xv.y - dec * kp[n][2 * hf + 1] : 0.f;
                pb[hf] += uf[n][2 * hf] * e0 + uf[n][2 * hf + 1] * e1;
                *reinterpret_cast<uint32_t *>(sm.e + i * kKS + c) = pack_bf16(e0, e1);
                *reinterpret_cast<uint32_t *>(sm.u + i * kKS + c) = pack_bf16(uf[n][2 * hf], uf[n][2 * hf + 1]);
            }
        // dv = beta U; the second direction adds to the first's with
        // reductions that return nothing (no load waits; one add per
        // element, so the sum does not depend on timing)
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int i = m0 + g8 + 8 * hf, c = n0 + 8 * n + 2 * t4;
                if (c >= V) continue;
                float2 *dst = reinterpret_cast<float2 *>(p.dv + ((((int64_t)b * p.T + t0 + i) * p.H + h) * V + c));
                const float2 val = make_float2(sm.beta[i] * uf[n][2 * hf], sm.beta[i] * uf[n][2 * hf + 1]);
                if (p.acc)
                    atomicAdd(dst, val);
                else
                    *dst = val;
            }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float s = pb[hf];
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            if (t4 == 0) sm.dbp[warp >> 2][m0 + g8 + 8 * hf] = s;
        }
    } else if (!p.acc) {  // a frame this direction never writes: zero gradients
        for (int e = tid; e < kChunk * V; e += kThreads) {
            const int i = e / V, c = e % V;
            p.dv[(((int64_t)b * p.T + t0 + i) * p.H + h) * V + c] = 0.f;
        }
    }
    __syncthreads();
    // dk = beta (E Lam^T - U P^T) and dq = [dO | dden] R^T (64 tokens x K)
    const int nk0 = 64 * (warp >> 2);
    float dq[8][4];
    acc_zero(dq);
    if (nk0 < kq) warp_gemm(dq, Tile{sm.x, kKS}, false, Tile{sm.rd, kKS}, false, m0, nk0, kv, lane);
    float dk[8][4];
    acc_zero(dk);
    if (wr && nk0 < kq) {
        float c2[8][4];
        acc_zero(c2);
        warp_gemm(dk, Tile{sm.e, kKS}, false, Tile{sm.lam, kKS}, false, m0, nk0, kv, lane);
        warp_gemm(c2, Tile{sm.u, kKS}, false, Tile{sm.pre, kKS}, false, m0, nk0, kv, lane);
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) dk[n][e] = sm.beta[m0 + g8 + 8 * (e >> 1)] * (dk[n][e] - dec * c2[n][e]);
    }
    if (nk0 < kq) {  // (the second direction adds by reductions, as for dv)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int i = m0 + g8 + 8 * hf;
            const int64_t row = (((int64_t)b * p.T + t0 + i) * p.H + h) * K;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                const int c = nk0 + 8 * n + 2 * t4;
                if (c >= K) continue;
                float2 *oq = reinterpret_cast<float2 *>(p.dq + row + c), *ok = reinterpret_cast<float2 *>(p.dk + row + c);
                const float2 vq = make_float2(dq[n][2 * hf], dq[n][2 * hf + 1]);
                const float2 vk = make_float2(dk[n][2 * hf], dk[n][2 * hf + 1]);
                if (p.acc) {
                    atomicAdd(oq, vq);
                    atomicAdd(ok, vk);
                } else {
                    *oq = vq;
                    *ok = vk;
                }
            }
        }
    }
    if (tid < kChunk) {
        const int64_t row = ((int64_t)b * p.T + t0 + tid) * p.H + h;
        const float db = wr ? sm.dbp[0][tid] + sm.dbp[1][tid] : 0.f;
        if (p.acc)
            atomicAdd(p.dbeta + row, db);
        else
            p.dbeta[row] = db;
    }
    // dg_frame from the chain's parts, once per frame (its first chunk)
    if (tid == 0 && t0 % p.frame == 0) {
        const int ntile = (Vt + kFrameBwdCT - 1) / kFrameBwdCT;
        float s = 0.f;
        if (wr)
            for (int x = 0; x < ntile; ++x) s += p.dgp[((int64_t)bh * F + f) * ntile + x];
        const int64_t gi = ((int64_t)b * F + f) * p.H + h;
        if (p.g_frame[gi] < kLogGateMin) s = 0.f;  // the forward floors it
        p.dg_frame[gi] = p.acc ? p.dg_frame[gi] + s : s;
    }
    __syncthreads();  // the token tiles are refilled next
    }
}

}  // namespace

cudaError_t launch_frame_xt(const FrameBwdParams &p, cudaStream_t st) {
    const int bytes = (int)sizeof(XtSmem);
    cudaError_t e = cudaFuncSetAttribute(frame_xt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    frame_xt_kernel<<<dim3(p.B * p.H, p.F), kThreads, bytes, st>>>(p);
    return cudaGetLastError();
}
cudaError_t launch_frame_lam(const FrameBwdParams &p, cudaStream_t st) {
    const int bytes = (int)sizeof(LamSmem);
    cudaError_t e = cudaFuncSetAttribute(frame_lam_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    frame_lam_kernel<<<dim3(p.B * p.H, (p.Vt + kFrameBwdCT - 1) / kFrameBwdCT), kThreads, bytes, st>>>(p);
    return cudaGetLastError();
}
cudaError_t launch_frame_tokgrad(const FrameBwdParams &p, cudaStream_t st) {
    const int bytes = (int)sizeof(TokSmem);
    cudaError_t e = cudaFuncSetAttribute(frame_tokgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    frame_tokgrad_kernel<<<dim3(p.B * p.H, p.T / (kChunk * p.tok_group)), kThreads, bytes, st>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
