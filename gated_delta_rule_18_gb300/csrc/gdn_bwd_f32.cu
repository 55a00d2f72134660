// gdn_bwd_f32.cu -- the backward of the fp32 path: the token recurrence in
// reverse time, in IEEE fp32 on CUDA cores.
//
// Per logical position (the reverse scan remaps rows as the forward does),
// with d the decay (e^{g}, or e^{gk} per key row), q^, k^ the normalised
// rows and h the state (K x V) before the position:
//   P = d . h,  r = v - P^T k^,  h' = P + beta k^ r^T,  o = h'^T q^
// Reverse mode, with dh = dL/dh' from the later positions:
//   dh += q^ do^T,  dq^ = h' do,  s = dh^T k^,  dv = beta s,  dbeta = r . s,
//   dk^ = beta dh r - P (beta s),  dP = dh - k^ (beta s)^T,
//   dg = sum(dP . P) (per key: its row sums),  dL/dh = d . dP.
// The SANA `fused_cam_gdn.py` page's `_cam_scan_bwd_kernel` walks the same
// recurrence backwards by these per-step rules; the fp32 forward
// (gdn_chunk_f32.cu) computes the same states in chunked form.
//
// Structure. The value columns of the state evolve independently given k,
// beta and g, so a scan CTA runs one (sequence, head, 16-column range). A
// forward pass stores the state before every 16th position (checkpoints in
// the workspace); then, from the last group of 16 positions to the first,
// the group's states are recomputed into shared memory and the group is
// walked backwards. dv and dh0 are final per range. dq^, dk^, dbeta and dg
// are partial sums over a range's columns, which the reduction kernel adds
// over the ranges in a fixed order (bit-reproducible) and takes through the
// L2 normalisation.
//
// Scan thread layout: warp w holds state rows 16 w .. 16 w + 15; lane l
// holds column l % 16 of rows 16 w + 8 (l / 16) + j, j < 8.
#include "gdn_bwd_f32.cuh"
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int NT = kF32BwdThreads, NC = kF32BwdCols, NG = kF32BwdGroup, KP = kF32BwdKP;
static_assert(NT == 256 && KP == 128 && NC == 16, "8 warps x 16 rows, 16 columns per lane half");

struct ScanSmem {
    float hp[NG][kF32BwdState];  // the group's states before each position (per-thread slices)
    float q[NG][KP], k[NG][KP];  // q^ of the query row, k^ of the key row
    float dk[NG][KP];            // per-key decay e^{gk} (per-key gate)
    float v[NG][NC], dO[NG][NC], r[NG][NC];
    float dec[NG], beta[NG];
    int tq[NG], tk[NG];          // tokens within the sequence (tk = -1: the position reads no key)
    float red[2][8][NC];         // cross-warp column sums, double-buffered
    float gs[NG][8];             // scalar dg per position and warp
};

struct Seq {
    int b, len;
    int64_t tstart, row0, gbase;  // first token (packed index), its (B, T) row, first checkpoint slot
};

__device__ __forceinline__ bool seq_of(const F32BwdParams &p, int s, Seq &q) {
    if (p.cu_seqlens) {
        const int a = p.cu_seqlens[s], e = p.cu_seqlens[s + 1];
        if (a < 0 || e < a || e > p.T || (s == 0 && a != 0) || (s == p.n_seq - 1 && e != p.T)) return false;
        q.b = 0, q.len = e - a, q.tstart = a, q.row0 = a, q.gbase = a / NG + s;
    } else {
        q.b = s, q.len = p.T, q.tstart = 0, q.row0 = (int64_t)s * p.T;
        q.gbase = (int64_t)s * ((p.T + NG - 1) / NG);
    }
    return true;
}

// the sum over the CTA's rows of x (this thread's partial over its 8 rows),
// for this lane's column; one barrier
__device__ __forceinline__ float col_sum(float x, int buf, ScanSmem &sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    x += __shfl_xor_sync(0xffffffffu, x, 16);
    if (lane < NC) sm.red[buf][warp][lane] = x;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += sm.red[buf][w][lane & 15];
    return s;
}

// sums of x[j] over the 16 lanes of this half-warp (the same 8 rows, 16
// columns) by recursive halving: the lane ends with the sum for its row
// j = (lane % 16) / 2 (lanes l and l ^ 1 hold the same)
__device__ __forceinline__ float rows16(const float (&x)[8]) {
    const int cl = threadIdx.x & 15;
    const bool b8 = cl & 8, b4 = cl & 4, b2 = cl & 2;
    float y[4], z[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float keep = b8 ? x[i + 4] : x[i], send = b8 ? x[i] : x[i + 4];
        y[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float keep = b4 ? y[i + 2] : y[i], send = b4 ? y[i] : y[i + 2];
        z[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    float u = (b2 ? z[1] : z[0]) + __shfl_xor_sync(0xffffffffu, b2 ? z[0] : z[1], 2);
    return u + __shfl_xor_sync(0xffffffffu, u, 1);
}

// positions gp0 .. gp0 + n - 1 of the sequence into shared memory (rows past
// n zero): q^, k^, the decays, beta, and this range's v and do columns
__device__ void load_group(const F32BwdParams &p, const Seq &sq, int hh, int c0, int gp0, int n,
                           ScanSmem &sm) {
    const int tid = threadIdx.x, K = p.K, V = p.V;
    const bool den = p.dden != nullptr;
    const int i = tid >> 4, part = tid & 15;  // 16 threads per position
    const int tq = i < n ? q_token(p.reverse, sq.len, gp0 + i) : -1;
    const int tk = i < n ? kv_token(p.reverse, sq.len, gp0 + i) : -1;
    if (part == 0) {
        float b = 0.f, dec = 1.f;
        if (tk >= 0) {
            const int64_t row = (sq.row0 + tk) * p.H + hh;
            b = p.beta[row];
            if (p.g) dec = __expf(fmaxf(p.g[row], kLogGateMin));
        }
        sm.tq[i] = tq, sm.tk[i] = tk, sm.beta[i] = b, sm.dec[i] = dec;
    }
    {  // q and k rows, 8 keys per thread, then the L2 normalisation
        const int d0 = part * 8;
        const float *qr = tq >= 0 ? p.q + sq.b * p.qk_sb + (sq.tstart + tq) * p.qk_st + hh * p.qk_sh : nullptr;
        const float *kr = tk >= 0 ? p.k + sq.b * p.qk_sb + (sq.tstart + tk) * p.qk_st + hh * p.qk_sh : nullptr;
        float qv[8], kv[8], sq2 = 0.f, sk2 = 0.f;
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            const int d = d0 + x;
            qv[x] = (qr && d < K) ? qr[d] : 0.f;
            kv[x] = (kr && d < K) ? kr[d] : 0.f;
            sq2 = fmaf(qv[x], qv[x], sq2);
            sk2 = fmaf(kv[x], kv[x], sk2);
        }
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) {
            sq2 += __shfl_xor_sync(0xffffffffu, sq2, o);
            sk2 += __shfl_xor_sync(0xffffffffu, sk2, o);
        }
        const float rq = p.l2norm ? rsqrtf(sq2 + 1e-6f) : 1.f, rk = p.l2norm ? rsqrtf(sk2 + 1e-6f) : 1.f;
        const float *gr = (p.gk && tk >= 0) ? p.gk + ((sq.row0 + tk) * p.H + hh) * (int64_t)K : nullptr;
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            const int d = d0 + x;
            sm.q[i][d] = qv[x] * rq;
            sm.k[i][d] = kv[x] * rk;
            if (p.gk) sm.dk[i][d] = (gr && d < K) ? __expf(fmaxf(gr[d], kLogGateMin)) : 1.f;
        }
    }
    {  // this range's columns of v (the ones column of den: 1) and do (den: dden)
        const int c = c0 + part;
        float vv = 0.f, oo = 0.f;
        if (tk >= 0) {
            if (c < V) vv = p.v[sq.b * p.v_sb + (sq.tstart + tk) * p.v_st + hh * p.v_sh + c];
            else if (den && c == V) vv = 1.f;
        }
        if (tq >= 0) {
            if (c < V) oo = p.dout[sq.b * p.do_sb + (sq.tstart + tq) * p.do_st + hh * p.do_sh + c];
            else if (den && c == V) oo = p.dden[((int64_t)sq.b * p.H + hh) * p.T + sq.tstart + tq];
        }
        sm.v[i][part] = vv, sm.dO[i][part] = oo;
    }
}

// one forward position: P = d . h, r = v - P^T k^ (stored when keep_r),
// h <- P + beta k^ r^T
__device__ __forceinline__ void fwd_step(const F32BwdParams &p, ScanSmem &sm, int i, int r0, float (&h)[8],
                                         int &buf, bool keep_r) {
    const int lane = threadIdx.x & 31;
    float P[8], a = 0.f;
    const float ds = sm.dec[i];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        P[j] = (p.gk ? sm.dk[i][r0 + j] : ds) * h[j];
        a = fmaf(sm.k[i][r0 + j], P[j], a);
    }
    a = col_sum(a, buf, sm);
    buf ^= 1;
    const float rc = sm.v[i][lane & 15] - a, bk = sm.beta[i];
    if (keep_r && threadIdx.x < NC) sm.r[i][lane] = rc;
#pragma unroll
    for (int j = 0; j < 8; ++j) h[j] = fmaf(bk * sm.k[i][r0 + j], rc, P[j]);
}

__global__ void __launch_bounds__(NT, 1) bwd_f32_scan_kernel(const F32BwdParams p) {
    extern __shared__ __align__(16) unsigned char smraw[];
    ScanSmem &sm = *reinterpret_cast<ScanSmem *>(smraw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int s = blockIdx.x / p.H, hh = blockIdx.x % p.H, range = blockIdx.y;
    const int c0 = range * NC, cl = lane & 15, c = c0 + cl;
    const int r0 = 16 * warp + 8 * (lane >> 4);  // this thread's first state row
    const int K = p.K, V = p.V, Vs = p.Vs, NK = p.gk ? 3 : 2;
    const int64_t BTH = (int64_t)p.B * p.T * p.H;
    Seq sq;
    if (!seq_of(p, s, sq)) {
        if (tid == 0) atomicOr(p.err, kDevErrSeqlens);
        return;
    }
    const int ng = (sq.len + NG - 1) / NG;
    float *ck = p.ckpt + ((int64_t)hh * p.n_range + range) * p.ck_groups * kF32BwdState + tid * 8;
    auto state_at = [&](const float *base, float (&x)[8]) {  // (n_seq, H, K, Vs) slice, or 0
#pragma unroll
        for (int j = 0; j < 8; ++j)
            x[j] = (base && r0 + j < K && c < Vs) ? base[(((int64_t)s * p.H + hh) * K + r0 + j) * Vs + c] : 0.f;
    };
    auto ck_store = [&](int64_t slot, const float (&x)[8]) {
        float4 *d = reinterpret_cast<float4 *>(ck + (sq.gbase + slot) * kF32BwdState);
        d[0] = make_float4(x[0], x[1], x[2], x[3]);
        d[1] = make_float4(x[4], x[5], x[6], x[7]);
    };

    // ---- forward: the state before every group of NG positions
    float h[8];
    state_at(p.h0, h);
    int buf = 0;
    for (int gi = 0; gi < ng; ++gi) {
        ck_store(gi, h);
        if (gi == ng - 1) break;  // the last group's states are formed below
        __syncthreads();          // the previous group's readers are done
        load_group(p, sq, hh, c0, gi * NG, NG, sm);
        __syncthreads();
        for (int i = 0; i < NG; ++i) fwd_step(p, sm, i, r0, h, buf, false);
    }

    // ---- backward, group by group from the end
    float dh[8];
    state_at(p.dh_final, dh);
    for (int gi = ng - 1; gi >= 0; --gi) {
        const int n = min(NG, sq.len - gi * NG);
        __syncthreads();
        load_group(p, sq, hh, c0, gi * NG, n, sm);
        __syncthreads();
        {
            const float4 *src = reinterpret_cast<const float4 *>(ck + (sq.gbase + gi) * kF32BwdState);
            const float4 a = src[0], b = src[1];
            h[0] = a.x, h[1] = a.y, h[2] = a.z, h[3] = a.w, h[4] = b.x, h[5] = b.y, h[6] = b.z, h[7] = b.w;
        }
        for (int i = 0; i < n; ++i) {
            float4 *d = reinterpret_cast<float4 *>(&sm.hp[i][tid * 8]);
            d[0] = make_float4(h[0], h[1], h[2], h[3]);
            d[1] = make_float4(h[4], h[5], h[6], h[7]);
            fwd_step(p, sm, i, r0, h, buf, true);
        }
        __syncthreads();  // r of every position
        for (int i = n - 1; i >= 0; --i) {
            float P[8], xq[8], xk[8], xg[8], kk[8], dd[8];
            {
                const float4 *hs = reinterpret_cast<const float4 *>(&sm.hp[i][tid * 8]);
                const float4 a = hs[0], b = hs[1];
                const float hp[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    dd[j] = p.gk ? sm.dk[i][r0 + j] : sm.dec[i];
                    P[j] = dd[j] * hp[j];
                    kk[j] = sm.k[i][r0 + j];
                }
            }
            const float rc = sm.r[i][cl], bk = sm.beta[i], oc = sm.dO[i][cl];
            float s_part = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float hpost = fmaf(bk * kk[j], rc, P[j]);  // the state after the position
                xq[j] = hpost * oc;                                // dq^ = h' do
                dh[j] = fmaf(sm.q[i][r0 + j], oc, dh[j]);          // the output reads h'
                s_part = fmaf(kk[j], dh[j], s_part);
            }
            const float sc = col_sum(s_part, buf, sm);
            buf ^= 1;
            const float dr = bk * sc;
            const int tq = sm.tq[i], tk = sm.tk[i];
            float gsum = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                xk[j] = fmaf(bk * dh[j], rc, -P[j] * dr);  // dk^ = beta dh r - P dr
                const float dp = fmaf(-kk[j], dr, dh[j]);   // dP = dh - k^ dr^T
                xg[j] = dp * P[j];
                gsum += xg[j];
                dh[j] = dd[j] * dp;
            }
            // row sums over this range's columns: dq^ (query row), dk^ and dgk (key row)
            const float sq_ = rows16(xq), sk_ = rows16(xk);
            const float sg_ = p.gk ? rows16(xg) : 0.f;
            const int krow = r0 + (cl >> 1);
            if ((cl & 1) == 0 && krow < K) {
                float *pq = p.part_k + (((int64_t)range * BTH + (sq.row0 + tq) * p.H + hh) * NK) * K;
                pq[krow] = sq_;
                if (tk >= 0) {
                    float *pk = p.part_k + (((int64_t)range * BTH + (sq.row0 + tk) * p.H + hh) * NK) * K;
                    pk[K + krow] = sk_;
                    if (p.gk) pk[2 * K + krow] = sg_;
                }
            }
            if (warp == 0) {  // dv = beta s and dbeta = r . s over this range's columns
                float db = lane < NC ? rc * sc : 0.f;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) db += __shfl_xor_sync(0xffffffffu, db, o);
                if (tk >= 0) {
                    const int64_t row = (sq.row0 + tk) * p.H + hh;
                    if (lane < NC && c < V) p.dv[row * V + c] = dr;
                    if (lane == 0) p.part_s[((int64_t)range * BTH + row) * 2] = db;
                }
            }
            if (!p.gk) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) gsum += __shfl_xor_sync(0xffffffffu, gsum, o);
                if (lane == 0) sm.gs[i][warp] = gsum;
            }
        }
        __syncthreads();  // the group's scalar dg parts
        if (!p.gk && tid < n && sm.tk[tid] >= 0) {
            float gsum = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) gsum += sm.gs[tid][w];
            p.part_s[((int64_t)range * BTH + (sq.row0 + sm.tk[tid]) * p.H + hh) * 2 + 1] = gsum;
        }
    }
    // dL/dh0 of this range's columns
    if (p.dh0 && c < Vs)
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (r0 + j < K) p.dh0[(((int64_t)s * p.H + hh) * K + r0 + j) * Vs + c] = dh[j];
    // the reverse scan never reads token 0's key and value: zero parts and dv
    if (p.reverse && sq.len > 0) {
        const int64_t row = sq.row0 * p.H + hh;
        float *pk = p.part_k + (((int64_t)range * BTH + row) * NK) * K;
        for (int e = tid; e < (NK - 1) * K; e += NT) pk[K + e] = 0.f;
        if (tid == 0) p.part_s[((int64_t)range * BTH + row) * 2] = p.part_s[((int64_t)range * BTH + row) * 2 + 1] = 0.f;
        if (tid < NC && c0 + tid < V) p.dv[row * V + c0 + tid] = 0.f;
    }
}

// one warp per (token row, head): the ranges' parts summed in order, then
// through the L2 normalisation; floored gates get no gradient
__global__ void __launch_bounds__(NT) bwd_f32_reduce_kernel(const F32BwdParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t BTH = (int64_t)p.B * p.T * p.H;
    const int64_t idx = (int64_t)blockIdx.x * (NT / 32) + (threadIdx.x >> 5);
    if (idx >= BTH) return;
    const int K = p.K, NK = p.gk ? 3 : 2;
    const int64_t row = idx / p.H;
    const int hh = (int)(idx - row * p.H);
    const int b = (int)(row / p.T);
    const int64_t t = row - (int64_t)b * p.T;
    constexpr int PL = KP / 32;  // keys per lane
    float acc[3][PL];
#pragma unroll
    for (int cpt = 0; cpt < 3; ++cpt)
#pragma unroll
        for (int x = 0; x < PL; ++x) acc[cpt][x] = 0.f;
    for (int r = 0; r < p.n_range; ++r) {
        const float *src = p.part_k + ((int64_t)r * BTH + idx) * NK * K;
#pragma unroll
        for (int cpt = 0; cpt < 3; ++cpt) {
            if (cpt >= NK) break;
#pragma unroll
            for (int x = 0; x < PL; ++x) {
                const int d = lane + 32 * x;
                if (d < K) acc[cpt][x] += src[cpt * K + d];
            }
        }
    }
    // dx = r (dx^ - x^ (x^ . dx^)), r = (|x|^2 + eps)^{-1/2}
#pragma unroll
    for (int cpt = 0; cpt < 2; ++cpt) {
        const float *xr = (cpt == 0 ? p.q : p.k) + b * p.qk_sb + t * p.qk_st + hh * p.qk_sh;
        float xv[PL], ss = 0.f;
#pragma unroll
        for (int x = 0; x < PL; ++x) {
            const int d = lane + 32 * x;
            xv[x] = d < K ? xr[d] : 0.f;
            ss = fmaf(xv[x], xv[x], ss);
        }
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float rn = p.l2norm ? rsqrtf(ss + 1e-6f) : 1.f;
        float dot = 0.f;
#pragma unroll
        for (int x = 0; x < PL; ++x) dot = fmaf(xv[x] * rn, acc[cpt][x], dot);
        for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        float *dst = (cpt == 0 ? p.dq : p.dk) + idx * K;
#pragma unroll
        for (int x = 0; x < PL; ++x) {
            const int d = lane + 32 * x;
            if (d < K) dst[d] = p.l2norm ? rn * (acc[cpt][x] - xv[x] * rn * dot) : acc[cpt][x];
        }
    }
    if (p.gk) {
#pragma unroll
        for (int x = 0; x < PL; ++x) {
            const int d = lane + 32 * x;
            if (d < K) p.dg[idx * K + d] = p.gk[idx * K + d] < kLogGateMin ? 0.f : acc[2][x];
        }
    }
    if (lane == 0) {
        float db = 0.f, dg = 0.f;
        for (int r = 0; r < p.n_range; ++r) {
            db += p.part_s[((int64_t)r * BTH + idx) * 2];
            dg += p.part_s[((int64_t)r * BTH + idx) * 2 + 1];
        }
        p.dbeta[idx] = db;
        if (!p.gk) p.dg[idx] = p.g[idx] < kLogGateMin ? 0.f : dg;
    }
}

}  // namespace

cudaError_t launch_bwd_f32_scan(const F32BwdParams &p, cudaStream_t st) {
    const int bytes = (int)sizeof(ScanSmem);
    cudaError_t e = cudaFuncSetAttribute(bwd_f32_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    bwd_f32_scan_kernel<<<dim3((unsigned)(p.n_seq * p.H), (unsigned)p.n_range), NT, bytes, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_bwd_f32_reduce(const F32BwdParams &p, cudaStream_t st) {
    const int64_t n = (int64_t)p.B * p.T * p.H;
    const int64_t blocks = (n + NT / 32 - 1) / (NT / 32);
    bwd_f32_reduce_kernel<<<(unsigned)blocks, NT, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
