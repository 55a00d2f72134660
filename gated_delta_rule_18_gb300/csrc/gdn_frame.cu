// gdn_frame.cu -- the frame-causal form of the rule (SANA `fused_gdn.py` page,
// `_fused_gdn_kernel` with S tokens per frame; SANA `fused_cam_gdn.py` page,
// `_cam_scan_kernel`): every token of a frame predicts from the same
// pre-frame state, and the frame's outputs read the post-frame state.
//
// Per frame f, with the frame's keys K_f, values V_f, betas and log-decay g_f,
//   S_f = S_pre + K_f^T diag(beta) (V_f - K_f S_pre),   S_pre = e^{g_f} S_{f-1}
//       = A_f S_pre + B_f,  A_f = I - K_f^T diag(beta) K_f,
//                           B_f = K_f^T diag(beta) [V_f | 1]
// (the ones column carries the denominator's state z). A_f and B_f depend
// only on the frame's inputs, so they are formed for every frame at once;
// only the short chain over frames is serial, and the reverse direction
// (frame f reads frames f+1 .. F-1) runs the same chain backwards over the
// same A_f, B_f. Three kernels:
//   frame_gram   per (sequence, head, frame, 64-column block): C = K^T diag(beta)
//                [K | V | 1] over the frame's tokens on tensor cores (mma.sync
//                bf16, fp32 accumulate); A_f = I - C_KK, B_f = C_KV to the
//                workspace (fp32)
//   frame_chain  per (sequence, head, 16-column tile): the fp32 chains
//                S_f = A_f (e^{g_f} S_{f-1}) + B_f forward and / or reverse
//                (A_f staged in shared memory per step), the states each
//                frame's outputs read summed over directions
//   frame_out    per (sequence, head, 64-token chunk, 64-column block):
//                O = Q S_f on tensor cores; the ones column gives den
#include "gdn_common.cuh"

namespace gdn {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kKS = kKP + 8;  // bf16 row stride of a 128-key tile
constexpr int kXS = 64 + 8;   // bf16 row stride of a 64-column tile

__device__ __forceinline__ const bf16 *row_ptr(const void *base, int64_t sb, int64_t st, int64_t sh, int b,
                                               int64_t t, int h) {
    return (const bf16 *)base + b * sb + t * st + h * sh;
}

// ---------------------------------------------------------------- gram ---
__global__ void __launch_bounds__(128) frame_gram_kernel(const FrameParams p) {
    __shared__ __align__(16) bf16 sKb[kChunk * kKS];  // beta . k, [token][key]
    __shared__ __align__(16) bf16 sX[kChunk * kXS];   // [K | V | 1] columns of this block
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x / p.H, h = blockIdx.x % p.H, f = blockIdx.y, cb = blockIdx.z;
    const int K = p.K, V = p.V, Vt = p.Vt;
    const int col0 = cb * 64;  // columns [0, 128) are keys, [128, 128 + Vt) values (+ ones)
    float acc[2][8][4];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[m][n][e] = 0.f;

    for (int c = 0; c < p.frame / kChunk; ++c) {
        const int64_t t0 = (int64_t)f * p.frame + (int64_t)c * kChunk;
        __syncthreads();  // the previous chunk's tiles are no longer read
        for (int e = tid; e < kChunk * (kKP / 8); e += 128) {
            const int i = e / (kKP / 8), d = (e % (kKP / 8)) * 8;
            const float bt = p.beta[((int64_t)b * p.T + t0 + i) * p.H + h];
            float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (d < K) {
                const uint4 u = *reinterpret_cast<const uint4 *>(
                    row_ptr(p.k, p.qk_sb, p.qk_st, p.qk_sh, b, t0 + i, h) + d);
                const __nv_bfloat162 *u2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 t = __bfloat1622float2(u2[j]);
                    x[2 * j] = t.x * bt;
                    x[2 * j + 1] = t.y * bt;
                }
            }
            uint4 o;
            o.x = pack_bf16(x[0], x[1]);
            o.y = pack_bf16(x[2], x[3]);
            o.z = pack_bf16(x[4], x[5]);
            o.w = pack_bf16(x[6], x[7]);
            *reinterpret_cast<uint4 *>(sKb + i * kKS + d) = o;
        }
        for (int e = tid; e < kChunk * 8; e += 128) {
            const int i = e / 8, cc = (e % 8) * 8, col = col0 + cc;
            uint4 o = make_uint4(0, 0, 0, 0);
            if (col < kKP) {
                if (col < K) o = *reinterpret_cast<const uint4 *>(row_ptr(p.k, p.qk_sb, p.qk_st, p.qk_sh, b, t0 + i, h) + col);
            } else {
                const int vc = col - kKP;
                if (vc + 8 <= V) {
                    o = *reinterpret_cast<const uint4 *>(row_ptr(p.v, p.v_sb, p.v_st, p.v_sh, b, t0 + i, h) + vc);
                } else if (p.has_den && vc <= V && V < vc + 8) {
                    // the ones column sits at value column V (V is a multiple of 8)
                    o.x = pack_bf16(1.f, 0.f);
                }
            }
            *reinterpret_cast<uint4 *>(sX + i * kXS + cc) = o;
        }
        __syncthreads();
        // C[key m][col n] += sum_token Kb[token][m] X[token][n]; warp w: keys 32w..32w+31
#pragma unroll
        for (int ks = 0; ks < kChunk / 16; ++ks) {
            uint32_t a[2][4];
#pragma unroll
            for (int m = 0; m < 2; ++m)
                ldsm_x4_t(a[m], sKb + (ks * 16 + (lane & 7) + ((lane >> 4) << 3)) * kKS + 32 * warp + 16 * m +
                                    ((lane >> 3) & 1) * 8);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t bb[4];
                ldsm_x4_t(bb, sX + (ks * 16 + (lane & 15)) * kXS + 16 * np + (lane >> 4) * 8);
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    mma_bf16(acc[m][2 * np], a[m], bb[0], bb[1]);
                    mma_bf16(acc[m][2 * np + 1], a[m], bb[2], bb[3]);
                }
            }
        }
    }
    // A_f = I - C (key columns), B_f = C (value columns)
    const int64_t fi = ((int64_t)blockIdx.x * p.F + f);
    const int g8 = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = 32 * warp + 16 * m + g8 + 8 * (e >> 1);
                const int col = col0 + 8 * n + 2 * t4 + (e & 1);
                if (row >= K) continue;
                if (col < kKP) {
                    if (col < K) p.amat[(fi * K + row) * K + col] = (row == col ? 1.f : 0.f) - acc[m][n][e];
                } else if (col - kKP < Vt) {
                    p.bmat[(fi * K + row) * Vt + (col - kKP)] = acc[m][n][e];
                }
            }
}

// --------------------------------------------------------------- chain ---
constexpr int kCT = 16;        // state columns per chain CTA
constexpr int kAS = kKP + 1;   // fp32 row stride of A_f in shared memory (conflict-free rows)
struct ChainSmem {
    float a[kKP * kAS];        // A_f, [key][key]
    float s[kKP * kCT];        // the state tile, [key][column]
    float n[kKP * kCT];
};
__global__ void __launch_bounds__(256) frame_chain_kernel(const FrameParams p) {
    extern __shared__ __align__(16) unsigned char smraw[];
    ChainSmem &sm = *reinterpret_cast<ChainSmem *>(smraw);
    const int tid = threadIdx.x;
    const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
    const int j0 = blockIdx.y * kCT;
    const int K = p.K, Vt = p.Vt, F = p.F;
    // thread: key row r = tid / 2, columns (tid & 1) * 8 .. + 7
    const int r = tid >> 1, cs = (tid & 1) * 8;
    auto run = [&](bool rev) {
        for (int e = tid; e < kKP * kCT; e += 256) {
            const int rr = e / kCT, j = j0 + e % kCT;
            float v0 = 0.f;
            if (!rev && p.h0 && rr < K && j < p.V) v0 = p.h0[(((int64_t)b * p.H + h) * K + rr) * p.V + j];
            sm.s[e] = v0;
        }
        __syncthreads();
        for (int i = 0; i < F; ++i) {
            // forward: absorb frame i, outputs of frame i read it; reverse:
            // step i outputs frame F-1-i after absorbing frame F-i (none at i = 0)
            const int af = rev ? F - i : i, of = rev ? F - 1 - i : i;
            if (!rev || i > 0) {
                const int64_t fi = (int64_t)bh * F + af;
                const float *amat = p.amat + fi * K * K;
                for (int e = tid; e < K * K; e += 256) sm.a[(e / K) * kAS + e % K] = amat[e];
                const float dec = __expf(fmaxf(p.g_frame[((int64_t)b * F + af) * p.H + h], kLogGateMin));
                __syncthreads();
                float accv[8];
#pragma unroll
                for (int x = 0; x < 8; ++x) accv[x] = 0.f;
                if (r < K) {
                    const float *arow = sm.a + r * kAS;
#pragma unroll 4
                    for (int a = 0; a < K; ++a) {
                        const float av = arow[a];
                        const float4 s0 = *reinterpret_cast<const float4 *>(sm.s + a * kCT + cs);
                        const float4 s1 = *reinterpret_cast<const float4 *>(sm.s + a * kCT + cs + 4);
                        accv[0] = fmaf(av, s0.x, accv[0]);
                        accv[1] = fmaf(av, s0.y, accv[1]);
                        accv[2] = fmaf(av, s0.z, accv[2]);
                        accv[3] = fmaf(av, s0.w, accv[3]);
                        accv[4] = fmaf(av, s1.x, accv[4]);
                        accv[5] = fmaf(av, s1.y, accv[5]);
                        accv[6] = fmaf(av, s1.z, accv[6]);
                        accv[7] = fmaf(av, s1.w, accv[7]);
                    }
                }
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    const int j = j0 + cs + x;
                    const bool in = r < K && j < Vt;
                    const float bv = in ? p.bmat[(fi * K + r) * Vt + j] : 0.f;
                    sm.n[r * kCT + cs + x] = in ? fmaf(dec, accv[x], bv) : 0.f;
                }
                __syncthreads();
#pragma unroll
                for (int x = 0; x < 8; ++x) sm.s[r * kCT + cs + x] = sm.n[r * kCT + cs + x];
                __syncthreads();
            }
            // the state frame `of` reads, summed over the directions
            if (r < K) {
                float *dst = p.sout + (((int64_t)bh * F + of) * K + r) * Vt;
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    const int j = j0 + cs + x;
                    if (j < Vt) dst[j] = (rev && p.direction == 2) ? dst[j] + sm.s[r * kCT + cs + x] : sm.s[r * kCT + cs + x];
                }
            }
        }
        if (!rev && p.h_final && r < K) {
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                const int j = j0 + cs + x;
                if (j < p.V) p.h_final[(((int64_t)b * p.H + h) * K + r) * p.V + j] = sm.s[r * kCT + cs + x];
            }
        }
        __syncthreads();
    };
    if (p.direction != 1) run(false);
    if (p.direction != 0) run(true);
}

// ----------------------------------------------------------------- out ---
__global__ void __launch_bounds__(128) frame_out_kernel(const FrameParams p) {
    __shared__ __align__(16) bf16 sQ[kChunk * kKS];   // [token][key]
    __shared__ __align__(16) bf16 sSt[kKP * kXS];     // state block, [key][column]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x / p.H, h = blockIdx.x % p.H, c = blockIdx.y, cb = blockIdx.z;
    const int K = p.K, V = p.V, Vt = p.Vt;
    const int64_t t0 = (int64_t)c * kChunk;
    const int f = (int)(t0 / p.frame);
    const int col0 = cb * 64;
    for (int e = tid; e < kChunk * (kKP / 8); e += 128) {
        const int i = e / (kKP / 8), d = (e % (kKP / 8)) * 8;
        uint4 o = make_uint4(0, 0, 0, 0);
        if (d < K) o = *reinterpret_cast<const uint4 *>(row_ptr(p.q, p.qk_sb, p.qk_st, p.qk_sh, b, t0 + i, h) + d);
        *reinterpret_cast<uint4 *>(sQ + i * kKS + d) = o;
    }
    const float *S = p.sout + ((int64_t)blockIdx.x * p.F + f) * K * Vt;
    for (int e = tid; e < kKP * 32; e += 128) {
        const int rr = e / 32, cc = (e % 32) * 2, j = col0 + cc;
        const float s0 = (rr < K && j < Vt) ? S[(int64_t)rr * Vt + j] : 0.f;
        const float s1 = (rr < K && j + 1 < Vt) ? S[(int64_t)rr * Vt + j + 1] : 0.f;
        *reinterpret_cast<uint32_t *>(sSt + rr * kXS + cc) = pack_bf16(s0, s1);
    }
    __syncthreads();
    float acc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < kKP / 16; ++ks) {
        uint32_t a[4];
        ldsm_x4(a, sQ + (16 * warp + (lane & 15)) * kKS + ks * 16 + (lane >> 4) * 8);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
            uint32_t bb[4];
            ldsm_x4_t(bb, sSt + (ks * 16 + (lane & 15)) * kXS + 16 * np + (lane >> 4) * 8);
            mma_bf16(acc[2 * np], a, bb[0], bb[1]);
            mma_bf16(acc[2 * np + 1], a, bb[2], bb[3]);
        }
    }
    const int g8 = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int64_t t = t0 + 16 * warp + g8 + 8 * hf;
            const int j = col0 + 8 * n + 2 * t4;
            const float o0 = acc[n][2 * hf], o1 = acc[n][2 * hf + 1];
            if (j + 1 < V) {  // both columns are values (V is a multiple of 8)
                const int64_t off = b * p.o_sb + t * p.o_st + h * p.o_sh + j;
                if (p.out_f32) {
                    float *op = (float *)p.out + off;
                    op[0] = p.accumulate ? op[0] + o0 : o0;
                    op[1] = p.accumulate ? op[1] + o1 : o1;
                } else {
                    bf16 *op = (bf16 *)p.out + off;
                    float y0 = o0, y1 = o1;
                    if (p.accumulate) {
                        y0 += __bfloat162float(op[0]);
                        y1 += __bfloat162float(op[1]);
                    }
                    *reinterpret_cast<uint32_t *>(op) = pack_bf16(y0, y1);
                }
            } else if (p.has_den && j == V) {
                float *dp = p.den + ((int64_t)b * p.H + h) * p.T + t;
                *dp = p.accumulate ? *dp + o0 : o0;
            }
        }
}

}  // namespace

cudaError_t launch_frame_gram(const FrameParams &p, cudaStream_t st) {
    const int ncb = (kKP + p.Vt + 63) / 64;
    frame_gram_kernel<<<dim3(p.B * p.H, p.F, ncb), 128, 0, st>>>(p);
    return cudaGetLastError();
}
cudaError_t launch_frame_chain(const FrameParams &p, cudaStream_t st) {
    const int bytes = (int)sizeof(ChainSmem);
    cudaError_t e = cudaFuncSetAttribute(frame_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    frame_chain_kernel<<<dim3(p.B * p.H, (p.Vt + kCT - 1) / kCT), 256, bytes, st>>>(p);
    return cudaGetLastError();
}
cudaError_t launch_frame_out(const FrameParams &p, cudaStream_t st) {
    frame_out_kernel<<<dim3(p.B * p.H, p.T / kChunk, (p.Vt + 63) / 64), 128, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
