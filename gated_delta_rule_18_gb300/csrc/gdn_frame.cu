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
//   frame_gram   per (sequence, head, frame, 128-column block): C = K^T diag(beta)
//                [K | V | 1] over the frame's tokens on tensor cores (mma.sync
//                bf16, fp32 accumulate), chunks streamed one ahead; A_f = I -
//                C_KK, B_f = C_KV to the workspace (fp32)
//   frame_chain  per (sequence, head, 32-column tile): the fp32 chains
//                S_f = A_f (e^{g_f} S_{f-1}) + B_f forward and / or reverse
//                (the next A_f copied in while the current one is applied),
//                the states each frame's outputs read summed over directions
//   frame_out    per (sequence, head, up to 4 chunks of one frame, 128-column
//                block): O = Q S_f on tensor cores; the ones column gives den
#include "gdn_common.cuh"

namespace gdn {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kKS = kKP + 8;  // bf16 row stride of a 128-key tile

// ---------------------------------------------------------------- gram ---
// One CTA (8 warps) per (sequence x head, frame, 128-column block of
// [K | V | 1]); warp w owns keys 32 (w & 3) .. + 31 and the block's column
// half w >> 2. The frame's 64-token chunks stream through two stages
// (cp.async one chunk ahead): raw k rows and the block's columns, the latter
// scaled by beta in place once they land, so C = K^T (diag(beta) X).
constexpr int kXB = 128 + 8;  // bf16 row stride of a 128-column tile
struct GramStage {
    bf16 k[kChunk * kKS];  // raw k, [token][key]
    bf16 x[kChunk * kXB];  // [K | V | 1] columns of this block, [token][column]
    float beta[kChunk];
};
struct GramSmem {
    GramStage st[2];
};
__global__ void __launch_bounds__(256) frame_gram_kernel(const FrameParams p) {
    extern __shared__ __align__(16) unsigned char smraw[];
    GramSmem &sm = *reinterpret_cast<GramSmem *>(smraw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x / p.H, h = blockIdx.x % p.H, f = blockIdx.y, cb = blockIdx.z;
    const int K = p.K, V = p.V, Vt = p.Vt;
    const int col0 = cb * 128;  // columns [0, 128) are keys, [128, 128 + Vt) values (+ ones)
    const int nc = p.frame / kChunk;
    const bf16 *kp = (const bf16 *)p.k, *vp = (const bf16 *)p.v;

    auto stage = [&](int c) {
        GramStage &S = sm.st[c & 1];
        const int64_t t0 = (int64_t)f * p.frame + (int64_t)c * kChunk;
        for (int e = tid; e < kChunk * (kKP / 8); e += 256) {  // k rows
            const int i = e / (kKP / 8), d = (e % (kKP / 8)) * 8;
            const bool in = d < K;
            const bf16 *src = kp + b * p.qk_sb + (t0 + i) * p.qk_st + h * p.qk_sh + d;
            cp_async16(S.k + i * kKS + d, in ? src : kp, in ? 16 : 0);
        }
        for (int e = tid; e < kChunk * 16; e += 256) {  // the block's 128 columns
            const int i = e >> 4, cc = (e & 15) * 8, col = col0 + cc;
            const bf16 *src = kp;
            int nb = 0;
            if (col < kKP) {
                if (col < K) src = kp + b * p.qk_sb + (t0 + i) * p.qk_st + h * p.qk_sh + col, nb = 16;
            } else if (col - kKP + 8 <= V) {
                src = vp + b * p.v_sb + (t0 + i) * p.v_st + h * p.v_sh + (col - kKP), nb = 16;
            }
            cp_async16(S.x + i * kXB + cc, src, nb);
        }
        cp_async_commit();
        if (tid < kChunk) S.beta[tid] = p.beta[((int64_t)b * p.T + t0 + tid) * p.H + h];
    };

    float acc[2][8][4];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[m][n][e] = 0.f;
    const int mw = 32 * (warp & 3), nw = 64 * (warp >> 2);
    stage(0);
    for (int c = 0; c < nc; ++c) {
        GramStage &S = sm.st[c & 1];
        if (c + 1 < nc) {
            stage(c + 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();  // chunk c landed everywhere
        // beta . X in place (and the ones column of the denominator)
        for (int e = tid; e < kChunk * 16; e += 256) {
            const int i = e >> 4, cc = (e & 15) * 8, col = col0 + cc;
            uint4 u = *reinterpret_cast<const uint4 *>(S.x + i * kXB + cc);
            if (p.has_den && col >= kKP && col - kKP <= V && V < col - kKP + 8) {
                // the ones column sits at value column V (V is a multiple of 8)
                u = make_uint4(pack_bf16(1.f, 0.f), 0, 0, 0);
            }
            __nv_bfloat162 *h2 = reinterpret_cast<__nv_bfloat162 *>(&u);
            const float bt = S.beta[i];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const float2 t = __bfloat1622float2(h2[x]);
                h2[x] = __floats2bfloat162_rn(t.x * bt, t.y * bt);
            }
            *reinterpret_cast<uint4 *>(S.x + i * kXB + cc) = u;
        }
        __syncthreads();
        // C[key m][col n] += sum_token K[token][m] (beta X)[token][n]
#pragma unroll
        for (int ks = 0; ks < kChunk / 16; ++ks) {
            uint32_t a[2][4];
#pragma unroll
            for (int m = 0; m < 2; ++m)
                ldsm_x4_t(a[m], S.k + (ks * 16 + (lane & 7) + ((lane >> 4) << 3)) * kKS + mw + 16 * m +
                                    ((lane >> 3) & 1) * 8);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t bb[4];
                ldsm_x4_t(bb, S.x + (ks * 16 + (lane & 15)) * kXB + nw + 16 * np + (lane >> 4) * 8);
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    mma_bf16(acc[m][2 * np], a[m], bb[0], bb[1]);
                    mma_bf16(acc[m][2 * np + 1], a[m], bb[2], bb[3]);
                }
            }
        }
        __syncthreads();  // this stage is refilled next
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
                const int row = mw + 16 * m + g8 + 8 * (e >> 1);
                const int col = col0 + nw + 8 * n + 2 * t4 + (e & 1);
                if (row >= K) continue;
                if (col < kKP) {
                    if (col < K) p.amat[(fi * K + row) * K + col] = (row == col ? 1.f : 0.f) - acc[m][n][e];
                } else if (col - kKP < Vt) {
                    p.bmat[(fi * K + row) * Vt + (col - kKP)] = acc[m][n][e];
                }
            }
}

// --------------------------------------------------------------- chain ---
// Thread (rb, cq) keeps rows 4 rb .. 4 rb + 3 and columns 4 cq .. 4 cq + 3 of
// the CTA's 32-column state tile (one wave of CTAs for the video shapes);
// A_f is symmetric (I - K^T diag(beta) K), so row a of A_f holds column a,
// and a thread's four rows of A_f S come from one 16-byte load of row a per
// step of the sum. The next frame's A_f is copied in (cp.async) while the
// current one is applied.
constexpr int kCT = 32;  // state columns per chain CTA
struct ChainSmem {
    float a[2][kKP * kKP];  // A_f of this step and of the next
    float s[kKP * kCT];     // the state tile, [key][column]
};
__device__ __forceinline__ void stage_a(const FrameParams &p, ChainSmem &sm, int buf, int64_t fi) {
    // thread t copies 16-byte piece t % 32 of rows t / 32, t / 32 + 8, ...
    const int K = p.K, c = (threadIdx.x & 31) * 4;
    const float *A = p.amat + fi * K * K;
    if (c < K)
        for (int r = threadIdx.x >> 5; r < K; r += 8)
            cp_async16(sm.a[buf] + r * kKP + c, A + (int64_t)r * K + c, 16);
    cp_async_commit();
}
__global__ void __launch_bounds__(256, 1) frame_chain_kernel(const FrameParams p) {
    extern __shared__ __align__(16) unsigned char smraw[];
    ChainSmem &sm = *reinterpret_cast<ChainSmem *>(smraw);
    const int tid = threadIdx.x;
    const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
    const int j0 = blockIdx.y * kCT;
    const int K = p.K, Vt = p.Vt, F = p.F;
    const int rb = tid >> 3, cq = tid & 7, r0 = 4 * rb, c0 = 4 * cq;
    // columns K .. 127 of A_f are never copied: zero them once
    if (K < kKP)
        for (int e = tid; e < 2 * kKP * kKP; e += 256)
            if (e % kKP >= K) (&sm.a[0][0])[e] = 0.f;
    __syncthreads();
    auto run = [&](bool rev) {
        // step i absorbs frame af(i) (none for the reverse direction's first
        // step) and gives the state frame of(i) reads
        auto af = [&](int i) { return rev ? F - i : i; };
        const int first = rev ? 1 : 0;  // first step that absorbs a frame
        if (first < F) stage_a(p, sm, first & 1, (int64_t)bh * F + af(first));
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int r = r0 + i, j = j0 + c0 + c;
                acc[i][c] = (!rev && p.h0 && r < K && j < p.Vt) ? p.h0[(((int64_t)b * p.H + h) * K + r) * p.Vt + j] : 0.f;
            }
        for (int i = 0; i < F; ++i) {
            const int of = rev ? F - 1 - i : i;
            if (i >= first) {
                const int64_t fi = (int64_t)bh * F + af(i);
#pragma unroll
                for (int x = 0; x < 4; ++x)
                    *reinterpret_cast<float4 *>(sm.s + (r0 + x) * kCT + c0) =
                        make_float4(acc[x][0], acc[x][1], acc[x][2], acc[x][3]);
                const bool next = i + 1 < F;
                if (next) stage_a(p, sm, (i + 1) & 1, (int64_t)bh * F + af(i + 1));
                float bv[4][4];
#pragma unroll
                for (int x = 0; x < 4; ++x)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int r = r0 + x, j = j0 + c0 + c;
                        bv[x][c] = (r < K && j < Vt) ? p.bmat[(fi * K + r) * Vt + j] : 0.f;
                    }
                const float dec = __expf(fmaxf(p.g_frame[((int64_t)b * F + af(i)) * p.H + h], kLogGateMin));
                if (next) cp_async_wait<1>();
                else cp_async_wait<0>();
                __syncthreads();  // A_f and the tile are complete
                const float *A = sm.a[i & 1];
#pragma unroll
                for (int x = 0; x < 4; ++x)
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[x][c] = 0.f;
#pragma unroll 8
                for (int a = 0; a < K; ++a) {
                    const float4 m4 = *reinterpret_cast<const float4 *>(A + a * kKP + r0);
                    const float4 s4 = *reinterpret_cast<const float4 *>(sm.s + a * kCT + c0);
                    const float mv[4] = {m4.x, m4.y, m4.z, m4.w}, sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                    for (int x = 0; x < 4; ++x)
#pragma unroll
                        for (int c = 0; c < 4; ++c) acc[x][c] = fmaf(mv[x], sv[c], acc[x][c]);
                }
#pragma unroll
                for (int x = 0; x < 4; ++x)
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[x][c] = fmaf(dec, acc[x][c], bv[x][c]);
                __syncthreads();  // the tile and this buffer are rewritten next
            }
            // the state frame `of` reads, summed over the directions (the
            // forward run's values all loaded before the first store)
            float prev[4][4];
            const bool add = rev && p.direction == 2;
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int r = r0 + x, j = j0 + c0 + c;
                    prev[x][c] = (add && r < K && j < Vt) ? p.sout[(((int64_t)bh * F + of) * K + r) * p.Vs + j] : 0.f;
                }
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const int r = r0 + x;
                if (r >= K) continue;
                float *dst = p.sout + (((int64_t)bh * F + of) * K + r) * p.Vs;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int j = j0 + c0 + c;
                    if (j < Vt) dst[j] = prev[x][c] + acc[x][c];
                }
            }
        }
        if (!rev && p.h_final) {
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int r = r0 + x, j = j0 + c0 + c;
                    if (r < K && j < p.Vt) p.h_final[(((int64_t)b * p.H + h) * K + r) * p.Vt + j] = acc[x][c];
                }
        }
    };
    if (p.direction != 1) run(false);
    if (p.direction != 0) run(true);
}

// ----------------------------------------------------------------- out ---
// One CTA (8 warps) per (sequence x head, up to kOutChunks consecutive
// 64-token chunks of one frame, 128 value columns). The frame's state is
// converted to bf16 once per CTA, from 16-byte fp32 loads; the chunks' q rows
// stream through two cp.async buffers, the next chunk's copy in flight while
// the current one is multiplied and stored. Warp w computes tokens
// 16 (w & 3) .. + 15 of column half w >> 2.
constexpr int kOutChunks = 4;
struct OutSmem {
    bf16 q[2][kChunk * kKS];  // [token][key], two chunks
    bf16 st[kKP * kXB];       // state block, [key][column]
};
__global__ void __launch_bounds__(256) frame_out_kernel(const FrameParams p) {
    extern __shared__ __align__(16) unsigned char smraw[];
    OutSmem &sm = *reinterpret_cast<OutSmem *>(smraw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x / p.H, h = blockIdx.x % p.H, cb = blockIdx.z;
    const int K = p.K, V = p.V, Vt = p.Vt;
    // chunks per frame, CTAs per frame; this CTA's frame and chunks
    const int cpf = p.frame / kChunk, gpf = (cpf + kOutChunks - 1) / kOutChunks;
    const int f = blockIdx.y / gpf;
    const int c_begin = f * cpf + (blockIdx.y % gpf) * kOutChunks;
    const int n_ch = min(kOutChunks, (f + 1) * cpf - c_begin);
    const int col0 = cb * 128;
    const bf16 *qp = (const bf16 *)p.q;
    auto load_q = [&](int c, bf16 *dst) {
        const int64_t t0 = (int64_t)c * kChunk;
        for (int e = tid; e < kChunk * (kKP / 8); e += 256) {
            const int i = e >> 4, d = (e & 15) * 8;
            const bool in = d < K;
            cp_async16(dst + i * kKS + d, in ? qp + b * p.qk_sb + (t0 + i) * p.qk_st + h * p.qk_sh + d : qp,
                       in ? 16 : 0);
        }
        cp_async_commit();
    };
    load_q(c_begin, sm.q[0]);
    const float *S = p.sout + ((int64_t)blockIdx.x * p.F + f) * K * p.Vs;
#pragma unroll 4
    for (int e = tid; e < kKP * 32; e += 256) {  // 4 columns per step
        const int rr = e >> 5, cc = (e & 31) * 4, j = col0 + cc;
        float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (rr < K && j < Vt) v4 = *reinterpret_cast<const float4 *>(S + (int64_t)rr * p.Vs + j);
        if (j + 1 >= Vt) v4.y = 0.f;  // padding columns of the state rows
        if (j + 2 >= Vt) v4.z = 0.f;
        if (j + 3 >= Vt) v4.w = 0.f;
        *reinterpret_cast<uint2 *>(sm.st + rr * kXB + cc) = make_uint2(pack_bf16(v4.x, v4.y), pack_bf16(v4.z, v4.w));
    }
    const int m0 = 16 * (warp & 3), n0 = 64 * (warp >> 2);
    const int g8 = lane >> 2, t4 = lane & 3;
    for (int it = 0; it < n_ch; ++it) {
        if (it + 1 < n_ch) {
            load_q(c_begin + it + 1, sm.q[(it + 1) & 1]);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const bf16 *qs = sm.q[it & 1];
        const int64_t t0 = (int64_t)(c_begin + it) * kChunk;
        float acc[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < kKP / 16; ++ks) {
            uint32_t a[4];
            ldsm_x4(a, qs + (m0 + (lane & 15)) * kKS + ks * 16 + (lane >> 4) * 8);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t bb[4];
                ldsm_x4_t(bb, sm.st + (ks * 16 + (lane & 15)) * kXB + n0 + 16 * np + (lane >> 4) * 8);
                mma_bf16(acc[2 * np], a, bb[0], bb[1]);
                mma_bf16(acc[2 * np + 1], a, bb[2], bb[3]);
            }
        }
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int64_t t = t0 + m0 + g8 + 8 * hf;
                const int j = col0 + n0 + 8 * n + 2 * t4;
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
        __syncthreads();  // every warp is done with this q buffer before it is refilled
    }
}

}  // namespace

cudaError_t launch_frame_gram(const FrameParams &p, cudaStream_t st) {
    const int bytes = (int)sizeof(GramSmem);
    cudaError_t e = cudaFuncSetAttribute(frame_gram_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    const int ncb = (kKP + p.Vt + 127) / 128;
    frame_gram_kernel<<<dim3(p.B * p.H, p.F, ncb), 256, bytes, st>>>(p);
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
    const int bytes = (int)sizeof(OutSmem);
    cudaError_t e = cudaFuncSetAttribute(frame_out_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    const int gpf = (p.frame / kChunk + kOutChunks - 1) / kOutChunks;  // CTAs per frame
    frame_out_kernel<<<dim3(p.B * p.H, p.F * gpf, (p.Vt + 127) / 128), 256, bytes, st>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
