// gdn_prep.cu -- q/k preparation: per-(token, head) L2 normalisation, or the
// full-channel RMSNorm of the SANA `fused_gdn.py` page (`_precompute_inv_rms`,
// `_fused_qk_inv_rms_kernel`: inv_rms = rsqrt(sum_{h,d} x^2 / (H*D) + eps) per
// token, weight 1), optionally followed by ReLU and a scale (the k_scale of
// `_fused_gdn_kernel`).
//
// HBM-bound: one warp per row (L2: a (token, head) row of D channels; RMS: a
// token's H*D channels), 16-byte vector loads, fp32 sums reduced with warp
// shuffles. Each row is read once for L2; RMS reads the token's channels once
// for the sum and again (from L1/L2) for the store.
#include "gdn_common.cuh"

namespace gdn {
namespace {

template <typename T>
struct Vec;
template <>
struct Vec<float> {
    static constexpr int N = 4;
};
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
};

template <typename T>
__device__ __forceinline__ void unpack(const uint4 &u, float *f) {
    if constexpr (sizeof(T) == 4) {
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
    } else {
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 t = __bfloat1622float2(h[i]);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
}

template <typename T>
__device__ __forceinline__ uint4 pack(const float *f) {
    uint4 u;
    if constexpr (sizeof(T) == 4) {
        u.x = __float_as_uint(f[0]);
        u.y = __float_as_uint(f[1]);
        u.z = __float_as_uint(f[2]);
        u.w = __float_as_uint(f[3]);
    } else {
        u.x = pack_bf16(f[0], f[1]);
        u.y = pack_bf16(f[2], f[3]);
        u.z = pack_bf16(f[4], f[5]);
        u.w = pack_bf16(f[6], f[7]);
    }
    return u;
}

// L2 mode: warp per (b, t, h) row; D / VE <= 64 vectors, two per lane.
template <typename T>
__global__ void __launch_bounds__(256) prep_l2_kernel(const T *__restrict__ x, int64_t xsb,
                                                      int64_t xst, int64_t xsh,
                                                      T *__restrict__ y, int64_t ysb,
                                                      int64_t yst, int64_t ysh, int B, int Tn,
                                                      int H, int D, int relu, float scale,
                                                      float eps) {
    constexpr int VE = Vec<T>::N;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= (int64_t)B * Tn * H) return;
    const int h = (int)(row % H);
    const int64_t bt = row / H;
    const int t = (int)(bt % Tn);
    const int b = (int)(bt / Tn);
    const T *xr = x + b * xsb + t * xst + h * xsh;
    T *yr = y + b * ysb + t * yst + h * ysh;
    const int nv = D / VE;
    float f[2][VE];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int vi = lane + 32 * i;
        if (vi < nv) {
            uint4 u = *reinterpret_cast<const uint4 *>(xr + vi * VE);
            unpack<T>(u, f[i]);
#pragma unroll
            for (int e = 0; e < VE; ++e) ss += f[i][e] * f[i][e];
        }
    }
    ss = warp_sum(ss);
    const float inv = rsqrtf(ss + eps);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int vi = lane + 32 * i;
        if (vi < nv) {
#pragma unroll
            for (int e = 0; e < VE; ++e) {
                float t2 = f[i][e] * inv;
                if (relu) t2 = fmaxf(t2, 0.f);
                f[i][e] = t2 * scale;
            }
            *reinterpret_cast<uint4 *>(yr + vi * VE) = pack<T>(f[i]);
        }
    }
}

// RMS mode: warp per (b, t) token over its H*D channels.
template <typename T>
__global__ void __launch_bounds__(256) prep_rms_kernel(const T *__restrict__ x, int64_t xsb,
                                                       int64_t xst, int64_t xsh, T *y,
                                                       int64_t ysb, int64_t yst, int64_t ysh,
                                                       int B, int Tn, int H, int D, int relu,
                                                       float scale, float eps,
                                                       float *__restrict__ inv_rms) {
    constexpr int VE = Vec<T>::N;
    const int64_t tok = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (tok >= (int64_t)B * Tn) return;
    const int t = (int)(tok % Tn);
    const int b = (int)(tok / Tn);
    const T *xb = x + b * xsb + t * xst;
    T *yb = y + b * ysb + t * yst;
    const int nv = D / VE;
    const int total = H * nv;
    float ss = 0.f;
    for (int idx = lane; idx < total; idx += 32) {
        const int h = idx / nv, vi = idx - h * nv;
        float f[VE];
        unpack<T>(*reinterpret_cast<const uint4 *>(xb + h * xsh + vi * VE), f);
#pragma unroll
        for (int e = 0; e < VE; ++e) ss += f[e] * f[e];
    }
    ss = warp_sum(ss);
    const float inv = rsqrtf(ss / (float)(H * D) + eps);
    if (lane == 0 && inv_rms) inv_rms[tok] = inv;
    for (int idx = lane; idx < total; idx += 32) {
        const int h = idx / nv, vi = idx - h * nv;
        float f[VE];
        unpack<T>(*reinterpret_cast<const uint4 *>(xb + h * xsh + vi * VE), f);
#pragma unroll
        for (int e = 0; e < VE; ++e) {
            float t2 = f[e] * inv;
            if (relu) t2 = fmaxf(t2, 0.f);
            f[e] = t2 * scale;
        }
        *reinterpret_cast<uint4 *>(yb + h * ysh + vi * VE) = pack<T>(f);
    }
}

// Backward of y = relu?(x * inv) * scale: with dt = scale * dy (zero where
// the ReLU cut, i.e. where x <= 0) and inv = (m sum x^2 + eps)^{-1/2} (m = 1
// for the per-(token, head) L2 form, 1 / (H D) for the full-channel RMS
// form), dx = inv dt - x inv^3 m sum(dt x). One warp per row, two passes
// (the second reads the row again from L1/L2); dy and dx fp32 contiguous.
template <typename T>
__global__ void __launch_bounds__(256) prep_bwd_kernel(const T *__restrict__ x, int64_t xsb, int64_t xst,
                                                       int64_t xsh, const float *__restrict__ dy,
                                                       float *__restrict__ dx, int B, int T_, int H, int D,
                                                       int rms, int relu, float scale, float eps) {
    constexpr int N = Vec<T>::N;
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t rows = rms ? (int64_t)B * T_ : (int64_t)B * T_ * H;
    if (row >= rows) return;
    const int heads = rms ? H : 1;                 // heads in this row
    const int64_t tok = rms ? row : row / H;       // flat token b * T + t
    const int h0 = rms ? 0 : (int)(row % H);
    const int b = (int)(tok / T_), t = (int)(tok % T_);
    const int per = D / N;                         // vectors per head
    const float m = rms ? 1.f / (float)(H * D) : 1.f;
    float ss = 0.f, sd = 0.f;
    for (int e = lane; e < heads * per; e += 32) {
        const int hh = h0 + e / per, d0 = (e % per) * N;
        float xf[N], gf[N];
        unpack<T>(*reinterpret_cast<const uint4 *>(x + b * xsb + (int64_t)t * xst + hh * xsh + d0), xf);
        const float *g = dy + ((tok * H + hh) * D + d0);
#pragma unroll
        for (int i = 0; i < N; ++i) {
            gf[i] = (relu && xf[i] <= 0.f) ? 0.f : scale * g[i];
            ss = fmaf(xf[i], xf[i], ss);
            sd = fmaf(gf[i], xf[i], sd);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ss += __shfl_xor_sync(0xffffffffu, ss, o);
        sd += __shfl_xor_sync(0xffffffffu, sd, o);
    }
    const float inv = rsqrtf(m * ss + eps);
    const float c = inv * inv * inv * m * sd;
    for (int e = lane; e < heads * per; e += 32) {
        const int hh = h0 + e / per, d0 = (e % per) * N;
        float xf[N];
        unpack<T>(*reinterpret_cast<const uint4 *>(x + b * xsb + (int64_t)t * xst + hh * xsh + d0), xf);
        const float *g = dy + ((tok * H + hh) * D + d0);
        float *o = dx + ((tok * H + hh) * D + d0);
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const float dt = (relu && xf[i] <= 0.f) ? 0.f : scale * g[i];
            o[i] = inv * dt - xf[i] * c;
        }
    }
}

}  // namespace

cudaError_t launch_prep(const void *x, int64_t xsb, int64_t xst, int64_t xsh, void *y,
                        int64_t ysb, int64_t yst, int64_t ysh, int B, int T, int H, int D,
                        int bf16, int mode, float scale, float eps, float *inv_rms,
                        cudaStream_t st) {
    const int relu = (mode & 0x10) ? 1 : 0;
    const int rms = mode & 0x1;
    const int64_t rows = rms ? (int64_t)B * T : (int64_t)B * T * H;
    if (rows == 0) return cudaSuccess;
    const int wpb = 8;
    const unsigned grid = (unsigned)((rows + wpb - 1) / wpb);
    if (bf16) {
        using E = __nv_bfloat16;
        if (rms)
            prep_rms_kernel<E><<<grid, 32 * wpb, 0, st>>>((const E *)x, xsb, xst, xsh, (E *)y,
                                                          ysb, yst, ysh, B, T, H, D, relu,
                                                          scale, eps, inv_rms);
        else
            prep_l2_kernel<E><<<grid, 32 * wpb, 0, st>>>((const E *)x, xsb, xst, xsh, (E *)y,
                                                         ysb, yst, ysh, B, T, H, D, relu,
                                                         scale, eps);
    } else {
        if (rms)
            prep_rms_kernel<float><<<grid, 32 * wpb, 0, st>>>(
                (const float *)x, xsb, xst, xsh, (float *)y, ysb, yst, ysh, B, T, H, D, relu,
                scale, eps, inv_rms);
        else
            prep_l2_kernel<float><<<grid, 32 * wpb, 0, st>>>((const float *)x, xsb, xst, xsh,
                                                             (float *)y, ysb, yst, ysh, B, T,
                                                             H, D, relu, scale, eps);
    }
    return cudaGetLastError();
}

}  // namespace gdn

namespace gdn {
cudaError_t launch_prep_bwd(const void *x, int64_t xsb, int64_t xst, int64_t xsh, const float *dy,
                            float *dx, int B, int T, int H, int D, int bf16, int mode, float scale,
                            float eps, cudaStream_t st) {
    const int relu = (mode & 0x10) ? 1 : 0;
    const int rms = mode & 0x1;
    const int64_t rows = rms ? (int64_t)B * T : (int64_t)B * T * H;
    if (rows == 0) return cudaSuccess;
    const int wpb = 8;
    const unsigned grid = (unsigned)((rows + wpb - 1) / wpb);
    if (bf16)
        prep_bwd_kernel<__nv_bfloat16><<<grid, 32 * wpb, 0, st>>>((const __nv_bfloat16 *)x, xsb, xst, xsh, dy, dx,
                                                                  B, T, H, D, rms, relu, scale, eps);
    else
        prep_bwd_kernel<float><<<grid, 32 * wpb, 0, st>>>((const float *)x, xsb, xst, xsh, dy, dx, B, T, H, D,
                                                          rms, relu, scale, eps);
    return cudaGetLastError();
}
}  // namespace gdn
