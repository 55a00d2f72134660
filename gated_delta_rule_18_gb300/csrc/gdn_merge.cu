// gdn_merge.cu -- the bidirectional merge of the SANA `fused_gdn.py` page
// (`fused_bigdn_func`: out = (num_fwd + num_bwd) / (den_fwd + den_bwd + eps);
// `_fused_bidi_merge_kernel`, PRE_SUMMED, with the optional APPLY_GATE
// factor silu(gate) = gate / (1 + e^{-gate})). The scan has already summed
// both directions into num (B, T, H, V) and den (B, H, T).
//
// HBM-bound elementwise pass: one 16-byte vector of a (token, head) row per
// thread and step of a grid-stride loop, fp32 arithmetic.
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
__device__ __forceinline__ void load_vec(const T *p, float *f) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    if constexpr (sizeof(T) == 4) {
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
    } else {
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 t = __bfloat1622float2(h[i]);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
}
template <typename T>
__device__ __forceinline__ void store_vec(T *p, const float *f) {
    uint4 u;
    if constexpr (sizeof(T) == 4) {
        u = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
    } else {
        u.x = pack_bf16(f[0], f[1]);
        u.y = pack_bf16(f[2], f[3]);
        u.z = pack_bf16(f[4], f[5]);
        u.w = pack_bf16(f[6], f[7]);
    }
    *reinterpret_cast<uint4 *>(p) = u;
}

template <typename TI, typename TO>
__global__ void __launch_bounds__(256) merge_kernel(const MergeParams m) {
    constexpr int N = Vec<TI>::N;
    const int vpr = m.V / N;  // vectors per (token, head) row
    const int64_t total = (int64_t)m.B * m.T * m.H * vpr;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(e % vpr) * N;
        int64_t row = e / vpr;
        const int h = (int)(row % m.H);
        row /= m.H;
        const int t = (int)(row % m.T);
        const int b = (int)(row / m.T);
        const float inv = 1.f / (m.den[((int64_t)b * m.H + h) * m.T + t] + m.eps);
        float x[8];
        load_vec<TI>((const TI *)m.num + b * m.n_sb + (int64_t)t * m.n_st + h * m.n_sh + c, x);
#pragma unroll
        for (int i = 0; i < N; ++i) x[i] *= inv;
        if (m.gate) {
            float gt[8];
            load_vec<TI>((const TI *)m.gate + b * m.g_sb + (int64_t)t * m.g_st + h * m.g_sh + c, gt);
#pragma unroll
            for (int i = 0; i < N; ++i) x[i] *= gt[i] / (1.f + __expf(-gt[i]));
        }
        if constexpr (sizeof(TO) == sizeof(TI)) {
            store_vec<TO>((TO *)m.out + b * m.o_sb + (int64_t)t * m.o_st + h * m.o_sh + c, x);
        } else {  // fp32 in, bf16 out: two 8-byte halves
            TO *o = (TO *)m.out + b * m.o_sb + (int64_t)t * m.o_st + h * m.o_sh + c;
            *reinterpret_cast<uint2 *>(o) = make_uint2(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]));
        }
    }
}

}  // namespace

cudaError_t launch_merge(const MergeParams &m, cudaStream_t st) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int vec = m.num_bf16 ? 8 : 4;
    const int64_t total = (int64_t)m.B * m.T * m.H * (m.V / vec);
    const int64_t want = (total + 255) / 256;
    const int grid = (int)(want < 8LL * sms ? (want > 0 ? want : 1) : 8LL * sms);
    if (m.num_bf16) {
        if (m.out_bf16) merge_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, 256, 0, st>>>(m);
        else return cudaErrorInvalidValue;  // bf16 in, fp32 out: not offered
    } else {
        if (m.out_bf16) merge_kernel<float, __nv_bfloat16><<<grid, 256, 0, st>>>(m);
        else merge_kernel<float, float><<<grid, 256, 0, st>>>(m);
    }
    return cudaGetLastError();
}

}  // namespace gdn
