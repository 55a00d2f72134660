// gdn_merge.cu -- the bidirectional merge of the SANA `fused_gdn.py` page
// (`fused_bigdn_func`: out = (num_fwd + num_bwd) / (den_fwd + den_bwd + eps);
// `_fused_bidi_merge_kernel`, PRE_SUMMED, with the optional APPLY_GATE
// factor silu(gate) = gate / (1 + e^{-gate})). The scan has already summed
// both directions into num (B, T, H, V) and den (B, H, T).
//
// HBM-bound elementwise pass: each block takes whole (token, head) rows, one
// 16-byte vector per thread, fp32 arithmetic.
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
__global__ void __launch_bounds__(256) merge_kernel(const MergeParams m, int vpr, int rows_per_block) {
    constexpr int N = Vec<TI>::N;
    // a block covers rows_per_block whole (token, head) rows of vpr vectors
    const int lr = threadIdx.x / vpr, c = (threadIdx.x - lr * vpr) * N;
    const int row = blockIdx.x * rows_per_block + lr;
    if (lr >= rows_per_block || row >= m.B * m.T * m.H) return;
    const int h = row % m.H, bt = row / m.H;
    const int t = bt % m.T, b = bt / m.T;
    const float inv = 1.f / (__ldg(m.den + ((int64_t)b * m.H + h) * m.T + t) + m.eps);
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
    } else {  // fp32 in, bf16 out: one 8-byte half
        TO *o = (TO *)m.out + b * m.o_sb + (int64_t)t * m.o_st + h * m.o_sh + c;
        *reinterpret_cast<uint2 *>(o) = make_uint2(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]));
    }
}

// out += add (rows of V, 16-byte vectors; add contiguous (B, T, H, V) in
// out's dtype) and den += den_add (B * H * T), fp32 arithmetic
template <class T>
__global__ void __launch_bounds__(256) sum_kernel(const SumParams a, int vpr, int rows_per_block) {
    constexpr int kVec = 16 / sizeof(T);
    const int tid = threadIdx.x;
    const int64_t row = (int64_t)blockIdx.x * rows_per_block + tid / vpr;
    const int c = (tid % vpr) * kVec;
    const int64_t rows = (int64_t)a.B * a.T * a.H;
    if (tid < rows_per_block * vpr && row < rows) {
        const int64_t h = row % a.H, t = (row / a.H) % a.T, b = row / ((int64_t)a.H * a.T);
        T *o = (T *)a.out + b * a.o_sb + t * a.o_st + h * a.o_sh + c;
        const T *x = (const T *)a.add + row * a.V + c;
        uint4 uo = *reinterpret_cast<const uint4 *>(o);
        const uint4 ux = __ldg(reinterpret_cast<const uint4 *>(x));
        if (sizeof(T) == 2) {
            __nv_bfloat162 *po = reinterpret_cast<__nv_bfloat162 *>(&uo);
            const __nv_bfloat162 *px = reinterpret_cast<const __nv_bfloat162 *>(&ux);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 fo = __bfloat1622float2(po[i]), fx = __bfloat1622float2(px[i]);
                po[i] = __floats2bfloat162_rn(fo.x + fx.x, fo.y + fx.y);
            }
        } else {
            float *po = reinterpret_cast<float *>(&uo);
            const float *px = reinterpret_cast<const float *>(&ux);
#pragma unroll
            for (int i = 0; i < 4; ++i) po[i] += px[i];
        }
        *reinterpret_cast<uint4 *>(o) = uo;
    }
    if (a.den)
        for (int64_t i = (int64_t)blockIdx.x * 256 + tid; i < (int64_t)a.B * a.H * a.T; i += (int64_t)gridDim.x * 256)
            a.den[i] += a.den_add[i];
}

}  // namespace

cudaError_t launch_sum(const SumParams &a, cudaStream_t st) {
    const int vec = a.bf16 ? 8 : 4;
    const int vpr = a.V / vec;
    const int rows_per_block = vpr <= 256 ? 256 / vpr : 0;
    if (rows_per_block == 0) return cudaErrorInvalidValue;
    const int64_t rows = (int64_t)a.B * a.T * a.H;
    if (rows > INT32_MAX) return cudaErrorInvalidValue;
    const unsigned grid = (unsigned)((rows + rows_per_block - 1) / rows_per_block);
    if (grid == 0) return cudaSuccess;
    if (a.bf16) sum_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(a, vpr, rows_per_block);
    else sum_kernel<float><<<grid, 256, 0, st>>>(a, vpr, rows_per_block);
    return cudaGetLastError();
}

cudaError_t launch_merge(const MergeParams &m, cudaStream_t st) {
    const int vec = m.num_bf16 ? 8 : 4;
    const int vpr = m.V / vec;  // vectors per row (V <= 1024 keeps it <= 256)
    const int rows_per_block = vpr <= 256 ? 256 / vpr : 0;
    if (rows_per_block == 0) return cudaErrorInvalidValue;
    const int64_t rows = (int64_t)m.B * m.T * m.H;
    if (rows > INT32_MAX) return cudaErrorInvalidValue;
    const unsigned grid = (unsigned)((rows + rows_per_block - 1) / rows_per_block);
    if (m.num_bf16) {
        if (m.out_bf16) merge_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, 256, 0, st>>>(m, vpr, rows_per_block);
        else return cudaErrorInvalidValue;  // bf16 in, fp32 out: not offered
    } else {
        if (m.out_bf16) merge_kernel<float, __nv_bfloat16><<<grid, 256, 0, st>>>(m, vpr, rows_per_block);
        else merge_kernel<float, float><<<grid, 256, 0, st>>>(m, vpr, rows_per_block);
    }
    return cudaGetLastError();
}

}  // namespace gdn

// ------------------------------------------------------------ backward ---
// Gradients of out = num / (den + eps) * s, s = silu(gate) (or 1), for an
// upstream dout: with r = 1 / (den + eps),
//   dnum = dout s r,  dden = -sum_v dout num s r^2,
//   dgate = dout num r silu'(gate),  silu'(x) = sig(x) (1 + x (1 - sig(x))).
// One warp per (b, t, h) row of V values (dden summed by the warp, in a
// fixed order); num and gate through their strides, dout and the outputs
// fp32 contiguous.
namespace gdn {
namespace {
template <typename T>
__device__ __forceinline__ float ld_f(const T *p) {
    if constexpr (sizeof(T) == 4) return *p;
    else return __bfloat162float(*p);
}
template <typename T>
__global__ void __launch_bounds__(256) merge_bwd_kernel(const T *num, int64_t n_sb, int64_t n_st, int64_t n_sh,
                                                        const float *den, const T *gate, int64_t g_sb,
                                                        int64_t g_st, int64_t g_sh, const float *dout,
                                                        float *dnum, float *dden, float *dgate, int B, int T_,
                                                        int H, int V, float eps) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= (int64_t)B * T_ * H) return;
    const int h = (int)(row % H);
    const int64_t tok = row / H;
    const int b = (int)(tok / T_), t = (int)(tok % T_);
    const int64_t di = ((int64_t)b * H + h) * T_ + t;
    const float r = 1.f / (den[di] + eps);
    const T *nrow = num + b * n_sb + (int64_t)t * n_st + h * n_sh;
    const T *grow = gate ? gate + b * g_sb + (int64_t)t * g_st + h * g_sh : nullptr;
    const float *orow = dout + row * V;
    float acc = 0.f;
    for (int c = lane; c < V; c += 32) {
        const float n = ld_f(nrow + c), go = orow[c];
        float s = 1.f, ds = 0.f;
        if (grow) {
            const float x = ld_f(grow + c);
            const float sg = 1.f / (1.f + __expf(-x));
            s = x * sg;
            ds = sg * (1.f + x * (1.f - sg));
        }
        dnum[row * V + c] = go * s * r;
        if (dgate) dgate[row * V + c] = go * n * r * ds;
        acc = fmaf(go * n, s, acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) dden[di] = -acc * r * r;
}
}  // namespace

cudaError_t launch_merge_bwd(const void *num, int64_t n_sb, int64_t n_st, int64_t n_sh, int bf16,
                             const float *den, const void *gate, int64_t g_sb, int64_t g_st, int64_t g_sh,
                             const float *dout, float *dnum, float *dden, float *dgate, int B, int T,
                             int H, int V, float eps, cudaStream_t st) {
    const int64_t rows = (int64_t)B * T * H;
    if (rows == 0) return cudaSuccess;
    const unsigned grid = (unsigned)((rows + 7) / 8);
    if (bf16)
        merge_bwd_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
            (const __nv_bfloat16 *)num, n_sb, n_st, n_sh, den, (const __nv_bfloat16 *)gate, g_sb, g_st, g_sh,
            dout, dnum, dden, dgate, B, T, H, V, eps);
    else
        merge_bwd_kernel<float><<<grid, 256, 0, st>>>((const float *)num, n_sb, n_st, n_sh, den,
                                                      (const float *)gate, g_sb, g_st, g_sh, dout, dnum,
                                                      dden, dgate, B, T, H, V, eps);
    return cudaGetLastError();
}
}  // namespace gdn
