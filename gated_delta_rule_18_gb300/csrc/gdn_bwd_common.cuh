// gdn_bwd_common.cuh -- pieces shared by the chunk-parallel backward
// kernels (scalar and per-key gates): chunk addressing through the forward's
// chunk table, row loads, L2 normalisation of tiles, and the 64 x 64
// triangular solve T = (I + A)^{-1} by 16 x 16 blocks.
#pragma once
#include "gdn_mma.cuh"

namespace gdn {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kThreads = 256;
constexpr int kLK = kKP + 8;   // row stride of 128-column tiles (keys or values)
constexpr int kL6 = 64 + 8;    // row stride of 64-column tiles
constexpr int kPS = kChunk + 1;  // fp32 64 x 64 row stride

__device__ __forceinline__ int round16(int x) { return (x + 15) & ~15; }

// common per-chunk addressing: chunk c of sequence s (s < 0: no chunk in
// this slot), its tokens at flat rows row0 + t (row0 = b * T + tstart)
struct ChunkCtx {
    int s, hh, c, pos0, Lc, len, b, tstart;
    int64_t row0;
    int64_t gch;  // [head][global chunk] image / snapshot slot
};
__device__ __forceinline__ ChunkCtx chunk_ctx(const BwdParams &p) {
    ChunkCtx x;
    x.hh = blockIdx.x % p.H;
    const int gid = blockIdx.x / p.H;
    x.s = -1;
    if (p.cu_seqlens) {  // the forward's chunk table (a bad cu_seqlens leaves it empty)
        if (gid >= *p.n_chunks) return x;
        const int2 e = p.chunk_tab[gid];
        x.s = e.x, x.c = e.y;
        x.b = 0, x.tstart = p.cu_seqlens[x.s], x.len = p.cu_seqlens[x.s + 1] - x.tstart;
    } else {
        const int nts = (p.T + kChunk - 1) / kChunk;
        x.s = gid / nts, x.c = gid - x.s * nts;
        x.b = x.s, x.tstart = 0, x.len = p.T;
    }
    x.pos0 = x.c * kChunk;
    x.Lc = min(kChunk, x.len - x.pos0);
    x.row0 = (int64_t)x.b * p.T + x.tstart;
    x.gch = (int64_t)x.hh * p.max_chunks + gid;
    return x;
}

// 16-byte pieces of a (rows x ncol) bf16 block into a row-major 128-column
// tile: thread t copies piece t % 16 of rows t / 16, t / 16 + NT / 16, ...;
// rows with no source (row_ptr NULL) and columns >= ncol are zero-filled
template <int NT = kThreads, class RowPtr>
__device__ __forceinline__ void load_rows(bf16 *dst, int ld, int rows, int ncol, RowPtr row_ptr) {
    const int c8 = (threadIdx.x & 15) * 8;
    for (int i = threadIdx.x >> 4; i < rows; i += NT / 16) {
        const bf16 *src = row_ptr(i);
        const bool in = src != nullptr && c8 < ncol;
        cp_async16(dst + i * ld + c8, in ? src + c8 : dst, in ? 16 : 0);
    }
}

// row sums of a warp's 16 x (8 NF) fragment set c (see gdn_mma.cuh) stored
// into row_dst[m0 ..], and column sums times col_sign into col_dst[n0 ..]:
// the gate-gradient terms of entries that depend on G_i - G_j. Every row and
// column has one writer per warp, so the caller's slots are summed in a
// fixed order (bit-reproducible runs).
template <int NF>
__device__ __forceinline__ void rowcol_store(const float (&c)[NF][4], int m0, int n0, float *row_dst,
                                             float *col_dst, float col_sign) {
    const int lane = threadIdx.x & 31, g8 = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        float r = 0.f;
#pragma unroll
        for (int n = 0; n < NF; ++n) r += c[n][2 * hf] + c[n][2 * hf + 1];
        r += __shfl_xor_sync(0xffffffffu, r, 1);
        r += __shfl_xor_sync(0xffffffffu, r, 2);
        if (t4 == 0) row_dst[m0 + g8 + 8 * hf] = r;
    }
#pragma unroll
    for (int n = 0; n < NF; ++n)
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            float v = c[n][b] + c[n][2 + b];
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            if (g8 == 0) col_dst[n0 + 8 * n + 2 * t4 + b] = col_sign * v;
        }
}

// L2 norms of 64 rows of a tile (1 when not normalising), then the rows
// scaled in place (bf16); NT threads call it (threads past 256 only scale)
template <int NT = kThreads>
__device__ __forceinline__ void norm_rows(bf16 *t, int ld, int ncol, float *r_out, bool l2) {
    const int tid = threadIdx.x;
    if (tid < 4 * kChunk) {  // four threads per row, each a quarter of the columns (whole warps)
        const int row = tid >> 2, q4 = tid & 3;
        float ss = 0.f;
        for (int d = 8 * q4; d < ncol; d += 32) {
            const uint4 u = *reinterpret_cast<const uint4 *>(t + row * ld + d);
            const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const float2 f = __bfloat1622float2(h2[x]);
                ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
            }
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        if (q4 == 0) r_out[row] = l2 ? rsqrtf(ss + 1e-6f) : 1.f;
    }
    __syncthreads();
    if (!l2) return;
    for (int e = tid; e < kChunk * (ncol / 8); e += NT) {
        const int i = e / (ncol / 8), d = (e % (ncol / 8)) * 8;
        uint4 u = *reinterpret_cast<const uint4 *>(t + i * ld + d);
        __nv_bfloat162 *h2 = reinterpret_cast<__nv_bfloat162 *>(&u);
        const float r = r_out[i];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const float2 f = __bfloat1622float2(h2[x]);
            h2[x] = __floats2bfloat162_rn(f.x * r, f.y * r);
        }
        *reinterpret_cast<uint4 *>(t + i * ld + d) = u;
    }
}

// The denominator's column of a range that carries it: dden into the dout
// tile (query rows), and the ones value into the value tile (key rows). Rows
// 0 .. 63 by threads 0 .. 63; a barrier must follow before the tiles are read.
__device__ __forceinline__ void fill_den_dout(const BwdParams &p, const ChunkCtx &x, bf16 *dout, int ld) {
    const int i = threadIdx.x;
    if (p.den_col < 0 || i >= kChunk) return;
    float d = 0.f;
    if (i < x.Lc)
        d = p.dden[((int64_t)x.b * p.H + x.hh) * p.T + x.tstart + q_token(p.reverse, x.len, x.pos0 + i)];
    dout[i * ld + p.den_col] = __float2bfloat16_rn(d);
}
__device__ __forceinline__ void fill_den_v(const BwdParams &p, const ChunkCtx &x, bf16 *vt, int ld) {
    const int i = threadIdx.x;
    if (p.den_col < 0 || i >= kChunk) return;
    const int tk = i < x.Lc ? kv_token(p.reverse, x.len, x.pos0 + i) : -1;
    vt[i * ld + p.den_col] = __float2bfloat16_rn(tk >= 0 ? 1.f : 0.f);
}
// value columns of this range that come from v / dout (the rest: the ones column)
__device__ __forceinline__ int value_cols(const BwdParams &p) { return p.den_col >= 0 ? p.den_col : p.V; }

// The per-key sums (dq or dk, (B*T, H, K) fp32) that an earlier value range
// left at this thread's fragment positions: chunk rows r0 and r0 + 8, keys
// k0 + 8n + 2 (lane & 3), n < NF. Zero on the first range, where `on` is
// false, past K, or where tok_of(row) < 0. All loads go out together, ahead
// of the stores that add them: a load placed after a store through the same
// pointer would otherwise wait for the one before it.
template <int NF, class TokOf>
__device__ __forceinline__ void acc_rows_load(float2 (&prev)[2][NF], const BwdParams &p, const ChunkCtx &x,
                                              const float *base, int r0, int k0, bool on, TokOf tok_of) {
    const int t4 = threadIdx.x & 3;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        const int tk = p.acc && on ? tok_of(r0 + 8 * hf) : -1;
        const float *src = tk >= 0 ? base + ((x.row0 + tk) * p.H + x.hh) * p.K : nullptr;
#pragma unroll
        for (int n = 0; n < NF; ++n) {
            const int d = k0 + 8 * n + 2 * t4;
            prev[hf][n] = src && d < p.K ? *reinterpret_cast<const float2 *>(src + d) : make_float2(0.f, 0.f);
        }
    }
}

// T = (I + A)^{-1} with A_ij = beta_i kkg_ij (i > j; kkg fp32 with row
// stride kPS), by 16 x 16 blocks as in the forward's solve: diagonal
// inverses T_II in fp32 by forward substitution, B_IM = -T_II A_IM, then
// block row I of T is sum_{M<I} B_IM (block row M) next to T_II (bf16
// products, fp32 sums). T goes to sTb (bf16, row stride kL6); sAb and sBb
// (same shape) hold A and the B_IM meanwhile. Every thread of the CTA calls
// it (NT threads); it ends with a barrier.
template <int NT = kThreads>
__device__ __forceinline__ void solve_t(const float *kkg, const float *beta, bf16 *sTb, bf16 *sAb,
                                        bf16 *sBb) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g8 = lane >> 2, t4 = lane & 3;
    for (int e = tid; e < kChunk * 32; e += NT) {
        const int i = e >> 5, j = (e & 31) * 2;
        const float a0 = j < i ? beta[i] * kkg[i * kPS + j] : 0.f;
        const float a1 = j + 1 < i ? beta[i] * kkg[i * kPS + j + 1] : 0.f;
        *reinterpret_cast<uint32_t *>(sAb + i * kL6 + j) = pack_bf16(a0, a1);
        *reinterpret_cast<uint32_t *>(sTb + i * kL6 + j) = 0u;
    }
    __syncthreads();
    if (warp < 4 && lane < 16) {  // diagonal blocks: forward substitution, lane = column
        const int o = 16 * warp;
        float t[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            // t_r = e_r - beta_r sum_{j<r} kkg_rj t_j, in two independent halves
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int j = 0; j < r; ++j) {
                if (j & 1) a1 = fmaf(kkg[(o + r) * kPS + o + j], t[j], a1);
                else a0 = fmaf(kkg[(o + r) * kPS + o + j], t[j], a0);
            }
            t[r] = ((r == lane) ? 1.f : 0.f) - beta[o + r] * (a0 + a1);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) sTb[(o + r) * kL6 + o + lane] = __float2bfloat16_rn(t[r]);
    }
    __syncthreads();
    if (warp >= 1 && warp < 4) {  // B_IM = -T_II A_IM for M < I = warp
        const int I = warp;
        uint32_t a[4];
        frag_a(a, Tile{sTb, kL6}, false, 16 * I, 16 * I, lane);
#pragma unroll
        for (int x2 = 0; x2 < 4; ++x2) a[x2] ^= 0x80008000u;  // -T_II
        for (int M = 0; M < I; ++M) {
            uint32_t b[4];
            ldsm_x4_t(b, sAb + (16 * I + (lane & 15)) * kL6 + 16 * M + (lane >> 4) * 8);
            float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
            mma_bf16(c0, a, b[0], b[1]);
            mma_bf16(c1, a, b[2], b[3]);
            bf16 *dst = sBb + (16 * I) * kL6 + 16 * M;
            *reinterpret_cast<uint32_t *>(dst + g8 * kL6 + 2 * t4) = pack_bf16(c0[0], c0[1]);
            *reinterpret_cast<uint32_t *>(dst + (g8 + 8) * kL6 + 2 * t4) = pack_bf16(c0[2], c0[3]);
            *reinterpret_cast<uint32_t *>(dst + g8 * kL6 + 8 + 2 * t4) = pack_bf16(c1[0], c1[1]);
            *reinterpret_cast<uint32_t *>(dst + (g8 + 8) * kL6 + 8 + 2 * t4) = pack_bf16(c1[2], c1[3]);
        }
    }
    __syncthreads();
    for (int I = 1; I < 4; ++I) {  // block row I left of the diagonal
        if (warp == I) {
            float tr[8][4];
            acc_zero(tr);
            warp_gemm(tr, Tile{sBb, kL6}, false, Tile{sTb, kL6}, true, 16 * I, 0, 16 * I, lane);
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                if (8 * n >= 16 * I) break;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
                    *reinterpret_cast<uint32_t *>(sTb + (16 * I + g8 + 8 * hf) * kL6 + 8 * n + 2 * t4) =
                        pack_bf16(tr[n][2 * hf], tr[n][2 * hf + 1]);
            }
        }
        __syncthreads();
    }
}

}  // namespace
}  // namespace gdn
