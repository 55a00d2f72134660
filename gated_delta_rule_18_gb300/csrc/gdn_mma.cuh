// gdn_mma.cuh -- warp-level bf16 tile products (mma.sync m16n8k16, fp32
// accumulate) on row-major shared-memory tiles, for the backward kernels.
//
// A tile is a row-major bf16 array with a leading dimension in elements
// (padded so that ldmatrix rows fall in different banks). An operand may be
// read straight or transposed: "A stored [m][k]" is the plain case, "A
// stored [k][m]" (at = true) reads the transpose of the stored tile through
// ldmatrix.trans; likewise B stored [k][n] (bt = true) or [n][k] (bt = false).
//
// Accumulator fragment layout (per warp, one 16 x 8 tile per acc[n]): element
// e of acc[n] sits at row m0 + g8 + 8 (e >> 1), column n0 + 8 n + 2 t4 + (e & 1),
// with g8 = lane / 4 and t4 = lane % 4.
#pragma once

#include "gdn_common.cuh"

namespace gdn {

struct Tile {
    const __nv_bfloat16 *p;
    int ld;
};

// A fragment for rows m0 .. m0+15, k = k0 .. k0+15
__device__ __forceinline__ void frag_a(uint32_t (&a)[4], const Tile &t, bool at, int m0, int k0, int lane) {
    if (!at)
        ldsm_x4(a, t.p + (m0 + (lane & 15)) * t.ld + k0 + (lane >> 4) * 8);
    else
        ldsm_x4_t(a, t.p + (k0 + (lane & 7) + ((lane >> 4) << 3)) * t.ld + m0 + ((lane >> 3) & 1) * 8);
}

// B fragments of the two 8-column tiles n0 and n0+8, k = k0 .. k0+15:
// b[0], b[1] for n0, b[2], b[3] for n0+8
__device__ __forceinline__ void frag_b2(uint32_t (&b)[4], const Tile &t, bool bt, int n0, int k0, int lane) {
    if (!bt)
        ldsm_x4(b, t.p + (n0 + (lane & 7) + ((lane >> 4) << 3)) * t.ld + k0 + ((lane >> 3) & 1) * 8);
    else
        ldsm_x4_t(b, t.p + (k0 + (lane & 15)) * t.ld + n0 + (lane >> 4) * 8);
}

// acc[NT] += A[m0 .. m0+15][0 .. kdim) . B[0 .. kdim)[n0 .. n0 + 8 NT)
template <int NT>
__device__ __forceinline__ void warp_gemm(float (&acc)[NT][4], const Tile &A, bool at, const Tile &B, bool bt,
                                          int m0, int n0, int kdim, int lane) {
    static_assert(NT % 2 == 0, "pairs of 8-column tiles");
    for (int k0 = 0; k0 < kdim; k0 += 16) {
        uint32_t a[4];
        frag_a(a, A, at, m0, k0, lane);
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
            uint32_t b[4];
            frag_b2(b, B, bt, n0 + 16 * np, k0, lane);
            mma_bf16(acc[2 * np], a, b[0], b[1]);
            mma_bf16(acc[2 * np + 1], a, b[2], b[3]);
        }
    }
}

template <int NT>
__device__ __forceinline__ void acc_zero(float (&acc)[NT][4]) {
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
}

}  // namespace gdn
