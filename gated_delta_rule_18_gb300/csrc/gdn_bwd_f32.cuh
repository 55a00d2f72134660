// gdn_bwd_f32.cuh -- parameters of the fp32 backward (gdn_bwd_f32.cu),
// shared with the C ABI in gdn_api.cu.
#pragma once
#include <cstdint>

#include <cuda_runtime.h>

namespace gdn {

constexpr int kF32BwdCols = 16;     // state columns per scan CTA
constexpr int kF32BwdGroup = 16;    // positions between state checkpoints
constexpr int kF32BwdThreads = 256;
constexpr int kF32BwdKP = 128;      // largest K
// floats of one checkpointed state slice: each thread's 8 rows x 1 column
constexpr int kF32BwdState = kF32BwdThreads * 8;

struct F32BwdParams {
    const float *q, *k, *v, *dout;  // fp32, strides in elements
    int64_t qk_sb, qk_st, qk_sh, v_sb, v_st, v_sh, do_sb, do_st, do_sh;
    const float *beta;              // (B, T, H)
    const float *g;                 // (B, T, H) or null (per-key gate)
    const float *gk;                // (B, T, H, K) or null
    const float *h0, *dh_final;     // (n_seq, H, K, Vs) or null
    const float *dden;              // (B, H, T) or null: column V of the state is the ones column
    const int32_t *cu_seqlens;      // (n_seq + 1) or null (dense: sequence = batch row)
    float *dv, *dh0;                // written by the scan
    float *dq, *dk, *dbeta, *dg;    // written by the reduction
    float *ckpt;                    // states before every kF32BwdGroup-th position
    float *part_k;                  // [range][row][h][NK][K]: dq^, dk^ (and dgk) per column range
    float *part_s;                  // [range][row][h][2]: dbeta, dg (scalar gate) per column range
    int *err;
    int B, T, H, K, V, Vs, n_seq, n_range, reverse, l2norm;
    int64_t ck_groups;              // checkpoint slots per (head, range)
};

cudaError_t launch_bwd_f32_scan(const F32BwdParams &p, cudaStream_t st);
cudaError_t launch_bwd_f32_reduce(const F32BwdParams &p, cudaStream_t st);

}  // namespace gdn
