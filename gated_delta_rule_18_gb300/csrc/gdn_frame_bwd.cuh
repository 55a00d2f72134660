// gdn_frame_bwd.cuh -- parameters of the frame-causal backward kernels
// (gdn_frame_bwd.cu), shared with the C ABI in gdn_api.cu.
#pragma once
#include "gdn_common.cuh"

namespace gdn {

struct FrameBwdParams {
    const void *q, *k, *v, *dout;  // bf16 (B, T, H, D)
    int64_t qk_sb, qk_st, qk_sh, v_sb, v_st, v_sh, do_sb, do_st, do_sh;
    const float *beta;      // (B, T, H)
    const float *g_frame;   // (B, F, H)
    const float *h0;        // (B, H, K, V) or null (direction 0)
    const float *dden;      // (B, H, T) or null: the state then carries the ones column
    const float *dh_final;  // (B, H, K, V) or null (direction 0)
    float *dq, *dk, *dv, *dbeta, *dg_frame, *dh0;
    int B, T, H, K, V, Vt, Vs, F, frame;
    int direction;  // of this pass: 0 causal, 1 reverse
    int acc;        // add into the outputs (the second direction of a summed pair)
    int tok_group;  // 64-token chunks per token-gradient CTA (dividing a frame's)
    // the forward's per-frame matrices and states (workspace): A_f (K x K),
    // the states each frame's outputs read (K x Vs) per direction
    // (direction 0: frame f writes onto frame f-1's read state, or h0;
    // direction 1: frame f writes onto the state it reads itself)
    const float *amat, *sread;
    float *cmat;          // Q_f^T [dO_f | dden_f] (K x Vs) per frame
    float *lam;           // dL/d(state after frame f's write), per written frame (K x Vs)
    float *dgp;           // per (sequence x head, frame, 32-column tile) parts of dg_frame
};

constexpr int kFrameBwdCT = 32;  // state columns per chain CTA

cudaError_t launch_frame_xt(const FrameBwdParams &p, cudaStream_t st);
cudaError_t launch_frame_lam(const FrameBwdParams &p, cudaStream_t st);
cudaError_t launch_frame_tokgrad(const FrameBwdParams &p, cudaStream_t st);

}  // namespace gdn
