// gdn_common.cuh -- shared definitions of the sm_103a kernels behind gdn.h:
// the launch parameter block, sequence/token addressing (including the
// flip-and-shift reverse scan done by index remapping), and thin inline-PTX
// wrappers (cp.async, bulk async copies, mbarriers, ldmatrix, movmatrix,
// bf16 mma).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr int kChunk = 64;  // tokens per chunk

// Floors applied to log gates on load. A decay below e^-30 (~1e-13) is
// indistinguishable from 0 in fp32 next to O(1) terms, and the floor keeps
// exp(G_i - G_j) of cumulative gates finite for g = -inf (a full reset).
// The bf16 per-key path splits e^{G_i - G_j} into two factors about a point
// at most 8 tokens away (see gdn_intra_bf16.cu); a floor of -10 per token
// bounds each factor by e^80, below the fp32/bf16 overflow at e^88. It
// changes the result only for per-key decays below e^-10 = 4.5e-5 per token,
// by less than that relative amount.
constexpr float kLogGateMin = -30.f;
constexpr float kLogGateMinPerKeyTC = -10.f;

// Everything a forward launch needs. Strides are in elements.
struct FwdParams {
    const void *q, *k, *v;
    int64_t qk_sb, qk_st, qk_sh;
    int64_t v_sb, v_st, v_sh;
    const float *g, *gk, *beta, *h0;
    const int32_t *cu_seqlens;
    void *out;
    int64_t o_sb, o_st, o_sh;
    int out_f32;
    float *h_final, *den;
    int B, T, H, K, V, n_seq;
    int reverse, accumulate, l2norm, has_den;
    int Vt;  // V + has_den: value columns carried by the scan
    int snap_ld;  // row stride of the h / v_new snapshots: Vt rounded up to 8 (16-byte rows)
    int h_ld;  // row stride (floats) of h0 / h_final in the bf16 state pass: Vt, or the
               // full width when a backward pass recomputes one value-column range
    // workspace
    int *err;         // device error word
    int *n_chunks;    // number of valid chunk-table entries (varlen)
    int2 *chunk_tab;  // (seq, chunk index within seq) per global chunk
    int *seq_chunk0;  // first global chunk of each sequence
    int max_chunks;
    // Per-chunk operand images, indexed [head][global chunk], each laid out
    // exactly as the state kernel's shared-memory MMA operand (see the
    // image layout helpers below) so that one bulk copy stages it.
    unsigned char *w_img, *qg_img, *kg_img, *p_img, *u_img;
    float *dec;       // [H][max_chunks][kKP] chunk decay e^{G_last}
    int n_vt;         // 64-column value tiles (ceil(Vt / 64))
    // Segment-parallel state passing (dense batches): the chunks of every
    // sequence are cut into segments of seg_chunks chunks (0: one segment),
    // one state-kernel CTA per segment (grid z). With summary set the kernel
    // emits each segment's affine summary h_out = M h_in + E instead of
    // outputs: value tiles run from h = 0 (E), n_kt extra 64-column tiles run
    // the same recurrence with u = 0 from h = I (the transition M). Otherwise
    // segment s starts from h_in[s] when h_in is given. summary 1 covers every
    // segment and stores M; summary 2 all but the last and stores M^T.
    int seg_chunks, summary, n_kt;
    float *sum_ext;      // (segments, n_seq * H, K, Vt)
    float *sum_tr;       // (segments, n_seq * H, K, K)
    const float *h_in;   // (segments, n_seq * H, K, Vt)
    // Recompute pass of the backward: when set, the state kernel also stores
    // the state entering every chunk and the chunk's v_new, bf16, indexed
    // [head][global chunk]: h_snap (K, V) rows, vn_snap (64, V) rows.
    __nv_bfloat16 *h_snap, *vn_snap;
    // testing aid for the bounded-wait path: block stall_cta (linear index)
    // of the intra-chunk and state kernels stalls instead of working (-1: off)
    int stall_cta, stall_us;
};

// Everything the backward kernels need (dense batches, scalar gate). The
// gradient outputs are fp32 and contiguous: dq, dk (B, T, H, K), dv (B, T,
// H, V), dbeta, dg (B, T, H), dh0 (B, H, K, V).
struct BwdParams {
    const void *q, *k, *v, *dout;
    int64_t qk_sb, qk_st, qk_sh;
    int64_t v_sb, v_st, v_sh;
    int64_t do_sb, do_st, do_sh;
    const float *g, *gk, *beta, *dh_final;  // gk: per-key gates (then dg is (B, T, H, K))
    float *dq, *dk, *dv, *dbeta, *dg, *dh0;
    int B, T, H, K, V, reverse, l2norm;
    int max_chunks;  // chunk slots per head (the forward's)
    // variable-length batches: the forward's chunk table (B == 1)
    const int32_t *cu_seqlens;
    const int *n_chunks, *seq_chunk0;
    const int2 *chunk_tab;
    int n_seq;
    // one pass covers value columns [v_off, v_off + V) of vfull: dout, v, dv,
    // dh_final and dh0 point at column v_off and keep rows of vfull columns
    int vfull, v_off;
    int dv_ld;  // row stride of dv (the value columns, without the denominator's)
    int snap_ld;  // row stride of the snapshots: V rounded up to 8 (16-byte rows)
    int acc;                 // add dq, dk, dbeta, dg into the outputs (a later value range)
    // the denominator: its upstream gradient (B, H, T), and the column of this
    // range that carries the ones value (-1: none; then V = the value columns)
    const float *dden;
    int den_col;
    float *dk_part, *dg_part;  // bwd_dq's shares of dk and dG, read by bwd_dk (workspace)
    // the forward's per-chunk operand images and snapshots (workspace)
    const unsigned char *w_img, *qg_img, *kg_img, *p_img;
    const float *dec;
    const __nv_bfloat16 *h_snap, *vn_snap;
    __nv_bfloat16 *dh_snap, *dvn_snap;  // state gradient at each chunk's end, dL/dv_new
    int *err;                           // device error word (bounded waits that gave up)
};

// ----------------------------------------------------- operand images -------
// The tensor-core MMAs read bf16 operands from shared memory in the
// no-swizzle canonical layout: 8 x 16-byte "core" blocks, addressed by a
// descriptor (start, LBO = byte stride between cores along K, SBO = byte
// stride between cores along M/N). The images below use LBO = 128 bytes,
// i.e. the cores along K are adjacent.
constexpr int kKP = 128;                 // keys per image (zero padded)
constexpr uint32_t kImgW = 64 * kKP * 2;  // w, qg (64 tokens x 128 keys), kg^T
constexpr uint32_t kImgP = 64 * 64 * 2;   // P (64 x 64)
constexpr uint32_t kImgU = 64 * 64 * 2;   // one 64-column u tile
constexpr uint32_t kDecB = kKP * 4;       // chunk decay vector

// w / qg: K-major A operand, M = token i, K = key d: core (i/8, d/8).
__host__ __device__ __forceinline__ uint32_t img_w_off(int i, int d) {
    return (uint32_t)((i >> 3) * 2048 + (d >> 3) * 128 + (i & 7) * 16 + (d & 7) * 2);
}
// kg^T: MN-major A operand, M = key d, K = token i: core (d/8, i/8).
__host__ __device__ __forceinline__ uint32_t img_kt_off(int i, int d) {
    return (uint32_t)((d >> 3) * 1024 + i * 16 + (d & 7) * 2);
}
// u (one 64-column tile): MN-major B operand, N = column j, K = token i:
// core (j/8, i/8), so a warp's stores of 8 rows x 8 columns fill 128 bytes.
__host__ __device__ __forceinline__ uint32_t img_u_off(int i, int j) {
    return (uint32_t)((j >> 3) * 1024 + i * 16 + (j & 7) * 2);
}
// P: K-major A operand, M = token i, K = token j.
__host__ __device__ __forceinline__ uint32_t img_p_off(int i, int j) {
    return (uint32_t)((i >> 3) * 1024 + (j >> 3) * 128 + (i & 7) * 16 + (j & 7) * 2);
}

// Sequence s: first flat token row, length, batch index, first token in
// its batch row.
struct SeqInfo {
    int64_t row0;  // flat token index b*T + tstart
    int len;
    int b;
    int tstart;
};

__device__ __forceinline__ bool seq_info(const FwdParams &p, int s, SeqInfo &si) {
    if (p.cu_seqlens) {
        int a = p.cu_seqlens[s], e = p.cu_seqlens[s + 1];
        if (a < 0 || e < a || e > p.T) return false;
        si.b = 0;
        si.tstart = a;
        si.len = e - a;
        si.row0 = a;
    } else {
        si.b = s;
        si.tstart = 0;
        si.len = p.T;
        si.row0 = (int64_t)s * p.T;
    }
    return true;
}

// Physical token (within the sequence) that feeds logical position `pos`.
// Query rows and output rows: the reverse scan flips. Key/value/beta/gate
// rows: the reverse scan flips and shifts by one; position 0 reads nothing
// (returns -1: zero key/value/beta and a zero log-gate).
__device__ __forceinline__ int q_token(int reverse, int len, int pos) {
    return reverse ? len - 1 - pos : pos;
}
__device__ __forceinline__ int kv_token(int reverse, int len, int pos) {
    return reverse ? (pos == 0 ? -1 : len - pos) : pos;
}

// ---------------------------------------------------------------- PTX ------

__device__ __forceinline__ uint32_t smem_u32(const void *ptr) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}

// 16-byte async copy global -> shared; src_bytes < 16 zero-fills the rest.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)),
                 "l"(gmem), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// ---- mbarriers and 1-D bulk async copies (global -> shared)

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// order this thread's generic-proxy shared-memory accesses before later
// async-proxy ones (bulk copies, tensor-core operand reads)
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// one arrival that also announces `bytes` of copies counted on the barrier
__device__ __forceinline__ void arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// bytes: a multiple of 16; both addresses 16-byte aligned
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
// pull global bytes into L2 ahead of a later bulk copy (no completion signal)
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
// Wait for the mbarrier phase `parity`; false after ~0.5 s or once *abort is
// set by another role (no hang either way). abort may be null.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
        if ((it & 255) == 0) {
            if (abort && *abort) return false;
            const uint64_t t = now_ns();
            if (t0 == 0) t0 = t;
            else if (t - t0 > 500000000ull) {
                if (abort) *abort = 1;
                return false;
            }
        }
    }
}

// Device error word bits (the same values as GDN_DEVERR_* in gdn.h).
constexpr int kDevErrSeqlens = 1, kDevErrTimeout = 2;

// Testing aid for the time-out path: the block whose linear index is
// stall_cta waits on an mbarrier that nothing completes until its stall_us
// limit runs out, records a time-out in the error word and reports true, so
// that the kernel leaves before issuing any copy or MMA. Every other block
// returns false at once. The decision depends only on the block index, so a
// block's threads all take the same branch. (Scalars, not the parameter
// block, are passed: taking the address of a kernel's parameters would move
// them to local memory.)
static __device__ __forceinline__ bool stall_test(int stall_cta, int stall_us, int *err) {
    const int b = (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
    if (stall_cta < 0 || b != stall_cta) return false;
    __shared__ __align__(8) uint64_t never;
    const uint32_t bar = smem_u32(&never);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        const uint64_t t0 = now_ns(), lim = (uint64_t)max(stall_us, 1) * 1000ull;
        for (;;) {
            uint32_t ok;
            asm volatile(
                "{\n .reg .pred q;\n mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2;\n"
                " selp.u32 %0, 1, 0, q;\n}"
                : "=r"(ok)
                : "r"(bar), "r"(0u)
                : "memory");
            if (ok || now_ns() - t0 > lim) break;
        }
        atomicOr(err, kDevErrTimeout);
    }
    __syncthreads();
    return true;
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *smem) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(smem)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *smem) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(smem)));
}

// 8x8 b16 transpose across the warp: in and out in the mma fragment layout
// (lane holds row lane/4, columns 2*(lane%4) and 2*(lane%4)+1).
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
        "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float bf16_to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

// Load a value of the storage type as float.
template <typename T>
__device__ __forceinline__ float ldf(const T *p);
template <>
__device__ __forceinline__ float ldf<float>(const float *p) { return *p; }
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

}  // namespace gdn

// Host-side launchers, defined in the .cu files and called by gdn_api.cu.
namespace gdn {
cudaError_t launch_chunk_table(const FwdParams &p, cudaStream_t st);
// The bidirectional merge: out = num / (den + eps) * (gate ? silu(gate) : 1).
struct MergeParams {
    const void *num;  // (B, T, H, V), fp32 or bf16
    int64_t n_sb, n_st, n_sh;
    const float *den;  // (B, H, T) contiguous
    const void *gate;  // like num, or null
    int64_t g_sb, g_st, g_sh;
    void *out;  // (B, T, H, V)
    int64_t o_sb, o_st, o_sh;
    int B, T, H, V;
    float eps;
    int num_bf16, out_bf16;
};
cudaError_t launch_merge(const MergeParams &m, cudaStream_t st);

// out += add, den += den_add (the two directions of a concurrent
// bidirectional scan)
struct SumParams {
    void *out;  // (B, T, H, V), fp32 or bf16
    int64_t o_sb, o_st, o_sh;
    const void *add;  // contiguous (B, T, H, V), out's dtype
    float *den;       // (B, H, T) or null
    const float *den_add;
    int B, T, H, V, bf16;
};
cudaError_t launch_sum(const SumParams &a, cudaStream_t st);
// The frame-causal form (gdn_frame.cu).
struct FrameParams {
    const void *q, *k, *v;  // bf16 (B, T, H, D)
    int64_t qk_sb, qk_st, qk_sh, v_sb, v_st, v_sh;
    const float *beta;     // (B, T, H)
    const float *g_frame;  // (B, F, H) log decay per frame
    const float *h0;       // (B, H, K, V) or null (forward only)
    float *h_final;        // (B, H, K, V) or null (forward only)
    void *out;
    int64_t o_sb, o_st, o_sh;
    int out_f32;
    float *den;  // (B, H, T) or null
    int B, T, H, K, V, Vt, F, frame;
    int Vs;  // row stride of sout: Vt rounded up to a multiple of 8
    int has_den, accumulate, direction;  // direction: 0 forward, 1 reverse, 2 both summed
    float *amat, *bmat, *sout;           // workspace: A_f (K x K), B_f (K x Vt), read states (K x Vt)
};
cudaError_t launch_frame_gram(const FrameParams &p, cudaStream_t st);
cudaError_t launch_frame_chain(const FrameParams &p, cudaStream_t st);
cudaError_t launch_frame_out(const FrameParams &p, cudaStream_t st);
cudaError_t launch_intra_bf16(const FwdParams &p, int perkey, cudaStream_t st);
// The bf16 forward of one direction in one kernel (gdn_fused_tc.cu): the
// tensor maps of q, k and v, built by fused_prepare, which returns false when
// the call needs the split path (per-key gate, segments, summaries,
// snapshots, layouts a tensor map cannot express, or the path switched off).
struct FusedMaps {
    CUtensorMap q, k, v;
};
bool fused_prepare(const FwdParams &p, FusedMaps *m);
cudaError_t launch_fused_tc(const FwdParams &p, const FusedMaps &m, cudaStream_t st);
void set_fused(int on);
cudaError_t launch_state_tc(const FwdParams &p, cudaStream_t st);
// value columns per state-kernel CTA: 0 chooses by the grid, 64 or 128 force one
void set_state_tile(int bv);

// The serial step of segment-parallel state passing: per (sequence x head),
// h_in[0] = h0 (or 0) and h_in[s+1] = M_s h_in[s] + E_s, fp32.
struct SegParams {
    const float *h0;       // (n_bh, K, V) or NULL
    const float *sum_ext;  // (n_seg, n_bh, K, Vt)
    const float *sum_tr;   // (n_seg, n_bh, K, K), each M_s transposed
    float *h_in;           // (n_seg, n_bh, K, Vt)
    int n_bh, K, V, Vt, n_seg;
};
cudaError_t launch_seg_combine(const SegParams &p, cudaStream_t st);
cudaError_t launch_bwd_dh(const BwdParams &p, cudaStream_t st);
cudaError_t launch_bwd_dq(const BwdParams &p, cudaStream_t st);
cudaError_t launch_bwd_dk(const BwdParams &p, cudaStream_t st);
cudaError_t launch_bwd_dq_gk(const BwdParams &p, cudaStream_t st);
cudaError_t launch_bwd_dk_gk(const BwdParams &p, cudaStream_t st);
cudaError_t launch_fused_f32(const FwdParams &p, int KP, int perkey, cudaStream_t st);
// the fp32 path in two kernels (chunk-parallel prep, chunk-serial pass) for
// problems whose fused grid would leave the GPU mostly idle
cudaError_t launch_f32_prep(const FwdParams &p, int KP, int perkey, cudaStream_t st);
cudaError_t launch_f32_serial(const FwdParams &p, int KP, cudaStream_t st);
// value columns of the fp32 u image (a multiple of 32)
__host__ __device__ __forceinline__ int f32_vp32(int vt) { return (vt + 31) / 32 * 32; }
// the fp32 path splits when its fused grid has at most this many CTAs
constexpr int kF32SplitMaxCtas = 32;
__host__ __device__ __forceinline__ bool f32_split(int n_seq, int H, int vt) {
    return (int64_t)n_seq * H * ((vt + 31) / 32) <= kF32SplitMaxCtas;
}
cudaError_t launch_prep(const void *x, int64_t xsb, int64_t xst, int64_t xsh, void *y,
                        int64_t ysb, int64_t yst, int64_t ysh, int B, int T, int H, int D,
                        int bf16, int mode, float scale, float eps, float *inv_rms,
                        cudaStream_t st);
}  // namespace gdn
