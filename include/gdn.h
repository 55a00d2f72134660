/*
 * gdn.h -- C ABI of libgdn.so, the GB300 (sm_103a) chunked gated delta rule
 * forward scan.
 *
 * The operation (per sequence and head, state S of K x V, fp32):
 *   S_t = (I - beta_t k_t k_t^T) e^{g_t} S_{t-1} + beta_t k_t v_t^T,
 *   o_t = S_t^T q_t, i.e. token by token
 *     S <- diag(e^{gk_t}) S            (scalar gate: e^{g_t} S)
 *     d  = beta_t (v_t - S^T k_t)
 *     S <- S + k_t d^T
 *     o_t = S^T q_t                    (inclusive: reads the updated state)
 * as defined by the SANA `fused_gdn.py` page (`_fused_gdn_kernel`, "Pass 1 --
 * State Accumulation" and "Pass 2 -- Output (reads state_curr, inclusive)")
 * and the SANA `fused_cam_gdn.py` page (`_cam_scan_kernel`, with its
 * init/final state contract). It is computed in chunks of 64 tokens with a
 * WY representation: per chunk, T = (I + strictly_lower(diag(beta)
 * (K K^T . Gamma)))^{-1}, w = T (beta e^{G} . K), u = T (beta . V), then
 * v_new = u - w h and h <- e^{G_last} h + (e^{G_last - G} . K)^T v_new, the
 * state-passing step of the hyper-parallel coverage_diff page
 * (`chunk_gated_delta_rule_fwd_kernel_h_blockdim64`).
 *
 * Conventions for every entry point:
 *   - All pointers are DEVICE pointers unless stated. The caller owns every
 *     buffer; the library never allocates device memory. Scratch space is a
 *     caller-provided workspace of gdn_workspace_size() bytes.
 *   - Calls are asynchronous on `stream`. All argument checks run on the host
 *     before any launch; a call that returns an error launched nothing.
 *   - Tensor layouts are row-major with the last dimension contiguous; the
 *     other strides are given in ELEMENTS by gdn_tensor_desc. Base pointers
 *     and strides must give 16-byte aligned rows (GDN_ERR_LAYOUT otherwise).
 *   - Errors mirror the pages' contract (SANA `fused_gdn.py` page,
 *     `fused_gdn_func`): bad shapes, dtypes, strides -> GDN_ERR_SHAPE /
 *     GDN_ERR_DTYPE / GDN_ERR_LAYOUT (the pages' ValueError); a reverse scan
 *     combined with initial/final state -> GDN_ERR_UNSUPPORTED (the pages'
 *     NotImplementedError); launch failures -> GDN_ERR_CUDA (RuntimeError).
 *     Problems only the device can see (a malformed cu_seqlens) set an error
 *     word in the workspace, skip the affected work, and are reported by
 *     gdn_last_device_error(). No kernel traps.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_NULL = 1,        /* a required pointer is NULL */
    GDN_ERR_SHAPE = 2,       /* sizes out of range or inconsistent */
    GDN_ERR_DTYPE = 3,       /* unsupported or mismatched element type */
    GDN_ERR_LAYOUT = 4,      /* stride / alignment / contiguity */
    GDN_ERR_UNSUPPORTED = 5, /* e.g. reverse scan with state input/output */
    GDN_ERR_CUDA = 6,        /* a CUDA call failed */
    GDN_ERR_TIMEOUT = 7,     /* a bounded device-side wait gave up */
    GDN_ERR_WORKSPACE = 8,   /* workspace missing, too small or misaligned */
    GDN_ERR_DEVICE = 9       /* a device-side argument check failed */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

/* Element strides of a (B, T, H, D) view; D is contiguous (stride 1). */
typedef struct {
    int32_t dtype; /* gdn_dtype */
    int32_t reserved;
    int64_t stride_b;
    int64_t stride_t;
    int64_t stride_h;
} gdn_tensor_desc;

/* gdn_prep modes */
#define GDN_PREP_L2 0x0   /* per (token, head): y = x / sqrt(sum_d x^2 + eps) */
#define GDN_PREP_RMS 0x1  /* per token over all H*D channels:
                             inv = 1/sqrt(sum_{h,d} x^2 / (H*D) + eps), y = x*inv */
#define GDN_PREP_RELU 0x10 /* then y = max(y, 0) */

/* gdn_chunk_fwd flags */
#define GDN_ACCUMULATE 0x1 /* add into out (and den_out) instead of storing */
#define GDN_QK_L2NORM 0x2  /* L2-normalise q and k per (token, head) on load
                              (eps 1e-6), fusing GDN_PREP_L2 into the scan */

/* device error word bits (gdn_last_device_error) */
#define GDN_DEVERR_SEQLENS 0x1 /* cu_seqlens not 0 = c0 <= c1 <= ... = T */
#define GDN_DEVERR_TIMEOUT 0x2 /* a bounded wait inside a kernel gave up */

/*
 * gdn_prep -- q/k preparation (SANA `fused_gdn.py` page: `_precompute_inv_rms`,
 * `_fused_qk_inv_rms_kernel`, and the ReLU / k_scale of `_fused_gdn_kernel`;
 * the per-(token, head) L2 form is the one the workload statement asks for).
 *   x, y: (B, T, H, D) with descriptors xd, yd (same dtype; may alias when
 *         the strides are equal). y = relu?(normalised x) * scale.
 *   mode: GDN_PREP_L2 or GDN_PREP_RMS, optionally | GDN_PREP_RELU.
 *   inv_rms: (B, T) fp32 output for GDN_PREP_RMS, or NULL.
 *   D <= 256 (L2) and H*D <= 16384 (RMS); D a multiple of 8 (bf16) or 4 (fp32).
 */
gdn_status gdn_prep(const void *x, gdn_tensor_desc xd, void *y,
                    gdn_tensor_desc yd, int B, int T, int H, int D, int mode,
                    float scale, float eps, float *inv_rms,
                    cudaStream_t stream);

/*
 * gdn_prep_bwd -- the gradient of gdn_prep: dx = dL/dx for an upstream dy =
 * dL/dy, with the same mode, scale and eps (the backward of the pages'
 * RMSNorm / L2 normalisation, ReLU and k_scale). With t = x inv (inv the
 * normalisation factor of x's row), dt = scale dy where the ReLU passed,
 * dx = inv dt - x inv^3 m sum_row(dt x), m = 1 (L2) or 1 / (H D) (RMS).
 *   x: (B, T, H, D), descriptor xd (the forward's input); dy, dx: (B, T, H,
 *   D) fp32, contiguous, 4-byte aligned. Limits as for gdn_prep.
 */
gdn_status gdn_prep_bwd(const void *x, gdn_tensor_desc xd, const float *dy,
                        float *dx, int B, int T, int H, int D, int mode,
                        float scale, float eps, cudaStream_t stream);

/*
 * gdn_workspace_size -- bytes of scratch gdn_chunk_fwd needs for this shape.
 *   varlen != 0: B must be 1 and T is the packed token count.
 *   with_den != 0: the call will also compute the denominator.
 * Returns 0 for sizes gdn_chunk_fwd would reject.
 */
size_t gdn_workspace_size(int B, int T, int H, int K, int V, int n_seq,
                          int varlen, int dtype, int with_den);

/*
 * gdn_chunk_fwd -- one direction of the chunked gated delta rule.
 *   q, k: (B, T, H, K), descriptor qkd (shared); v: (B, T, H, V), vd.
 *         All three have the same dtype: GDN_F32 runs the fp32 CUDA-core path
 *         (IEEE fp32 products), GDN_BF16 the bf16 tensor-core path with an
 *         fp32 state.
 *   g:    (B, T, H) fp32 natural-log gate, or NULL when gk is given.
 *   gk:   (B, T, H, K) fp32 per-key natural-log gate, or NULL.
 *   beta: (B, T, H) fp32.
 *   h0:   (n_seq, H, K, V) fp32 initial state (state at the end of a prefix,
 *         decayed by this call's first gate), or NULL for zero. With den_out
 *         the state is (n_seq, H, K, V + 1): column V is the denominator's
 *         z state (SANA `fused_gdn.py` page, `_fused_gdn_kernel`,
 *         init_state_z / the final z), the state of the same scan over
 *         v = 1, so that a stream split into calls carries both. h0 and
 *         h_final may start at any 4-byte boundary; the bf16 path moves
 *         their rows by 16-byte accesses when the start is 16-byte aligned.
 *   cu_seqlens: device int32 (n_seq + 1) offsets of packed sequences, or NULL
 *         for B dense sequences of length T (n_seq must then equal B).
 *         With cu_seqlens, B must be 1; chunks never cross sequences.
 *   out:  (B, T, H, V), descriptor od, dtype GDN_F32 or GDN_BF16.
 *   h_final: (n_seq, H, K, V) fp32 state after the last token (V + 1
 *         columns with den_out, as h0), or NULL.
 *   den_out: (B, H, T) fp32 denominator (the same scan with v = 1, SANA
 *         `fused_gdn.py` page, z state), or NULL. With T = 0 any non-NULL
 *         pointer selects the (V + 1)-column state; nothing is written.
 *   chunk: must be 64. K <= 128 (a multiple of 8), V (+1 with den_out) <= 256.
 *   reverse: 0 causal; 1 anti-causal flip-and-shift scan (SANA
 *         `fused_cam_gdn.py` page, `_flip_and_shift` and
 *         `_torch_cam_scan_reference`): o_t reads tokens t+1 .. end, token
 *         t+1's gate decays the state before its write, and no token reads
 *         itself. reverse with h0 or h_final -> GDN_ERR_UNSUPPORTED, as on
 *         the pages.
 *   flags: GDN_ACCUMULATE, GDN_QK_L2NORM.
 *   workspace: >= gdn_workspace_size() bytes, 256-byte aligned.
 */
gdn_status gdn_chunk_fwd(const void *q, const void *k, gdn_tensor_desc qkd,
                         const void *v, gdn_tensor_desc vd, const float *g,
                         const float *gk, const float *beta, const float *h0,
                         const int32_t *cu_seqlens, int n_seq, void *out,
                         gdn_tensor_desc od, float *h_final, float *den_out,
                         int B, int T, int H, int K, int V, int chunk,
                         int reverse, int flags, void *workspace,
                         size_t ws_bytes, cudaStream_t stream);

/*
 * gdn_chunk_fwd_noalloc -- gdn_chunk_fwd for callers that cannot allocate
 * device memory. The pages have no counterpart; this is a library service.
 *
 * Who needs it: code running inside a host that forbids cudaMalloc once it
 * is up (allocation would break its memory accounting or synchronise other
 * streams), runtimes whose device memory belongs to someone else, and
 * plug-ins that are handed only input and output pointers. Such callers
 * cannot provide gdn_chunk_fwd's workspace.
 *
 * Same arguments and results as gdn_chunk_fwd, minus the workspace: scratch
 * comes from a buffer of GDN_NOALLOC_SCRATCH_BYTES built into the library
 * (a file-scope device array; every GPU that loads the library holds it
 * until the process exits). Nothing is allocated: no cudaMalloc/cudaFree and
 * no allocating library routine is called (leave gdn_profile_enable off,
 * since profiling creates CUDA events).
 *   - Argument checks are gdn_chunk_fwd's and return its status codes.
 *     Problems that pass them but whose gdn_workspace_size() exceeds
 *     GDN_NOALLOC_SCRATCH_BYTES are rejected with GDN_ERR_WORKSPACE before
 *     anything runs.
 *   - The first call on each device looks up the buffer's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.
 *   - All calls share the one buffer, which keeps the last call's contents;
 *     the kernels write every scratch word they read, so nothing has to be
 *     cleared between calls. Calls that overlap on the GPU (different
 *     streams, or different host threads on the same device) race on the
 *     buffer: serialise them.
 *   - The device error word (malformed cu_seqlens, bounded waits that gave
 *     up) lives in the buffer too: read it with
 *     gdn_noalloc_last_device_error() after the call.
 */
#define GDN_NOALLOC_SCRATCH_BYTES (64u << 20)
gdn_status gdn_chunk_fwd_noalloc(const void *q, const void *k,
                                 gdn_tensor_desc qkd, const void *v,
                                 gdn_tensor_desc vd, const float *g,
                                 const float *gk, const float *beta,
                                 const float *h0, const int32_t *cu_seqlens,
                                 int n_seq, void *out, gdn_tensor_desc od,
                                 float *h_final, float *den_out, int B, int T,
                                 int H, int K, int V, int chunk, int reverse,
                                 int flags, cudaStream_t stream);

/*
 * gdn_noalloc_last_device_error -- gdn_last_device_error for the built-in
 * buffer of gdn_chunk_fwd_noalloc on the current device: synchronise
 * `stream`, store the error word in *word (may be NULL), clear it, and
 * return GDN_ERR_TIMEOUT / GDN_ERR_DEVICE / GDN_OK as gdn_last_device_error
 * does. Allocates nothing.
 */
gdn_status gdn_noalloc_last_device_error(cudaStream_t stream, int *word);

/*
 * gdn_seg_workspace_size / gdn_chunk_fwd_seg -- gdn_chunk_fwd for dense
 * batches with segment-parallel state passing (hyper-parallel coverage_diff
 * page: `kda_state_summary_forward_from_prepared` forms a piece's summary
 * (state_ext, transition), the initial state of a piece is the previous
 * piece's final state transition . h_in + state_ext, and
 * `chunk_gated_delta_rule_fwd_h` re-runs the piece from it). Each sequence
 * is cut into segments of segment_len tokens; every segment's summary
 * (E = the segment's state from h = 0, M = its transition) is formed in
 * parallel, a short fp32 chain gives the state entering each segment
 * (h_in[0] = h0, h_in[s+1] = M_s h_in[s] + E_s), and every segment is then
 * re-run from its h_in in parallel, writing the outputs. The result is the
 * token recurrence's, as for gdn_chunk_fwd (rounding differs: the states
 * entering segments are formed in fp32 from fp32 summaries). It pays when
 * B * H * ceil((V + den) / 64) is small next to the SM count.
 *   Arguments as gdn_chunk_fwd with cu_seqlens = NULL and n_seq = B; bf16
 *   q/k/v only (GDN_ERR_DTYPE for fp32). segment_len: a positive multiple of
 *   64 (GDN_ERR_SHAPE otherwise); a sequence of at most segment_len tokens
 *   runs as gdn_chunk_fwd does.
 *   workspace: >= gdn_seg_workspace_size() bytes, 256-byte aligned.
 */
size_t gdn_seg_workspace_size(int B, int T, int H, int K, int V, int with_den,
                              int segment_len);
gdn_status gdn_chunk_fwd_seg(const void *q, const void *k, gdn_tensor_desc qkd,
                             const void *v, gdn_tensor_desc vd, const float *g,
                             const float *gk, const float *beta,
                             const float *h0, void *out, gdn_tensor_desc od,
                             float *h_final, float *den_out, int B, int T,
                             int H, int K, int V, int chunk, int reverse,
                             int flags, int segment_len, void *workspace,
                             size_t ws_bytes, cudaStream_t stream);

/*
 * gdn_seg_choose -- a segment_len for gdn_chunk_fwd_seg on a GPU with n_sm
 * SMs (host arithmetic only, no CUDA call): the length that minimises the
 * estimated time of the summary pass, the chain and the re-run, counted in
 * chunk steps of state-kernel CTAs at one per SM. A result >= T means the
 * plain one-segment pass is estimated fastest. Returns 0 for bad sizes.
 */
int gdn_seg_choose(int B, int T, int H, int K, int V, int with_den, int n_sm);

/*
 * gdn_state_summary -- the affine summary of each segment of each sequence
 * (hyper-parallel coverage_diff page, `kda_state_summary_forward_from_prepared`
 * returning state_ext and transition): for segment s of segment_len tokens
 * (the last one ragged), the state after the segment is
 *   h_out = transition_s . h_in + state_ext_s
 * for any state h_in entering it (h in [K, V] orientation, causal scan).
 *   k: (B, T, H, K) bf16, kd; v: (B, T, H, V) bf16, vd; g / gk / beta as for
 *   gdn_chunk_fwd. flags: GDN_QK_L2NORM (normalise k) or 0.
 *   state_ext: (n_seg, B, H, K, V) fp32 output; transition: (n_seg, B, H, K,
 *   K) fp32 output or NULL (not formed); n_seg = ceil(T / segment_len).
 *   segment_len: a positive multiple of 64.
 *   workspace: >= gdn_workspace_size(B, T, H, K, V, B, 0, GDN_BF16, 0) bytes.
 */
gdn_status gdn_state_summary(const void *k, gdn_tensor_desc kd, const void *v,
                             gdn_tensor_desc vd, const float *g,
                             const float *gk, const float *beta,
                             float *state_ext, float *transition, int B, int T,
                             int H, int K, int V, int chunk, int segment_len,
                             int flags, void *workspace, size_t ws_bytes,
                             cudaStream_t stream);

/*
 * gdn_bwd_workspace_size / gdn_chunk_bwd -- gradients of one direction of
 * the chunked scan (gdn_chunk_fwd's bf16 path; fp32 below) for the loss
 * L = sum(dout . o) + sum(dh_final . h_final): the reverse-time chunked state
 * gradient of the hyper-parallel coverage_diff page
 * (`chunk_gated_delta_rule_bwd_dhu`, with its varlen offsets) and the
 * per-chunk input gradients of the WY form (`chunk_bwd_dqkwg`,
 * `prepare_wy_repr_bwd` on the same page; the per-step rules of the SANA
 * `fused_cam_gdn.py` page's `_cam_scan_bwd_kernel` at one token per frame).
 * The forward is recomputed first (its per-chunk operands and the state
 * entering every chunk are kept in the workspace). The value columns of the
 * state evolve independently given k, beta and g, so V > 128 runs as two
 * ranges of columns: dv and dh0 per range, dq, dk, dbeta and dg summed.
 *   q, k, v, g, beta, h0, cu_seqlens, n_seq, reverse, flags: as for
 *     gdn_chunk_fwd (bf16 q/k/v); flags: GDN_QK_L2NORM (the gradients are
 *     then with respect to the raw q and k). With gk (per-key gates, g
 *     NULL) dg is dL/dgk, (B, T, H, K): the chunk products that carry
 *     e^{G_i - G_j} per key are split about 16-row block middles, as in the
 *     forward, and dgk is 0 where the forward floors gk at -10.
 *   dout: (B, T, H, V) bf16 upstream gradient of o, descriptor dod.
 *   dden: (B, H, T) fp32 upstream gradient of den_out (the same scan over
 *     v = 1), or NULL when the loss does not involve den. With dden the state
 *     carries the ones column: h0, dh_final and dh0 are then (n_seq, H, K,
 *     V + 1), as for gdn_chunk_fwd with den_out.
 *   dh_final: (n_seq, H, K, V) fp32 upstream gradient of h_final, or NULL (0).
 *   dq, dk: (B, T, H, K); dv: (B, T, H, V); dbeta, dg: (B, T, H) (dg
 *     (B, T, H, K) with gk); dh0:
 *     (n_seq, H, K, V) or NULL -- fp32, contiguous, 8-byte aligned. dg is 0
 *     where g is below the -30 floor the forward applies.
 *   K <= 128 and V <= 256, both multiples of 8. reverse with h0, dh_final or
 *   dh0 -> GDN_ERR_UNSUPPORTED.
 *   workspace: >= gdn_bwd_workspace_size(B, T, H, K, V, n_seq, varlen,
 *   perkey, with_den) bytes (0 for an unsupported shape), 256-byte aligned.
 *
 * fp32 (qkd, vd and dod GDN_F32, the dtype of gdn_chunk_fwd's fp32 path):
 * the same arguments, loss and outputs, computed by the token recurrence in
 * reverse time in IEEE fp32 on CUDA cores. Per position, with P the decayed
 * state before it and r = v - P^T k the correction: dh += q do^T,
 * dq = h' do, dv = beta dh^T k, dbeta = r . (dh^T k), dk = beta dh r -
 * P dv, dg = sum((dh - k dv^T) . P), and the state gradient carries back as
 * e^{g} (dh - k dv^T) (the SANA `fused_cam_gdn.py` page's
 * `_cam_scan_bwd_kernel` rules). The state is checkpointed every 16
 * positions and each group of 16 recomputed before it is walked back. Any
 * K <= 128 and V <= 256; any non-negative strides; pointers 4-byte aligned;
 * gates floored at -30 as in the fp32 forward (g and gk: 0 gradient there).
 * A malformed cu_seqlens leaves that sequence's outputs unwritten and sets
 * GDN_DEVERR_SEQLENS in the word gdn_last_device_error() reads.
 *   workspace: >= gdn_bwd_f32_workspace_size(B, T, H, K, V, n_seq, varlen,
 *   perkey, with_den) bytes (0 for an unsupported shape), 256-byte aligned:
 *   checkpoints of (T / 16 + n_seq) x 2,048 floats per head and 16 state
 *   columns, and per-16-column partial sums of dq, dk (dgk), dbeta and dg.
 */
size_t gdn_bwd_workspace_size(int B, int T, int H, int K, int V, int n_seq,
                              int varlen, int perkey, int with_den);
size_t gdn_bwd_f32_workspace_size(int B, int T, int H, int K, int V, int n_seq,
                                  int varlen, int perkey, int with_den);
gdn_status gdn_chunk_bwd(const void *q, const void *k, gdn_tensor_desc qkd,
                         const void *v, gdn_tensor_desc vd, const float *g,
                         const float *gk, const float *beta, const float *h0,
                         const int32_t *cu_seqlens, int n_seq,
                         const void *dout, gdn_tensor_desc dod,
                         const float *dden, const float *dh_final,
                         float *dq, float *dk,
                         float *dv, float *dbeta, float *dg, float *dh0,
                         int B, int T, int H, int K, int V, int chunk,
                         int reverse, int flags, void *workspace,
                         size_t ws_bytes, cudaStream_t stream);

/*
 * gdn_frame_bwd_workspace_size / gdn_frame_bwd -- gradients of the
 * frame-causal rule of gdn_frame_fwd (SANA `fused_gdn.py` page,
 * `_fused_gdn_bwd_kernel`; SANA `fused_cam_gdn.py` page, `_cam_scan_bwd_kernel`)
 * for L = sum(dout . o) + sum(dden . den) + sum(dh_final . h_final), with
 * respect to q and k as gdn_frame_fwd takes them (prepared), v, beta,
 * g_frame and h0. The forward's per-frame matrices and states are
 * recomputed first; then, per direction, a reverse chain over the frames
 * forms the state gradient after every frame's write and the per-token
 * gradients follow from it in parallel.
 *   q, k, v, g_frame, beta, h0, frame, direction: as for gdn_frame_fwd
 *     (direction 2: both directions summed); h0 (B, H, K, V), or V + 1
 *     columns with dden, direction 0 only.
 *   dout: (B, T, H, V) bf16, descriptor dod. dden: (B, H, T) fp32 upstream
 *     gradient of den, or NULL (no denominator). dh_final: like h0, or NULL.
 *   dq, dk: (B, T, H, K); dv: (B, T, H, V); dbeta: (B, T, H); dg_frame:
 *     (B, T / frame, H); dh0: like h0, or NULL -- fp32, contiguous, 8-byte
 *     aligned. dg_frame is 0 where g_frame is below the -30 floor.
 *   K <= 128 and V (+1 with dden) <= 128; K and V multiples of 8. flags: 0.
 *   workspace: >= gdn_frame_bwd_workspace_size() bytes (0: unsupported
 *   shape), 256-byte aligned.
 */
size_t gdn_frame_bwd_workspace_size(int B, int T, int H, int K, int V, int frame,
                                    int with_den);
gdn_status gdn_frame_bwd(const void *q, const void *k, gdn_tensor_desc qkd,
                         const void *v, gdn_tensor_desc vd, const float *g_frame,
                         const float *beta, const float *h0, const void *dout,
                         gdn_tensor_desc dod, const float *dden,
                         const float *dh_final, float *dq, float *dk, float *dv,
                         float *dbeta, float *dg_frame, float *dh0, int B, int T,
                         int H, int K, int V, int frame, int direction, int flags,
                         void *workspace, size_t ws_bytes, cudaStream_t stream);

/* Human-readable name of a status code (static storage). */
/*
 * gdn_bidir_workspace_size / gdn_chunk_fwd_bidir -- both directions of the
 * bidirectional scan in one call (SANA `fused_gdn.py` page, `fused_bigdn_func`
 * forms num_fwd + num_bwd and den_fwd + den_bwd before any divide), with the
 * two directions running concurrently: the reverse scan is launched on a
 * second stream the library owns for the current device (forked from and
 * joined back to `stream` with events, so the call stays asynchronous and
 * capturable), writes its half into the workspace, and a last kernel on
 * `stream` adds it into out (and den_out). The result equals gdn_chunk_fwd
 * (reverse = 0) followed by gdn_chunk_fwd (reverse = 1, GDN_ACCUMULATE) up to
 * rounding.
 *   Arguments as gdn_chunk_fwd (no h0 / h_final, out overwritten); out has
 *   q's dtype. g_bwd / beta_bwd: the reverse direction's log gates and betas
 *   (the chunk-causal form's decay_bwd / beta_bwd), or NULL for g / beta;
 *   g_bwd only with a scalar gate. flags: GDN_QK_L2NORM.
 *   workspace: >= gdn_bidir_workspace_size() bytes, 256-byte aligned; the
 *   device error word of gdn_last_device_error() is the forward half's.
 * Calls on one device serialise their launches on a host lock (the side
 * stream and its events are shared).
 */
size_t gdn_bidir_workspace_size(int B, int T, int H, int K, int V, int n_seq,
                                int varlen, int dtype, int with_den);
gdn_status gdn_chunk_fwd_bidir(const void *q, const void *k, gdn_tensor_desc qkd,
                               const void *v, gdn_tensor_desc vd,
                               const float *g, const float *gk,
                               const float *beta, const float *g_bwd,
                               const float *beta_bwd,
                               const int32_t *cu_seqlens, int n_seq,
                               void *out, gdn_tensor_desc od, float *den_out,
                               int B, int T, int H, int K, int V, int chunk,
                               int flags, void *workspace, size_t ws_bytes,
                               cudaStream_t stream);

/*
 * gdn_merge -- the bidirectional merge (SANA `fused_gdn.py` page,
 * `fused_bigdn_func`: out = (num_fwd + num_bwd) / (den_fwd + den_bwd + eps),
 * and `_fused_bidi_merge_kernel` with APPLY_GATE: times silu(gate) =
 * gate / (1 + e^{-gate})). The scan has already summed both directions
 * (gdn_chunk_fwd with GDN_ACCUMULATE on the reverse call), so
 *   out = num / (den + eps) * (gate ? silu(gate) : 1)
 * elementwise, in fp32.
 *   num, gate, out: (B, T, H, V) with descriptors nd, gd, od. num is fp32 or
 *       bf16; gate (or NULL) has num's dtype; out is bf16, or fp32 when num
 *       is fp32 (GDN_ERR_DTYPE otherwise). out may alias num when the
 *       descriptors are equal.
 *   den: (B, H, T) fp32, contiguous.
 *   V a multiple of 8 (bf16 num) or 4 (fp32 num), at most 1024; B*T*H < 2^31;
 *   eps >= 0.
 * The chunk-causal variant of the page (state zeroed at chunk boundaries in
 * the backward direction only) needs nothing here: the reverse gdn_chunk_fwd
 * call takes its own gates, with a log-gate of -inf at each boundary token.
 */
gdn_status gdn_merge(const void *num, gdn_tensor_desc nd, const float *den,
                     const void *gate, gdn_tensor_desc gd, void *out,
                     gdn_tensor_desc od, int B, int T, int H, int V, float eps,
                     cudaStream_t stream);

/*
 * gdn_merge_bwd -- the gradient of gdn_merge for an upstream dout: with
 * r = 1 / (den + eps) and s = silu(gate) (or 1),
 *   dnum = dout s r,  dden = -sum_v dout num s r^2,
 *   dgate = dout num r silu'(gate),  silu'(x) = sig(x) (1 + x (1 - sig(x))).
 *   num, gate: as for gdn_merge (gate NULL: no dgate); den: (B, H, T) fp32;
 *   dout, dnum, dgate: (B, T, H, V) fp32 contiguous; dden: (B, H, T) fp32.
 *   V <= 1024; eps >= 0.
 */
gdn_status gdn_merge_bwd(const void *num, gdn_tensor_desc nd, const float *den,
                         const void *gate, gdn_tensor_desc gd, const float *dout,
                         float *dnum, float *dden, float *dgate, int B, int T,
                         int H, int V, float eps, cudaStream_t stream);

/*
 * gdn_frame_workspace_size / gdn_frame_fwd -- the frame-causal form of the
 * rule (SANA `fused_gdn.py` page, `_fused_gdn_kernel` with S tokens per frame;
 * SANA `fused_cam_gdn.py` page, `_cam_scan_kernel`): per (sequence, head),
 * frames of `frame` tokens and one log-decay per frame,
 *   S_pre = e^{g_f} S;  S <- S_pre + sum_{t in frame} k_t beta_t (v_t - S_pre^T k_t)^T
 *   o_t = S^T q_t for every token t of the frame (the post-frame state)
 * i.e. every token of a frame predicts from the same pre-frame state. With
 * direction 1 (reverse) frame f reads frames f+1 .. F-1 (each frame's decay
 * applied before its tokens); direction 2 sums both directions (the
 * bidirectional num, and den when den_out is given).
 *   q, k: (B, T, H, K) bf16 (prepared: gdn_prep); v: (B, T, H, V) bf16;
 *   g_frame: (B, T / frame, H) fp32 log decays (floored at -30);
 *   beta: (B, T, H) fp32; out: (B, T, H, V) bf16 or fp32; den_out: (B, H, T)
 *   fp32 or NULL; h0 / h_final: (B, H, K, V) fp32 (V + 1 columns with
 *   den_out, column V the z state, as for gdn_chunk_fwd), direction 0 only.
 *   frame a multiple of 64 dividing T; K <= 128, V <= 256, both multiples
 *   of 8. flags: GDN_ACCUMULATE adds into out / den_out.
 * Workspace: gdn_frame_workspace_size() bytes (with_den as for the call).
 */
size_t gdn_frame_workspace_size(int B, int T, int H, int K, int V, int frame,
                                int with_den);
gdn_status gdn_frame_fwd(const void *q, const void *k, gdn_tensor_desc qkd,
                         const void *v, gdn_tensor_desc vd, const float *g_frame,
                         const float *beta, const float *h0, void *out,
                         gdn_tensor_desc od, float *h_final, float *den_out,
                         int B, int T, int H, int K, int V, int frame,
                         int direction, int flags, void *workspace,
                         size_t ws_bytes, cudaStream_t stream);

const char *gdn_status_string(gdn_status s);

/*
 * gdn_last_device_error -- synchronise `stream`, read the device error word
 * that gdn_chunk_fwd keeps in `workspace`, store it in *word (GDN_DEVERR_*
 * bits, may be NULL) and clear it. Returns GDN_ERR_TIMEOUT if a bounded
 * wait gave up, GDN_ERR_DEVICE for other set bits, GDN_ERR_CUDA on a CUDA
 * failure, else GDN_OK. The word describes the last call that used this
 * workspace: every call clears it on its stream before its first kernel
 * (both directions of gdn_chunk_fwd_bidir report into the same word).
 */
gdn_status gdn_last_device_error(void *workspace, cudaStream_t stream,
                                 int *word);

/*
 * Launch accounting and per-kernel timing, for benchmarks.
 *   gdn_profile_enable(1) makes every later launch record a CUDA event pair
 *   on its own stream; gdn_profile_collect() synchronises those events and
 *   returns, per kernel kind (0 .. gdn_kernel_kinds()-1), the summed device
 *   milliseconds and launch counts, then clears them.
 *   gdn_launch_count() counts every kernel this library launched.
 */
int gdn_kernel_kinds(void);
const char *gdn_kernel_name(int kind);
void gdn_profile_enable(int on);
gdn_status gdn_profile_collect(float *ms, int *launches, int n);
long long gdn_launch_count(void);

/*
 * Value columns per CTA of the tensor-core state pass (the chunk-serial
 * recurrence of the chunked form, hyper-parallel coverage_diff page,
 * `chunk_gated_delta_rule_fwd_kernel_h_blockdim64`).
 *   bv = 0 (the default) chooses by the grid: 64-column CTAs, or 128-column
 *   CTAs (both 64-column tiles of a head in one CTA) for passes without
 *   summaries or snapshots whose 64-column grid has more CTAs than the GPU
 *   has SMs. bv = 64 or 128 forces one (128 only where the pass allows it);
 *   any other value means 0. Process-wide; affects later launches. Both
 *   compute the same recurrence (results agree to rounding order).
 */
void gdn_set_state_tile(int bv);

/*
 * Path of the bf16 forward with a scalar gate. on = 0 (the default) runs the
 * split path: an intra-chunk pass writing per-chunk operand images, then the
 * chunk-serial state pass. on = 1 runs each scan direction as one kernel in
 * which the intra-chunk WY factors are formed on the tensor cores (tcgen05,
 * TMA-loaded tiles) inside the state pass's CTAs and never leave the SM; it
 * falls back to the split path where it does not apply (per-key gates,
 * segment-parallel passes, summaries, gradient snapshots, layouts a TMA
 * tensor map cannot express). Both compute the same recurrence; results
 * agree to rounding order. On GB300 the fused kernel is correct but slower
 * than the split path (every value-tile CTA of a head repeats the head's
 * intra-chunk work, and that work per chunk exceeds the chain's step), so it
 * is not the default. Process-wide; affects later launches.
 */
void gdn_set_fused(int on);

/*
 * Testing aid for the device-side time-out path; the pages have no
 * counterpart. While set (cta >= 0), the block with linear index `cta` of
 * every later intra-chunk and state-pass launch of the bf16 path waits on a
 * barrier that nothing completes, gives up after about `limit_us`
 * microseconds, records GDN_DEVERR_TIMEOUT in the call's error word and
 * leaves without issuing any copy or tensor-core operation; every other
 * block works as usual (the call's results are then incomplete).
 * cta < 0 turns it off (the default). Process-wide; affects later launches.
 */
void gdn_set_stall_test(int cta, int limit_us);

#ifdef __cplusplus
}
#endif
#endif /* GDN_H_ */
