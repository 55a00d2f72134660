// gdn_api.cu -- the C ABI declared in include/gdn.h: host-side argument
// checks (everything is validated before the first launch), workspace
// layout, kernel dispatch and optional per-kernel CUDA-event timing.
#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/gdn.h"
#include "gdn_common.cuh"
#include "gdn_bwd_f32.cuh"
#include "gdn_frame_bwd.cuh"

namespace gdn {
cudaError_t launch_prep_bwd(const void *x, int64_t xsb, int64_t xst, int64_t xsh, const float *dy,
                            float *dx, int B, int T, int H, int D, int bf16, int mode, float scale,
                            float eps, cudaStream_t st);
cudaError_t launch_merge_bwd(const void *num, int64_t n_sb, int64_t n_st, int64_t n_sh, int bf16,
                             const float *den, const void *gate, int64_t g_sb, int64_t g_st, int64_t g_sh,
                             const float *dout, float *dnum, float *dden, float *dgate, int B, int T,
                             int H, int V, float eps, cudaStream_t st);
}

namespace {

using gdn::FwdParams;

// ------------------------------------------------------------ profiling ----

enum Kind {
    KPrepL2 = 0, KPrepRms, KTable, KIntra, KState, KFusedF32, KMerge, KFrameGram, KFrameChain,
    KFrameOut, KSegSummary, KSegCombine, KBwdDh, KBwdDq, KBwdDk, KSum, KF32Prep, KF32Serial, KFused,
    KFrameXt, KFrameLam, KFrameTok, KPrepBwd, KMergeBwd, KBwdF32Scan, KBwdF32Reduce, KNumKinds
};
const char *kKindNames[KNumKinds] = {"prep_l2",  "prep_rms", "chunk_table", "intra_bf16",
                                     "state_tc", "fused_f32", "merge",      "frame_gram",
                                     "frame_chain", "frame_out", "seg_summary", "seg_combine",
                                     "bwd_dh", "bwd_dq", "bwd_dk", "dir_sum", "f32_prep", "f32_serial",
                                     "fused_tc", "frame_xt", "frame_lam", "frame_tokgrad", "prep_bwd", "merge_bwd",
                                     "bwd_f32_scan", "bwd_f32_reduce"};

struct Profiler {
    std::mutex mu;
    bool on = false;
    std::vector<cudaEvent_t> pool;
    struct Rec {
        int kind;
        cudaEvent_t a, b;
    };
    std::vector<Rec> recs;
};
Profiler &prof() {
    static Profiler *p = new Profiler();  // never destroyed: safe at exit
    return *p;
}
std::atomic<long long> g_launches{0};
// the testing aid of gdn_set_stall_test (-1: off)
std::atomic<int> g_stall_cta{-1}, g_stall_us{1000};

cudaEvent_t take_event(Profiler &P) {
    if (!P.pool.empty()) {
        cudaEvent_t e = P.pool.back();
        P.pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

template <class F>
cudaError_t launch(int kind, cudaStream_t st, F &&f) {
    Profiler &P = prof();
    cudaEvent_t a = nullptr, b = nullptr;
    {
        std::lock_guard<std::mutex> g(P.mu);
        if (P.on) {
            a = take_event(P);
            b = take_event(P);
        }
    }
    if (a && b) cudaEventRecord(a, st);
    cudaError_t e = f();
    if (e == cudaSuccess) g_launches.fetch_add(1);
    if (a && b) {
        cudaEventRecord(b, st);
        std::lock_guard<std::mutex> g(P.mu);
        P.recs.push_back({kind, a, b});
    }
    return e;
}

// ------------------------------------------------------------- workspace ---

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Ws {
    size_t err, tab, seq0, w, qg, kg, pm, u, dec, total;
    int max_chunks, KP, Vt, n_vt;
};

bool ws_layout(int B, int T, int H, int K, int V, int n_seq, int varlen, int dtype,
               int with_den, Ws &L) {
    if (B < 1 || T < 0 || H < 1 || K < 1 || K > 128 || V < 1 || n_seq < 0) return false;
    if (varlen && (B != 1 || n_seq < 1)) return false;
    if (!varlen && n_seq != B) return false;
    if (dtype != GDN_F32 && dtype != GDN_BF16) return false;
    L.Vt = V + (with_den ? 1 : 0);
    if (L.Vt > 256) return false;
    L.KP = (dtype == GDN_BF16 || K > 64) ? 128 : 64;  // the bf16 path always pads keys to 128
    L.n_vt = (L.Vt + 63) / 64;
    const int64_t nts = ((int64_t)T + gdn::kChunk - 1) / gdn::kChunk;
    const int64_t mc = varlen ? nts + n_seq : (int64_t)B * nts;
    if (mc > (1 << 30)) return false;
    L.max_chunks = (int)mc;
    size_t off = 0;
    L.err = off;
    off += kAlign;
    L.tab = off;
    off = align_up(off + (varlen ? sizeof(int2) * (size_t)mc : 0));
    L.seq0 = off;
    off = align_up(off + (varlen ? sizeof(int) * (size_t)(n_seq + 1) : 0));
    L.w = L.qg = L.kg = L.pm = L.u = L.dec = off;
    if (dtype == GDN_F32 && gdn::f32_split(n_seq, H, L.Vt)) {  // fp32 images of the split path
        const size_t hmc = (size_t)H * (size_t)mc, f = sizeof(float);
        L.w = off;
        off = align_up(off + hmc * gdn::kChunk * L.KP * f);
        L.qg = off;
        off = align_up(off + hmc * gdn::kChunk * L.KP * f);
        L.kg = off;
        off = align_up(off + hmc * gdn::kChunk * L.KP * f);
        L.pm = off;
        off = align_up(off + hmc * gdn::kChunk * gdn::kChunk * f);
        L.u = off;
        off = align_up(off + hmc * gdn::kChunk * gdn::f32_vp32(L.Vt) * f);
        L.dec = off;
        off = align_up(off + hmc * L.KP * f);
    }
    if (dtype == GDN_BF16) {  // per-(head, chunk) operand images
        const size_t hmc = (size_t)H * (size_t)mc;
        L.w = off;
        off = align_up(off + hmc * gdn::kImgW);
        L.qg = off;
        off = align_up(off + hmc * gdn::kImgW);
        L.kg = off;
        off = align_up(off + hmc * gdn::kImgW);
        L.pm = off;
        off = align_up(off + hmc * gdn::kImgP);
        L.u = off;
        off = align_up(off + hmc * L.n_vt * gdn::kImgU);
        L.dec = off;
        off = align_up(off + hmc * gdn::kDecB);
    }
    L.total = off;
    return true;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
int elem_size(int dtype) { return dtype == GDN_BF16 ? 2 : 4; }
// strides must keep every row start 16-byte aligned
bool strides_ok(const gdn_tensor_desc &d) {
    const int64_t vec = 16 / elem_size(d.dtype);
    return d.stride_b % vec == 0 && d.stride_t % vec == 0 && d.stride_h % vec == 0 &&
           d.stride_b >= 0 && d.stride_t >= 0 && d.stride_h >= 0;
}
bool dtype_ok(int t) { return t == GDN_F32 || t == GDN_BF16; }

gdn_status cuda_status(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA; }

// The fp32 path: one fused kernel, or, for grids that would leave the GPU
// mostly idle, the chunk-parallel prep and the chunk-serial pass (the
// workspace holds their images exactly then, see ws_layout).
cudaError_t launch_f32(const gdn::FwdParams &p, int KP, int perkey, cudaStream_t s) {
    if (!gdn::f32_split(p.n_seq, p.H, p.Vt))
        return launch(KFusedF32, s, [&] { return gdn::launch_fused_f32(p, KP, perkey, s); });
    cudaError_t e = cudaSuccess;
    if (p.max_chunks > 0) e = launch(KF32Prep, s, [&] { return gdn::launch_f32_prep(p, KP, perkey, s); });
    if (e != cudaSuccess) return e;
    return launch(KF32Serial, s, [&] { return gdn::launch_f32_serial(p, KP, s); });
}

}  // namespace

extern "C" {

const char *gdn_status_string(gdn_status s) {
    switch (s) {
        case GDN_OK: return "ok";
        case GDN_ERR_NULL: return "a required pointer is NULL";
        case GDN_ERR_SHAPE: return "sizes out of range or inconsistent";
        case GDN_ERR_DTYPE: return "unsupported or mismatched element type";
        case GDN_ERR_LAYOUT: return "stride, alignment or contiguity not supported";
        case GDN_ERR_UNSUPPORTED: return "unsupported combination of arguments";
        case GDN_ERR_CUDA: return "a CUDA call failed";
        case GDN_ERR_TIMEOUT: return "a bounded device-side wait timed out";
        case GDN_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        case GDN_ERR_DEVICE: return "a device-side argument check failed";
    }
    return "unknown status";
}

size_t gdn_workspace_size(int B, int T, int H, int K, int V, int n_seq, int varlen, int dtype,
                          int with_den) {
    Ws L;
    if (!ws_layout(B, T, H, K, V, n_seq, varlen, dtype, with_den, L)) return 0;
    return L.total;
}

gdn_status gdn_prep(const void *x, gdn_tensor_desc xd, void *y, gdn_tensor_desc yd, int B,
                    int T, int H, int D, int mode, float scale, float eps, float *inv_rms,
                    cudaStream_t stream) {
    if (!x || !y) return GDN_ERR_NULL;
    if (B < 1 || T < 0 || H < 1 || D < 1) return GDN_ERR_SHAPE;
    if (!dtype_ok(xd.dtype) || xd.dtype != yd.dtype) return GDN_ERR_DTYPE;
    const int base = mode & 0xF;
    if ((mode & ~0x1F) != 0 || (base != GDN_PREP_L2 && base != GDN_PREP_RMS))
        return GDN_ERR_UNSUPPORTED;
    const int vec = 16 / elem_size(xd.dtype);
    if (D % vec != 0) return GDN_ERR_SHAPE;
    if (base == GDN_PREP_L2 && D > 256) return GDN_ERR_SHAPE;
    if (base == GDN_PREP_RMS && (int64_t)H * D > 16384) return GDN_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(y) || !strides_ok(xd) || !strides_ok(yd))
        return GDN_ERR_LAYOUT;
    if (inv_rms && (reinterpret_cast<uintptr_t>(inv_rms) & 3)) return GDN_ERR_LAYOUT;
    if (T == 0) return GDN_OK;
    const int kind = base == GDN_PREP_RMS ? KPrepRms : KPrepL2;
    return cuda_status(launch(kind, stream, [&] {
        return gdn::launch_prep(x, xd.stride_b, xd.stride_t, xd.stride_h, y, yd.stride_b,
                                yd.stride_t, yd.stride_h, B, T, H, D, xd.dtype == GDN_BF16, mode,
                                scale, eps, base == GDN_PREP_RMS ? inv_rms : nullptr, stream);
    }));
}

gdn_status gdn_prep_bwd(const void *x, gdn_tensor_desc xd, const float *dy, float *dx, int B,
                        int T, int H, int D, int mode, float scale, float eps,
                        cudaStream_t stream) {
    if (T > 0 && (!x || !dy || !dx)) return GDN_ERR_NULL;
    if (B < 1 || T < 0 || H < 1 || D < 1) return GDN_ERR_SHAPE;
    if (!dtype_ok(xd.dtype)) return GDN_ERR_DTYPE;
    const int base = mode & 0xF;
    if ((mode & ~0x1F) != 0 || (base != GDN_PREP_L2 && base != GDN_PREP_RMS))
        return GDN_ERR_UNSUPPORTED;
    if (D % (16 / elem_size(xd.dtype)) != 0) return GDN_ERR_SHAPE;
    if (base == GDN_PREP_L2 && D > 256) return GDN_ERR_SHAPE;
    if (base == GDN_PREP_RMS && (int64_t)H * D > 16384) return GDN_ERR_SHAPE;
    if (!aligned16(x) || !strides_ok(xd)) return GDN_ERR_LAYOUT;
    if ((reinterpret_cast<uintptr_t>(dy) & 3) || (reinterpret_cast<uintptr_t>(dx) & 3)) return GDN_ERR_LAYOUT;
    if (T == 0) return GDN_OK;
    return cuda_status(launch(KPrepBwd, stream, [&] {
        return gdn::launch_prep_bwd(x, xd.stride_b, xd.stride_t, xd.stride_h, dy, dx, B, T, H, D,
                                    xd.dtype == GDN_BF16, mode, scale, eps, stream);
    }));
}

}  // extern "C"

namespace {
// Argument checks and the launch parameter block shared by gdn_chunk_fwd,
// gdn_chunk_fwd_seg and gdn_state_summary; on GDN_OK, L and p describe the
// problem (workspace pointers are bound by bind_ws). With need_out unset the
// output may be NULL (summary passes write none).
gdn_status fwd_setup(const void *q, const void *k, gdn_tensor_desc qkd, const void *v,
                     gdn_tensor_desc vd, const float *g, const float *gk, const float *beta,
                     const float *h0, const int32_t *cu_seqlens, int n_seq, void *out,
                     gdn_tensor_desc od, float *h_final, float *den_out, int B, int T, int H,
                     int K, int V, int chunk, int reverse, int flags, bool need_out, Ws &L,
                     gdn::FwdParams &p) {
    // With no tokens the per-token tensors may be empty (NULL); only the
    // state pass-through h0 -> h_final runs.
    const bool empty = T == 0;
    if (!empty && (!q || !k || !v || !beta || (need_out && !out))) return GDN_ERR_NULL;
    if (g && gk) return GDN_ERR_UNSUPPORTED;
    if (!empty && !g && !gk) return GDN_ERR_NULL;
    if (chunk != gdn::kChunk) return GDN_ERR_SHAPE;
    if ((flags & ~(GDN_ACCUMULATE | GDN_QK_L2NORM)) != 0) return GDN_ERR_UNSUPPORTED;
    if (!dtype_ok(qkd.dtype) || !dtype_ok(vd.dtype) || !dtype_ok(od.dtype))
        return GDN_ERR_DTYPE;
    if (qkd.dtype != vd.dtype) return GDN_ERR_DTYPE;
    if (B < 1 || T < 0 || H < 1 || K < 1 || K > 128 || V < 1) return GDN_ERR_SHAPE;
    if (K % 8 != 0 || V % 8 != 0) return GDN_ERR_SHAPE;
    if (V + (den_out ? 1 : 0) > 256) return GDN_ERR_SHAPE;
    const int varlen = cu_seqlens != nullptr;
    if (varlen && (B != 1 || n_seq < 1)) return GDN_ERR_SHAPE;
    if (!varlen && n_seq != B) return GDN_ERR_SHAPE;
    if (reverse != 0 && reverse != 1) return GDN_ERR_SHAPE;
    if (reverse && (h0 || h_final)) return GDN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return GDN_ERR_LAYOUT;  // (NULL counts as aligned)
    if (!strides_ok(qkd) || !strides_ok(vd) || !strides_ok(od)) return GDN_ERR_LAYOUT;
    if (!aligned16(gk)) return GDN_ERR_LAYOUT;  // gk tiles are copied in 16-byte pieces
    for (const void *f : {(const void *)g, (const void *)gk, (const void *)beta,
                          (const void *)h0, (const void *)h_final, (const void *)den_out,
                          (const void *)cu_seqlens})
        if (f && (reinterpret_cast<uintptr_t>(f) & 3)) return GDN_ERR_LAYOUT;
    if (!ws_layout(B, T, H, K, V, n_seq, varlen, qkd.dtype, den_out != nullptr, L))
        return GDN_ERR_SHAPE;
    p = gdn::FwdParams{};
    p.q = q;
    p.k = k;
    p.v = v;
    p.qk_sb = qkd.stride_b;
    p.qk_st = qkd.stride_t;
    p.qk_sh = qkd.stride_h;
    p.v_sb = vd.stride_b;
    p.v_st = vd.stride_t;
    p.v_sh = vd.stride_h;
    p.g = g;
    p.gk = gk;
    p.beta = beta;
    p.h0 = h0;
    p.cu_seqlens = cu_seqlens;
    p.out = out;
    p.o_sb = od.stride_b;
    p.o_st = od.stride_t;
    p.o_sh = od.stride_h;
    p.out_f32 = od.dtype == GDN_F32;
    p.h_final = h_final;
    p.den = den_out;
    p.B = B;
    p.T = T;
    p.H = H;
    p.K = K;
    p.V = V;
    p.n_seq = n_seq;
    p.reverse = reverse;
    p.accumulate = (flags & GDN_ACCUMULATE) ? 1 : 0;
    p.l2norm = (flags & GDN_QK_L2NORM) ? 1 : 0;
    p.has_den = den_out != nullptr;
    p.Vt = L.Vt;
    p.h_ld = L.Vt;
    p.snap_ld = (L.Vt + 7) / 8 * 8;
    p.max_chunks = L.max_chunks;
    p.n_vt = L.n_vt;
    p.stall_cta = g_stall_cta.load();
    p.stall_us = g_stall_us.load();
    return GDN_OK;
}

// The device error word describes one call: it is cleared in stream order
// before the call's first kernel, so no kernel of the call clears it while
// another block may already have recorded an error.
cudaError_t clear_err(const gdn::FwdParams &p, cudaStream_t s) {
    return cudaMemsetAsync(p.err, 0, sizeof(int), s);
}

void bind_ws(unsigned char *ws, const Ws &L, gdn::FwdParams &p) {
    p.err = reinterpret_cast<int *>(ws + L.err);
    p.n_chunks = reinterpret_cast<int *>(ws + L.err) + 1;
    p.chunk_tab = reinterpret_cast<int2 *>(ws + L.tab);
    p.seq_chunk0 = reinterpret_cast<int *>(ws + L.seq0);
    p.w_img = ws + L.w;
    p.qg_img = ws + L.qg;
    p.kg_img = ws + L.kg;
    p.p_img = ws + L.pm;
    p.u_img = ws + L.u;
    p.dec = reinterpret_cast<float *>(ws + L.dec);
}

bool ws_ok(const void *workspace, size_t ws_bytes, size_t need) {
    return workspace && ws_bytes >= need && (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) == 0;
}

// segment-parallel sections after the forward workspace: the summaries and
// the state entering each segment, fp32
struct SegWs {
    size_t ext, tr, hin, total;
    int seg_chunks, n_seg;
};
bool seg_layout(const Ws &L, int B, int T, int H, int K, int segment_len, SegWs &S) {
    if (segment_len < gdn::kChunk || segment_len % gdn::kChunk != 0) return false;
    S.seg_chunks = segment_len / gdn::kChunk;
    const int nall = (T + gdn::kChunk - 1) / gdn::kChunk;
    S.n_seg = (nall + S.seg_chunks - 1) / S.seg_chunks;
    const size_t per = (size_t)S.n_seg * B * H * K * 4;
    size_t off = L.total;
    S.ext = off;
    off = align_up(off + per * L.Vt);
    S.tr = off;
    off = align_up(off + per * K);
    S.hin = off;
    off = align_up(off + per * L.Vt);
    S.total = off;
    return true;
}
}  // namespace

extern "C" {

gdn_status gdn_chunk_fwd(const void *q, const void *k, gdn_tensor_desc qkd, const void *v,
                         gdn_tensor_desc vd, const float *g, const float *gk, const float *beta,
                         const float *h0, const int32_t *cu_seqlens, int n_seq, void *out,
                         gdn_tensor_desc od, float *h_final, float *den_out, int B, int T,
                         int H, int K, int V, int chunk, int reverse, int flags,
                         void *workspace, size_t ws_bytes, cudaStream_t stream) {
    Ws L;
    gdn::FwdParams p;
    const gdn_status st = fwd_setup(q, k, qkd, v, vd, g, gk, beta, h0, cu_seqlens, n_seq, out, od,
                                    h_final, den_out, B, T, H, K, V, chunk, reverse, flags, true, L, p);
    if (st != GDN_OK) return st;
    if (!ws_ok(workspace, ws_bytes, L.total)) return GDN_ERR_WORKSPACE;
    bind_ws(static_cast<unsigned char *>(workspace), L, p);
    const int perkey = gk != nullptr;
    const int varlen = cu_seqlens != nullptr;

    cudaError_t e = clear_err(p, stream);
    if (e == cudaSuccess && varlen) e = launch(KTable, stream, [&] { return gdn::launch_chunk_table(p, stream); });
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    if (qkd.dtype == GDN_F32) {
        e = launch_f32(p, L.KP, perkey, stream);
        return cuda_status(e);
    }
    gdn::FusedMaps maps;
    if (gdn::fused_prepare(p, &maps))
        return cuda_status(launch(KFused, stream, [&] { return gdn::launch_fused_tc(p, maps, stream); }));
    if (L.max_chunks > 0) {
        e = launch(KIntra, stream, [&] { return gdn::launch_intra_bf16(p, perkey, stream); });
        if (e != cudaSuccess) return GDN_ERR_CUDA;
    }
    e = launch(KState, stream, [&] { return gdn::launch_state_tc(p, stream); });
    return cuda_status(e);
}

size_t gdn_seg_workspace_size(int B, int T, int H, int K, int V, int with_den, int segment_len) {
    Ws L;
    SegWs S;
    if (!ws_layout(B, T, H, K, V, B, 0, GDN_BF16, with_den, L)) return 0;
    if (!seg_layout(L, B, T, H, K, segment_len, S)) return 0;
    return S.total;
}

gdn_status gdn_chunk_fwd_seg(const void *q, const void *k, gdn_tensor_desc qkd, const void *v,
                             gdn_tensor_desc vd, const float *g, const float *gk,
                             const float *beta, const float *h0, void *out, gdn_tensor_desc od,
                             float *h_final, float *den_out, int B, int T, int H, int K, int V,
                             int chunk, int reverse, int flags, int segment_len, void *workspace,
                             size_t ws_bytes, cudaStream_t stream) {
    if (!workspace) return GDN_ERR_WORKSPACE;
    Ws L;
    gdn::FwdParams p;
    gdn_status st = fwd_setup(q, k, qkd, v, vd, g, gk, beta, h0, nullptr, B, out, od, h_final,
                              den_out, B, T, H, K, V, chunk, reverse, flags, true, L, p);
    if (st != GDN_OK) return st;
    if (qkd.dtype != GDN_BF16) return GDN_ERR_DTYPE;  // the fp32 path is one fused kernel
    SegWs S;
    if (!seg_layout(L, B, T, H, K, segment_len, S)) return GDN_ERR_SHAPE;
    if (!ws_ok(workspace, ws_bytes, S.total)) return GDN_ERR_WORKSPACE;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    bind_ws(ws, L, p);
    const int perkey = gk != nullptr;
    cudaError_t e = clear_err(p, stream);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    if (L.max_chunks > 0) {
        e = launch(KIntra, stream, [&] { return gdn::launch_intra_bf16(p, perkey, stream); });
        if (e != cudaSuccess) return GDN_ERR_CUDA;
    }
    if (S.n_seg <= 1) {  // one segment: the plain state pass
        e = launch(KState, stream, [&] { return gdn::launch_state_tc(p, stream); });
        return cuda_status(e);
    }
    p.seg_chunks = S.seg_chunks;
    p.sum_ext = reinterpret_cast<float *>(ws + S.ext);
    p.sum_tr = reinterpret_cast<float *>(ws + S.tr);
    p.n_kt = (K + 63) / 64;
    // 1. every segment's summary but the last one's, in parallel
    gdn::FwdParams ps = p;
    ps.summary = 2;
    e = launch(KSegSummary, stream, [&] { return gdn::launch_state_tc(ps, stream); });
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    // 2. the chain over segments
    gdn::SegParams c{};
    c.h0 = h0;
    c.sum_ext = p.sum_ext;
    c.sum_tr = p.sum_tr;
    c.h_in = reinterpret_cast<float *>(ws + S.hin);
    c.n_bh = B * H, c.K = K, c.V = V, c.Vt = L.Vt, c.n_seg = S.n_seg;
    e = launch(KSegCombine, stream, [&] { return gdn::launch_seg_combine(c, stream); });
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    // 3. every segment again from its entering state, with the outputs
    p.h_in = c.h_in;
    e = launch(KState, stream, [&] { return gdn::launch_state_tc(p, stream); });
    return cuda_status(e);
}

int gdn_seg_choose(int B, int T, int H, int K, int V, int with_den, int n_sm) {
    if (B < 1 || T < 1 || H < 1 || K < 1 || V < 1 || n_sm < 1) return 0;
    const int64_t nall = (T + gdn::kChunk - 1) / gdn::kChunk;
    const int64_t bh = (int64_t)B * H, n_vt = (V + (with_den ? 1 : 0) + 63) / 64, n_kt = (K + 63) / 64;
    // time in chunk steps of one state-kernel CTA (one CTA per SM): the
    // summary pass, the chain (about one step per segment) and the re-run
    auto cost = [&](int64_t n_seg, int64_t seg) {
        if (n_seg == 1) return ((bh * n_vt + n_sm - 1) / n_sm) * nall;
        return ((bh * (n_vt + n_kt) * (n_seg - 1) + n_sm - 1) / n_sm) * seg + n_seg +
               ((bh * n_vt * n_seg + n_sm - 1) / n_sm) * seg;
    };
    int64_t best_seg = nall, best = cost(1, nall);
    for (int64_t n = 2; n <= 256 && n <= nall; ++n) {
        const int64_t seg = (nall + n - 1) / n;
        const int64_t n_seg = (nall + seg - 1) / seg;
        const int64_t c = cost(n_seg, seg);
        if (c < best) best = c, best_seg = seg;
    }
    return (int)(best_seg * gdn::kChunk);
}

gdn_status gdn_state_summary(const void *k, gdn_tensor_desc kd, const void *v, gdn_tensor_desc vd,
                             const float *g, const float *gk, const float *beta, float *state_ext,
                             float *transition, int B, int T, int H, int K, int V, int chunk,
                             int segment_len, int flags, void *workspace, size_t ws_bytes,
                             cudaStream_t stream) {
    if (!workspace) return GDN_ERR_WORKSPACE;
    if (T > 0 && !state_ext) return GDN_ERR_NULL;
    if ((flags & ~GDN_QK_L2NORM) != 0) return GDN_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(state_ext) & 3) || (reinterpret_cast<uintptr_t>(transition) & 3))
        return GDN_ERR_LAYOUT;
    if (kd.dtype != GDN_BF16) return GDN_ERR_DTYPE;
    Ws L;
    gdn::FwdParams p;
    // the keys stand in for the queries: the summary reads no query
    gdn_status st = fwd_setup(k, k, kd, v, vd, g, gk, beta, nullptr, nullptr, B, nullptr,
                              gdn_tensor_desc{GDN_F32, 0, 0, 0, 0}, nullptr, nullptr, B, T, H, K,
                              V, chunk, 0, flags, false, L, p);
    if (st != GDN_OK) return st;
    SegWs S;
    if (!seg_layout(L, B, T, H, K, segment_len, S)) return GDN_ERR_SHAPE;
    if (!ws_ok(workspace, ws_bytes, L.total)) return GDN_ERR_WORKSPACE;
    if (T == 0) return GDN_OK;
    bind_ws(static_cast<unsigned char *>(workspace), L, p);
    cudaError_t e = clear_err(p, stream);
    if (e == cudaSuccess)
        e = launch(KIntra, stream, [&] { return gdn::launch_intra_bf16(p, gk != nullptr, stream); });
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    p.seg_chunks = S.seg_chunks;
    p.summary = 1;
    p.sum_ext = state_ext;
    p.sum_tr = transition;
    p.n_kt = transition ? (K + 63) / 64 : 0;
    e = launch(KSegSummary, stream, [&] { return gdn::launch_state_tc(p, stream); });
    return cuda_status(e);
}

}  // extern "C"

namespace {
// backward sections after the forward workspace: bf16 snapshots of the state
// entering each chunk, v_new, the state gradient at each chunk's end, dv_new
struct BwdWs {
    size_t h, vn, dh, dvn, dkp, dgp, total;
};
// after the forward's workspace L (of one value range of at most 128
// columns): the snapshots of that range, then bwd_dq's shares of dk and dG
bool bwd_layout(const Ws &L, int B, int T, int H, int K, int Vp, int perkey, BwdWs &S) {
    const size_t hc = (size_t)H * L.max_chunks;
    Vp = (Vp + 7) / 8 * 8;  // the snapshots' 16-byte rows
    size_t off = L.total;
    S.h = off;
    off = align_up(off + hc * K * Vp * 2);
    S.vn = off;
    off = align_up(off + hc * gdn::kChunk * Vp * 2);
    S.dh = off;
    off = align_up(off + hc * K * Vp * 2);
    S.dvn = off;
    off = align_up(off + hc * gdn::kChunk * Vp * 2);
    S.dkp = off;
    off = align_up(off + (size_t)B * T * H * K * 4);
    S.dgp = off;
    off = align_up(off + (size_t)B * T * H * (perkey ? K : 1) * 4);  // dG per key with gk
    S.total = off;
    return true;
}
}  // namespace

extern "C" {

}  // extern "C"

namespace {
// The value columns of a backward pass in ranges of at most 128 (the state
// columns evolve independently); with the denominator the last range also
// carries the ones column, so it keeps at most 120 value columns.
struct BwdRange {
    int off, w, den;
};
int bwd_ranges(int V, int den, BwdRange (&r)[4]) {
    int n = 0, off = 0, rem = V;
    const int cap_last = den ? 120 : 128;
    while (rem > cap_last && n < 3) {
        const int take = rem - 8 < 128 ? rem - 8 : 128;
        r[n++] = {off, take, 0};
        off += take, rem -= take;
    }
    r[n++] = {off, rem, den};
    return n;
}
size_t bwd_ws_total(int B, int T, int H, int K, int V, int n_seq, int varlen, int perkey, int den) {
    BwdRange r[4];
    const int n = bwd_ranges(V, den, r);
    size_t tot = 0;
    for (int i = 0; i < n; ++i) {
        Ws L;
        BwdWs S;
        if (!ws_layout(B, T, H, K, r[i].w, n_seq, varlen, GDN_BF16, r[i].den, L)) return 0;
        bwd_layout(L, B, T, H, K, r[i].w + r[i].den, perkey, S);
        if (S.total > tot) tot = S.total;
    }
    return tot;
}

// The fp32 backward's workspace: the error word, the state checkpoints (one
// per kF32BwdGroup positions, per head and 16-column range; a packed
// sequence s starts at slot c_s / 16 + s, which never overlaps the one
// before), and the per-range parts of dq^, dk^ (dgk) and of dbeta, dg.
struct F32BwdWs {
    size_t err, ck, pk, ps, total;
    int n_range;
    int64_t ck_groups;
};
bool f32_bwd_layout(int B, int T, int H, int K, int V, int n_seq, int varlen, int perkey, int den,
                    F32BwdWs &S) {
    if (B < 0 || T < 0 || H < 1 || K < 1 || K > gdn::kF32BwdKP || V < 1 || V > 256) return false;
    if (varlen ? (B != 1 || n_seq < 1) : n_seq != B) return false;
    const int Vs = V + (den ? 1 : 0);
    S.n_range = (Vs + gdn::kF32BwdCols - 1) / gdn::kF32BwdCols;
    S.ck_groups = varlen ? (int64_t)T / gdn::kF32BwdGroup + n_seq
                         : (int64_t)n_seq * ((T + gdn::kF32BwdGroup - 1) / gdn::kF32BwdGroup);
    const size_t rows = (size_t)B * T * H;
    size_t off = 0;
    S.err = off;
    off = align_up(off + 2 * sizeof(int));
    S.ck = off;
    off = align_up(off + (size_t)H * S.n_range * S.ck_groups * gdn::kF32BwdState * sizeof(float));
    S.pk = off;
    off = align_up(off + (size_t)S.n_range * rows * (perkey ? 3 : 2) * K * sizeof(float));
    S.ps = off;
    off = align_up(off + (size_t)S.n_range * rows * 2 * sizeof(float));
    S.total = off;
    return true;
}

// gdn_chunk_bwd for fp32 q, k, v and dout (the token recurrence in reverse
// time, gdn_bwd_f32.cu); the same arguments and checks as the bf16 path
gdn_status chunk_bwd_f32(const void *q, const void *k, gdn_tensor_desc qkd, const void *v,
                         gdn_tensor_desc vd, const float *g, const float *gk, const float *beta,
                         const float *h0, const int32_t *cu_seqlens, int n_seq, const void *dout,
                         gdn_tensor_desc dod, const float *dden, const float *dh_final, float *dq,
                         float *dk, float *dv, float *dbeta, float *dg, float *dh0, int B, int T,
                         int H, int K, int V, int chunk, int reverse, int flags, void *workspace,
                         size_t ws_bytes, cudaStream_t stream) {
    if (vd.dtype != GDN_F32 || (T > 0 && dod.dtype != GDN_F32)) return GDN_ERR_DTYPE;
    if ((flags & ~GDN_QK_L2NORM) != 0) return GDN_ERR_UNSUPPORTED;
    if (reverse && (h0 || dh_final || dh0)) return GDN_ERR_UNSUPPORTED;
    if (g && gk) return GDN_ERR_UNSUPPORTED;
    if (chunk != gdn::kChunk) return GDN_ERR_SHAPE;
    if (T > 0 && (!q || !k || !v || !beta || (!g && !gk))) return GDN_ERR_NULL;
    const int den = dden != nullptr;
    F32BwdWs S;
    if (!f32_bwd_layout(B, T, H, K, V, n_seq, cu_seqlens != nullptr, gk != nullptr, den, S))
        return GDN_ERR_SHAPE;
    for (const gdn_tensor_desc *d : {&qkd, &vd, &dod})
        if (d->stride_b < 0 || d->stride_t < 0 || d->stride_h < 0) return GDN_ERR_LAYOUT;
    for (const void *f : {q, k, v, dout, (const void *)g, (const void *)gk, (const void *)beta,
                          (const void *)h0, (const void *)dden, (const void *)dh_final, (const void *)dq,
                          (const void *)dk, (const void *)dv, (const void *)dbeta, (const void *)dg,
                          (const void *)dh0})
        if (f && (reinterpret_cast<uintptr_t>(f) & 3)) return GDN_ERR_LAYOUT;
    if (!ws_ok(workspace, ws_bytes, S.total)) return GDN_ERR_WORKSPACE;
    const int Vs = V + den;
    if (T == 0) {  // dL/dh0 = dL/dh_final
        if (!dh0) return GDN_OK;
        const size_t n = (size_t)n_seq * H * K * Vs * sizeof(float);
        cudaError_t e = dh_final ? cudaMemcpyAsync(dh0, dh_final, n, cudaMemcpyDeviceToDevice, stream)
                                 : cudaMemsetAsync(dh0, 0, n, stream);
        return cuda_status(e);
    }
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    gdn::F32BwdParams p{};
    p.q = static_cast<const float *>(q), p.k = static_cast<const float *>(k);
    p.v = static_cast<const float *>(v), p.dout = static_cast<const float *>(dout);
    p.qk_sb = qkd.stride_b, p.qk_st = qkd.stride_t, p.qk_sh = qkd.stride_h;
    p.v_sb = vd.stride_b, p.v_st = vd.stride_t, p.v_sh = vd.stride_h;
    p.do_sb = dod.stride_b, p.do_st = dod.stride_t, p.do_sh = dod.stride_h;
    p.beta = beta, p.g = g, p.gk = gk, p.h0 = h0, p.dh_final = dh_final, p.dden = dden;
    p.cu_seqlens = cu_seqlens;
    p.dv = dv, p.dh0 = dh0, p.dq = dq, p.dk = dk, p.dbeta = dbeta, p.dg = dg;
    p.err = reinterpret_cast<int *>(ws + S.err);
    p.ckpt = reinterpret_cast<float *>(ws + S.ck);
    p.part_k = reinterpret_cast<float *>(ws + S.pk);
    p.part_s = reinterpret_cast<float *>(ws + S.ps);
    p.B = B, p.T = T, p.H = H, p.K = K, p.V = V, p.Vs = Vs, p.n_seq = n_seq, p.n_range = S.n_range;
    p.reverse = reverse, p.l2norm = (flags & GDN_QK_L2NORM) != 0, p.ck_groups = S.ck_groups;
    cudaError_t e = cudaMemsetAsync(p.err, 0, sizeof(int), stream);
    if (e == cudaSuccess) e = launch(KBwdF32Scan, stream, [&] { return gdn::launch_bwd_f32_scan(p, stream); });
    if (e == cudaSuccess)
        e = launch(KBwdF32Reduce, stream, [&] { return gdn::launch_bwd_f32_reduce(p, stream); });
    return cuda_status(e);
}
}  // namespace

extern "C" {

size_t gdn_bwd_workspace_size(int B, int T, int H, int K, int V, int n_seq, int varlen,
                              int perkey, int with_den) {
    if (V < 1 || V > 256) return 0;
    return bwd_ws_total(B, T, H, K, V, n_seq, varlen, perkey != 0, with_den != 0);
}

size_t gdn_bwd_f32_workspace_size(int B, int T, int H, int K, int V, int n_seq, int varlen,
                                  int perkey, int with_den) {
    F32BwdWs S;
    if (!f32_bwd_layout(B, T, H, K, V, n_seq, varlen != 0, perkey != 0, with_den != 0, S)) return 0;
    return S.total;
}

gdn_status gdn_chunk_bwd(const void *q, const void *k, gdn_tensor_desc qkd, const void *v,
                         gdn_tensor_desc vd, const float *g, const float *gk, const float *beta,
                         const float *h0, const int32_t *cu_seqlens, int n_seq, const void *dout,
                         gdn_tensor_desc dod, const float *dden, const float *dh_final, float *dq,
                         float *dk, float *dv, float *dbeta, float *dg, float *dh0, int B, int T,
                         int H, int K, int V, int chunk, int reverse, int flags, void *workspace,
                         size_t ws_bytes, cudaStream_t stream) {
    if (T > 0 && (!dout || !dq || !dk || !dv || !dbeta || !dg)) return GDN_ERR_NULL;
    if (qkd.dtype == GDN_F32)
        return chunk_bwd_f32(q, k, qkd, v, vd, g, gk, beta, h0, cu_seqlens, n_seq, dout, dod, dden,
                             dh_final, dq, dk, dv, dbeta, dg, dh0, B, T, H, K, V, chunk, reverse, flags,
                             workspace, ws_bytes, stream);
    if (qkd.dtype != GDN_BF16 || vd.dtype != GDN_BF16 || (T > 0 && dod.dtype != GDN_BF16))
        return GDN_ERR_DTYPE;
    if ((flags & ~GDN_QK_L2NORM) != 0) return GDN_ERR_UNSUPPORTED;
    if (reverse && (h0 || dh_final || dh0)) return GDN_ERR_UNSUPPORTED;
    if (V < 1 || V > 256 || V % 8 != 0) return GDN_ERR_SHAPE;
    if (!aligned16(dout) || !strides_ok(dod)) return GDN_ERR_LAYOUT;
    for (const void *f : {(const void *)dq, (const void *)dk, (const void *)dv, (const void *)dbeta,
                          (const void *)dg, (const void *)dh0, (const void *)dh_final})
        if (f && (reinterpret_cast<uintptr_t>(f) & 7)) return GDN_ERR_LAYOUT;
    if (dden && (reinterpret_cast<uintptr_t>(dden) & 3)) return GDN_ERR_LAYOUT;
    const int den = dden != nullptr;
    const int Vs = V + den;  // columns of h0, h_final, dh0, dh_final
    // The value columns of the state evolve independently given k, beta and
    // g, so the gradient is formed over ranges of at most 128 columns: dv
    // and dh0 per range, dq, dk, dbeta and dg summed over the ranges.
    BwdRange rg[4];
    const int nrg = bwd_ranges(V, den, rg);
    Ws L;
    gdn::FwdParams p;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    // the forward recompute of a range: no outputs, the snapshots instead (a
    // range with the ones column is run as with a denominator, which it then
    // never writes)
    auto setup = [&](const BwdRange &r) {
        return fwd_setup(q, k, qkd, static_cast<const __nv_bfloat16 *>(v) + r.off, vd, g, gk, beta,
                         h0 ? h0 + r.off : nullptr, cu_seqlens, n_seq, nullptr,
                         gdn_tensor_desc{GDN_BF16, 0, 0, 0, 0}, nullptr,
                         r.den ? reinterpret_cast<float *>(ws ? ws : reinterpret_cast<unsigned char *>(16))
                               : nullptr,
                         B, T, H, K, r.w, chunk, reverse, flags, false, L, p);
    };
    gdn_status st = setup(rg[0]);
    if (st != GDN_OK) return st;
    const int perkey = gk != nullptr;
    const size_t need = bwd_ws_total(B, T, H, K, V, n_seq, cu_seqlens != nullptr, perkey, den);
    if (need == 0) return GDN_ERR_SHAPE;
    if (!ws_ok(workspace, ws_bytes, need)) return GDN_ERR_WORKSPACE;
    if (T == 0) {  // dL/dh0 = dL/dh_final
        if (!dh0) return GDN_OK;
        const size_t n = (size_t)n_seq * H * K * Vs * sizeof(float);
        cudaError_t e = dh_final ? cudaMemcpyAsync(dh0, dh_final, n, cudaMemcpyDeviceToDevice, stream)
                                 : cudaMemsetAsync(dh0, 0, n, stream);
        return cuda_status(e);
    }
    cudaError_t e = cudaSuccess;
    for (int ri = 0; ri < nrg && e == cudaSuccess; ++ri) {
        const BwdRange &r = rg[ri];
        if (ri > 0) {  // the same checks passed for the first range
            st = setup(r);
            if (st != GDN_OK) return st;
        }
        BwdWs S;
        bwd_layout(L, B, T, H, K, r.w + r.den, perkey, S);
        p.h_ld = Vs;  // h0 rows keep all the state's columns
        bind_ws(ws, L, p);
        p.h_snap = reinterpret_cast<__nv_bfloat16 *>(ws + S.h);
        p.vn_snap = reinterpret_cast<__nv_bfloat16 *>(ws + S.vn);
        if (ri == 0) e = clear_err(p, stream);
        if (e == cudaSuccess && cu_seqlens)
            e = launch(KTable, stream, [&] { return gdn::launch_chunk_table(p, stream); });
        if (e == cudaSuccess) e = launch(KIntra, stream, [&] { return gdn::launch_intra_bf16(p, perkey, stream); });
        if (e == cudaSuccess) e = launch(KState, stream, [&] { return gdn::launch_state_tc(p, stream); });
        if (e != cudaSuccess) return GDN_ERR_CUDA;
        gdn::BwdParams b{};
        b.q = q, b.k = k, b.v = static_cast<const __nv_bfloat16 *>(v) + r.off;
        b.dout = static_cast<const __nv_bfloat16 *>(dout) + r.off;
        b.qk_sb = qkd.stride_b, b.qk_st = qkd.stride_t, b.qk_sh = qkd.stride_h;
        b.v_sb = vd.stride_b, b.v_st = vd.stride_t, b.v_sh = vd.stride_h;
        b.do_sb = dod.stride_b, b.do_st = dod.stride_t, b.do_sh = dod.stride_h;
        b.g = g, b.gk = gk, b.beta = beta, b.dh_final = dh_final ? dh_final + r.off : nullptr;
        b.dq = dq, b.dk = dk, b.dv = dv + r.off, b.dbeta = dbeta, b.dg = dg;
        b.dh0 = dh0 ? dh0 + r.off : nullptr;
        b.B = B, b.T = T, b.H = H, b.K = K, b.V = r.w + r.den, b.reverse = reverse, b.l2norm = p.l2norm;
        b.max_chunks = L.max_chunks;
        b.cu_seqlens = cu_seqlens, b.n_seq = n_seq;
        b.n_chunks = p.n_chunks, b.chunk_tab = p.chunk_tab, b.seq_chunk0 = p.seq_chunk0;
        b.vfull = Vs, b.v_off = r.off, b.dv_ld = V, b.acc = ri > 0;
        b.dden = dden, b.den_col = r.den ? r.w : -1;
        b.snap_ld = (r.w + r.den + 7) / 8 * 8;
        b.dk_part = reinterpret_cast<float *>(ws + S.dkp);
        b.dg_part = reinterpret_cast<float *>(ws + S.dgp);
        b.w_img = p.w_img, b.qg_img = p.qg_img, b.kg_img = p.kg_img, b.p_img = p.p_img, b.dec = p.dec;
        b.h_snap = p.h_snap, b.vn_snap = p.vn_snap;
        b.dh_snap = reinterpret_cast<__nv_bfloat16 *>(ws + S.dh);
        b.dvn_snap = reinterpret_cast<__nv_bfloat16 *>(ws + S.dvn);
        b.err = p.err;
        e = launch(KBwdDh, stream, [&] { return gdn::launch_bwd_dh(b, stream); });
        if (e == cudaSuccess)
            e = launch(KBwdDq, stream, [&] { return perkey ? gdn::launch_bwd_dq_gk(b, stream) : gdn::launch_bwd_dq(b, stream); });
        if (e == cudaSuccess)
            e = launch(KBwdDk, stream, [&] { return perkey ? gdn::launch_bwd_dk_gk(b, stream) : gdn::launch_bwd_dk(b, stream); });
    }
    return cuda_status(e);
}

}  // extern "C"

namespace {
// A library-owned second stream per device (and the events that fork it
// from, and join it back to, the caller's stream), for the reverse direction
// of a concurrent bidirectional scan. Created on first use, never destroyed.
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr, mid_main = nullptr, mid_side = nullptr;
};
std::mutex &side_mutex() {
    static std::mutex *m = new std::mutex();
    return *m;
}
cudaError_t side_stream(SideStream *&out) {
    static SideStream *per_dev = new SideStream[64];
    int d = 0;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess) return e;
    if (d < 0 || d >= 64) return cudaErrorInvalidDevice;
    SideStream &x = per_dev[d];
    if (!x.s) {
        if ((e = cudaStreamCreateWithFlags(&x.s, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&x.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&x.join, cudaEventDisableTiming)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&x.mid_main, cudaEventDisableTiming)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&x.mid_side, cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    out = &x;
    return cudaSuccess;
}

struct BidirWs {
    size_t fwd, rev, out2, den2, total;
};
bool bidir_layout(const Ws &L, int B, int T, int H, int V, int dtype, int with_den, BidirWs &S) {
    S.fwd = 0;
    S.rev = align_up(L.total);
    size_t off = S.rev + align_up(L.total);
    S.out2 = off;
    off = align_up(off + (size_t)B * T * H * V * (dtype == GDN_BF16 ? 2 : 4));
    S.den2 = off;
    off = align_up(off + (with_den ? (size_t)B * H * T * 4 : 0));
    S.total = off;
    return true;
}
}  // namespace

extern "C" {

size_t gdn_bidir_workspace_size(int B, int T, int H, int K, int V, int n_seq, int varlen, int dtype,
                                int with_den) {
    Ws L;
    BidirWs S;
    if (!ws_layout(B, T, H, K, V, n_seq, varlen, dtype, with_den, L)) return 0;
    bidir_layout(L, B, T, H, V, dtype, with_den, S);
    return S.total;
}

gdn_status gdn_chunk_fwd_bidir(const void *q, const void *k, gdn_tensor_desc qkd, const void *v,
                               gdn_tensor_desc vd, const float *g, const float *gk,
                               const float *beta, const float *g_bwd, const float *beta_bwd,
                               const int32_t *cu_seqlens, int n_seq, void *out, gdn_tensor_desc od,
                               float *den_out, int B, int T, int H, int K, int V, int chunk,
                               int flags, void *workspace, size_t ws_bytes, cudaStream_t stream) {
    if ((flags & ~GDN_QK_L2NORM) != 0) return GDN_ERR_UNSUPPORTED;
    if (g_bwd && !g) return GDN_ERR_UNSUPPORTED;  // backward gates replace a scalar gate only
    if (od.dtype != qkd.dtype) return GDN_ERR_DTYPE;  // the reverse half is staged in out's dtype
    for (const void *f : {(const void *)g_bwd, (const void *)beta_bwd})
        if (f && (reinterpret_cast<uintptr_t>(f) & 3)) return GDN_ERR_LAYOUT;
    Ws L;
    gdn::FwdParams pf, pr;
    gdn_status st = fwd_setup(q, k, qkd, v, vd, g, gk, beta, nullptr, cu_seqlens, n_seq, out, od,
                              nullptr, den_out, B, T, H, K, V, chunk, 0, flags, true, L, pf);
    if (st != GDN_OK) return st;
    BidirWs S;
    bidir_layout(L, B, T, H, V, qkd.dtype, den_out != nullptr, S);
    if (!ws_ok(workspace, ws_bytes, S.total)) return GDN_ERR_WORKSPACE;
    if (T == 0) return GDN_OK;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    // the reverse direction writes its own contiguous output, summed in after
    gdn_tensor_desc od2{};
    od2.dtype = od.dtype;
    od2.stride_b = (int64_t)T * H * V;
    od2.stride_t = (int64_t)H * V;
    od2.stride_h = V;
    float *den2 = den_out ? reinterpret_cast<float *>(ws + S.den2) : nullptr;
    st = fwd_setup(q, k, qkd, v, vd, g_bwd ? g_bwd : g, gk, beta_bwd ? beta_bwd : beta, nullptr,
                   cu_seqlens, n_seq, ws + S.out2, od2, nullptr, den2, B, T, H, K, V, chunk, 1, flags,
                   true, L, pr);
    if (st != GDN_OK) return st;
    bind_ws(ws + S.fwd, L, pf);
    bind_ws(ws + S.rev, L, pr);
    pr.err = pf.err;  // both directions report into the word at the workspace start
    const int perkey = gk != nullptr, varlen = cu_seqlens != nullptr;

    std::lock_guard<std::mutex> lock(side_mutex());
    SideStream *side = nullptr;
    if (side_stream(side) != cudaSuccess) return GDN_ERR_CUDA;
    // one kernel per direction where the fused path applies, else the split
    // intra-chunk and state passes
    gdn::FusedMaps mf, mr;
    const bool fused = qkd.dtype == GDN_BF16 && gdn::fused_prepare(pf, &mf) && gdn::fused_prepare(pr, &mr);
    // everything of a direction up to its state pass
    auto first = [&](gdn::FwdParams &p, cudaStream_t s) -> cudaError_t {
        cudaError_t e = cudaSuccess;
        if (varlen) e = launch(KTable, s, [&] { return gdn::launch_chunk_table(p, s); });
        if (e != cudaSuccess) return e;
        if (qkd.dtype == GDN_F32)
            return launch_f32(p, L.KP, perkey, s);
        if (!fused && L.max_chunks > 0)
            e = launch(KIntra, s, [&] { return gdn::launch_intra_bf16(p, perkey, s); });
        return e;
    };
    auto second = [&](gdn::FwdParams &p, cudaStream_t s) -> cudaError_t {
        if (qkd.dtype == GDN_F32) return cudaSuccess;
        if (fused) {
            const gdn::FusedMaps &m = &p == &pf ? mf : mr;
            return launch(KFused, s, [&] { return gdn::launch_fused_tc(p, m, s); });
        }
        return launch(KState, s, [&] { return gdn::launch_state_tc(p, s); });
    };
    // fork: the reverse direction on the side stream, the forward on the
    // caller's. Each state pass waits for both directions' intra passes, so
    // the two intra passes share the whole GPU and the two state passes (one
    // CTA per SM each) then start together, instead of one direction's state
    // CTAs taking SMs from the other's intra pass.
    cudaError_t e = clear_err(pf, stream);
    if (e == cudaSuccess) e = cudaEventRecord(side->fork, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side->s, side->fork, 0);
    if (e == cudaSuccess) e = first(pr, side->s);
    if (e == cudaSuccess) e = first(pf, stream);
    if (e == cudaSuccess && qkd.dtype != GDN_F32) {
        e = cudaEventRecord(side->mid_side, side->s);
        if (e == cudaSuccess) e = cudaEventRecord(side->mid_main, stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, side->mid_side, 0);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(side->s, side->mid_main, 0);
    }
    if (e == cudaSuccess) e = second(pr, side->s);
    if (e == cudaSuccess) e = second(pf, stream);
    // join, then out += the reverse half, den += its denominator
    if (e == cudaSuccess) e = cudaEventRecord(side->join, side->s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, side->join, 0);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    gdn::SumParams a{};
    a.out = out, a.o_sb = od.stride_b, a.o_st = od.stride_t, a.o_sh = od.stride_h;
    a.add = ws + S.out2;
    a.den = den_out, a.den_add = den2;
    a.B = B, a.T = T, a.H = H, a.V = V, a.bf16 = od.dtype == GDN_BF16;
    return cuda_status(launch(KSum, stream, [&] { return gdn::launch_sum(a, stream); }));
}

gdn_status gdn_merge(const void *num, gdn_tensor_desc nd, const float *den, const void *gate,
                     gdn_tensor_desc gd, void *out, gdn_tensor_desc od, int B, int T, int H, int V,
                     float eps, cudaStream_t stream) {
    if (B < 1 || T < 0 || H < 1 || V < 1) return GDN_ERR_SHAPE;
    if (T > 0 && (!num || !den || !out)) return GDN_ERR_NULL;
    if (!dtype_ok(nd.dtype) || !dtype_ok(od.dtype)) return GDN_ERR_DTYPE;
    if (nd.dtype == GDN_BF16 && od.dtype != GDN_BF16) return GDN_ERR_DTYPE;
    if (gate && gd.dtype != nd.dtype) return GDN_ERR_DTYPE;
    if (V % (16 / elem_size(nd.dtype)) != 0 || V > 1024) return GDN_ERR_SHAPE;
    if ((int64_t)B * T * H > INT32_MAX) return GDN_ERR_SHAPE;
    if (!aligned16(num) || !aligned16(out) || !aligned16(gate) || !strides_ok(nd) || !strides_ok(od) ||
        (gate && !strides_ok(gd)))
        return GDN_ERR_LAYOUT;
    if (den && (reinterpret_cast<uintptr_t>(den) & 3)) return GDN_ERR_LAYOUT;
    if (!(eps >= 0.f)) return GDN_ERR_SHAPE;
    if (T == 0) return GDN_OK;
    gdn::MergeParams m{};
    m.num = num;
    m.n_sb = nd.stride_b, m.n_st = nd.stride_t, m.n_sh = nd.stride_h;
    m.den = den;
    m.gate = gate;
    m.g_sb = gd.stride_b, m.g_st = gd.stride_t, m.g_sh = gd.stride_h;
    m.out = out;
    m.o_sb = od.stride_b, m.o_st = od.stride_t, m.o_sh = od.stride_h;
    m.B = B, m.T = T, m.H = H, m.V = V;
    m.eps = eps;
    m.num_bf16 = nd.dtype == GDN_BF16;
    m.out_bf16 = od.dtype == GDN_BF16;
    return cuda_status(launch(KMerge, stream, [&] { return gdn::launch_merge(m, stream); }));
}

gdn_status gdn_merge_bwd(const void *num, gdn_tensor_desc nd, const float *den, const void *gate,
                         gdn_tensor_desc gd, const float *dout, float *dnum, float *dden,
                         float *dgate, int B, int T, int H, int V, float eps,
                         cudaStream_t stream) {
    if (B < 1 || T < 0 || H < 1 || V < 1 || V > 1024) return GDN_ERR_SHAPE;
    if (T > 0 && (!num || !den || !dout || !dnum || !dden)) return GDN_ERR_NULL;
    if (!dtype_ok(nd.dtype) || (gate && gd.dtype != nd.dtype)) return GDN_ERR_DTYPE;
    if (!(eps >= 0.f)) return GDN_ERR_SHAPE;
    if (gate && !dgate) return GDN_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(num) % elem_size(nd.dtype) ||
        (gate && reinterpret_cast<uintptr_t>(gate) % elem_size(gd.dtype)))
        return GDN_ERR_LAYOUT;
    for (const void *f : {(const void *)den, (const void *)dout, (const void *)dnum, (const void *)dden,
                          (const void *)dgate})
        if (f && (reinterpret_cast<uintptr_t>(f) & 3)) return GDN_ERR_LAYOUT;
    if (T == 0) return GDN_OK;
    return cuda_status(launch(KMergeBwd, stream, [&] {
        return gdn::launch_merge_bwd(num, nd.stride_b, nd.stride_t, nd.stride_h, nd.dtype == GDN_BF16, den,
                                     gate, gd.stride_b, gd.stride_t, gd.stride_h, dout, dnum, dden,
                                     gate ? dgate : nullptr, B, T, H, V, eps, stream);
    }));
}

namespace {
// frame-causal workspace: A_f, B_f and the read states, fp32, 256-byte sections
struct FrameWs {
    size_t amat, bmat, sout, total;
};
bool frame_ws(int B, int T, int H, int K, int V, int frame, int with_den, FrameWs &L) {
    if (B < 1 || T < 0 || H < 1 || K < 1 || K > 128 || V < 1 || V > 256 || frame < gdn::kChunk ||
        frame % gdn::kChunk != 0 || T % frame != 0)
        return false;
    const size_t F = (size_t)(T / frame), bh = (size_t)B * H, Vt = (size_t)V + (with_den ? 1 : 0);
    size_t off = 0;
    L.amat = off;
    off = align_up(off + bh * F * K * K * 4);
    L.bmat = off;
    off = align_up(off + bh * F * K * Vt * 4);
    L.sout = off;
    off = align_up(off + bh * F * K * ((Vt + 7) / 8 * 8) * 4);
    L.total = off > 0 ? off : kAlign;
    return true;
}
}  // namespace

size_t gdn_frame_workspace_size(int B, int T, int H, int K, int V, int frame, int with_den) {
    FrameWs L;
    return frame_ws(B, T, H, K, V, frame, with_den, L) ? L.total : 0;
}

gdn_status gdn_frame_fwd(const void *q, const void *k, gdn_tensor_desc qkd, const void *v,
                         gdn_tensor_desc vd, const float *g_frame, const float *beta,
                         const float *h0, void *out, gdn_tensor_desc od, float *h_final,
                         float *den_out, int B, int T, int H, int K, int V, int frame,
                         int direction, int flags, void *workspace, size_t ws_bytes,
                         cudaStream_t stream) {
    if (B < 1 || T < 0 || H < 1 || K < 1 || V < 1) return GDN_ERR_SHAPE;
    if (direction < 0 || direction > 2) return GDN_ERR_UNSUPPORTED;
    if ((flags & ~GDN_ACCUMULATE) != 0) return GDN_ERR_UNSUPPORTED;
    if ((h0 || h_final) && direction != 0) return GDN_ERR_UNSUPPORTED;
    if (T > 0 && (!q || !k || !v || !g_frame || !beta || !out)) return GDN_ERR_NULL;
    if (qkd.dtype != GDN_BF16 || vd.dtype != GDN_BF16) return GDN_ERR_DTYPE;
    if (!dtype_ok(od.dtype)) return GDN_ERR_DTYPE;
    if (K % 8 != 0 || V % 8 != 0 || K > 128 || V > 256) return GDN_ERR_SHAPE;
    if (frame < gdn::kChunk || frame % gdn::kChunk != 0 || T % frame != 0) return GDN_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !strides_ok(qkd) ||
        !strides_ok(vd) || !strides_ok(od))
        return GDN_ERR_LAYOUT;
    FrameWs L;
    if (!frame_ws(B, T, H, K, V, frame, den_out != nullptr, L)) return GDN_ERR_SHAPE;
    if (!workspace || ws_bytes < L.total || !aligned16(workspace)) return GDN_ERR_WORKSPACE;
    if (T == 0) return GDN_OK;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    gdn::FrameParams p{};
    p.q = q, p.k = k, p.v = v;
    p.qk_sb = qkd.stride_b, p.qk_st = qkd.stride_t, p.qk_sh = qkd.stride_h;
    p.v_sb = vd.stride_b, p.v_st = vd.stride_t, p.v_sh = vd.stride_h;
    p.beta = beta, p.g_frame = g_frame, p.h0 = h0, p.h_final = h_final;
    p.out = out, p.o_sb = od.stride_b, p.o_st = od.stride_t, p.o_sh = od.stride_h;
    p.out_f32 = od.dtype == GDN_F32;
    p.den = den_out;
    p.B = B, p.T = T, p.H = H, p.K = K, p.V = V, p.Vt = V + (den_out ? 1 : 0);
    p.Vs = (p.Vt + 7) / 8 * 8;
    p.F = T / frame, p.frame = frame;
    p.has_den = den_out != nullptr;
    p.accumulate = (flags & GDN_ACCUMULATE) != 0;
    p.direction = direction;
    p.amat = reinterpret_cast<float *>(ws + L.amat);
    p.bmat = reinterpret_cast<float *>(ws + L.bmat);
    p.sout = reinterpret_cast<float *>(ws + L.sout);
    cudaError_t e = launch(KFrameGram, stream, [&] { return gdn::launch_frame_gram(p, stream); });
    if (e == cudaSuccess) e = launch(KFrameChain, stream, [&] { return gdn::launch_frame_chain(p, stream); });
    if (e == cudaSuccess) e = launch(KFrameOut, stream, [&] { return gdn::launch_frame_out(p, stream); });
    return cuda_status(e);
}

namespace {
struct FrameBwdWs {
    FrameWs fwd;  // A_f, B_f and direction 0's read states
    size_t sread1, cmat, lam, dgp, total;
};
bool frame_bwd_ws(int B, int T, int H, int K, int V, int frame, int with_den, FrameBwdWs &L) {
    if (!frame_ws(B, T, H, K, V, frame, with_den, L.fwd)) return false;
    const size_t F = (size_t)(T / frame), bh = (size_t)B * H, Vt = (size_t)V + (with_den ? 1 : 0);
    const size_t Vs = (Vt + 7) / 8 * 8, st = bh * F * K * Vs * 4;
    size_t off = align_up(L.fwd.total);
    L.sread1 = off;
    off = align_up(off + st);
    L.cmat = off;
    off = align_up(off + st);
    L.lam = off;
    off = align_up(off + st);
    L.dgp = off;
    off = align_up(off + bh * F * ((Vt + gdn::kFrameBwdCT - 1) / gdn::kFrameBwdCT) * 4);
    L.total = off;
    return true;
}
}  // namespace

size_t gdn_frame_bwd_workspace_size(int B, int T, int H, int K, int V, int frame, int with_den) {
    FrameBwdWs L;
    if (V + (with_den ? 1 : 0) > 128) return 0;
    return frame_bwd_ws(B, T, H, K, V, frame, with_den, L) ? L.total : 0;
}

gdn_status gdn_frame_bwd(const void *q, const void *k, gdn_tensor_desc qkd, const void *v,
                         gdn_tensor_desc vd, const float *g_frame, const float *beta, const float *h0,
                         const void *dout, gdn_tensor_desc dod, const float *dden,
                         const float *dh_final, float *dq, float *dk, float *dv, float *dbeta,
                         float *dg_frame, float *dh0, int B, int T, int H, int K, int V, int frame,
                         int direction, int flags, void *workspace, size_t ws_bytes,
                         cudaStream_t stream) {
    if (B < 1 || T < 0 || H < 1 || K < 1 || V < 1) return GDN_ERR_SHAPE;
    if (direction < 0 || direction > 2 || flags != 0) return GDN_ERR_UNSUPPORTED;
    if ((h0 || dh_final || dh0) && direction != 0) return GDN_ERR_UNSUPPORTED;
    if (T > 0 && (!q || !k || !v || !g_frame || !beta || !dout || !dq || !dk || !dv || !dbeta || !dg_frame))
        return GDN_ERR_NULL;
    if (qkd.dtype != GDN_BF16 || vd.dtype != GDN_BF16 || dod.dtype != GDN_BF16) return GDN_ERR_DTYPE;
    const int Vt = V + (dden ? 1 : 0);
    if (K % 8 != 0 || V % 8 != 0 || K > 128 || Vt > 128) return GDN_ERR_SHAPE;
    if (frame < gdn::kChunk || frame % gdn::kChunk != 0 || T % frame != 0) return GDN_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !strides_ok(qkd) ||
        !strides_ok(vd) || !strides_ok(dod))
        return GDN_ERR_LAYOUT;
    for (const void *f : {(const void *)dq, (const void *)dk, (const void *)dv, (const void *)dbeta,
                          (const void *)dg_frame, (const void *)dh0, (const void *)dh_final,
                          (const void *)h0, (const void *)dden, (const void *)g_frame, (const void *)beta})
        if (f && (reinterpret_cast<uintptr_t>(f) & 7)) return GDN_ERR_LAYOUT;
    FrameBwdWs L;
    if (!frame_bwd_ws(B, T, H, K, V, frame, dden != nullptr, L)) return GDN_ERR_SHAPE;
    if (!workspace || ws_bytes < L.total || !aligned16(workspace)) return GDN_ERR_WORKSPACE;
    if (T == 0) {  // dL/dh0 = dL/dh_final
        if (!dh0) return GDN_OK;
        const size_t n = (size_t)B * H * K * Vt * sizeof(float);
        return cuda_status(dh_final ? cudaMemcpyAsync(dh0, dh_final, n, cudaMemcpyDeviceToDevice, stream)
                                    : cudaMemsetAsync(dh0, 0, n, stream));
    }
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    // the forward's A_f, B_f and the read states of each direction
    gdn::FrameParams p{};
    p.q = q, p.k = k, p.v = v;
    p.qk_sb = qkd.stride_b, p.qk_st = qkd.stride_t, p.qk_sh = qkd.stride_h;
    p.v_sb = vd.stride_b, p.v_st = vd.stride_t, p.v_sh = vd.stride_h;
    p.beta = beta, p.g_frame = g_frame;
    p.B = B, p.T = T, p.H = H, p.K = K, p.V = V, p.Vt = Vt;
    p.Vs = (Vt + 7) / 8 * 8;
    p.F = T / frame, p.frame = frame;
    p.has_den = dden != nullptr;
    p.amat = reinterpret_cast<float *>(ws + L.fwd.amat);
    p.bmat = reinterpret_cast<float *>(ws + L.fwd.bmat);
    float *sread[2] = {reinterpret_cast<float *>(ws + L.fwd.sout), reinterpret_cast<float *>(ws + L.sread1)};
    cudaError_t e = launch(KFrameGram, stream, [&] { return gdn::launch_frame_gram(p, stream); });
    gdn::FrameBwdParams b{};
    b.q = q, b.k = k, b.v = v, b.dout = dout;
    b.qk_sb = qkd.stride_b, b.qk_st = qkd.stride_t, b.qk_sh = qkd.stride_h;
    b.v_sb = vd.stride_b, b.v_st = vd.stride_t, b.v_sh = vd.stride_h;
    b.do_sb = dod.stride_b, b.do_st = dod.stride_t, b.do_sh = dod.stride_h;
    b.beta = beta, b.g_frame = g_frame, b.h0 = h0, b.dden = dden, b.dh_final = dh_final;
    b.dq = dq, b.dk = dk, b.dv = dv, b.dbeta = dbeta, b.dg_frame = dg_frame, b.dh0 = dh0;
    b.B = B, b.T = T, b.H = H, b.K = K, b.V = V, b.Vt = Vt, b.Vs = p.Vs, b.F = p.F, b.frame = frame;
    b.tok_group = 1;  // the largest of 4, 3, 2 chunks dividing the frame's
    for (int g = 4; g > 1; --g)
        if ((frame / gdn::kChunk) % g == 0) {
            b.tok_group = g;
            break;
        }
    b.amat = p.amat;
    b.cmat = reinterpret_cast<float *>(ws + L.cmat);
    b.lam = reinterpret_cast<float *>(ws + L.lam);
    b.dgp = reinterpret_cast<float *>(ws + L.dgp);
    // Q_f^T [dO_f | dden_f] serves both directions
    if (e == cudaSuccess) e = launch(KFrameXt, stream, [&] { return gdn::launch_frame_xt(b, stream); });
    int pass = 0;
    for (int d = 0; d < 2 && e == cudaSuccess; ++d) {
        if (direction != 2 && direction != d) continue;
        p.direction = d;
        p.sout = sread[d];
        p.h0 = d == 0 ? h0 : nullptr;
        e = launch(KFrameChain, stream, [&] { return gdn::launch_frame_chain(p, stream); });
        b.direction = d, b.acc = pass++ > 0, b.sread = sread[d];
        if (e == cudaSuccess) e = launch(KFrameLam, stream, [&] { return gdn::launch_frame_lam(b, stream); });
        if (e == cudaSuccess) e = launch(KFrameTok, stream, [&] { return gdn::launch_frame_tokgrad(b, stream); });
    }
    return cuda_status(e);
}

gdn_status gdn_last_device_error(void *workspace, cudaStream_t stream, int *word) {
    if (!workspace) return GDN_ERR_WORKSPACE;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GDN_ERR_CUDA;
    int w = 0;
    if (cudaMemcpy(&w, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (cudaMemset(workspace, 0, sizeof(int)) != cudaSuccess) return GDN_ERR_CUDA;
    if (word) *word = w;
    if (w & GDN_DEVERR_TIMEOUT) return GDN_ERR_TIMEOUT;
    return w ? GDN_ERR_DEVICE : GDN_OK;
}

int gdn_kernel_kinds(void) { return KNumKinds; }

const char *gdn_kernel_name(int kind) {
    return (kind >= 0 && kind < KNumKinds) ? kKindNames[kind] : "unknown";
}

void gdn_set_state_tile(int bv) { gdn::set_state_tile(bv); }

void gdn_set_fused(int on) { gdn::set_fused(on); }

void gdn_set_stall_test(int cta, int limit_us) {
    g_stall_us.store(limit_us > 0 ? limit_us : 1);
    g_stall_cta.store(cta >= 0 ? cta : -1);
}

void gdn_profile_enable(int on) {
    Profiler &P = prof();
    std::lock_guard<std::mutex> g(P.mu);
    P.on = on != 0;
}

gdn_status gdn_profile_collect(float *ms, int *launches, int n) {
    Profiler &P = prof();
    std::lock_guard<std::mutex> g(P.mu);
    for (int i = 0; i < n; ++i) {
        if (ms) ms[i] = 0.f;
        if (launches) launches[i] = 0;
    }
    gdn_status st = GDN_OK;
    for (auto &r : P.recs) {
        float t = 0.f;
        if (cudaEventSynchronize(r.b) != cudaSuccess ||
            cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess)
            st = GDN_ERR_CUDA;
        if (r.kind < n) {
            if (ms) ms[r.kind] += t;
            if (launches) launches[r.kind] += 1;
        }
        P.pool.push_back(r.a);
        P.pool.push_back(r.b);
    }
    P.recs.clear();
    return st;
}

long long gdn_launch_count(void) { return g_launches.load(); }

}  // extern "C"
