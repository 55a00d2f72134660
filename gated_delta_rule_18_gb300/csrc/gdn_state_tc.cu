// gdn_state_tc.cu -- chunk-serial state passing and output of the bf16 path
// on the fifth-generation tensor cores (tcgen05, accumulators in TMEM).
//
// One CTA (4 warps) per (sequence, head, 64-column value tile), walking the
// sequence's 64-token chunks in order. Thread r keeps row r of the fp32 state
// h (128 keys x 64 columns) in registers. Per chunk (hyper-parallel
// coverage_diff page, `chunk_gated_delta_rule_fwd_kernel_h_blockdim64`:
// b_v = u - w h, h *= exp(g_last), h += k^T v_new; the output adds the
// in-chunk term and reads the state after each token's own write, as the
// SANA `fused_gdn.py` page's Pass 2 does):
//
//   [Xw; O] = [w; qg] h      one MMA chain, M=128 (w and qg stacked), K=128
//   v_new   = u - Xw         threads of warps 0-1 (bf16 operand below)
//   dh      = kg^T v_new     MMA, M=128 keys, K=64 tokens
//   h       = dec . h + dh   every thread, fp32
//   [.; O] += [0; P] v_new   MMA, M=128 (a zero block stacked over P)
//
// Only the recurrence (the first product, v_new, dh, the h update) is on the
// critical path. Its MMAs are issued by thread 0; the output of chunk c
// (P v_new, then storing O) runs one chunk later on warps 2-3 while warps 0-1
// compute chunk c+1's v_new, so the [Xw; O] accumulator and v_new are double
// buffered. Copies are issued by a thread of warp 1; each MMA group completes
// on its own mbarrier. The intra-chunk kernel stores w, qg, kg^T, P, u and dec
// as per-chunk images already in the shared-memory operand layouts, so a
// chunk's operands arrive by six 1-D bulk async copies (cp.async.bulk,
// completion counted in bytes on an mbarrier), double-buffered one chunk
// ahead; w and qg land back to back, so one descriptor spans both.
//
// Every wait is bounded: on a timeout the kernel records GDN_DEVERR_TIMEOUT in
// the workspace error word, drains what it issued (again bounded), frees its
// tensor memory and returns.
#include "gdn_common.cuh"

namespace gdn {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kThreads = 128;
constexpr int kBVt = 64;  // value columns per CTA

struct Lay {
    // one stage: w | qg | kg^T | zero block | P | u | dec
    static constexpr uint32_t w = 0;
    static constexpr uint32_t qg = w + kImgW;  // directly after w: [w; qg] is one M=128 operand
    static constexpr uint32_t kg = qg + kImgW;
    static constexpr uint32_t z = kg + kImgW;  // 64 zero rows stacked over P
    static constexpr uint32_t pm = z + kImgP;
    static constexpr uint32_t u = pm + kImgP;
    static constexpr uint32_t dec = u + kImgU;
    static constexpr uint32_t stage = dec + kDecB;
    static constexpr uint32_t copy_bytes = stage - kImgP;  // everything but the zero block
    static constexpr uint32_t h = 2 * stage;               // h as the MMA B operand (MN-major)
    static constexpr uint32_t vn = h + 64 * kKP * 2;       // 2 x v_new as the MMA B operand (MN-major)
    static constexpr uint32_t vn_bytes = 64 * 64 * 2;
    static constexpr uint32_t bytes = vn + 2 * vn_bytes;
};

// TMEM columns: [Xw; O] of even / odd chunks [0,64) / [64,128) (lane = row:
// 0-63 Xw, 64-127 O), dh [128,192)
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColD = 0, kColDh = 128;

// instruction descriptors (kind::f16: bf16 inputs, fp32 accumulate)
constexpr uint32_t idesc(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t kIdescK = idesc(128, 64, 0, 1);   // A K-major ([w;qg], [0;P]), B MN-major
constexpr uint32_t kIdescMN = idesc(128, 64, 1, 1);  // A = kg^T MN-major, B = v_new MN-major

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
// Wait for the mbarrier phase `parity`; false after ~0.5 s (no hang).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity) {
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
            const uint64_t t = now_ns();
            if (t0 == 0) t0 = t;
            else if (t - t0 > 500000000ull) return false;
        }
    }
}

// 64 consecutive TMEM columns of this warp's 32 lanes -> 64 registers
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
    uint32_t r[64];
#define GDN_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
        "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
        : GDN_R8(0), GDN_R8(8), GDN_R8(16), GDN_R8(24), GDN_R8(32), GDN_R8(40), GDN_R8(48), GDN_R8(56)
        : "r"(taddr));
#undef GDN_R8
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint4 pack8(const float *f) {
    uint4 u;
    u.x = pack_bf16(f[0], f[1]);
    u.y = pack_bf16(f[2], f[3]);
    u.z = pack_bf16(f[4], f[5]);
    u.w = pack_bf16(f[6], f[7]);
    return u;
}

__global__ void __launch_bounds__(kThreads, 1) state_tc_kernel(const FwdParams p) {
    extern __shared__ __align__(1024) unsigned char sm[];
    __shared__ __align__(8) uint64_t bar_stage[2];
    __shared__ __align__(8) uint64_t bar_a, bar_dh, bar_o;
    __shared__ uint32_t tmem_base_s;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = p.H, K = p.K, V = p.V;
    const int s = blockIdx.x / H, hh = blockIdx.x % H;
    const int vt = blockIdx.y, v0 = vt * kBVt;
    if (!p.cu_seqlens && blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) *p.err = 0;
    if (p.cu_seqlens && *p.n_chunks < 0) return;
    SeqInfo si;
    if (!seq_info(p, s, si)) return;
    const int nchunks = (si.len + kChunk - 1) / kChunk;
    const int gc0 = p.cu_seqlens ? p.seq_chunk0[s] : s * ((p.T + kChunk - 1) / kChunk);
    const uint32_t sbase = smem_u32(sm);
    const uint32_t bar_st0 = smem_u32(&bar_stage[0]), bar_st1 = smem_u32(&bar_stage[1]);
    const uint32_t b_a = smem_u32(&bar_a), b_dh = smem_u32(&bar_dh), b_o = smem_u32(&bar_o);

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_base_s)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar_st0));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar_st1));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b_a));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b_dh));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b_o));
        asm volatile("fence.mbarrier_init.release.cluster;");
    }
    // the zero blocks stacked over P (never overwritten by the copies)
    for (int e = tid; e < (int)(kImgP / 16); e += kThreads) {
        *reinterpret_cast<uint4 *>(sm + Lay::z + 16 * e) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(sm + Lay::stage + Lay::z + 16 * e) = make_uint4(0, 0, 0, 0);
    }
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = tmem_base_s;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

    // state row r = tid (TMEM lane of the M=128 accumulator), columns v0..v0+63
    const int r = tid;
    float h[64];
#pragma unroll
    for (int c = 0; c < 64; ++c)
        h[c] = (p.h0 && r < K && v0 + c < V) ? p.h0[(((int64_t)s * H + hh) * K + r) * V + v0 + c] : 0.f;

    // chunk c's operands: part 0 = w, qg, kg^T, u, dec; part 1 = P (P of the
    // stage's previous chunk is read by the deferred output MMA, so it is
    // copied later). Both parts complete on the stage's mbarrier.
    auto issue_stage = [&](int c, int part) {  // one thread
        const int st = c & 1;
        const uint32_t dst = sbase + st * Lay::stage;
        const uint32_t bar = st ? bar_st1 : bar_st0;
        const size_t gch = (size_t)hh * p.max_chunks + gc0 + c;
        if (part == 0) {
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                         "r"(Lay::copy_bytes)
                         : "memory");
            const void *src[5] = {p.w_img + gch * kImgW, p.qg_img + gch * kImgW, p.kg_img + gch * kImgW,
                                  p.u_img + (gch * p.n_vt + vt) * kImgU, p.dec + gch * kKP};
            const uint32_t off[5] = {Lay::w, Lay::qg, Lay::kg, Lay::u, Lay::dec};
            const uint32_t len[5] = {kImgW, kImgW, kImgW, kImgU, kDecB};
#pragma unroll
            for (int x = 0; x < 5; ++x)
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                        dst + off[x]),
                    "l"(src[x]), "r"(len[x]), "r"(bar)
                    : "memory");
        } else {
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    dst + Lay::pm),
                "l"(p.p_img + gch * kImgP), "r"(kImgP), "r"(bar)
                : "memory");
        }
    };
    // output of chunk c (warps 2-3): O += P v_new, then store O's rows
    auto output = [&](int c, bool &okc) {
        const int st = c & 1;
        const uint32_t dcol = kColD + (uint32_t)(c & 1) * 64;
        if (tid == 64) {
            const uint32_t vb = sbase + Lay::vn + (uint32_t)(c & 1) * Lay::vn_bytes;
            const uint32_t stg = sbase + st * Lay::stage;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma(tmem + dcol, sdesc(stg + Lay::z + ks * 256, 128, 1024), sdesc(vb + ks * 256, 128, 1024),
                    kIdescK, 1);
            commit(b_o);
        }
        okc = wait_bar(b_o, c & 1) && okc;
        fence_after();
        float t[64];
        tmem_ld64(tmem + lane_base + dcol, t);
        const int i = tid - 64;
        const int pos0 = c * kChunk;
        const int Lc = min(kChunk, si.len - pos0);
        if (i < Lc && okc) {
            const int tq = q_token(p.reverse, si.len, pos0 + i);
            const int64_t off = si.b * p.o_sb + (int64_t)(si.tstart + tq) * p.o_st + hh * p.o_sh + v0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int col = v0 + 8 * j;
                if (col + 8 <= V) {
                    if (p.out_f32) {
                        float4 *op = reinterpret_cast<float4 *>((float *)p.out + off + 8 * j);
                        float4 a = make_float4(t[8 * j], t[8 * j + 1], t[8 * j + 2], t[8 * j + 3]);
                        float4 b = make_float4(t[8 * j + 4], t[8 * j + 5], t[8 * j + 6], t[8 * j + 7]);
                        if (p.accumulate) {
                            const float4 y0 = op[0], y1 = op[1];
                            a.x += y0.x; a.y += y0.y; a.z += y0.z; a.w += y0.w;
                            b.x += y1.x; b.y += y1.y; b.z += y1.z; b.w += y1.w;
                        }
                        op[0] = a;
                        op[1] = b;
                    } else {
                        uint4 *op = reinterpret_cast<uint4 *>((bf16 *)p.out + off + 8 * j);
                        float f[8];
#pragma unroll
                        for (int x = 0; x < 8; ++x) f[x] = t[8 * j + x];
                        if (p.accumulate) {
                            const uint4 y = *op;
                            const __nv_bfloat162 *y2 = reinterpret_cast<const __nv_bfloat162 *>(&y);
#pragma unroll
                            for (int x = 0; x < 4; ++x) {
                                const float2 fy = __bfloat1622float2(y2[x]);
                                f[2 * x] += fy.x;
                                f[2 * x + 1] += fy.y;
                            }
                        }
                        *op = pack8(f);
                    }
                } else if (p.has_den && col == V) {
                    float *dp = p.den + ((int64_t)si.b * H + hh) * p.T + si.tstart + tq;
                    *dp = p.accumulate ? *dp + t[8 * j] : t[8 * j];
                }
            }
        }
    };

    int timed_out = 0;
    if (nchunks > 0 && tid == 32) {
        issue_stage(0, 0);
        issue_stage(0, 1);
    }
    int c = 0;
    for (; c < nchunks; ++c) {
        const int st = c & 1;
        const uint32_t par = c & 1;  // phase of the per-chunk barriers
        const uint32_t stg = sbase + st * Lay::stage;
        const int pos0 = c * kChunk;
        const int Lc = min(kChunk, si.len - pos0);

        // operands of chunk c have landed; h (bf16) -> MN-major B operand
        const bool ok_stage = wait_bar(st ? bar_st1 : bar_st0, (c >> 1) & 1);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4 *>(sm + Lay::h + j * 2048 + r * 16) = pack8(&h[8 * j]);
        fence_async_smem();
        fence_before();
        if (__syncthreads_or(!ok_stage)) {
            timed_out = 1;
            break;
        }
        fence_after();
        const uint32_t dcol = kColD + par * 64;  // this chunk's [Xw; O] columns
        if (tid == 0) {  // [Xw; O] = [w; qg] h, K = 128 keys in 8 steps
            const uint32_t hb = sbase + Lay::h;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma(tmem + dcol, sdesc(stg + Lay::w + ks * 256, 128, 2048), sdesc(hb + ks * 256, 128, 2048),
                    kIdescK, ks > 0);
            commit(b_a);
        } else if (tid == 32 && c + 1 < nchunks) {
            issue_stage(c + 1, 0);
        }
        bool ok = true;
        if (warp >= 2 && c > 0) output(c - 1, ok);  // the previous chunk's output, off the critical path
        if (warp < 2) {  // v_new = u - Xw for token row i = tid
            ok = wait_bar(b_a, par);
            fence_after();
            float xw[64];
            tmem_ld64(tmem + lane_base + dcol, xw);
            const int i = tid;
            const unsigned char *urow = sm + st * Lay::stage + Lay::u + i * (kUS * 2);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint4 uv = *reinterpret_cast<const uint4 *>(urow + 16 * j);
                const __nv_bfloat162 *u2 = reinterpret_cast<const __nv_bfloat162 *>(&uv);
                float f[8];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const float2 t = __bfloat1622float2(u2[x]);
                    f[2 * x] = t.x - xw[8 * j + 2 * x];
                    f[2 * x + 1] = t.y - xw[8 * j + 2 * x + 1];
                }
                // MN-major B operand (N = column, K = token): (col/8)*1024 + i*16
                *reinterpret_cast<uint4 *>(sm + Lay::vn + par * Lay::vn_bytes + j * 1024 + i * 16) = pack8(f);
            }
            fence_async_smem();
        }
        fence_before();
        if (__syncthreads_or(!ok)) {
            timed_out = 2;
            break;
        }
        fence_after();
        const uint32_t vb = sbase + Lay::vn + par * Lay::vn_bytes;
        if (tid == 0) {  // dh = kg^T v_new (M = 128 keys, K = 64 tokens)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma(tmem + kColDh, sdesc(stg + Lay::kg + ks * 256, 128, 1024), sdesc(vb + ks * 256, 128, 1024),
                    kIdescMN, ks > 0);
            commit(b_dh);
        } else if (tid == 32 && c + 1 < nchunks) {
            issue_stage(c + 1, 1);  // the previous chunk's output MMA no longer reads this stage's P
        }
        // h = dec . h + dh (row r)
        bool ok2 = wait_bar(b_dh, par);
        fence_after();
        {
            float t[64];
            tmem_ld64(tmem + lane_base + kColDh, t);
            const float d = reinterpret_cast<const float *>(sm + st * Lay::stage + Lay::dec)[r];
#pragma unroll
            for (int x = 0; x < 64; ++x) h[x] = fmaf(d, h[x], t[x]);
        }
        fence_before();
        if (__syncthreads_or(!ok2)) {
            timed_out = 3;
            break;
        }
    }
    if (!timed_out && nchunks > 0) {  // the last chunk's output
        fence_after();
        bool ok = true;
        if (warp >= 2) output(nchunks - 1, ok);
        fence_before();
        if (__syncthreads_or(!ok)) timed_out = 4;
    }

    if (timed_out) {
        // record, then drain what this CTA issued (bounded) before freeing TMEM
        if (tid == 0) {
            atomicOr(p.err, 2);
            const uint32_t par = c & 1;
            if (timed_out == 1) {
                wait_bar((c & 1) ? bar_st1 : bar_st0, (c >> 1) & 1);
            } else if (timed_out == 4) {
                wait_bar(b_o, (nchunks - 1) & 1);
            } else {
                wait_bar(b_a, par);
                if (c > 0) wait_bar(b_o, (c - 1) & 1);
                if (timed_out == 3) wait_bar(b_dh, par);
                if (c + 1 < nchunks) wait_bar(((c + 1) & 1) ? bar_st1 : bar_st0, ((c + 1) >> 1) & 1);
            }
        }
    } else if (p.h_final && r < K) {
#pragma unroll
        for (int x = 0; x < 64; ++x)
            if (v0 + x < V) p.h_final[(((int64_t)s * H + hh) * K + r) * V + v0 + x] = h[x];
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

}  // namespace

cudaError_t launch_state_tc(const FwdParams &p, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(state_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Lay::bytes);
    if (e != cudaSuccess) return e;
    dim3 grid(p.n_seq * p.H, p.n_vt);
    state_tc_kernel<<<grid, kThreads, Lay::bytes, st>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
