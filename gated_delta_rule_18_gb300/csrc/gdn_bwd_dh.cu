// gdn_bwd_dh.cu -- the serial part of the backward on the fifth-generation
// tensor cores (tcgen05, accumulators in TMEM): the state gradient walked back
// over the chunks (hyper-parallel coverage_diff page,
// `chunk_gated_delta_rule_bwd_dhu`: dh accumulates q do^T and - w dv each
// chunk and is decayed by the chunk's e^{g_last}; dv gains k dh).
//
// The forward per chunk (state h entering it, G the in-chunk cumulative gate):
//   v_new = u - w h,   o = qg h + P v_new,   h' = e^{G_C} h + kg^T v_new.
// For the loss gradient dh' at the chunk's end and do of its outputs:
//   dv_new = P^T do + kg dh'                     M = 64 tokens, N = 64 columns
//   dh     = e^{G_C} dh' + qg^T do - w^T dv_new   M = 128 keys
// The forward's per-chunk images serve as the transposed operands: P^T, qg^T
// and w^T are the P, qg and w images read MN-major, kg is the kg^T image
// read K-major.
//
// One CTA per (sequence, head, 64-column tile) walks the chunks last to
// first, warp-specialised (9 warps):
//   warps 0-3  the recurrence: thread d keeps row d of dh (64 fp32) in
//              registers, writes dh' as the bf16 B operand of kg dh' (and its
//              snapshot) and applies dh = dec . dh' + [qg^T do - w^T dv_new]
//              read from TMEM; while they wait for those products they copy
//              the do tiles (cp.async) two chunks ahead and store the
//              previous chunk's dv_new snapshot from TMEM.
//   warps 4-7  dv_new: read from TMEM (M = 64 layout: rows 16q .. 16q+15 at
//              lanes 32q ..), written negated as the B operand of w^T dv_new.
//   warp 8     lane 0 issues every MMA and the images' bulk copies.
// Per chunk the do-only products (P^T do, qg^T do) are issued as soon as the
// chunk's operands have landed, ahead of dh'; what is left on the chain is
// dh' -> 8 MMAs -> dv_new -> 4 MMAs -> dh. Operands arrive in three slots,
// two chunks ahead; the TMEM accumulators are double buffered.
//
// Every wait is bounded: a wait that gives up raises a shared abort flag that
// makes every role leave its loop; the kernel records GDN_DEVERR_TIMEOUT,
// drains what it issued (again bounded), frees its tensor memory and returns.
#include "gdn_mma.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kThreadsTc = 288;  // 9 warps
constexpr int kNS = 3;           // operand slots
// one slot: qg | w | kg^T | P | do (64 x 64, MN-major B) | dec
constexpr uint32_t kOffQg = 0, kOffW = kImgW, kOffKg = 2 * kImgW, kOffP = 3 * kImgW;
constexpr uint32_t kOffDo = kOffP + kImgP, kOffDec = kOffDo + 64 * 64 * 2;
constexpr uint32_t kSlot = 65 * 1024;
static_assert(kOffDec + kDecB <= kSlot, "slot layout");
constexpr uint32_t kOffDh = kNS * kSlot;               // dh' (128 keys x 64 columns, MN-major B)
constexpr uint32_t kOffDvn = kOffDh + kKP * 64 * 2;     // -dv_new (64 tokens x 64 columns, MN-major B)
constexpr uint32_t kBytesTc = kOffDvn + 64 * 64 * 2;
static_assert(kBytesTc <= 226 * 1024, "shared memory per CTA");
// TMEM columns: dv_new of even / odd chunks at 0 / 64 (M = 64 layout), dh's
// products at 128 / 192 (lane = key)
constexpr uint32_t kTmemCols = 256, kColDv = 0, kColDh = 128;

__device__ __forceinline__ uint4 pack8(const float *f) {
    uint4 u;
    u.x = pack_bf16(f[0], f[1]);
    u.y = pack_bf16(f[2], f[3]);
    u.z = pack_bf16(f[4], f[5]);
    u.w = pack_bf16(f[6], f[7]);
    return u;
}

__global__ void __launch_bounds__(kThreadsTc, 1) bwd_dh_kernel(const BwdParams p) {
    extern __shared__ __align__(1024) unsigned char sm[];
    __shared__ __align__(8) uint64_t bar_full[kNS], bar_dvd[2], bar_dhd[2], bar_dhr, bar_dvr;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = blockIdx.x / p.H, hh = blockIdx.x % p.H;
    const int v0 = blockIdx.y * 64;
    const int K = p.K, V = p.V;
    if (p.cu_seqlens && *p.n_chunks < 0) return;  // a bad cu_seqlens: nothing was recomputed
    // the sequence: its tokens at flat rows b * T + tstart + t, its chunks at
    // global chunk slots c0 .. c0 + nts - 1
    const int b = p.cu_seqlens ? 0 : s, tstart = p.cu_seqlens ? p.cu_seqlens[s] : 0;
    const int T = p.cu_seqlens ? p.cu_seqlens[s + 1] - tstart : p.T;
    const int nts = (T + kChunk - 1) / kChunk;
    const int c0 = p.cu_seqlens ? p.seq_chunk0[s] : s * nts;
    const int vcols = p.den_col >= 0 ? p.den_col : V;  // columns from do (the rest: the ones column)
    const bf16 *dout = (const bf16 *)p.dout;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t b_full = smem_u32(&bar_full[0]), b_dvd = smem_u32(&bar_dvd[0]), b_dhd = smem_u32(&bar_dhd[0]);
    const uint32_t b_dhr = smem_u32(&bar_dhr), b_dvr = smem_u32(&bar_dvr);
    volatile int *abort = &abort_s;

    if (warp == 0) tc_alloc(&tmem_base_s, kTmemCols);
    if (tid == 0) {
        abort_s = 0;
        // a slot fills by the issuer's bulk copies (one arrival with their
        // bytes) and the do tile's 128 copying threads
        for (int x = 0; x < kNS; ++x) mbar_init(b_full + 8 * x, 129);
        for (int x = 0; x < 2; ++x) {
            mbar_init(b_dvd + 8 * x, 1);
            mbar_init(b_dhd + 8 * x, 1);
        }
        mbar_init(b_dhr, 128);
        mbar_init(b_dvr, 128);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    // step `it` handles chunk nts - 1 - it, in slot it % kNS
    auto gch_of = [&](int it) { return (int64_t)hh * p.max_chunks + c0 + (nts - 1 - it); };
    // (the do tiles are copied by the recurrence warps, in the time they
    // wait for dh's products)
    // chunk it's do tile into its slot: 64 tokens x 8 pieces of 16 bytes,
    // MN-major B ((col/8)*1024 + i*16); one cp.async group
    auto load_do = [&](int it) {
        const int c = nts - 1 - it, pos0 = c * kChunk, Lc = min(kChunk, T - pos0);
        unsigned char *dst = sm + (it % kNS) * kSlot + kOffDo;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
        const int e = (tid & 127) + 128 * j, i = e >> 3, pc = e & 7, col = 8 * pc;
        unsigned char *dp = dst + pc * 1024 + i * 16;
        if (p.den_col == v0 + col) {  // the ones column's piece: dden, then zeros
            float dd = 0.f;
            if (i < Lc)
            dd = p.dden[((int64_t)b * p.H + hh) * p.T + tstart + q_token(p.reverse, T, pos0 + i)];
            *reinterpret_cast<uint4 *>(dp) = make_uint4(pack_bf16(dd, 0.f), 0u, 0u, 0u);
            continue;
        }
        const bool in = i < Lc && v0 + col < vcols;
        const bf16 *src = in ? dout + b * p.do_sb + (int64_t)(tstart + q_token(p.reverse, T, pos0 + i)) * p.do_st +
                       hh * p.do_sh + v0 + col
                     : dout;
        cp_async16(dp, src, in ? 16 : 0);
        }
        cp_async_commit();
    };
    // the do tile of chunk j has landed: make it visible to the tensor
    // cores and count it on the slot's barrier (newer: groups issued after)
    auto publish = [&](int j, bool newer) {
        if (newer) cp_async_wait<1>();
        else cp_async_wait<0>();
        fence_async_smem();
        arrive(b_full + 8 * (j % kNS));
    };

    if (warp < 4) {
        // ------------------------------------------------ recurrence warps
        const int d = tid;
        float h[64];
#pragma unroll
        for (int c = 0; c < 64; ++c)
            h[c] = (p.dh_final && d < K && v0 + c < V)
                       ? p.dh_final[(((int64_t)s * p.H + hh) * K + d) * p.vfull + v0 + c]
                       : 0.f;
        // chunk j's dv_new (TMEM, M = 64 layout: token row 16 q + l at lane
        // 32 q + l, l < 16) to its snapshot, by this warp's lanes 0-15; here
        // rather than in the dv_new warps, whose proxy fence would otherwise
        // wait for these global stores
        auto dvn_snapshot = [&](int j) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float v[32];
                tc_ld32(tmem + lane_base + kColDv + 64 * (j & 1) + 32 * half, v);
                if (lane < 16) {
                    const int i = 16 * warp + lane;
                    bf16 *vs = p.dvn_snap + (gch_of(j) * kChunk + i) * p.snap_ld + v0 + 32 * half;
#pragma unroll
                    for (int x = 0; x < 4; ++x)
                        if (v0 + 32 * half + 8 * x < V) *reinterpret_cast<uint4 *>(vs + 8 * x) = pack8(&v[8 * x]);
                }
            }
            tc_fence_before();
        };
        if (nts > 0) load_do(0);
        if (nts > 1) load_do(1);
        if (nts > 0) publish(0, nts > 1);
        bool ok = true;
        for (int it = 0; it < nts && ok; ++it) {
            const int sl = it % kNS;
            // the slot's decay (the slot is refilled only after this chunk's
            // products, which wait for the arrival below)
            ok = warp_all(wait_bar(b_full + 8 * sl, (it / kNS) & 1, abort));
            if (!ok) break;
            const float dec = reinterpret_cast<const float *>(sm + sl * kSlot + kOffDec)[d];
            // dh' -> the MN-major B operand ((col/8)*2048 + d*16; its last
            // reader, chunk it-1's kg dh', finished before that chunk's dh),
            // handed over before its snapshot is stored (a proxy fence after
            // the global stores would wait for them)
#pragma unroll
            for (int j = 0; j < 8; ++j)
                *reinterpret_cast<uint4 *>(sm + kOffDh + j * 2048 + d * 16) = pack8(&h[8 * j]);
            fence_async_smem();
            arrive(b_dhr);
            // chunk it-1's dv_new snapshot from its TMEM buffer (chunk it+1's
            // products overwrite that buffer only after the publish below)
            if (it >= 1) dvn_snapshot(it - 1);
            // chunk it+2's do tile (its slot was chunk it-1's, whose products
            // are done), then chunk it+1's, copied a chunk ago, is published
            if (it + 2 < nts) load_do(it + 2);
            if (it + 1 < nts) publish(it + 1, it + 2 < nts);
            if (d < K) {
                bf16 *hs = p.dh_snap + (gch_of(it) * K + d) * p.snap_ld + v0;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (v0 + 8 * j < V) *reinterpret_cast<uint4 *>(hs + 8 * j) = pack8(&h[8 * j]);
            }
            ok = warp_all(wait_bar(b_dhd + 8 * (it & 1), (it >> 1) & 1, abort));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float t[32];
                tc_ld32(tmem + lane_base + kColDh + 64 * (it & 1) + 32 * half, t);
#pragma unroll
                for (int x = 0; x < 32; ++x) h[32 * half + x] = fmaf(dec, h[32 * half + x], t[x]);
            }
            tc_fence_before();
        }
        if (ok && nts > 0) dvn_snapshot(nts - 1);
        cp_async_wait<0>();  // no copy outlives the CTA
        if (ok && p.dh0 && d < K) {
#pragma unroll
            for (int c = 0; c < 64; ++c)
                if (v0 + c < V) p.dh0[(((int64_t)s * p.H + hh) * K + d) * p.vfull + v0 + c] = h[c];
        }
    } else if (warp < 8) {
        // ------------------------------------------------ dv_new (warps 4-7)
        const int q4 = warp & 3;
        bool ok = true;
        for (int it = 0; it < nts && ok; ++it) {
            ok = warp_all(wait_bar(b_dvd + 8 * (it & 1), (it >> 1) & 1, abort));
            tc_fence_after();
            float v[64];
            if (ok) {
                tc_ld64(tmem + lane_base + kColDv + 64 * (it & 1), v);
                if (lane < 16) {  // token row i of the M = 64 accumulator: -dv_new
                    const int i = 16 * q4 + lane;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint4 u = pack8(&v[8 * j]);
                        u.x ^= 0x80008000u, u.y ^= 0x80008000u, u.z ^= 0x80008000u, u.w ^= 0x80008000u;
                        *reinterpret_cast<uint4 *>(sm + kOffDvn + j * 1024 + i * 16) = u;
                    }
                }
            }
            fence_async_smem();
            tc_fence_before();
            arrive(b_dvr);
        }
    } else if (tid == 8 * 32) {
        // ------------------------------------------------------ the MMA issuer
        auto issue_imgs = [&](int it) {
            const uint32_t slot = sbase + (uint32_t)(it % kNS) * kSlot, bar = b_full + 8 * (it % kNS);
            const int64_t gch = gch_of(it);
            arrive_expect_tx(bar, 3 * kImgW + kImgP + kDecB);
            bulk_g2s(slot + kOffQg, p.qg_img + gch * kImgW, kImgW, bar);
            bulk_g2s(slot + kOffW, p.w_img + gch * kImgW, kImgW, bar);
            bulk_g2s(slot + kOffKg, p.kg_img + gch * kImgW, kImgW, bar);
            bulk_g2s(slot + kOffP, p.p_img + gch * kImgP, kImgP, bar);
            bulk_g2s(slot + kOffDec, p.dec + gch * kKP, kDecB, bar);
        };
        // instruction descriptors: P^T do (A MN-major), kg dh' (A K-major),
        // qg^T do and w^T dv_new (M = 128, A MN-major); B always MN-major
        constexpr uint32_t kIdPd = tc_idesc(64, 64, 1, 1), kIdKg = tc_idesc(64, 64, 0, 1);
        constexpr uint32_t kIdDh = tc_idesc(128, 64, 1, 1);
        // B descriptors (lbo: core stride along K, sbo: along N); a K step of
        // 16 advances them by 256 bytes
        const uint64_t dDh = tc_sdesc(sbase + kOffDh, 128, 2048), dDv = tc_sdesc(sbase + kOffDvn, 128, 1024);
        int issued = min(nts, kNS);
        for (int j = 0; j < issued; ++j) issue_imgs(j);
        bool ok = true;
        int it = 0;
        for (; it < nts && ok; ++it) {
            const int sl = it % kNS;
            const uint32_t bb = (uint32_t)(it & 1);
            const uint32_t slot = sbase + (uint32_t)sl * kSlot;
            // A descriptors: P^T (K = token i: cores 1024 apart, M = j: 128),
            // qg^T / w^T (K = i: 2048, M = key: 128), kg (K = key: 1024, M = i: 128)
            const uint64_t dP = tc_sdesc(slot + kOffP, 1024, 128), dQ = tc_sdesc(slot + kOffQg, 2048, 128);
            const uint64_t dW = tc_sdesc(slot + kOffW, 2048, 128), dK = tc_sdesc(slot + kOffKg, 1024, 128);
            const uint64_t dO = tc_sdesc(slot + kOffDo, 128, 1024);
            const uint32_t tdv = tmem + kColDv + 64 * bb, tdh = tmem + kColDh + 64 * bb;
            ok = wait_bar(b_full + 8 * sl, (it / kNS) & 1, abort);
            if (!ok) break;
            tc_fence_after();
            // the do-only products (the accumulators' previous readers,
            // chunk it-2's, were done before chunk it-1's dh' arrived)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) tc_mma(tdv, dP + 128 * ks, dO + 16 * ks, kIdPd, ks > 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) tc_mma(tdh, dQ + 256 * ks, dO + 16 * ks, kIdDh, ks > 0);
            ok = wait_bar(b_dhr, (uint32_t)it & 1, abort);
            if (!ok) break;
            tc_fence_after();
            // dv_new += kg dh' (K = 128 keys)
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) tc_mma(tdv, dK + 128 * ks, dDh + 16 * ks, kIdKg, 1);
            tc_commit(b_dvd + 8 * bb);
            // chunk it+2's images into chunk it-1's slot (dh' of chunk it
            // followed that chunk's last product), while dv_new is read out
            if (it >= 1 && issued < nts) issue_imgs(issued++);
            ok = wait_bar(b_dvr, (uint32_t)it & 1, abort);
            if (!ok) break;
            tc_fence_after();
            // dh += w^T (-dv_new) (K = 64 tokens)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) tc_mma(tdh, dW + 256 * ks, dDv + 16 * ks, kIdDh, 1);
            tc_commit(b_dhd + 8 * bb);
        }
        if (!ok) {
            // drain: one more commit covers every MMA issued so far; its
            // barrier (chunk it's dv_new barrier) completes the phase of
            // parity (it / 2) & 1 at the latest with it. Then the bulk copies
            // of the chunks not yet consumed land (bounded waits).
            *abort = 1;
            tc_commit(b_dvd + 8 * (uint32_t)(it & 1));
            wait_bar(b_dvd + 8 * (uint32_t)(it & 1), (uint32_t)(it >> 1) & 1, nullptr);
            for (int j = it; j < issued; ++j) wait_bar(b_full + 8 * (j % kNS), (j / kNS) & 1, nullptr);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0 && *abort) atomicOr(p.err, kDevErrTimeout);
    if (warp == 0) tc_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_bwd_dh(const BwdParams &p, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(bwd_dh_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBytesTc);
    if (e != cudaSuccess) return e;
    bwd_dh_kernel<<<dim3(p.n_seq * p.H, (p.V + 63) / 64), kThreadsTc, kBytesTc, st>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
