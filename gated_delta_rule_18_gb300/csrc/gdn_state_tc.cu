// gdn_state_tc.cu -- chunk-serial state passing and output of the bf16 path
// on the fifth-generation tensor cores (tcgen05, accumulators in TMEM).
//
// One CTA per (sequence, head, 64-column value tile), the tiles of a head
// adjacent in the grid, walking the sequence's 64-token chunks in order,
// warp-specialised (9 warps):
//
//   warps 0-3  the recurrence. Thread r keeps row r of the fp32 state h
//              (128 keys x 64 columns) in registers; per chunk it writes h as
//              the bf16 B operand and applies h = dec . h + dh.
//   warps 0,1  with warps 4,5 (same TMEM lanes 0-63): v_new = u - Xw, each
//   + 4,5      warp pair splitting a row's 64 columns in halves.
//   warps 6-7  the output: read O for TMEM lanes 64-127 and store it; one of
//              their threads also issues the operand copies once chunk c's
//              last MMA is done: chunk c+3's [w; qg], u and dec, chunk
//              c+2's kg^T and P.
//   warp 8     lane 0 issues every tcgen05.mma and does nothing else, so it
//              answers each hand-over at once and no v_new warp waits on
//              its issuing.
//
// Per chunk (hyper-parallel coverage_diff page,
// `chunk_gated_delta_rule_fwd_kernel_h_blockdim64`: b_v = u - w h,
// h *= exp(g_last), h += k^T v_new; the output adds the in-chunk term and
// reads the state after each token's own write, as the SANA `fused_gdn.py`
// page's Pass 2 does):
//
//   [Xw; O] = [w; qg] h      MMA chain, M=128 (w and qg stacked), K=128 keys
//   v_new   = u - Xw         warps 0-1 (bf16 MN-major operand)
//   dh      = kg^T v_new     MMA, M=128 keys, K=64 tokens
//   h       = dec . h + dh   warps 0-3, fp32
//   [.; O] += [0; P] v_new   MMA, M=128 (a zero block stacked over P)
//
// Roles hand over through mbarriers only (thread arrivals for "operand
// written", tcgen05.commit for "MMA done", transaction bytes for copies), so
// only the recurrence is on the critical path; the output of a chunk overlaps
// the next chunk. [Xw; O] and v_new are double buffered. The intra-chunk
// kernel stores w, qg, kg^T, P, u and dec as per-chunk images in the
// shared-memory operand layouts, so a chunk's operands arrive by six 1-D bulk
// async copies (cp.async.bulk) in two rings, each with its own barriers:
// ring A ([w; qg], u; dec in a ring of four) three chunks (two for the
// 128-column tiles) ahead of the first product, ring B (kg^T, P) two chunks
// ahead of the dh product, so that every buffer a copy overwrites was
// released before the copy is issued. (With one two-slot ring for all six, a
// chunk's first product waited ~280 cycles for its copies after h was ready.)
//
// Every wait is bounded: a wait that gives up raises a shared abort flag that
// makes every role leave its loop, the kernel records GDN_DEVERR_TIMEOUT in
// the workspace error word, drains what it issued (again bounded), frees its
// tensor memory and returns.
#include <atomic>

#include "gdn_tc.cuh"

namespace gdn {
namespace {

using bf16 = __nv_bfloat16;

// BV value columns per CTA: 64 (the default), or 128 for grids with more
// (sequence, head, 64-column tile) units than SMs, where one CTA carrying
// both 64-column tiles of a head (N = 128 products, the head's w / qg / kg /
// P staged once) does the two tiles' chains in about the time of one.
template <int BV>
struct Cfg;
template <>
struct Cfg<64> {
    static constexpr int kThreads = 288;  // 9 warps
    // [w; qg], u and dec are copied kRingA chunks ahead of their first
    // product; kg^T and P, read later in a chunk, two chunks ahead
    static constexpr int kRingA = 3, kVnBuf = 2;
    static constexpr uint32_t kTmemCols = 256;
};
template <>
struct Cfg<128> {
    static constexpr int kThreads = 384;  // 12 warps
    // rings of two [w; qg] / u slots and one v_new buffer fit the 128-column
    // tiles in shared memory; chunk c+1's v_new is written after its first
    // product, whose commit covers chunk c's products that read the v_new
    // buffer (one issuing thread, products in order)
    static constexpr int kRingA = 2, kVnBuf = 1;
    static constexpr uint32_t kTmemCols = 512;
};

template <int BV>
struct Lay {
    // ring A (kRingA slots): w | qg, then ring B (two slots): kg^T | zero block | P
    static constexpr uint32_t w = 0;
    static constexpr uint32_t qg = w + kImgW;  // directly after w: [w; qg] is one M=128 operand
    static constexpr uint32_t a_slot = 2 * kImgW;
    static constexpr uint32_t b_ring = Cfg<BV>::kRingA * a_slot;
    static constexpr uint32_t kg = 0;              // within a ring B slot
    static constexpr uint32_t z = kg + kImgW;      // 64 zero rows stacked over P
    static constexpr uint32_t pm = z + kImgP;
    static constexpr uint32_t b_slot = pm + kImgP;
    static constexpr uint32_t u_slot = kImgU * (BV / 64);      // BV/64 u image tiles side by side
    static constexpr uint32_t u = b_ring + 2 * b_slot;          // ring of u slots (ring A's chunks)
    static constexpr uint32_t dec = u + Cfg<BV>::kRingA * u_slot;  // ring of 4 decay vectors
    static constexpr uint32_t h = dec + 4 * kDecB;              // h as the MMA B operand (MN-major)
    static constexpr uint32_t vn = h + BV * kKP * 2;            // v_new as the MMA B operand (MN-major)
    static constexpr uint32_t vn_bytes = 64 * BV * 2;
    static constexpr uint32_t bytes = vn + Cfg<BV>::kVnBuf * vn_bytes;
};
static_assert(Lay<64>::bytes <= 226 * 1024 && Lay<128>::bytes <= 226 * 1024, "shared memory per CTA");

// TMEM columns: [Xw; O] of even / odd chunks [0,BV) / [BV,2BV) (lane = row:
// 0-63 Xw, 64-127 O), dh [2BV,3BV)
constexpr uint32_t kColD = 0;

__device__ __forceinline__ uint4 pack8(const float *f) {
    uint4 u;
    u.x = pack_bf16(f[0], f[1]);
    u.y = pack_bf16(f[2], f[3]);
    u.z = pack_bf16(f[4], f[5]);
    u.w = pack_bf16(f[6], f[7]);
    return u;
}

// columns v1 .. v1+63 of one fp32 state row (n columns; columns past n read
// as 0 and are not written), by 16-byte accesses when the row start is
// 16-byte aligned and n a multiple of 4 (v1 is a multiple of 64)
__device__ __forceinline__ void load_row64(float (&h)[64], const float *row, int v1, int n) {
    if ((reinterpret_cast<uintptr_t>(row) & 15) == 0 && (n & 3) == 0) {
#pragma unroll
        for (int x = 0; x < 64; x += 4) {
            const float4 t = v1 + x < n ? *reinterpret_cast<const float4 *>(row + v1 + x) : make_float4(0.f, 0.f, 0.f, 0.f);
            h[x] = t.x, h[x + 1] = t.y, h[x + 2] = t.z, h[x + 3] = t.w;
        }
    } else {
#pragma unroll
        for (int x = 0; x < 64; ++x) h[x] = v1 + x < n ? row[v1 + x] : 0.f;
    }
}
__device__ __forceinline__ void store_row64(float *row, const float (&h)[64], int v1, int n) {
    if ((reinterpret_cast<uintptr_t>(row) & 15) == 0 && (n & 3) == 0) {
#pragma unroll
        for (int x = 0; x < 64; x += 4)
            if (v1 + x < n) *reinterpret_cast<float4 *>(row + v1 + x) = make_float4(h[x], h[x + 1], h[x + 2], h[x + 3]);
    } else {
#pragma unroll
        for (int x = 0; x < 64; ++x)
            if (v1 + x < n) row[v1 + x] = h[x];
    }
}

// STALL: the instantiation with the stall testing aid (launched only while it
// is on, so that the working kernel carries none of its code)
template <int BV, bool STALL>
__global__ void __launch_bounds__(Cfg<BV>::kThreads, 1) state_tc_kernel(const FwdParams p) {
    using Lay = gdn::Lay<BV>;
    constexpr int kThreads = Cfg<BV>::kThreads;
    constexpr uint32_t kTmemCols = Cfg<BV>::kTmemCols;
    constexpr uint32_t kColDh = 2 * BV;
    constexpr uint32_t kIdescK = tc_idesc(128, BV, 0, 1);   // A K-major ([w;qg], [0;P]), B MN-major
    constexpr uint32_t kIdescMN = tc_idesc(128, BV, 1, 1);  // A = kg^T MN-major, B = v_new MN-major
    constexpr int kUT = BV / 64;                            // u image tiles per CTA
    constexpr int kOutW = BV == 64 ? 6 : 10;                // first output warp (TMEM lanes 64-127)
    extern __shared__ __align__(1024) unsigned char sm[];
    constexpr int kRingA = Cfg<BV>::kRingA;
    __shared__ __align__(8) uint64_t bar_ra[kRingA], bar_rb[2], bar_ofree[2];
    __shared__ __align__(8) uint64_t bar_h, bar_vn, bar_a, bar_dh, bar_o;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;

    const int tid = threadIdx.x, warp = tid >> 5;
    const int H = p.H, K = p.K, V = p.V;
    // the column tiles of one (sequence, head) are adjacent in launch order,
    // so they run together and all but the first read the head's operand
    // images from L2 rather than HBM
    // (the 128-column tiles serve plain forward passes only: no summary)
    const int n_tiles = BV == 64 ? p.n_vt + (p.summary ? p.n_kt : 0) : (p.n_vt + kUT - 1) / kUT;
    const int bhx = blockIdx.x / n_tiles;
    const int s = bhx / H, hh = bhx % H;
    const int vt = blockIdx.x % n_tiles, v0 = vt * BV;
    const int seg = blockIdx.z;
    // a transition tile of a summary pass: columns t0 .. t0+63 of M
    const bool trt = BV == 64 && p.summary && vt >= p.n_vt;
    const int t0 = trt ? (vt - p.n_vt) * BV : 0;
    // u image tiles of this CTA present in the images (a 128-column CTA over
    // an odd last tile keeps the second half of its u slots zero)
    const int n_ut = trt ? 0 : min(kUT, p.n_vt - vt * kUT);
    if (STALL && stall_test(p.stall_cta, p.stall_us, p.err)) return;
    if (p.cu_seqlens && *p.n_chunks < 0) return;
    SeqInfo si;
    if (!seq_info(p, s, si)) return;
    const int nall = (si.len + kChunk - 1) / kChunk;
    // this CTA's chunks: cb .. cb + nchunks - 1 of the sequence
    const int cb = p.seg_chunks ? seg * p.seg_chunks : 0;
    const int nchunks = p.seg_chunks ? max(0, min(p.seg_chunks, nall - cb)) : nall;
    const int64_t bh = (int64_t)s * H + hh, n_bh = (int64_t)p.n_seq * H;
    const int gc0 = (p.cu_seqlens ? p.seq_chunk0[s] : s * ((p.T + kChunk - 1) / kChunk)) + cb;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t b_ra0 = smem_u32(&bar_ra[0]), b_rb0 = smem_u32(&bar_rb[0]);  // 8-byte barriers in a row
    const uint32_t b_of[2] = {smem_u32(&bar_ofree[0]), smem_u32(&bar_ofree[1])};
    const uint32_t b_h = smem_u32(&bar_h), b_vn = smem_u32(&bar_vn), b_a = smem_u32(&bar_a);
    const uint32_t b_dh = smem_u32(&bar_dh);
    const uint32_t b_o = smem_u32(&bar_o);
    volatile int *abort = &abort_s;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_base_s)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        abort_s = 0;
        for (int x = 0; x < kRingA; ++x) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b_ra0 + 8 * x));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b_rb0));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b_rb0 + 8));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 64;" ::"r"(b_of[0]));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 64;" ::"r"(b_of[1]));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(b_h), "r"(32 * 4 * kUT));  // recurrence
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 128;" ::"r"(b_vn));  // warps 0, 1, 4, 5
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b_a));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b_dh));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b_o));
        asm volatile("fence.mbarrier_init.release.cluster;");
    }
    // the zero blocks stacked over P (never overwritten by the copies)
    for (int e = tid; e < (int)(kImgP / 16); e += kThreads) {
        *reinterpret_cast<uint4 *>(sm + Lay::b_ring + Lay::z + 16 * e) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(sm + Lay::b_ring + Lay::b_slot + Lay::z + 16 * e) = make_uint4(0, 0, 0, 0);
    }
    if (n_ut < kUT)  // u = 0 for transition columns and absent tiles: those parts stay zero
        for (int e = tid; e < (int)(kRingA * Lay::u_slot / 16); e += kThreads)
            *reinterpret_cast<uint4 *>(sm + Lay::u + 16 * e) = make_uint4(0, 0, 0, 0);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

    // chunk c's operands of the first product and of v_new ([w; qg], u, dec)
    // into ring A slot c % kRingA, counted on that slot's barrier (dec into
    // ring slot c % 4)
    auto issue_a = [&](int c) {
        const uint32_t ra = (uint32_t)(c % kRingA), bar = b_ra0 + 8 * ra;
        const uint32_t dst = sbase + ra * Lay::a_slot;
        const size_t gch = (size_t)hh * p.max_chunks + gc0 + c;
        arrive_expect_tx(bar, 2 * kImgW + kDecB + (uint32_t)n_ut * kImgU);
        bulk_g2s(dst + Lay::w, p.w_img + gch * kImgW, kImgW, bar);
        bulk_g2s(dst + Lay::qg, p.qg_img + gch * kImgW, kImgW, bar);
        const uint32_t us = sbase + Lay::u + ra * Lay::u_slot;
        for (int x = 0; x < n_ut; ++x)
            bulk_g2s(us + x * kImgU, p.u_img + (gch * p.n_vt + vt * kUT + x) * kImgU, kImgU, bar);
        bulk_g2s(sbase + Lay::dec + (uint32_t)(c % 4) * kDecB, p.dec + gch * kKP, kDecB, bar);
    };
    // chunk c's operands of the dh and output products (kg^T, P) into ring B
    // slot c & 1
    auto issue_b = [&](int c) {
        const uint32_t bar = b_rb0 + 8 * (c & 1);
        const uint32_t dst = sbase + Lay::b_ring + (c & 1) * Lay::b_slot;
        const size_t gch = (size_t)hh * p.max_chunks + gc0 + c;
        arrive_expect_tx(bar, kImgW + kImgP);
        bulk_g2s(dst + Lay::kg, p.kg_img + gch * kImgW, kImgW, bar);
        bulk_g2s(dst + Lay::pm, p.p_img + gch * kImgP, kImgP, bar);
    };
    // v_new = u - Xw for token row i, columns c0 .. c0+31 (warps 0,1 / 4,5)
    // token row i, columns c0 .. c0+31 of chunk c's u, read ahead of the
    // product it is combined with
    auto load_u = [&](int c, int i, int c0, uint4 (&uv)[4]) {
        const unsigned char *urow = sm + Lay::u + (c % kRingA) * Lay::u_slot + img_u_off(i, c0);
#pragma unroll
        for (int j = 0; j < 4; ++j) uv[j] = *reinterpret_cast<const uint4 *>(urow + 1024 * j);
    };
    // (the packed values also go to keep[], for the snapshot the caller
    // stores after its hand-over)
    auto vnew_half = [&](int c, int i, int c0, const uint4 (&uvs)[4], uint4 (&keep)[4]) {
        const uint32_t par = c & 1;
        uint32_t rr[32];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
            "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
            "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
            : "=r"(rr[0]), "=r"(rr[1]), "=r"(rr[2]), "=r"(rr[3]), "=r"(rr[4]), "=r"(rr[5]), "=r"(rr[6]),
              "=r"(rr[7]), "=r"(rr[8]), "=r"(rr[9]), "=r"(rr[10]), "=r"(rr[11]), "=r"(rr[12]), "=r"(rr[13]),
              "=r"(rr[14]), "=r"(rr[15]), "=r"(rr[16]), "=r"(rr[17]), "=r"(rr[18]), "=r"(rr[19]),
              "=r"(rr[20]), "=r"(rr[21]), "=r"(rr[22]), "=r"(rr[23]), "=r"(rr[24]), "=r"(rr[25]),
              "=r"(rr[26]), "=r"(rr[27]), "=r"(rr[28]), "=r"(rr[29]), "=r"(rr[30]), "=r"(rr[31])
            : "r"(tmem + lane_base + kColD + par * BV + c0));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 uv = uvs[j];
            const __nv_bfloat162 *u2 = reinterpret_cast<const __nv_bfloat162 *>(&uv);
            float f[8];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const float2 t = __bfloat1622float2(u2[x]);
                f[2 * x] = t.x - __uint_as_float(rr[8 * j + 2 * x]);
                f[2 * x + 1] = t.y - __uint_as_float(rr[8 * j + 2 * x + 1]);
            }
            // MN-major B operand (N = column, K = token): (col/8)*1024 + i*16
            const uint4 pv = pack8(f);
            *reinterpret_cast<uint4 *>(sm + Lay::vn + (Cfg<BV>::kVnBuf == 2 ? par : 0u) * Lay::vn_bytes +
                                       (c0 / 8 + j) * 1024 + i * 16) = pv;
            keep[j] = pv;
        }
    };
    // v_new's snapshot (the ones column's too), stored after the hand-over: a
    // proxy fence after global stores would wait for them
    auto vnew_snapshot = [&](int c, int i, int c0, const uint4 (&keep)[4]) {
        if (!p.vn_snap) return;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (v0 + c0 + 8 * j < p.Vt)
                *reinterpret_cast<uint4 *>(p.vn_snap + (((int64_t)hh * p.max_chunks + gc0 + c) * kChunk + i) * p.snap_ld +
                                           v0 + c0 + 8 * j) = keep[j];
    };

    if (warp < 4 * kUT) {
        // ------------------------------------------------ recurrence warps
        // thread r of warp group hg keeps row r, columns 64 hg .. 64 hg + 63
        const int r = BV == 64 ? tid : tid & 127, hc = BV == 64 ? 0 : (warp >> 2) * 64, v1 = v0 + hc;
        float h[64];
        if (p.summary) {  // E from h = 0, M from h = I
#pragma unroll
            for (int c = 0; c < 64; ++c) h[c] = (trt && r < K && r == t0 + c) ? 1.f : 0.f;
        } else if (p.h_in && r < K) {
            load_row64(h, p.h_in + (((int64_t)seg * n_bh + bh) * K + r) * p.Vt, v1, p.Vt);
        } else if (p.h0 && r < K) {
            load_row64(h, p.h0 + (bh * K + r) * p.h_ld, v1, p.Vt);
        } else {
#pragma unroll
            for (int c = 0; c < 64; ++c) h[c] = 0.f;
        }
        bool ok = true;
        for (int c = 0; c < nchunks && ok; ++c) {
            const uint32_t par = c & 1;
            // h (bf16) -> MN-major B operand: (col/8)*2048 + r*16; its last
            // reader, chunk c-1's first product, finished before that chunk's dh
#pragma unroll
            for (int j = 0; j < 8; ++j)
                *reinterpret_cast<uint4 *>(sm + Lay::h + (hc / 8 + j) * 2048 + r * 16) = pack8(&h[8 * j]);
            fence_async_smem();
            arrive(b_h);
            // its snapshot after the hand-over (a proxy fence after global
            // stores would wait for them)
            if (p.h_snap && r < K) {
                bf16 *hs = p.h_snap + (((int64_t)hh * p.max_chunks + gc0 + c) * K + r) * p.snap_ld + v1;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (v1 + 8 * j < p.Vt) *reinterpret_cast<uint4 *>(hs + 8 * j) = pack8(&h[8 * j]);
            }
            if ((warp & 3) < 2) {  // v_new for token row r (TMEM lanes 0-63)
                // Only the v_new warps (and the issuer) wait for ring A: chunk
                // c+kRingA's copies into the same slot follow this chunk's
                // v_new, so the barrier cannot run a phase ahead of them;
                // warps 2-3 take dec after the dh product, which follows it.
                ok = warp_all(wait_bar(b_ra0 + 8 * (c % kRingA), (c / kRingA) & 1, abort));  // u, dec of chunk c
                if (!ok) break;
                // 64 columns: columns 0..31 (the 64-column tile: its helpers
                // take 32..63), or this group's 64 of the 128-column tile
                uint4 uv[4], uw[4], kv[4], kw[4];
                load_u(c, r, hc, uv);
                if (BV == 128) load_u(c, r, hc + 32, uw);
                ok = warp_all(wait_bar(b_a, par, abort));
                tc_fence_after();
                if (ok) {
                    vnew_half(c, r, hc, uv, kv);
                    if (BV == 128) vnew_half(c, r, hc + 32, uw, kw);
                }
                fence_async_smem();
                tc_fence_before();
                arrive(b_vn);
                if (!ok) break;
                if (BV == 64) vnew_snapshot(c, r, hc, kv);  // (128-column tiles run without snapshots)
            }
            ok = warp_all(wait_bar(b_dh, par, abort));
            if (!ok) break;
            const float d = reinterpret_cast<const float *>(sm + Lay::dec + (c % 4) * kDecB)[r];
            tc_fence_after();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float t[32];
                tc_ld32(tmem + lane_base + kColDh + hc + 32 * half, t);
#pragma unroll
                for (int x = 0; x < 32; ++x) h[32 * half + x] = fmaf(d, h[32 * half + x], t[x]);
            }
            tc_fence_before();
        }
        if (ok && p.summary && r < K) {
            if (trt) {  // summary 1: M row-major; summary 2: M^T (the chain's operand)
                float *dst = p.sum_tr + ((int64_t)seg * n_bh + bh) * K * K;
                const int64_t rs = p.summary == 2 ? 1 : K, cs = p.summary == 2 ? K : 1;
#pragma unroll
                for (int x = 0; x < 64; ++x)
                    if (t0 + x < K) dst[r * rs + (t0 + x) * cs] = h[x];
            } else {
                store_row64(p.sum_ext + (((int64_t)seg * n_bh + bh) * K + r) * p.Vt, h, v1, p.Vt);
            }
        } else if (ok && p.h_final && r < K && cb + nchunks == nall) {
            store_row64(p.h_final + (bh * K + r) * p.h_ld, h, v1, p.Vt);
        }
    } else if (BV == 64 && (warp == 4 || warp == 5)) {
        // ------------------------------------- v_new helpers (columns 32..63)
        bool ok = true;
        for (int c = 0; c < nchunks && ok; ++c) {
            const uint32_t par = c & 1;
            ok = warp_all(wait_bar(b_ra0 + 8 * (c % kRingA), (c / kRingA) & 1, abort));
            uint4 uv[4], kv[4];
            if (ok) load_u(c, tid - 128, 32, uv);
            ok = ok && warp_all(wait_bar(b_a, par, abort));
            tc_fence_after();
            if (ok) vnew_half(c, tid - 128, 32, uv, kv);
            fence_async_smem();
            tc_fence_before();
            arrive(b_vn);
            if (ok) vnew_snapshot(c, tid - 128, 32, kv);
        }
    } else if (tid == 8 * 32) {
        // ------------------------------------------------------ the MMA issuer
        bool ok = true;
        int c = 0;
        // operand descriptors of every slot / buffer, built once: a K step
        // of 16 advances the start address by 256 bytes, i.e. the descriptor
        // by 16 (the 14-bit address field cannot carry: shared addresses stay
        // below 256 KB)
        const uint64_t dW0 = tc_sdesc(sbase + Lay::w, 128, 2048),
                       dW1 = tc_sdesc(sbase + Lay::a_slot + Lay::w, 128, 2048),
                       dW2 = tc_sdesc(sbase + (kRingA - 1) * Lay::a_slot + Lay::w, 128, 2048);
        const uint32_t b1 = sbase + Lay::b_ring + Lay::b_slot;
        const uint64_t dK0 = tc_sdesc(sbase + Lay::b_ring + Lay::kg, 128, 1024), dK1 = tc_sdesc(b1 + Lay::kg, 128, 1024);
        const uint64_t dZ0 = tc_sdesc(sbase + Lay::b_ring + Lay::z, 128, 1024), dZ1 = tc_sdesc(b1 + Lay::z, 128, 1024);
        const uint64_t dV0 = tc_sdesc(sbase + Lay::vn, 128, 1024),
                       dV1 = tc_sdesc(sbase + Lay::vn + (Cfg<BV>::kVnBuf - 1) * Lay::vn_bytes, 128, 1024);
        const uint64_t dH = tc_sdesc(sbase + Lay::h, 128, 2048);
        for (; c < nchunks && ok; ++c) {
            const uint32_t par = c & 1;
            const int ra = c % kRingA;
            const uint32_t dcol = kColD + par * BV;
            const uint64_t dW = ra == 0 ? dW0 : ra == 1 ? dW1 : dW2;
            const uint64_t dK = par ? dK1 : dK0, dZ = par ? dZ1 : dZ0, dV = par ? dV1 : dV0;
            // [Xw; O] = [w; qg] h once h_c is written and chunk c's ring A
            // copies landed (this accumulator set's previous user, chunk c-2,
            // was read out before P v_new of chunk c-1 was issued, below)
            ok = wait_bar(b_ra0 + 8 * ra, (c / kRingA) & 1, abort) && wait_bar(b_h, par, abort);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) tc_mma(tmem + dcol, dW + 16 * ks, dH + 16 * ks, kIdescK, ks > 0);
            tc_commit(b_a);
            // dh = kg^T v_new, then [.; O] += [0; P] v_new (ring B: kg^T, P,
            // landed long before; polled while v_new is still being formed)
            ok = wait_bar(b_rb0 + 8 * par, (c >> 1) & 1, abort) && wait_bar(b_vn, par, abort);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) tc_mma(tmem + kColDh, dK + 16 * ks, dV + 16 * ks, kIdescMN, ks > 0);
            tc_commit(b_dh);
            // b_o must not run two phases ahead of the output warps: chunk
            // c-1's output has to be read out before chunk c's is committed
            // (this also keeps the output warps, which issue the copies, in
            // step with the chain)
            if (c >= 1) ok = wait_bar(b_of[(c - 1) & 1], ((c - 1) >> 1) & 1, abort);
            if (!ok) break;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) tc_mma(tmem + dcol, dZ + 16 * ks, dV + 16 * ks, kIdescK, 1);
            tc_commit(b_o);
        }
        if (!ok) {
            // drain the last MMA groups (the copier drains the copies)
            *abort = 1;
            wait_bar(b_a, (uint32_t)c & 1, nullptr);
            wait_bar(b_o, (uint32_t)(c - 1) & 1, nullptr);
        }
    } else if (warp == kOutW || warp == kOutW + 1) {
        // ------------------------------------------------ output warps (lanes 64-127)
        const int i = tid - 32 * kOutW;  // token row within the chunk
        // one thread issues every copy once chunk c's last product is done:
        // ring A for chunk c+kRingA (its slot's readers, chunk c's first
        // product and v_new, are done), ring B for chunk c+2
        const bool copier = i == 0;
        int a_hi = 0, b_hi = 0;  // chunks issued on rings A and B
        if (copier) {
            for (; a_hi < 2 && a_hi < nchunks; ++a_hi) {
                issue_a(a_hi);
                if (b_hi < nchunks) issue_b(b_hi++);
            }
            for (; a_hi < kRingA && a_hi < nchunks; ++a_hi) issue_a(a_hi);
        }
        bool ok = true;
        for (int c = 0; c < nchunks && ok; ++c) {
            const uint32_t par = c & 1;
            const int pos0 = (cb + c) * kChunk;
            const int Lc = min(kChunk, si.len - pos0);
            const bool wr = i < Lc && !p.summary && p.out;  // no output: summary or recompute pass
            const int tq = wr ? q_token(p.reverse, si.len, pos0 + i) : 0;
            float *dp = p.den + ((int64_t)si.b * H + hh) * p.T + si.tstart + tq;
            // 64 columns at a time
#pragma unroll 1
            for (int hv = 0; hv < kUT; ++hv) {
                const int vo = v0 + 64 * hv;
                const int64_t off = si.b * p.o_sb + (int64_t)(si.tstart + tq) * p.o_st + hh * p.o_sh + vo;
                const bool den_here = p.has_den && vo <= V && V < vo + 64;
                // accumulating into bf16 rows: their old contents are loaded while
                // this chunk's products are still running
                uint4 prev[8];
                float dprev = 0.f;
                if (wr && p.accumulate && !p.out_f32) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        prev[j] = (vo + 8 * j + 8 <= V)
                                      ? *reinterpret_cast<const uint4 *>((const bf16 *)p.out + off + 8 * j)
                                      : make_uint4(0, 0, 0, 0);
                }
                if (wr && p.accumulate && den_here) dprev = *dp;
                if (hv == 0) {
                    ok = warp_all(wait_bar(b_o, par, abort));
                    tc_fence_after();
                    if (copier && ok) {
                        if (a_hi < nchunks) issue_a(a_hi++);  // chunk c + kRingA
                        if (b_hi < nchunks) issue_b(b_hi++);  // chunk c + 2
                    }
                }
                float t[64];
                tc_ld64(tmem + lane_base + kColD + par * BV + 64 * hv, t);
                if (hv == kUT - 1) {
                    tc_fence_before();
                    arrive(b_of[c & 1]);
                }
                if (!ok || !wr) continue;
                if (p.out_f32) {
#pragma unroll
                    for (int h4 = 0; h4 < 2; ++h4) {  // per half: every load before any store
                        float4 y[8];
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            const int j = 4 * h4 + jj;
                            const bool in = p.accumulate && vo + 8 * j + 8 <= V;
                            const float4 *op = reinterpret_cast<const float4 *>((const float *)p.out + off + 8 * j);
                            y[2 * jj] = in ? op[0] : make_float4(0.f, 0.f, 0.f, 0.f);
                            y[2 * jj + 1] = in ? op[1] : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            const int j = 4 * h4 + jj;
                            if (vo + 8 * j + 8 > V) continue;
                            float4 *op = reinterpret_cast<float4 *>((float *)p.out + off + 8 * j);
                            const float4 y0 = y[2 * jj], y1 = y[2 * jj + 1];
                            op[0] = make_float4(t[8 * j] + y0.x, t[8 * j + 1] + y0.y, t[8 * j + 2] + y0.z,
                                                t[8 * j + 3] + y0.w);
                            op[1] = make_float4(t[8 * j + 4] + y1.x, t[8 * j + 5] + y1.y, t[8 * j + 6] + y1.z,
                                                t[8 * j + 7] + y1.w);
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (vo + 8 * j + 8 > V) continue;
                        float f[8];
#pragma unroll
                        for (int x = 0; x < 8; ++x) f[x] = t[8 * j + x];
                        if (p.accumulate) {
                            const __nv_bfloat162 *y2 = reinterpret_cast<const __nv_bfloat162 *>(&prev[j]);
#pragma unroll
                            for (int x = 0; x < 4; ++x) {
                                const float2 fy = __bfloat1622float2(y2[x]);
                                f[2 * x] += fy.x;
                                f[2 * x + 1] += fy.y;
                            }
                        }
                        *reinterpret_cast<uint4 *>((bf16 *)p.out + off + 8 * j) = pack8(f);
                    }
                }
                if (den_here) {  // the ones column V sits at the start of an 8-column group
                    float dv = 0.f;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (vo + 8 * j == V) dv = t[8 * j];
                    *dp = (p.accumulate ? dprev : 0.f) + dv;
                }
            }
        }
        if (copier && !ok) {  // drain the outstanding copies
            for (int j = max(0, a_hi - kRingA); j < a_hi; ++j)
                wait_bar(b_ra0 + 8 * (j % kRingA), (j / kRingA) & 1, nullptr);
            for (int j = max(0, b_hi - 2); j < b_hi; ++j) wait_bar(b_rb0 + 8 * (j & 1), (j >> 1) & 1, nullptr);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0 && *abort) atomicOr(p.err, kDevErrTimeout);
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

}  // namespace

namespace {
std::atomic<int> g_state_tile{0};  // 0: by the grid, else 64 or 128

template <int BV>
cudaError_t launch_bv(const FwdParams &p, int n_tiles, cudaStream_t st) {
    auto kern = p.stall_cta >= 0 ? state_tc_kernel<BV, true> : state_tc_kernel<BV, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Lay<BV>::bytes);
    if (e != cudaSuccess) return e;
    const int nall = (p.T + kChunk - 1) / kChunk;
    // summary 2: every segment but the last (whose summary nothing reads)
    const int nseg = p.seg_chunks ? max(1, (nall + p.seg_chunks - 1) / p.seg_chunks) - (p.summary == 2 ? 1 : 0) : 1;
    if (nseg < 1) return cudaSuccess;
    dim3 grid(p.n_seq * p.H * n_tiles, 1, nseg);
    kern<<<grid, Cfg<BV>::kThreads, Lay<BV>::bytes, st>>>(p);
    return cudaGetLastError();
}
}  // namespace

void set_state_tile(int bv) { g_state_tile.store(bv == 64 || bv == 128 ? bv : 0); }

cudaError_t launch_state_tc(const FwdParams &p, cudaStream_t st) {
    // 128-column tiles: plain passes (no summary, no snapshots) over two or
    // more 64-column tiles whose 64-column grid would not fit one wave of
    // one CTA per SM
    bool wide = false;
    const int forced = g_state_tile.load();
    if (!p.summary && !p.h_snap && p.n_vt >= 2) {
        if (forced) {
            wide = forced == 128;
        } else {
            int dev = 0, n_sm = 0;
            cudaError_t e = cudaGetDevice(&dev);
            if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return e;
            const int64_t nall = (p.T + kChunk - 1) / kChunk;
            const int64_t nseg = p.seg_chunks ? (nall + p.seg_chunks - 1) / p.seg_chunks : 1;
            wide = (int64_t)p.n_seq * p.H * p.n_vt * nseg > n_sm;
        }
    }
    if (wide) return launch_bv<128>(p, (p.n_vt + 1) / 2, st);
    return launch_bv<64>(p, p.n_vt + (p.summary ? p.n_kt : 0), st);
}

}  // namespace gdn
