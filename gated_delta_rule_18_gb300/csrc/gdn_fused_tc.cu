// gdn_fused_tc.cu -- the bf16 forward of one scan direction in a single
// kernel: the intra-chunk WY factors of each chunk are formed on the tensor
// cores inside the CTA that runs the chunk-serial state pass, so they never
// leave shared and tensor memory (the split form writes them to HBM as
// per-chunk images and reads them back).
//
// One CTA per (sequence, head, 64-column value tile), 13 warps, one CTA per
// SM (~205 KB of shared memory, all 512 tensor-memory columns):
//
//   warps 0-3   the recurrence: thread r keeps row r of the fp32 state h
//               (128 keys x 64 columns) in registers; per chunk it writes h as
//               the bf16 B operand and applies h = dec . h + dh.
//   warps 0,1   with warps 4,5: v_new = u - Xw (warp pairs split a row's 64
//   + 4,5       columns).
//   warps 6-7   the output rows (tensor-memory lanes 64-127).
//   warp 12     lane 0 issues the chain's tcgen05 MMAs.
//   warps 8-11  the intra-chunk part, one chunk ahead of the chain:
//     1. q, k and v tiles of a chunk arrive by TMA (tensor maps over the
//        caller's (B, T, H, D) tensors, 128-byte swizzle) two chunks ahead,
//        into two stages; beta and the log gates by plain loads one chunk
//        ahead, with the in-chunk cumulative gate formed by a warp scan.
//     2. [K; Q] K^T on the tensor cores (M = 128: key rows over query rows).
//     3. From the Gram rows: the L2 row norms (diagonal of K K^T; the query
//        norms from the tile), A = strictly_lower(diag(beta) (k^ k^T . Gamma))
//        into shared memory and P = lower_incl(q^ k^T . Gamma) into tensor
//        memory as the A operand of the output product.
//     4. T = (I + A)^{-1}: 16 x 16 diagonal blocks by forward substitution
//        in fp32 registers, the blocks below by the block-triangular
//        inverse formula on mma.sync; written with its column scales as
//        T diag(beta e^G r_k) and T diag(beta).
//     5. W = T diag(beta e^G r_k) K and U = T diag(beta) V on the tensor
//        cores straight from the TMA tiles (K and V read as MN-major B).
//     6. Once the chain has finished with the previous chunk's operands, the
//        chunk's w, qg, u, dec and kg^T images are written in the operand
//        layouts the chain's MMAs read.
//
// The chain per chunk is the state pass of the split form (hyper-parallel
// coverage_diff page, `chunk_gated_delta_rule_fwd_kernel_h_blockdim64`:
// b_v = u - w h, h *= exp(g_last), h += k^T v_new, with the inclusive output
// of the SANA `fused_gdn.py` page's Pass 2):
//   [Xw; O] = [w; qg] h,  v_new = u - Xw,  dh = kg^T v_new,
//   h = dec . h + dh,     [.; O] += [P_tmem] v_new.
// The factors follow the token recurrence (SANA `fused_gdn.py` page,
// `_fused_gdn_kernel` Pass 1); the coverage_diff page's `chunk_kda_fwd_intra`
// returns the same w, u, kg and Aqk without showing their construction.
//
// The reverse scan (flip-and-shift) loads each chunk's rows as one TMA box
// in ascending token order, so shared row r holds logical position 63 - r;
// the state side (A, T, w, u, kg, v_new) is kept in logical order, the output
// side (qg, P, O) in shared-row order, which maps output row r back to its
// token directly.
//
// Every wait is bounded: a wait that gives up raises a shared abort flag that
// makes every role leave its loop; the kernel records GDN_DEVERR_TIMEOUT,
// waits (bounded) for the copies and MMAs it issued, frees its tensor memory
// and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "gdn_tc.cuh"

namespace gdn {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kThreads = 512;  // 16 warps: 4 per scheduler, 128 registers each
constexpr int kEW = 8;         // intra warps 8-15
constexpr int kNE = 256;       // intra threads
constexpr int kIssW = 6;       // chain MMA issuer (lane 0); warp 7 has no role
constexpr int kBS = 24;        // bf16 row stride of the 16 x 16 blocks
constexpr int kAdS = 20;       // fp32 row stride of A's diagonal blocks (16-byte aligned rows)
// Chunks whose in-chunk decay e^{G_last} is at least e^-64 take the
// pre-scaled Gram (no per-entry exponential); stronger decays take the
// per-entry form.
constexpr float kScaledGramMaxDecay = 64.f;

// tensor-memory columns
constexpr uint32_t kColXO = 0;    // [Xw; O], two sets of 64 (chunk parity)
constexpr uint32_t kColDh = 128;  // dh = kg^T v_new
constexpr uint32_t kColS = 192;   // the Gram [X1; Qg] X2^T
constexpr uint32_t kColW = 256;   // W, 128 key columns (M = 64 layout)
constexpr uint32_t kColU = 384;   // U (M = 64 layout)
constexpr uint32_t kColP = 448;   // P as bf16 pairs, two buffers of 32 (chunk parity)
constexpr uint32_t kTmemCols = 512;

// Shared memory, offsets from a 1024-byte aligned base (the swizzled TMA
// tiles need it). The q / k stage holds one chunk's tiles: per 64-key block
// kb the k rows (8 KB) then the q rows (8 KB); the v tiles have two stages.
// The chain's operands have two slots (chunk parity): [w; qg] (one M = 128
// operand; before its W product the w half holds the Gram's X1 rows), kg^T
// (also the Gram's B operand) and u.
struct FL {
    static constexpr uint32_t qk = 0, st_q = 8192, st_kb = 16384;
    static constexpr uint32_t v = 32768;               // two v stages of 8 KB
    static constexpr uint32_t wq = v + 2 * 8192;       // two [w; qg] slots of 32 KB
    static constexpr uint32_t kg = wq + 2 * 2 * kImgW;   // two kg^T slots
    static constexpr uint32_t u = kg + 2 * kImgW;        // two u slots
    static constexpr uint32_t dec = u + 2 * kImgU;       // ring of 4 decay vectors
    static constexpr uint32_t h = dec + 4 * kDecB;       // h, the MN-major B operand
    static constexpr uint32_t vn = h + 64 * kKP * 2;     // v_new, two buffers
    static constexpr uint32_t tu = vn + 2 * 8192;        // T diag(beta), K-major 64 x 64
    static constexpr uint32_t ad = tu + 8192;            // A's diagonal blocks, fp32 [4][16][20]
    static constexpr uint32_t ab = ad + 4 * 16 * kAdS * 4;  // A below the diagonal, bf16 [6][16][24]
    static constexpr uint32_t tb = ab + 6 * 16 * kBS * 2;   // T / temporary blocks, bf16 [10][16][24]
    static constexpr uint32_t gates = tb + 10 * 16 * kBS * 2;  // G, beta, r_k, r_q [64] fp32; misc
    static constexpr uint32_t bytes = gates + 4 * 256 + 16;
    static constexpr uint32_t alloc = bytes + 1024;  // slack for aligning the base
};
static_assert(FL::alloc <= 227 * 1024, "shared memory per CTA");
static_assert(FL::ad % 16 == 0 && FL::ab % 16 == 0 && FL::tb % 16 == 0 && FL::gates % 16 == 0, "alignment");
static_assert(FL::v % 1024 == 0, "swizzled tiles");
// slots of the bf16 block array
constexpr int kTbT = 0;   // T_II, I = 0..3
constexpr int kTb10 = 4, kTb32 = 5;
constexpr int kTbY = 6;   // Y blocks / level-2 temporaries, 4 slots

__device__ __forceinline__ int blk(int I, int M) { return I * (I - 1) / 2 + M; }

// Wait for mbarrier phase `parity` (try_wait suspends the thread for a
// while between polls). False after ~0.5 s or once *abort is set (abort may
// be null).
__device__ __forceinline__ bool wait_sleep(uint32_t bar, uint32_t parity, volatile int *abort) {
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
        if (abort && *abort) return false;
        const uint64_t t = now_ns();
        if (t0 == 0) t0 = t;
        else if (t - t0 > 500000000ull) {
            if (abort) *abort = 1;
            return false;
        }
    }
}

// shared-memory descriptor with 128-byte swizzle (both byte offsets 1024:
// the 8-row group stride, and the atom stride, never crossed by these MMAs)
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    return tc_sdesc(saddr, 1024, 1024) | (2ull << 61);
}
// D (+)= A B with A in tensor memory
__device__ __forceinline__ void tc_mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void tma_load4(uint32_t dst, const CUtensorMap *m, int c0, int c1, int c2, int c3,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
        "%5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}
// 32 consecutive tensor-memory columns of this warp's lanes <- 32 registers
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]));
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// 16 consecutive tensor-memory columns of this warp's lanes <-> 16 registers
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]));
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// barrier 1 over the 256 intra threads, with an AND of their flags
__device__ __forceinline__ bool e_sync_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n bar.red.and.pred po, 1, 256, pi;\n"
        " selp.u32 %0, 1, 0, po;\n}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void e_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ uint4 pack8(const float *f) {
    uint4 u;
    u.x = pack_bf16(f[0], f[1]);
    u.y = pack_bf16(f[2], f[3]);
    u.z = pack_bf16(f[4], f[5]);
    u.w = pack_bf16(f[6], f[7]);
    return u;
}
__device__ __forceinline__ void unpack8(const uint4 &u, float *f) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

// columns v1 .. v1+63 of one fp32 state row (n columns; columns past n read
// as 0 and are not written), by 16-byte accesses when the row start is
// 16-byte aligned and n a multiple of 4
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

// acc (16 x 16 as two m16n8 fragments) += A B for 16 x 16 bf16 blocks in
// shared memory (row-major, row stride kBS): A read as the row operand, B as
// the [k][n] column operand; neg negates A
__device__ __forceinline__ void blk_mma(float (&acc)[2][4], const bf16 *A, const bf16 *B, bool neg, int lane) {
    uint32_t a[4], b[4];
    ldsm_x4(a, A + (lane & 15) * kBS + (lane >> 4) * 8);
    if (neg) {
#pragma unroll
        for (int x = 0; x < 4; ++x) a[x] ^= 0x80008000u;
    }
    ldsm_x4_t(b, B + (lane & 15) * kBS + (lane >> 4) * 8);
    mma_bf16(acc[0], a, b[0], b[1]);
    mma_bf16(acc[1], a, b[2], b[3]);
}
__device__ __forceinline__ void blk_store(bf16 *D, const float (&acc)[2][4], int lane) {
    const int g8 = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int n = 0; n < 2; ++n) {
        *reinterpret_cast<uint32_t *>(D + g8 * kBS + 8 * n + 2 * t4) = pack_bf16(acc[n][0], acc[n][1]);
        *reinterpret_cast<uint32_t *>(D + (g8 + 8) * kBS + 8 * n + 2 * t4) = pack_bf16(acc[n][2], acc[n][3]);
    }
}

// STALL: the instantiation with the stall testing aid (launched only while it
// is on, so that the working kernel carries none of its code)
template <bool REV, bool STALL>
__global__ void __launch_bounds__(kThreads, 1)
    fused_tc_kernel(const FwdParams p, const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                    const __grid_constant__ CUtensorMap mv) {
    extern __shared__ __align__(1024) unsigned char sm_raw[];
    __shared__ __align__(8) uint64_t bar_h, bar_vn, bar_a, bar_dh, bar_o, bar_of[2];
    __shared__ __align__(8) uint64_t bar_ia[2], bar_ib[2], bar_free[2];
    __shared__ __align__(8) uint64_t bar_qk, bar_v[2], bar_gram, bar_wu;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H, K = p.K, V = p.V;
    const int n_tiles = p.n_vt;
    const int bhx = blockIdx.x / n_tiles;
    const int s = bhx / H, hh = bhx % H;
    const int vt = blockIdx.x % n_tiles, v0 = vt * 64;
    if (STALL && stall_test(p.stall_cta, p.stall_us, p.err)) return;
    if (p.cu_seqlens && *p.n_chunks < 0) return;
    SeqInfo si;
    if (!seq_info(p, s, si)) return;
    const int len = si.len;
    const int nchunks = (len + kChunk - 1) / kChunk;
    const int64_t bh = (int64_t)s * H + hh;
    const int n_kb = K > 64 ? 2 : 1;

    const uint32_t raw_base = smem_u32(sm_raw);
    const uint32_t sbase = (raw_base + 1023u) & ~1023u;
    unsigned char *sm = sm_raw + (sbase - raw_base);
    const uint32_t b_h = smem_u32(&bar_h), b_vn = smem_u32(&bar_vn), b_a = smem_u32(&bar_a);
    const uint32_t b_dh = smem_u32(&bar_dh), b_o = smem_u32(&bar_o);
    const uint32_t b_of0 = smem_u32(&bar_of[0]), b_ia0 = smem_u32(&bar_ia[0]), b_ib0 = smem_u32(&bar_ib[0]);
    const uint32_t b_free0 = smem_u32(&bar_free[0]), b_v0 = smem_u32(&bar_v[0]);  // pairs 8 bytes apart
    const uint32_t b_qk = smem_u32(&bar_qk), b_gram = smem_u32(&bar_gram), b_wu = smem_u32(&bar_wu);
    volatile int *abort = &abort_s;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_s)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        abort_s = 0;
        mbar_init(b_h, 128);
        mbar_init(b_vn, 128);
        mbar_init(b_a, 1);
        mbar_init(b_dh, 1);
        mbar_init(b_o, 1);
        for (int x = 0; x < 2; ++x) {
            mbar_init(b_of0 + 8 * x, 64);
            mbar_init(b_ia0 + 8 * x, 1);
            mbar_init(b_ib0 + 8 * x, 1);
            mbar_init(b_free0 + 8 * x, 1);
            mbar_init(b_v0 + 8 * x, 1);
        }
        mbar_init(b_qk, 1);
        mbar_init(b_gram, 1);
        mbar_init(b_wu, 1);
        fence_mbar_init();
    }
    // the blocks of T above the diagonal stay zero; with 64 keys or fewer the
    // second key block of the q / k stage stays zero
    for (int e = tid; e < (int)(8192 / 16); e += kThreads)
        *reinterpret_cast<uint4 *>(sm + FL::tu + 16 * e) = make_uint4(0, 0, 0, 0);
    if (n_kb == 1)
        for (int e = tid; e < (int)(FL::st_kb / 16); e += kThreads)
            *reinterpret_cast<uint4 *>(sm + FL::qk + FL::st_kb + 16 * e) = make_uint4(0, 0, 0, 0);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    float *const dec_s = reinterpret_cast<float *>(sm + FL::dec);

    // v_new = u - Xw for token row i, columns c0 .. c0+31 (u of slot par)
    auto load_u = [&](int par, int i, int c0, uint4 (&uv)[4]) {
        const unsigned char *urow = sm + FL::u + par * kImgU + img_u_off(i, c0);
#pragma unroll
        for (int j = 0; j < 4; ++j) uv[j] = *reinterpret_cast<const uint4 *>(urow + 1024 * j);
    };
    auto vnew_half = [&](int c, int i, int c0, const uint4 (&uvs)[4]) {
        const uint32_t par = c & 1;
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
            float t[16];
            tc_ld16(tmem + lane_base + kColXO + par * 64 + c0 + 16 * hq, t);
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int j = 2 * hq + jj;
                float f[8];
                unpack8(uvs[j], f);
#pragma unroll
                for (int x = 0; x < 8; ++x) f[x] -= t[8 * jj + x];
                *reinterpret_cast<uint4 *>(sm + FL::vn + par * 8192 + (c0 / 8 + j) * 1024 + i * 16) = pack8(f);
            }
        }
    };
    // the output rows of chunk c (tensor-memory lanes 64-127, shared-row
    // order), read by warps 2 and 3 one chunk late
    auto output = [&](int c, int i) -> bool {
        const uint32_t par = c & 1;
        const int pos0 = c * kChunk;
        const int Lc = min(kChunk, len - pos0);
        const int li = REV ? 63 - i : i;
        const bool wr = li < Lc && p.out;
        const int tq = wr ? q_token(REV, len, pos0 + li) : 0;
        float *dp = p.den + ((int64_t)si.b * H + hh) * p.T + si.tstart + tq;
        const int64_t off = si.b * p.o_sb + (int64_t)(si.tstart + tq) * p.o_st + hh * p.o_sh + v0;
        const bool den_here = p.has_den && v0 <= V && V < v0 + 64;
        const bool ok = warp_all(wait_sleep(b_o, par, abort));
        tc_fence_after();
        float dv = 0.f;
#pragma unroll 1
        for (int hv = 0; hv < 2; ++hv) {  // 32 columns at a time
            float t[32];
            tc_ld32(tmem + lane_base + kColXO + par * 64 + 32 * hv, t);
            if (hv == 1) {
                tc_fence_before();
                arrive(b_of0 + 8 * par);
            }
            if (!ok || !wr) continue;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int j = 4 * hv + jj;
                if (v0 + 8 * j == V) dv = t[8 * jj];  // the ones column starts an 8-column group
                if (v0 + 8 * j + 8 > V) continue;
                if (p.out_f32) {
                    float4 *op = reinterpret_cast<float4 *>((float *)p.out + off + 8 * j);
                    float4 y0 = make_float4(0.f, 0.f, 0.f, 0.f), y1 = y0;
                    if (p.accumulate) y0 = op[0], y1 = op[1];
                    const float *x = &t[8 * jj];
                    op[0] = make_float4(x[0] + y0.x, x[1] + y0.y, x[2] + y0.z, x[3] + y0.w);
                    op[1] = make_float4(x[4] + y1.x, x[5] + y1.y, x[6] + y1.z, x[7] + y1.w);
                } else {
                    float f[8];
#pragma unroll
                    for (int x = 0; x < 8; ++x) f[x] = t[8 * jj + x];
                    uint4 *op = reinterpret_cast<uint4 *>((bf16 *)p.out + off + 8 * j);
                    if (p.accumulate) {
                        float y[8];
                        unpack8(*op, y);
#pragma unroll
                        for (int x = 0; x < 8; ++x) f[x] += y[x];
                    }
                    *op = pack8(f);
                }
            }
        }
        if (ok && wr && den_here) *dp = (p.accumulate ? *dp : 0.f) + dv;
        return ok;
    };

    if (warp < 4) {
        // ---------------------------------------------------- recurrence
        const int r = tid;
        float h[64];
        if (p.h0 && r < K) {
            load_row64(h, p.h0 + (bh * K + r) * p.h_ld, v0, p.Vt);
        } else {
#pragma unroll
            for (int c = 0; c < 64; ++c) h[c] = 0.f;
        }
        bool ok = true;
        for (int c = 0; c < nchunks && ok; ++c) {
            const uint32_t par = c & 1;
            // chunk c's images (u, dec) are in
            ok = warp_all(wait_sleep(b_ia0 + 8 * par, (c >> 1) & 1, abort));
            if (!ok) break;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                *reinterpret_cast<uint4 *>(sm + FL::h + j * 2048 + r * 16) = pack8(&h[8 * j]);
            fence_async_smem();
            arrive(b_h);
            if (warp < 2) {  // v_new for token row r, columns 0..31
                uint4 uv[4];
                load_u(par, r, 0, uv);
                ok = warp_all(wait_sleep(b_a, par, abort));
                tc_fence_after();
                if (ok) vnew_half(c, r, 0, uv);
                fence_async_smem();
                tc_fence_before();
                arrive(b_vn);
                if (!ok) break;
            } else if (c >= 1) {  // the previous chunk's output
                ok = output(c - 1, tid - 64);
                if (!ok) break;
            }
            ok = warp_all(wait_sleep(b_dh, par, abort));
            if (!ok) break;
            const float d = dec_s[(c & 3) * kKP + r];
            tc_fence_after();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float t[32];
                tc_ld32(tmem + lane_base + kColDh + 32 * half, t);
#pragma unroll
                for (int x = 0; x < 32; ++x) h[32 * half + x] = fmaf(d, h[32 * half + x], t[x]);
            }
            tc_fence_before();
        }
        if (ok && warp >= 2 && nchunks > 0) ok = output(nchunks - 1, tid - 64);
        if (ok && p.h_final && r < K) store_row64(p.h_final + (bh * K + r) * p.h_ld, h, v0, p.Vt);
    } else if (warp == 4 || warp == 5) {
        // ------------------------------------- v_new helpers (columns 32..63)
        const int i = tid - 128;
        bool ok = true;
        for (int c = 0; c < nchunks && ok; ++c) {
            const uint32_t par = c & 1;
            ok = warp_all(wait_sleep(b_ia0 + 8 * par, (c >> 1) & 1, abort));
            uint4 uv[4];
            if (ok) load_u(par, i, 32, uv);
            ok = ok && warp_all(wait_sleep(b_a, par, abort));
            tc_fence_after();
            if (ok) vnew_half(c, i, 32, uv);
            fence_async_smem();
            tc_fence_before();
            arrive(b_vn);
        }
    } else if (warp == kIssW) {
        // -------------------------------------------------- chain MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdK = tc_idesc(128, 64, 0, 1);   // A K-major, B MN-major
            constexpr uint32_t kIdMN = tc_idesc(128, 64, 1, 1);  // A and B MN-major
            const uint64_t dH = tc_sdesc(sbase + FL::h, 128, 2048);
            bool ok = true;
            uint32_t last_bar = 0, last_par = 0;  // the last commit issued
            for (int c = 0; c < nchunks && ok; ++c) {
                const uint32_t par = c & 1;
                const uint32_t dcol = kColXO + par * 64;
                const uint64_t dW = tc_sdesc(sbase + FL::wq + par * 2 * kImgW, 128, 2048);
                const uint64_t dK = tc_sdesc(sbase + FL::kg + par * kImgW, 128, 1024);
                const uint64_t dV = tc_sdesc(sbase + FL::vn + par * 8192, 128, 1024);
                ok = wait_sleep(b_ia0 + 8 * par, (c >> 1) & 1, abort) && wait_sleep(b_h, par, abort);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) tc_mma(tmem + dcol, dW + 16 * ks, dH + 16 * ks, kIdK, ks > 0);
                tc_commit(b_a);
                last_bar = b_a, last_par = par;
                ok = wait_sleep(b_ib0 + 8 * par, (c >> 1) & 1, abort) && wait_sleep(b_vn, par, abort);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) tc_mma(tmem + kColDh, dK + 16 * ks, dV + 16 * ks, kIdMN, ks > 0);
                tc_commit(b_dh);
                last_bar = b_dh, last_par = par;
                // chunk c-1's output must be read out before chunk c's is added
                if (c >= 1) ok = wait_sleep(b_of0 + 8 * ((c - 1) & 1), ((c - 1) >> 1) & 1, abort);
                if (!ok) break;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc_mma_ta(tmem + dcol, tmem + kColP + par * 32 + 8 * ks, dV + 16 * ks, kIdK, 1);
                tc_commit(b_o);
                // every product of chunk c is done when this arrives: its slot
                // (and its P buffer) may take chunk c + 2
                tc_commit(b_free0 + 8 * par);
                last_bar = b_free0 + 8 * par, last_par = (c >> 1) & 1;
            }
            if (!ok) {
                *abort = 1;
                if (last_bar) wait_sleep(last_bar, last_par, nullptr);  // MMAs complete in issue order
            }
        }
    } else if (warp >= kEW) {
        // ---------------------------------------------- intra-chunk warps
        const int et = tid - 32 * kEW;  // 0..255
        const int e8 = warp - kEW;      // 0..7
        const int q4 = warp & 3;        // tensor-memory lane quarter
        const int hf = e8 >> 2;         // which half of a row's columns
        const int g8 = lane >> 2, t4 = lane & 3;
        float *const sG = reinterpret_cast<float *>(sm + FL::gates);
        float *const sB = sG + 64, *const sRk = sG + 128, *const sRq = sG + 192;
        float *const sMisc = sG + 256;  // G_last, scaled-Gram flag
        float *const sAd = reinterpret_cast<float *>(sm + FL::ad);
        bf16 *const sAb = reinterpret_cast<bf16 *>(sm + FL::ab);
        bf16 *const sTb = reinterpret_cast<bf16 *>(sm + FL::tb);
        unsigned char *const sTu = sm + FL::tu;
        const int tbase = p.cu_seqlens ? si.tstart : 0;
        const int wcoord = p.cu_seqlens ? 0 : si.b;
        // a value tile wholly past V (the denominator's own tile when V is a
        // multiple of 64) is not loaded: it is zero but for the ones column
        const bool v_in = v0 < V;
        auto issue_qk = [&](int m) {
            const int pos = m * kChunk;
            const int zq = REV ? tbase + len - 64 - pos : tbase + pos;
            const int zk = REV ? tbase + len - 63 - pos : tbase + pos;
            arrive_expect_tx(b_qk, (uint32_t)n_kb * FL::st_kb);
            for (int kb = 0; kb < n_kb; ++kb) {
                tma_load4(sbase + FL::qk + kb * FL::st_kb, &mk, 64 * kb, hh, zk, wcoord, b_qk);
                tma_load4(sbase + FL::qk + kb * FL::st_kb + FL::st_q, &mq, 64 * kb, hh, zq, wcoord, b_qk);
            }
        };
        auto issue_v = [&](int m) {
            const int pos = m * kChunk;
            const int zk = REV ? tbase + len - 63 - pos : tbase + pos;
            const uint32_t bar = b_v0 + 8 * (m & 1);
            arrive_expect_tx(bar, v_in ? 8192u : 0u);
            if (v_in) tma_load4(sbase + FL::v + (m & 1) * 8192, &mv, v0, hh, zk, wcoord, bar);
        };
        // beta and the raw log gate of logical rows 2 lane, 2 lane + 1 of
        // chunk m (warp 8; zero for rows without a token)
        auto load_bg = [&](int m, float (&b)[2], float (&g)[2]) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int pos = m * kChunk + 2 * lane + e;
                const int tk = (m < nchunks && pos < len) ? kv_token(REV, len, pos) : -1;
                b[e] = tk >= 0 ? p.beta[(si.row0 + tk) * H + hh] : 0.f;
                g[e] = tk >= 0 ? p.g[(si.row0 + tk) * H + hh] : 0.f;  // floored when used
            }
        };
        int qk_hi = 0, v_hi = 0;      // chunks whose loads were issued
        int qk_lo = 0, v_lo = 0;      // chunks whose loads were waited for
        if (et == 0 && nchunks > 0) {
            issue_qk(qk_hi++);
            for (; v_hi < 2 && v_hi < nchunks; ++v_hi) issue_v(v_hi);
        }
        // P's rows 0-63 (lanes 0-63) multiply into the Xw half of the
        // accumulator after v_new has read it; keep them zero
        if (q4 < 2) {
            uint32_t z[32];
#pragma unroll
            for (int x = 0; x < 32; ++x) z[x] = 0u;
            tc_st32(tmem + lane_base + kColP + 32 * hf, z);
        }
        float cb[2] = {0.f, 0.f}, cg[2] = {0.f, 0.f}, nb[2], ng[2];
        if (e8 == 0) load_bg(0, cb, cg);
        bool ok = true;
        uint32_t last_bar = 0, last_par = 0;  // the last intra commit
        for (int n = 0; n < nchunks && ok; ++n) {
            const int b = n & 1;
            const uint32_t np = n & 1;
            const int pos0 = n * kChunk;
            const int Lc = min(kChunk, len - pos0);
            unsigned char *const wq_s = sm + FL::wq + b * 2 * kImgW;  // w (X1 first) | qg
            unsigned char *const kg_s = sm + FL::kg + b * kImgW;
            // ---- 1. cumulative gates (warp 8)
            if (e8 == 0) {
                cg[0] = fmaxf(cg[0], kLogGateMin), cg[1] = fmaxf(cg[1], kLogGateMin);
                float incl = cg[0] + cg[1];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                sG[2 * lane] = incl - cg[1];
                sG[2 * lane + 1] = incl;
                sB[2 * lane] = cb[0];
                sB[2 * lane + 1] = cb[1];
                const float gl = __shfl_sync(0xffffffffu, (Lc - 1) & 1 ? incl : incl - cg[1], (Lc - 1) >> 1);
                if (lane == 0) {
                    sMisc[0] = gl;
                    sMisc[1] = -gl <= kScaledGramMaxDecay ? 1.f : 0.f;
                }
            }
            // ---- 2. the chunk's tiles
            ok = wait_sleep(b_qk, np, abort) && wait_sleep(b_v0 + 8 * b, (n >> 1) & 1, abort);
            ok = e_sync_and(ok);
            if (!ok) break;
            qk_lo = v_lo = n + 1;
            if (e8 == 0) load_bg(n + 1, nb, ng);  // used at the next chunk
            const float GL = sMisc[0];
            const bool scaled = sMisc[1] != 0.f;
            const float dec = __expf(GL);
            {  // rows without a token in the v tile are zeroed; the denominator's ones column
                const bool ragged = Lc < kChunk || (REV && pos0 == 0);
                const bool den_tile = p.has_den && v0 <= V && V < v0 + 64;
                if (ragged || den_tile || !v_in) {
                    unsigned char *vs = sm + FL::v + b * 8192;
                    for (int e = et; e < 64 * 8; e += kNE) {
                        const int r = e >> 3, ch = e & 7, li = REV ? 63 - r : r;
                        const bool kv = v_in && li < Lc && (!REV || pos0 + li >= 1);
                        if (!kv) *reinterpret_cast<uint4 *>(vs + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
                    }
                    e_sync();
                    if (den_tile && et < 64) {
                        const int r = et, li = REV ? 63 - r : r;
                        if (li < Lc && (!REV || pos0 + li >= 1)) {
                            const int col = V - v0, ch = col >> 3;
                            *reinterpret_cast<bf16 *>(vs + r * 128 + ((ch ^ (r & 7)) * 16) + (col & 7) * 2) =
                                __float2bfloat16_rn(1.f);
                        }
                    }
                }
            }
            if (REV) {
                // the reverse scan's v tile arrives in shared-row order (row r
                // holds logical position 63 - r); U takes it in logical order:
                // swap rows r and 63 - r, each thread one 16-byte piece of a pair
                e_sync();
                unsigned char *vs = sm + FL::v + b * 8192;
                const int r = et >> 3, ch = et & 7, r2 = 63 - r;
                unsigned char *pa = vs + r * 128 + ((ch ^ (r & 7)) * 16);
                unsigned char *pb = vs + r2 * 128 + ((ch ^ (r2 & 7)) * 16);
                const uint4 xa = *reinterpret_cast<const uint4 *>(pa), xb = *reinterpret_cast<const uint4 *>(pb);
                *reinterpret_cast<uint4 *>(pa) = xb;
                *reinterpret_cast<uint4 *>(pb) = xa;
            }
            // ---- 3. row norms and the scaled rows: thread (row rr, key half kb)
            //         holds the 8 16-byte pieces of its half row; k rows 0-63, q rows 64-127
            const int rr = et >> 1, kb = et & 1;
            const bool is_q = rr >= 64;
            const int r = rr & 63;                 // shared row of the tile
            const int li = REV ? 63 - r : r;       // its logical position in the chunk
            const bool valid = li < Lc && (is_q || !REV || pos0 + li >= 1);
            uint4 x8[8];
            {
                const unsigned char *row = sm + FL::qk + kb * FL::st_kb + (is_q ? FL::st_q : 0u) + r * 128;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) x8[ch] = *reinterpret_cast<const uint4 *>(row + ((ch ^ (r & 7)) * 16));
            }
            float nrm;
            {
                float ss = 0.f;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    float f[8];
                    unpack8(x8[ch], f);
#pragma unroll
                    for (int x = 0; x < 8; ++x) ss = fmaf(f[x], f[x], ss);
                }
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                nrm = p.l2norm ? rsqrtf(ss + 1e-6f) : 1.f;
            }
            if (kb == 0) (is_q ? sRq : sRk)[li] = nrm;
            // the slot of chunk n - 2 (and its P buffer) is free
            if (n >= 2) ok = wait_sleep(b_free0 + 8 * b, ((n - 2) >> 1) & 1, abort);
            ok = e_sync_and(ok);
            if (!ok) break;
            {
                const float Gi = sG[li];
                // scaled Gram: X1 = e^{G - G_last} k^, X2 = kg = e^{G_last - G} k^,
                // qg = e^{G} q^; per-entry form: X1 = k^, X2 = k^, qg = q^ first
                const float s1 = valid ? (scaled ? __expf(Gi - GL) * nrm : nrm) : 0.f;
                const float s2 = valid ? (scaled ? __expf(GL - Gi) * nrm : nrm) : 0.f;
                const float sq = valid ? (scaled ? __expf(Gi) * nrm : nrm) : 0.f;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    float f[8], o[8];
                    unpack8(x8[ch], f);
                    const int d = 64 * kb + 8 * ch;
                    if (is_q) {
#pragma unroll
                        for (int x = 0; x < 8; ++x) o[x] = f[x] * sq;
                        *reinterpret_cast<uint4 *>(wq_s + kImgW + img_w_off(r, d)) = pack8(o);
                    } else {
#pragma unroll
                        for (int x = 0; x < 8; ++x) o[x] = f[x] * s1;
                        *reinterpret_cast<uint4 *>(wq_s + img_w_off(li, d)) = pack8(o);
#pragma unroll
                        for (int x = 0; x < 8; ++x) o[x] = f[x] * s2;
                        *reinterpret_cast<uint4 *>(kg_s + img_kt_off(li, d)) = pack8(o);
                    }
                }
            }
            fence_async_smem();
            e_sync();
            if (et == 0) {
                // the q / k stage is free (the per-entry form rereads it
                // below): load the next chunk; the Gram
                if (scaled) {
                    if (qk_hi < nchunks) issue_qk(qk_hi++);
                    arrive(b_ib0 + 8 * b);  // kg^T of chunk n is final
                }
                tc_fence_after();
                constexpr uint32_t kIdG = tc_idesc(128, 64, 0, 0);
                const uint32_t a0 = sbase + FL::wq + b * 2 * kImgW, b0 = sbase + FL::kg + b * kImgW;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    tc_mma(tmem + kColS, tc_sdesc(a0 + 256 * ks, 128, 2048), tc_sdesc(b0 + 2048 * ks, 1024, 128),
                           kIdG, ks > 0);
                tc_commit(b_gram);
                last_bar = b_gram, last_par = np;
            }
            ok = wait_sleep(b_gram, np, abort);
            ok = e_sync_and(ok);
            if (!ok) break;
            tc_fence_after();
            // ---- 4. A (shared memory) and P (tensor memory) from the Gram
            //         rows; warp (q4, hf) takes lanes 32 q4.. and columns 32 hf..
            {
                float sv[32];
                tc_ld32(tmem + lane_base + kColS + 32 * hf, sv);
                if (q4 < 2) {
                    const int i = 32 * q4 + lane, I = i >> 4;  // logical row
                    const float Gi = sG[i], bi = sB[i];
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const int j0 = 32 * hf + 8 * g;
                        float a[8];
                        if (scaled) {
#pragma unroll
                            for (int y = 0; y < 8; ++y) a[y] = j0 + y < i ? bi * sv[8 * g + y] : 0.f;
                        } else {
                            const float4 G0 = *reinterpret_cast<const float4 *>(sG + j0);
                            const float4 G1 = *reinterpret_cast<const float4 *>(sG + j0 + 4);
                            const float gj[8] = {G0.x, G0.y, G0.z, G0.w, G1.x, G1.y, G1.z, G1.w};
#pragma unroll
                            for (int y = 0; y < 8; ++y) {
                                const float v = bi * sv[8 * g + y] * __expf(fminf(Gi - gj[y], 0.f));
                                a[y] = j0 + y < i ? v : 0.f;
                            }
                        }
                        const int M = j0 >> 4;
                        if (M == I) {
                            float *dd = sAd + (I * 16 + (i & 15)) * kAdS + (j0 & 15);
                            *reinterpret_cast<float4 *>(dd) = make_float4(a[0], a[1], a[2], a[3]);
                            *reinterpret_cast<float4 *>(dd + 4) = make_float4(a[4], a[5], a[6], a[7]);
                        } else if (M < I) {
                            *reinterpret_cast<uint4 *>(sAb + (blk(I, M) * 16 + (i & 15)) * kBS + (j0 & 15)) = pack8(a);
                        }
                    }
                } else {
                    const int m = 32 * (q4 - 2) + lane, i = REV ? 63 - m : m;  // shared row, logical row
                    const float Gi = sG[i], inv_dec = __expf(-GL);
                    uint32_t pr[16];
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const int j0 = 32 * hf + 8 * g;
                        float pv[8];
                        if (scaled) {
#pragma unroll
                            for (int y = 0; y < 8; ++y) pv[y] = j0 + y <= i ? sv[8 * g + y] * inv_dec : 0.f;
                        } else {
                            const float4 G0 = *reinterpret_cast<const float4 *>(sG + j0);
                            const float4 G1 = *reinterpret_cast<const float4 *>(sG + j0 + 4);
                            const float gj[8] = {G0.x, G0.y, G0.z, G0.w, G1.x, G1.y, G1.z, G1.w};
#pragma unroll
                            for (int y = 0; y < 8; ++y) {
                                const float v = sv[8 * g + y] * __expf(fminf(Gi - gj[y], 0.f));
                                pv[y] = j0 + y <= i ? v : 0.f;
                            }
                        }
#pragma unroll
                        for (int y = 0; y < 4; ++y) pr[4 * g + y] = pack_bf16(pv[2 * y], pv[2 * y + 1]);
                    }
                    tc_st16(tmem + lane_base + kColP + np * 32 + 16 * hf, pr);
                }
            }
            if (!scaled) {
                // per-entry form: the chain's operands get their gates now
                // (X1 -> e^{G} k^, qg -> e^{G} q^, kg -> e^{G_last - G} k^),
                // from the rows of the q / k stage
                {
                    const unsigned char *row = sm + FL::qk + kb * FL::st_kb + (is_q ? FL::st_q : 0u) + r * 128;
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch)
                        x8[ch] = *reinterpret_cast<const uint4 *>(row + ((ch ^ (r & 7)) * 16));
                }
                const float Gi = sG[li];
                const float s1 = valid ? __expf(Gi) * nrm : 0.f;
                const float s2 = valid ? __expf(GL - Gi) * nrm : 0.f;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    float f[8], o[8];
                    unpack8(x8[ch], f);
                    const int d = 64 * kb + 8 * ch;
#pragma unroll
                    for (int x = 0; x < 8; ++x) o[x] = f[x] * s1;
                    if (is_q) {
                        *reinterpret_cast<uint4 *>(wq_s + kImgW + img_w_off(r, d)) = pack8(o);
                    } else {
                        *reinterpret_cast<uint4 *>(wq_s + img_w_off(li, d)) = pack8(o);
#pragma unroll
                        for (int x = 0; x < 8; ++x) o[x] = f[x] * s2;
                        *reinterpret_cast<uint4 *>(kg_s + img_kt_off(li, d)) = pack8(o);
                    }
                }
                fence_async_smem();
            }
            tc_fence_before();
            e_sync();
            if (!scaled && et == 0) {
                arrive(b_ib0 + 8 * b);  // kg^T of chunk n is final
                if (qk_hi < nchunks) issue_qk(qk_hi++);
            }
            // ---- 5. T = (I + A)^{-1}, written as T diag(beta)
            auto put_frag = [&](int I, int J, const float (&acc)[2][4]) {
                float2 su[2];
#pragma unroll
                for (int nn = 0; nn < 2; ++nn) su[nn] = *reinterpret_cast<const float2 *>(sB + 16 * J + 8 * nn + 2 * t4);
#pragma unroll
                for (int nn = 0; nn < 2; ++nn)
#pragma unroll
                    for (int hf2 = 0; hf2 < 2; ++hf2) {
                        const int i = 16 * I + g8 + 8 * hf2, j = 16 * J + 8 * nn + 2 * t4;
                        *reinterpret_cast<uint32_t *>(sTu + img_p_off(i, j)) =
                            pack_bf16(acc[nn][2 * hf2] * su[nn].x, acc[nn][2 * hf2 + 1] * su[nn].y);
                    }
            };
            if (hf == 0) {  // level 1: warp q4 inverts diagonal block q4 (lane cc holds column cc)
                const int I = q4, cc = lane & 15;
                const float *Ad = sAd + I * 16 * kAdS;
                float t[16];
#pragma unroll
                for (int rr2 = 0; rr2 < 16; ++rr2) t[rr2] = (rr2 == cc) ? 1.f : 0.f;
#pragma unroll
                for (int rr2 = 1; rr2 < 16; ++rr2) {
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};  // independent partial sums
#pragma unroll
                    for (int j = 0; j < rr2; ++j) acc[j & 3] = fmaf(Ad[rr2 * kAdS + j], t[j], acc[j & 3]);
                    if (rr2 > cc) t[rr2] = -((acc[0] + acc[1]) + (acc[2] + acc[3]));
                }
                if (lane < 16) {
                    const int j = 16 * I + cc;
                    const float su = sB[j];
#pragma unroll
                    for (int rr2 = 0; rr2 < 16; ++rr2) {
                        sTb[((kTbT + I) * 16 + rr2) * kBS + cc] = __float2bfloat16_rn(t[rr2]);
                        *reinterpret_cast<bf16 *>(sTu + img_p_off(16 * I + rr2, j)) = __float2bfloat16_rn(t[rr2] * su);
                    }
                }
            }
            e_sync();
            if (e8 < 2) {  // level 2: T_10 = -T_11 A_10 T_00, T_32 = -T_33 A_32 T_22
                const int I = e8 == 0 ? 1 : 3, J = I - 1;
                float x[2][4] = {}, y[2][4] = {};
                blk_mma(x, sAb + blk(I, J) * 16 * kBS, sTb + (kTbT + J) * 16 * kBS, false, lane);
                bf16 *tmp = sTb + (kTbY + e8) * 16 * kBS;
                blk_store(tmp, x, lane);
                __syncwarp();
                blk_mma(y, sTb + (kTbT + I) * 16 * kBS, tmp, true, lane);
                blk_store(sTb + (e8 == 0 ? kTb10 : kTb32) * 16 * kBS, y, lane);
                put_frag(I, J, y);
            }
            e_sync();
            if (e8 < 4) {  // level 3a: Y = A_(2,3)(0,1) T_(0,1)(0,1)
                float y[2][4] = {};
                const bf16 *T00 = sTb + (kTbT + 0) * 16 * kBS, *T11 = sTb + (kTbT + 1) * 16 * kBS;
                const bf16 *T10 = sTb + kTb10 * 16 * kBS;
                const int I = 2 + (e8 >> 1);  // A rows block 2 (Y0x) or 3 (Y1x)
                if ((e8 & 1) == 0) {          // Y_x0 = A_I0 T00 + A_I1 T10
                    blk_mma(y, sAb + blk(I, 0) * 16 * kBS, T00, false, lane);
                    blk_mma(y, sAb + blk(I, 1) * 16 * kBS, T10, false, lane);
                } else {  // Y_x1 = A_I1 T11
                    blk_mma(y, sAb + blk(I, 1) * 16 * kBS, T11, false, lane);
                }
                blk_store(sTb + (kTbY + e8) * 16 * kBS, y, lane);
            }
            e_sync();
            if (e8 < 4) {  // level 3b: T_2x = -T22 Y_0x, T_3x = -(T32 Y_0x + T33 Y_1x)
                float y[2][4] = {};
                const int col = e8 & 1;  // x
                const bf16 *Y0 = sTb + (kTbY + col) * 16 * kBS, *Y1 = sTb + (kTbY + 2 + col) * 16 * kBS;
                if (e8 < 2) {
                    blk_mma(y, sTb + (kTbT + 2) * 16 * kBS, Y0, true, lane);
                    put_frag(2, col, y);
                } else {
                    blk_mma(y, sTb + kTb32 * 16 * kBS, Y0, true, lane);
                    blk_mma(y, sTb + (kTbT + 3) * 16 * kBS, Y1, true, lane);
                    put_frag(3, col, y);
                }
            }
            fence_async_smem();
            e_sync();
            // ---- 6. W = T diag(beta) X1 (128 key columns), U = T diag(beta) V
            if (et == 0) {
                tc_fence_after();
                const uint32_t a0 = sbase + FL::tu, x1 = sbase + FL::wq + b * 2 * kImgW;
                constexpr uint32_t kIdW = tc_idesc(64, 128, 0, 1), kIdU = tc_idesc(64, 64, 0, 1);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc_mma(tmem + kColW, tc_sdesc(a0 + 256 * ks, 128, 1024), tc_sdesc(x1 + 4096 * ks, 2048, 128), kIdW,
                           ks > 0);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc_mma(tmem + kColU, tc_sdesc(a0 + 256 * ks, 128, 1024),
                           sdesc_sw128(sbase + FL::v + b * 8192 + 2048 * ks), kIdU, ks > 0);
                tc_commit(b_wu);
                last_bar = b_wu, last_par = np;
            }
            ok = wait_sleep(b_wu, np, abort);
            ok = e_sync_and(ok);
            if (!ok) break;
            tc_fence_after();
            // ---- 7. w (over X1), u and dec; then the chain may take chunk n
            {
                const float ws = scaled ? dec : 1.f;  // the scaled form's W is w / e^{G_last}
#pragma unroll 1
                for (int q = 0; q < 2; ++q) {
                    float t[32];
                    tc_ld32(tmem + lane_base + kColW + 64 * hf + 32 * q, t);
                    if (lane < 16) {
                        const int i = 16 * q4 + lane;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            float f[8];
#pragma unroll
                            for (int x = 0; x < 8; ++x) f[x] = t[8 * j + x] * ws;
                            *reinterpret_cast<uint4 *>(wq_s + img_w_off(i, 64 * hf + 32 * q + 8 * j)) = pack8(f);
                        }
                    }
                }
                float t[32];
                tc_ld32(tmem + lane_base + kColU + 32 * hf, t);
                if (lane < 16) {
                    const int i = 16 * q4 + lane;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *reinterpret_cast<uint4 *>(sm + FL::u + b * kImgU + img_u_off(i, 32 * hf + 8 * j)) =
                            pack8(&t[8 * j]);
                }
            }
            if (et < 128) dec_s[(n & 3) * kKP + et] = dec;
            fence_async_smem();
            tc_fence_before();
            e_sync();
            if (et == 0) {
                arrive(b_ia0 + 8 * b);
                // the v stage of chunk n is free: chunk n + 2
                if (v_hi < nchunks) issue_v(v_hi++);
            }
            if (e8 == 0) {
                cb[0] = nb[0], cb[1] = nb[1], cg[0] = ng[0], cg[1] = ng[1];
            }
        }
        if (!ok) {
            *abort = 1;
            if (et == 0) {  // drain: the tile loads in flight and the last intra MMAs
                for (int m = qk_lo; m < qk_hi; ++m) wait_sleep(b_qk, m & 1, nullptr);
                for (int m = v_lo; m < v_hi; ++m) wait_sleep(b_v0 + 8 * (m & 1), (m >> 1) & 1, nullptr);
                if (last_bar) wait_sleep(last_bar, last_par, nullptr);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0 && *abort) atomicOr(p.err, kDevErrTimeout);
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

// ----------------------------------------------------------- tensor maps

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// A (D, H, T, B) bf16 view with element strides (sh, st, sb), boxes of 64
// rows of one head x 64 elements, 128-byte swizzle, zero fill outside
bool make_map(CUtensorMap *m, const void *ptr, int D, int H, int T, int B, int64_t sh, int64_t st, int64_t sb) {
    auto fn = encode_fn();
    if (!fn || T < 1) return false;
    const int64_t sb_b = B > 1 ? sb * 2 : ((int64_t)T * st * 2 + 15) / 16 * 16;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)(sh * 2), (cuuint64_t)(st * 2), (cuuint64_t)sb_b};
    for (int i = 0; i < 3; ++i)
        if (strides[i] == 0 || strides[i] % 16 != 0 || strides[i] >= (1ull << 40)) return false;
    cuuint32_t box[4] = {64, 1, 64, 1}, es[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

std::atomic<int> g_fused{0};

}  // namespace

void set_fused(int on) { g_fused.store(on ? 1 : 0); }

bool fused_prepare(const FwdParams &p, FusedMaps *m) {
    if (!g_fused.load() || p.gk != nullptr || p.g == nullptr || p.summary || p.seg_chunks != 0 || p.h_in ||
        p.h_snap || p.K > 128 || p.out == nullptr || p.T < 1)
        return false;
    const int B = p.cu_seqlens ? 1 : p.B;
    return make_map(&m->q, p.q, p.K, p.H, p.T, B, p.qk_sh, p.qk_st, p.qk_sb) &&
           make_map(&m->k, p.k, p.K, p.H, p.T, B, p.qk_sh, p.qk_st, p.qk_sb) &&
           make_map(&m->v, p.v, p.V, p.H, p.T, B, p.v_sh, p.v_st, p.v_sb);
}

cudaError_t launch_fused_tc(const FwdParams &p, const FusedMaps &m, cudaStream_t st) {
    auto kern = p.stall_cta >= 0 ? (p.reverse ? fused_tc_kernel<true, true> : fused_tc_kernel<false, true>)
                                 : (p.reverse ? fused_tc_kernel<true, false> : fused_tc_kernel<false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)FL::alloc);
    if (e != cudaSuccess) return e;
    const int grid = p.n_seq * p.H * p.n_vt;
    if (grid == 0) return cudaSuccess;
    kern<<<grid, kThreads, FL::alloc, st>>>(p, m.q, m.k, m.v);
    return cudaGetLastError();
}

}  // namespace gdn
