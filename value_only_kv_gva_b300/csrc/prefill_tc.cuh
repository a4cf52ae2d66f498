// prefill_tc.cuh -- causal chunked prefill on the fifth-generation tensor cores.
//
// Every new token of a chunk attends to the cached history and to the chunk up to and
// including itself (MQA/GQA page §1; GVA analysis page, 关键技巧一/二 for the scores:
// z = q~_h . v_{j,g(h)} + q^_h . k_rope_j).  The chunk's queries of one value group share
// that group's rows (MQA/GQA page §6.1), so one CTA per (history range, value group,
// sequence) holds the group's n r query rows and streams 128-token tiles of its rows once:
//
//   S[M x 128] = Q~ V_g^T + Q^ K_rope^T          tcgen05.mma, fp32 in tensor memory
//   online softmax in log2 units, a quarter of a query row per thread (tcgen05.ld)
//   O[M x d_h] += P V_g                          tcgen05.mma, O resident in tensor memory
//
// M = 64 (n r <= 64) or 128 rows.  The fp32 queries and probabilities enter as bf16 high
// and low parts (about 16 bits kept).  The query parts accumulate into the same S columns.
// With M = 64 the probability parts are stacked into one 128-row operand, so O += P V is
// one 128-row product per k-step: the high part of row r lands in tensor-memory lane
// 32 (r / 16) + r % 16 and the low part 16 lanes further, in the lane quadrant of the
// warps that own score row r, and the two are summed once at the end.
// The value tile is the B operand of both products: K-major (tokens x d_h) for the
// scores, MN-major for P V.  The positional keys come in as a 64-wide box of which the
// columns past d_r are zero (out of the tensor's bounds), matching zero columns of Q^;
// it is 16 (32-byte swizzle) or 32 (64-byte swizzle) columns wide.
// Warps: 0-15 softmax (four per tensor-memory lane quadrant, a quarter of the columns
// each), 16 the TMA producer, 17 the MMA issuer.  The ranges' partials use the layout of the mma.sync prefill kernel and its
// log-sum-exp merge (prefill_mma.cuh).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "decode_mma.cuh"
#include "decode_rope_keys.cuh"
#include "prefill_mma.cuh"

namespace gva {

constexpr int PT_TILE = 128;
constexpr int PT_SWARPS = 16;   // softmax warps: four per tensor-memory lane quadrant
constexpr int PT_THREADS = (PT_SWARPS + 2) * 32;
constexpr int PT_MAX_STAGES = 8;

struct PrefillTcParams {
    PrefillMmaParams p;   // shapes, inputs, partial layout (splits, wpg, rows_pad)
    int ch;               // cache rows per TMA box
    int nstages;
    int smem_bytes;
    int *tickets;         // [B][G], zero at launch: the last CTA of each (value group,
                          //   sequence) merges its ranges; null: a merge kernel follows
    int by_length;        // 1: the kernel instance in which CTA z takes the sequence with
                          //   the z-th most tiles (B <= PT_ORDER_MAX), so that the longest
                          //   ranges start first
};

constexpr int PT_ORDER_MAX = 256;

// Shared-memory matrix descriptor: layout 2 = 128-byte swizzle (rows of 128 B), 4 = 64-byte,
// 6 = 32-byte; sbo = bytes between groups of 8 rows, lbo = bytes between 64-element blocks
// along the contiguous dimension of an MN-major operand.
__device__ __forceinline__ uint64_t pt_sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                             uint32_t layout = 2) {
    uint64_t d = (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)layout << 61;
    return d;
}
// bf16 A and B, fp32 D; b_mn: B is MN-major (N contiguous)
__host__ __device__ constexpr uint32_t pt_idesc(int M, int N, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t *v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
          "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
          "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
        "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
        "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15])
        : "memory");
}
// 16 lanes x 256 bits per repeat: thread t gets lanes t/4 and 8 + t/4, columns 2 (t % 4)
// and 2 (t % 4) + 1 of each 8-column block (registers 4 j + 0, 1 and 4 j + 2, 3).
__device__ __forceinline__ void tc_ld16x256_x4(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tc_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// 2^x by the hardware approximation (relative error about 2^-22, far below the bf16
// split of P that follows); subnormal results flush to zero.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// Probability pair (x0, x1) >= 0 as bf16 high parts taken by truncation (the upper halves
// of the fp32 words: one byte permute) and the remainders x - hi (exact in fp32) rounded
// to bf16: hi + lo keeps about 16 bits, with one conversion per pair instead of two.
__device__ __forceinline__ void split_bf16_trunc(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const uint32_t u0 = __float_as_uint(x0), u1 = __float_as_uint(x1);
    hi = __byte_perm(u0, u1, 0x7632);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - __uint_as_float(u0 & 0xffff0000u),
                                                   x1 - __uint_as_float(u1 & 0xffff0000u));
    lo = *reinterpret_cast<const uint32_t *>(&l);
}
// Byte offset of the 16-byte chunk holding elements 8 c .. 8 c + 7 of row r of a K-major
// tile with `rows` rows, in 64-element (128-byte) swizzled blocks.
__device__ __forceinline__ uint32_t pt_chunk(int r, int c, int rows) {
    return (uint32_t)((c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// 128-token tiles of sequence b once the chunk is appended: positions up to L0[b] + n,
// capped by the capacity; none when L0[b] is out of range (the kernel's own rule).
__device__ __forceinline__ int pt_tiles(const PrefillMmaParams &p, int b) {
    const long long l0 = p.L0[b];
    const long long cap = min(seq_capacity(p.R, b), 0x7fffffffLL);
    const long long Lt = (l0 >= 0 && l0 <= cap) ? min(l0 + p.n, cap) : 0;
    return (int)((Lt + PT_TILE - 1) / PT_TILE);
}

// The sequence CTA z of the grid takes when the grid is ordered by length: sequences
// ranked by tile count, most first, ties by index (a permutation).  The tile counts are
// staged in `scratch` (B + 1 ints).  Called by every thread of the CTA.
__device__ __forceinline__ int pt_seq_by_length(const PrefillMmaParams &p, int *scratch, int tid,
                                                int nthreads) {
    for (int bb = tid; bb < p.B; bb += nthreads) scratch[bb] = pt_tiles(p, bb);
    __syncthreads();
    for (int bb = tid; bb < p.B; bb += nthreads) {
        const int t = scratch[bb];
        int rank = 0;
        for (int o = 0; o < p.B; ++o) {
            const int u = scratch[o];
            rank += (u > t || (u == t && o < bb)) ? 1 : 0;
        }
        if (rank == (int)blockIdx.z) scratch[p.B] = bb;   // exactly one thread
    }
    __syncthreads();
    return scratch[p.B];
}

template <int DH, int DR, int M>
struct PtSmem {
    static constexpr int KQ = DH / 64 + (DR > 0 ? 1 : 0);   // 64-wide K-blocks of a query row
    static constexpr int QPART = KQ * M * 128;               // one of the two query parts
    static constexpr int PPART = 2 * M * 128;                // P part: 128 tokens
    static constexpr int VT = RK_TILE * DH * 2;              // value tile
    // positional tile: 16 columns in 32-byte rows (d_r <= 16) or 32 in 64-byte rows
    static constexpr int KRW = DR <= 16 ? 16 : 32;
    static constexpr int KT = DR > 0 ? RK_TILE * KRW * 2 : 0;
    static constexpr int STAGE = VT + KT;
    static constexpr int XM = 2 * 4 * 4 * 32 * 4;            // row max parts [buf][quad][part][32]
    static constexpr int LS = 4 * 4 * 32 * 4;                // row sum parts [quad][part][32]
    // two P buffers (the products of tile k - 1 run while the softmax of tile k writes
    // its P) when four stages still fit beside them; otherwise the stages come first:
    // with two stages only one tile is in flight while the other is scored
    static constexpr int PB = 1024 + 2 * QPART + 4 * PPART + 4 * STAGE + XM + LS + 256 <= MMA_SMEM_LIMIT ? 2 : 1;
    static constexpr int fixed = 2 * QPART + PB * 2 * PPART + XM + LS;
};

// Warps 0-15 run the softmax: warp w reads tensor-memory lane quadrant q = w & 3 and
// handles quarter pt = w >> 2 of each tile's 128 columns and of O's d_h columns; the four
// warps of a quadrant exchange their rows' partial maxima (a 128-thread barrier).  Warp 16
// is the TMA producer, warp 17 the MMA issuer.
template <int DH, int DR, int M, bool ORD>
__global__ void __launch_bounds__(PT_THREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_k, const PrefillTcParams tp) {
    using SM = PtSmem<DH, DR, M>;
    constexpr int KB = DH / 64;
    constexpr int KR = (DR + 15) / 16;          // positional k-steps
    constexpr int PB = SM::PB;
    constexpr int TCOLS = 512;                  // S x 2 (128 each) + O (d_h)
    constexpr uint32_t O_COL = 256;
    const PrefillMmaParams &p = tp.p;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    unsigned char *sm = smem_raw + (base - raw_u32);
    const int ns = tp.nstages;
    const uint32_t q_s = base;                               // Q hi, Q lo
    const uint32_t p_s = q_s + 2 * SM::QPART;                // P buffers: hi, lo each
    const uint32_t st_s = p_s + PB * 2 * SM::PPART;          // value (+ positional) stages
    unsigned char *p8 = sm + 2 * SM::QPART;
    float *xm = reinterpret_cast<float *>(sm + (st_s - base) + ns * SM::STAGE);
    float *lsh = xm + SM::XM / 4;
    const uint32_t bars = st_s + ns * SM::STAGE + SM::XM + SM::LS;
    const uint32_t bar_full = bars, bar_empty = bars + 8 * ns;
    const uint32_t bar_sfull = bar_empty + 8 * ns, bar_sfree = bar_sfull + 16;
    const uint32_t bar_pfull = bar_sfree + 16, bar_pvdone = bar_pfull + 16;
    const uint32_t bar_done = bar_pvdone + 16;
    unsigned char *tail = sm + (bars - base) + (2 * ns + 9) * 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tail);
    volatile int *abort = reinterpret_cast<volatile int *>(tail + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, g = blockIdx.y;
    // ORD: CTAs start in block order, so CTA z takes the sequence with the z-th most tiles
    // (its tile counts staged in the first ring stage, which no copy has reached yet; the
    // start positions and capacities are inputs no kernel of the call writes)
    const int b = ORD ? pt_seq_by_length(p, reinterpret_cast<int *>(sm + (st_s - base)), tid,
                                         PT_THREADS)
                      : (int)blockIdx.z;
    const int nrows = p.n * p.r;
    if (tid == 0) GVA_TRACE_AT(0);
    if (tid == 0) {
        for (int s = 0; s < ns; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar_sfull + 8 * s, 1);
            mbar_init(bar_sfree + 8 * s, PT_SWARPS);
            mbar_init(bar_pfull + 8 * s, PT_SWARPS);
            mbar_init(bar_pvdone + 8 * s, 1);
        }
        mbar_init(bar_done, 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == PT_SWARPS && lane == 0) {
        prefetch_tmap(&tm_v);
        if (DR > 0) prefetch_tmap(&tm_k);
    }
    pdl_wait();
    pdl_launch_dependents();
    if (tid == 0) GVA_TRACE_AT(1);

    // this sequence's tokens once the chunk is appended (those past the capacity were
    // skipped by the append; their queries see nothing), and this CTA's range of tiles
    const long long l0 = p.L0[b];
    const long long cap = min(seq_capacity(p.R, b), 0x7fffffffLL);
    const bool l0_ok = l0 >= 0 && l0 <= cap;
    const long long Lt = l0_ok ? min(l0 + p.n, cap) : 0;
    if ((!l0_ok || l0 + p.n > cap) && split == 0 && g == 0 && tid == 0) dev_report(GVA_DEV_BAD_LENGTH);
    const int nt = (int)((Lt + PT_TILE - 1) / PT_TILE);
    const int per = (nt + p.splits - 1) / p.splits;
    const int k0 = min(nt, split * per), k1 = min(nt, k0 + per);
    const int ntile = k1 - k0;

    // the group's query rows: row q = i r + hl (head g r + hl of query i), as bf16 high and
    // low parts, the positional part in the last 64-wide K-block (zero past d_r); rows
    // past n r are zero
    for (int e = tid; e < M * SM::KQ * 8; e += PT_THREADS) {
        const int r = e / (SM::KQ * 8), c = e - r * (SM::KQ * 8);   // 16-byte chunk c of row r
        float x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = 0.f;
        if (r < nrows) {
            const int i = r / p.r, h = g * p.r + (r - i * p.r);
            const long long ent = (long long)b * p.n + i;
            const int col = c * 8;
            if (col < DH) {
                const float4 *src = reinterpret_cast<const float4 *>(p.qt + (ent * p.H + h) * DH + col);
                const float4 a = src[0], bq = src[1];
                x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
                x[4] = bq.x; x[5] = bq.y; x[6] = bq.z; x[7] = bq.w;
            } else if (DR > 0) {
                const int rc = col - DH;
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (rc + u < DR) x[u] = p.qh[(ent * p.H + h) * DR + rc + u];
            }
        }
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) split_bf16(x[2 * u], x[2 * u + 1], hw[u], lw[u]);
        const uint32_t off = pt_chunk(r, c, M);
        *reinterpret_cast<uint4 *>(sm + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4 *>(sm + SM::QPART + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");

    if (warp == PT_SWARPS + 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(TCOLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (tid == 0) GVA_TRACE_AT(2);

    if (warp == PT_SWARPS) {
        // ------------------------------ producer ------------------------------ //
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            const int nbox = PT_TILE / tp.ch;
            int k = 0;
            for (; k < ntile; ++k) {
                const int sl = k % ns;
                if (k >= ns && !mbar_wait(bar_empty + 8 * sl, (uint32_t)((k / ns) - 1) & 1u, abort)) break;
                const long long j0 = (long long)(k0 + k) * PT_TILE;
                const int nv = (int)min((long long)PT_TILE, Lt - j0);
                long long rows[PT_TILE / 16];
                int nl = 0;
                for (int c = 0; c < nbox; ++c) {
                    rows[c] = -2;
                    if (c * tp.ch < nv) {
                        rows[c] = row_of(p.R, b, j0 + c * tp.ch);
                        if (rows[c] == -1) dev_report(GVA_DEV_BAD_PAGE);
                        if (rows[c] >= 0) ++nl;
                    }
                }
                const uint32_t fb = bar_full + 8 * sl;
                mbar_expect_tx(fb, (uint32_t)(nl * tp.ch * (128 * KB + (DR > 0 ? SM::KRW * 2 : 0))));
                const uint32_t dst = st_s + sl * SM::STAGE;
                for (int c = 0; c < nbox; ++c) {
                    if (rows[c] < 0) continue;
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb)
                        tma_load_2d(dst + kb * (PT_TILE * 128) + c * tp.ch * 128, &tm_v,
                                    g * DH + kb * 64, (int)rows[c], fb, pol);
                    if (DR > 0)
                        tma_load_2d(dst + SM::VT + c * tp.ch * (SM::KRW * 2), &tm_k, 0, (int)rows[c], fb, pol);
                }
                GVA_TRACE_AT(200 + k);
            }
            for (int i = (k > ns ? k - ns : 0); i < k; ++i)
                rk_drain(bar_full + 8 * (i % ns), (uint32_t)(i / ns) & 1u);
        }
    } else if (warp == PT_SWARPS + 1) {
        // ------------------------------ MMA issuer ------------------------------ //
        if (lane == 0) {
            constexpr uint32_t id_s = pt_idesc(M, PT_TILE, 0);
            constexpr uint32_t id_o = pt_idesc(M == 64 ? 128 : M, DH, 1);
            const uint64_t qd = pt_sdesc(q_s, 16, 1024);
            // descriptors are built once per buffer; an operand offset within a buffer is
            // added to the descriptor's address field (bytes / 16; addresses stay < 256 KB)
            auto pv = [&](int k) -> bool {   // O += P V of tile k (P hi and lo)
                if (!mbar_wait(bar_pfull + 8 * (k & 1), (uint32_t)(k >> 1) & 1u, abort)) return false;
                tc_fence_after();
                const uint64_t pd = pt_sdesc(p_s + (k % PB) * 2 * SM::PPART, 16, 1024);
                const uint64_t vd = pt_sdesc(st_s + (k % ns) * SM::STAGE, PT_TILE * 128, 1024);
                if constexpr (M == 64) {
                    // the stacked parts: 128 rows per 64-token K-block
#pragma unroll
                    for (int kk = 0; kk < PT_TILE / 16; ++kk)
                        tc_mma(tmem + O_COL, pd + (uint64_t)(((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4),
                               vd + (uint64_t)((kk * 2048) >> 4), id_o, (k > 0 || kk > 0) ? 1u : 0u);
                } else {
#pragma unroll
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int kk = 0; kk < PT_TILE / 16; ++kk)
                            tc_mma(tmem + O_COL,
                                   pd + (uint64_t)((part * SM::PPART + (kk >> 2) * (M * 128) + (kk & 3) * 32) >> 4),
                                   vd + (uint64_t)((kk * 2048) >> 4), id_o,
                                   (k > 0 || part > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(bar_pvdone + 8 * (k & 1));
                tc_commit(bar_empty + 8 * (k % ns));
                return true;
            };
            int k = 0;
            bool ok = true;
            for (; k < ntile && ok; ++k) {
                const int sl = k % ns, sb = k & 1;
                ok = mbar_wait(bar_full + 8 * sl, (uint32_t)(k / ns) & 1u, abort);
                if (ok && k >= 2) ok = mbar_wait(bar_sfree + 8 * sb, (uint32_t)((k >> 1) - 1) & 1u, abort);
                if (!ok) break;
                tc_fence_after();
                const uint32_t vt = st_s + sl * SM::STAGE;
                const uint32_t d = tmem + sb * PT_TILE;
                const uint64_t vd = pt_sdesc(vt, 16, 1024);
                const uint64_t kd = pt_sdesc(vt + SM::VT, 16, 8 * SM::KRW * 2, SM::KRW == 16 ? 6u : 4u);
#pragma unroll
                for (int part = 0; part < 2; ++part) {
#pragma unroll
                    for (int kk = 0; kk < DH / 16; ++kk)
                        tc_mma(d, qd + (uint64_t)((part * SM::QPART + (kk >> 2) * (M * 128) + (kk & 3) * 32) >> 4),
                               vd + (uint64_t)(((kk >> 2) * (PT_TILE * 128) + (kk & 3) * 32) >> 4), id_s,
                               (part > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                    for (int kk = 0; kk < KR; ++kk)
                        tc_mma(d, qd + (uint64_t)((part * SM::QPART + KB * (M * 128) + kk * 32) >> 4),
                               kd + (uint64_t)((kk * 32) >> 4), id_s, 1u);
                }
                tc_commit(bar_sfull + 8 * sb);
                GVA_TRACE_AT(10 + 3 * k);
                if (k >= 1) ok = pv(k - 1);
                GVA_TRACE_AT(11 + 3 * k);
            }
            if (ok && ntile > 0) pv(ntile - 1);
            // every product issued has completed before the tensor memory is freed
            tc_commit(bar_done);
            rk_drain(bar_done, 0);
        }
    } else {
        // ------------------------------ softmax ------------------------------ //
        if constexpr (M == 64) {
        // M = 64: rows 16 q .. 16 q + 15 sit in lanes 0-15 of quadrant q; the 16x256b loads
        // spread them over all 32 threads: thread t holds rows A = 16 q + t/4 and
        // B = A + 8, column pairs 2 (t % 4) + {0, 1} of each 8-column block of the warp's
        // quarter (32 columns) of the tile
        const int q = warp & 3, pt = warp >> 2;
        const int tq = lane >> 2, tc = lane & 3;
        const int rA = 16 * q + tq, rB = rA + 8;
        const bool hA = rA < nrows, hB = rB < nrows;
        const long long limA = (hA && l0 + rA / p.r < Lt) ? l0 + rA / p.r : -1;
        const long long limB = (hB && l0 + rB / p.r < Lt) ? l0 + rB / p.r : -1;
        const uint32_t tq0 = tmem + ((uint32_t)(32 * q) << 16);
        const int cb = 32 * pt + 2 * tc;   // tile column of register 0
        float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
        bool ok = true;
        for (int k = 0; k < ntile; ++k) {
            const int sb = k & 1, sl = k % ns, pbuf = k % PB;
            const long long j0 = (long long)(k0 + k) * PT_TILE;
            const int nv = (int)min((long long)PT_TILE, Lt - j0);
            ok = ok && mbar_wait(bar_sfull + 8 * sb, (uint32_t)(k >> 1) & 1u, abort);
            ok = __all_sync(0xffffffffu, ok);
            if (tid == 0) GVA_TRACE_AT(100 + 3 * k);
            uint32_t v[16];
            if (ok) {
                tc_fence_after();
                tc_ld16x256_x4(tq0 + sb * PT_TILE + 32 * pt, v);
                tc_wait_ld();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_sfree + 8 * sb);
            // last visible tile column of rows A and B, clamped to [-1, 127]
            const int vA = (int)max(-1LL, min((long long)PT_TILE - 1, limA - j0));
            const int vB = (int)max(-1LL, min((long long)PT_TILE - 1, limB - j0));
            // the warp's whole quarter visible to all its rows (every history tile)
            const bool whole = __all_sync(0xffffffffu, vA >= cb + 31 - 2 * tc && vB >= cb + 31 - 2 * tc);
            float xA = -INFINITY, xB = -INFINITY;
            if (whole) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        xA = fmaxf(xA, __uint_as_float(v[4 * j + e]));
                        xB = fmaxf(xB, __uint_as_float(v[4 * j + 2 + e]));
                    }
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int col = cb + 8 * j + e;
                        if (col <= vA) xA = fmaxf(xA, __uint_as_float(v[4 * j + e]));
                        if (col <= vB) xB = fmaxf(xB, __uint_as_float(v[4 * j + 2 + e]));
                    }
            }
            xA = fmaxf(xA, __shfl_xor_sync(0xffffffffu, xA, 1));
            xB = fmaxf(xB, __shfl_xor_sync(0xffffffffu, xB, 1));
            xA = fmaxf(xA, __shfl_xor_sync(0xffffffffu, xA, 2));
            xB = fmaxf(xB, __shfl_xor_sync(0xffffffffu, xB, 2));
            float *xw = xm + (sb * 4 + q) * 64;   // [part][16 rows]
            if (tc == 0) {
                xw[pt * 16 + tq] = xA;
                xw[pt * 16 + 8 + tq] = xB;
            }
            named_sync(1 + q, 128);
            if (tid == 0) GVA_TRACE_AT(101 + 3 * k);
            const float tA = fmaxf(fmaxf(xw[tq], xw[16 + tq]), fmaxf(xw[32 + tq], xw[48 + tq]));
            const float tB = fmaxf(fmaxf(xw[8 + tq], xw[24 + tq]), fmaxf(xw[40 + tq], xw[56 + tq]));
            float aA = 1.f, aB = 1.f;
            if (tA > mA + RK_RESCALE_TH) {
                aA = exp2f(mA - tA);
                mA = tA;
            }
            if (tB > mB + RK_RESCALE_TH) {
                aB = exp2f(mB - tB);
                mB = tB;
            }
            float sA = 0.f, sB = 0.f;
            if (whole) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float pa = ex2_approx(__uint_as_float(v[4 * j + e]) - mA);
                        const float pb = ex2_approx(__uint_as_float(v[4 * j + 2 + e]) - mB);
                        v[4 * j + e] = __float_as_uint(pa);
                        v[4 * j + 2 + e] = __float_as_uint(pb);
                        sA += pa;
                        sB += pb;
                    }
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int col = cb + 8 * j + e;
                        const float pa = col <= vA ? ex2_approx(__uint_as_float(v[4 * j + e]) - mA) : 0.f;
                        const float pb = col <= vB ? ex2_approx(__uint_as_float(v[4 * j + 2 + e]) - mB) : 0.f;
                        v[4 * j + e] = __float_as_uint(pa);
                        v[4 * j + 2 + e] = __float_as_uint(pb);
                        sA += pa;
                        sB += pb;
                    }
            }
            lA = lA * aA + sA;
            lB = lB * aB + sB;
            // O is rescaled after the previous tile's products and before this one's; P's
            // buffer is rewritten after the products that last read it
            const bool rescale = __any_sync(0xffffffffu, aA != 1.f || aB != 1.f) && k >= 1;
            if (rescale)
                ok = ok && mbar_wait(bar_pvdone + 8 * ((k - 1) & 1), (uint32_t)((k - 1) >> 1) & 1u, abort);
            if (k >= PB)
                ok = ok && mbar_wait(bar_pvdone + 8 * ((k - PB) & 1), (uint32_t)((k - PB) >> 1) & 1u, abort);
            ok = __all_sync(0xffffffffu, ok);
            if (ok && rescale) {
                // O lane 32 q + t holds the high (t < 16) or low part of row 16 q + t % 16,
                // whose factor is aA (t % 16 < 8) or aB of the threads with tq = t % 8
                const int i = lane & 15;
                const float xa = __shfl_sync(0xffffffffu, aA, 4 * (i & 7));
                const float xb = __shfl_sync(0xffffffffu, aB, 4 * (i & 7));
                const float ar = i < 8 ? xa : xb;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < DH / 64; ++c) {
                    uint32_t o[16];
                    const uint32_t oa = tq0 + O_COL + pt * (DH / 4) + 16 * c;
                    tc_ld16(oa, o);
                    tc_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * ar);
                    tc_st16(oa, o);
                }
                tc_wait_st();
                tc_fence_before();
            }
            // P (bf16 high and low parts): this thread's column pairs of rows A and B
            {
                unsigned char *pb = p8 + pbuf * 2 * SM::PPART;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int chunk = 4 * pt + j;
                    uint32_t h0, l0w, h1, l1w;
                    split_bf16_trunc(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]), h0, l0w);
                    split_bf16_trunc(__uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]), h1, l1w);
                    // stacked operand rows: high part of row 16 q + i at 32 q + i, low at 32 q + 16 + i
                    const int ah = 32 * q + tq, bh = ah + 8;
                    *reinterpret_cast<uint32_t *>(pb + pt_chunk(ah, chunk, 128) + 4 * tc) = h0;
                    *reinterpret_cast<uint32_t *>(pb + pt_chunk(ah + 16, chunk, 128) + 4 * tc) = l0w;
                    *reinterpret_cast<uint32_t *>(pb + pt_chunk(bh, chunk, 128) + 4 * tc) = h1;
                    *reinterpret_cast<uint32_t *>(pb + pt_chunk(bh + 16, chunk, 128) + 4 * tc) = l1w;
                }
            }
            // value rows past the sequence's end hold whatever the staged boxes brought
            // (or nothing): zero them, so that P = 0 multiplies zeros
            if (nv < PT_TILE) {
                unsigned char *vt = sm + (st_s - base) + sl * SM::STAGE;
                for (int e = tid; e < (PT_TILE - nv) * (DH / 8); e += PT_SWARPS * 32) {
                    const int t = nv + e / (DH / 8), c = e % (DH / 8);
                    *reinterpret_cast<uint4 *>(vt + (c >> 3) * (PT_TILE * 128) + t * 128 + (((c & 7) ^ (t & 7)) << 4)) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_pfull + 8 * sb);
            if (tid == 0) GVA_TRACE_AT(102 + 3 * k);
        }
        // this range's partial of rows A and B: unnormalised O, running max, sum
        if (ntile > 0)
            ok = ok && mbar_wait(bar_pvdone + 8 * ((ntile - 1) & 1), (uint32_t)((ntile - 1) >> 1) & 1u, abort);
        ok = __all_sync(0xffffffffu, ok);
        const long long prow0 = ((long long)b * p.splits + split) * p.rows_pad + (long long)g * p.wpg * 16;
        if (ntile > 0 && ok) tc_fence_after();
        // O of row 16 q + t % 16: its high part in lane 32 q + t % 16, its low part 16 lanes on
        const int ro = 16 * q + (lane & 15);
#pragma unroll
        for (int c = 0; c < DH / 64; ++c) {
            uint32_t o[16];
            if (ntile > 0 && ok) {
                tc_ld16(tq0 + O_COL + pt * (DH / 4) + 16 * c, o);
                tc_wait_ld();
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) o[j] = 0u;
            }
            float f[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                f[j] = __uint_as_float(o[j]);
                f[j] += __shfl_down_sync(0xffffffffu, f[j], 16);
            }
            if (lane < 16 && ro < nrows) {
                float4 *dst = reinterpret_cast<float4 *>(p.part_o + (prow0 + ro) * DH + pt * (DH / 4) + 16 * c);
#pragma unroll
                for (int j = 0; j < 4; ++j) dst[j] = make_float4(f[4 * j], f[4 * j + 1], f[4 * j + 2], f[4 * j + 3]);
            }
        }
        lA += __shfl_xor_sync(0xffffffffu, lA, 1);
        lB += __shfl_xor_sync(0xffffffffu, lB, 1);
        lA += __shfl_xor_sync(0xffffffffu, lA, 2);
        lB += __shfl_xor_sync(0xffffffffu, lB, 2);
        float *lw = lsh + q * 64;   // [part][16 rows]
        if (tc == 0) {
            lw[pt * 16 + tq] = lA;
            lw[pt * 16 + 8 + tq] = lB;
        }
        named_sync(1 + q, 128);
        if (pt == 0 && tc == 0) {
            if (hA)
                *reinterpret_cast<float2 *>(p.part_ml + (prow0 + rA) * 2) =
                    make_float2(mA, (lw[tq] + lw[16 + tq]) + (lw[32 + tq] + lw[48 + tq]));
            if (hB)
                *reinterpret_cast<float2 *>(p.part_ml + (prow0 + rB) * 2) =
                    make_float2(mB, (lw[8 + tq] + lw[24 + tq]) + (lw[40 + tq] + lw[56 + tq]));
        }
        } else {
        // the thread's query row: M = 128 lanes = rows; M = 64 puts rows 16 q .. 16 q + 15
        // in lanes 0-15 of quadrant q
        const int q = warp & 3, pt = warp >> 2;   // quadrant, column quarter
        const int r = M == 128 ? 32 * q + lane : 16 * q + lane;
        const bool lane_row = M == 128 || lane < 16;
        const bool has_row = lane_row && r < nrows;
        const int qi = has_row ? r / p.r : 0;
        const long long lim = (has_row && l0 + qi < Lt) ? l0 + qi : -1;   // last visible position
        const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int k = 0; k < ntile; ++k) {
            const int sb = k & 1, sl = k % ns, pbuf = k % PB;
            const long long j0 = (long long)(k0 + k) * PT_TILE;
            const int nv = (int)min((long long)PT_TILE, Lt - j0);
            ok = ok && mbar_wait(bar_sfull + 8 * sb, (uint32_t)(k >> 1) & 1u, abort);
            ok = __all_sync(0xffffffffu, ok);
            if (tid == 0) GVA_TRACE_AT(100 + 3 * k);
            uint32_t s[32];
            if (ok) {
                tc_fence_after();
                tc_ld32(trow + sb * PT_TILE + 32 * pt, s);
                tc_wait_ld();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_sfree + 8 * sb);
            // masked maximum of this quarter (log2 units); tokens past lim are invisible
            const int vis = (int)max(-1LL, min(31LL, lim - j0 - 32 * pt));   // last visible column
            float hmax = -INFINITY;
            if (vis == 31) {
#pragma unroll
                for (int j = 0; j < 32; ++j) hmax = fmaxf(hmax, __uint_as_float(s[j]));
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j <= vis) hmax = fmaxf(hmax, __uint_as_float(s[j]));
            }
            float *xb = xm + (sb * 4 + q) * 128;
            xb[pt * 32 + lane] = hmax;
            named_sync(1 + q, 128);
            if (tid == 0) GVA_TRACE_AT(101 + 3 * k);
            const float tmax = fmaxf(fmaxf(xb[lane], xb[32 + lane]), fmaxf(xb[64 + lane], xb[96 + lane]));
            float alpha = 1.f;
            if (tmax > m + RK_RESCALE_TH) {
                alpha = exp2f(m - tmax);
                m = tmax;
            }
            float ls = 0.f;
            if (vis == 31) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float pj = ex2_approx(__uint_as_float(s[j]) - m);
                    s[j] = __float_as_uint(pj);
                    ls += pj;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float pj = j <= vis ? ex2_approx(__uint_as_float(s[j]) - m) : 0.f;
                    s[j] = __float_as_uint(pj);
                    ls += pj;
                }
            }
            l = l * alpha + ls;
            // O is rescaled after the previous tile's products and before this one's; P's
            // buffer is rewritten after the products that last read it
            const bool rescale = __any_sync(0xffffffffu, alpha != 1.f) && k >= 1;
            if (rescale)
                ok = ok && mbar_wait(bar_pvdone + 8 * ((k - 1) & 1), (uint32_t)((k - 1) >> 1) & 1u, abort);
            if (k >= PB)
                ok = ok && mbar_wait(bar_pvdone + 8 * ((k - PB) & 1), (uint32_t)((k - PB) >> 1) & 1u, abort);
            ok = __all_sync(0xffffffffu, ok);
            if (ok && rescale) {
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < DH / 64; ++c) {
                    uint32_t o[16];
                    const uint32_t oa = trow + O_COL + pt * (DH / 4) + 16 * c;
                    tc_ld16(oa, *reinterpret_cast<uint32_t(*)[16]>(o));
                    tc_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                    tc_st16(oa, o);
                }
                tc_wait_st();
                tc_fence_before();
            }
            // this quarter's P columns (bf16 high and low parts)
            if (lane_row) {
                unsigned char *pb = p8 + pbuf * 2 * SM::PPART;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        split_bf16_trunc(__uint_as_float(s[8 * c + 2 * u]), __uint_as_float(s[8 * c + 2 * u + 1]), hw[u], lw[u]);
                    const uint32_t off = pt_chunk(r, 4 * pt + c, M);
                    *reinterpret_cast<uint4 *>(pb + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4 *>(pb + SM::PPART + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
            }
            // value rows past the sequence's end hold whatever the staged boxes brought
            // (or nothing): zero them, so that P = 0 multiplies zeros
            if (nv < PT_TILE) {
                unsigned char *vt = sm + (st_s - base) + sl * SM::STAGE;
                for (int e = tid; e < (PT_TILE - nv) * (DH / 8); e += PT_SWARPS * 32) {
                    const int t = nv + e / (DH / 8), c = e % (DH / 8);
                    *reinterpret_cast<uint4 *>(vt + (c >> 3) * (PT_TILE * 128) + t * 128 + (((c & 7) ^ (t & 7)) << 4)) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_pfull + 8 * sb);
            if (tid == 0) GVA_TRACE_AT(102 + 3 * k);
        }
        // this range's partial of the row: unnormalised O, running max, sum of the quarters
        if (ntile > 0)
            ok = ok && mbar_wait(bar_pvdone + 8 * ((ntile - 1) & 1), (uint32_t)((ntile - 1) >> 1) & 1u, abort);
        ok = __all_sync(0xffffffffu, ok);
        const long long prow = ((long long)b * p.splits + split) * p.rows_pad + (long long)g * p.wpg * 16 + r;
        if (ntile > 0 && ok) tc_fence_after();
#pragma unroll
        for (int c = 0; c < DH / 64; ++c) {
            uint32_t o[16];
            if (ntile > 0 && ok) {
                tc_ld16(trow + O_COL + pt * (DH / 4) + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(o));
                tc_wait_ld();
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) o[j] = 0u;
            }
            if (has_row) {
                float4 *dst = reinterpret_cast<float4 *>(p.part_o + prow * DH + pt * (DH / 4) + 16 * c);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    dst[j] = make_float4(__uint_as_float(o[4 * j]), __uint_as_float(o[4 * j + 1]),
                                         __uint_as_float(o[4 * j + 2]), __uint_as_float(o[4 * j + 3]));
            }
        }
        lsh[(q * 4 + pt) * 32 + lane] = l;
        named_sync(1 + q, 128);
        if (pt == 0 && has_row)
            *reinterpret_cast<float2 *>(p.part_ml + prow * 2) =
                make_float2(m, (lsh[(q * 4) * 32 + lane] + lsh[(q * 4 + 1) * 32 + lane]) +
                                   (lsh[(q * 4 + 2) * 32 + lane] + lsh[(q * 4 + 3) * 32 + lane]));
            }
    }
    // every thread's partial writes are visible device-wide before the CTA's ticket
    if (tp.tickets != nullptr) __threadfence();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        GVA_TRACE_AT(300);
        GVA_TRACE_FLUSH(0, 320);
    }
    if (warp == PT_SWARPS + 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TCOLS)
                     : "memory");
    }
    if (tp.tickets == nullptr) return;

    // ---- the ranges' log-sum-exp merge, by the last CTA of this (value group, sequence) ----
    volatile int *last = reinterpret_cast<volatile int *>(tail + 8);
    if (tid == 0) *last = atomicAdd(tp.tickets + b * p.G + g, 1) == p.splits - 1;
    __syncthreads();
    if (!*last) return;
    __threadfence();
    // The ranges' (max, sum) of every row of the group (row q = i r + hl: query i, head
    // g r + hl) are staged in the P buffers, which no product reads any more; each row's
    // maximum and weights follow, then one thread per 4 output columns of a row sums the
    // ranges' parts with independent loads.
    const int S = p.splits;
    const long long at_b = (long long)b * S * p.rows_pad + (long long)g * p.wpg * 16;
    float *mls = reinterpret_cast<float *>(p8);   // [nrows][S] (max, sum), then weights
    float *dens = mls + 2 * nrows * S, *mxs = dens + nrows;
    for (int e = tid; e < nrows * S; e += PT_THREADS) {
        const int q = e / S, r = e - q * S;
        const float2 ml = __ldcg(reinterpret_cast<const float2 *>(p.part_ml + (at_b + q + (long long)r * p.rows_pad) * 2));
        mls[2 * e] = ml.x;
        mls[2 * e + 1] = ml.y;
    }
    __syncthreads();
    for (int q = tid; q < nrows; q += PT_THREADS) {
        float Mx = -INFINITY;
        for (int r = 0; r < S; ++r) Mx = fmaxf(Mx, mls[2 * (q * S + r)]);
        float den = 0.f;
        for (int r = 0; r < S; ++r) {
            const float m = mls[2 * (q * S + r)];
            const float wgt = (Mx == -INFINITY || m == -INFINITY) ? 0.f : exp2f(m - Mx);
            den += wgt * mls[2 * (q * S + r) + 1];
            mls[2 * (q * S + r)] = wgt;
        }
        dens[q] = den;
        mxs[q] = Mx;
    }
    __syncthreads();
    for (int e = tid; e < nrows * (DH / 4); e += PT_THREADS) {
        const int q = e / (DH / 4), c = e - q * (DH / 4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r = 0; r < S; ++r) {
            // a range whose rows saw nothing wrote zeros: weight 0 adds 0
            const float wgt = mls[2 * (q * S + r)];
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(p.part_o + (at_b + q + (long long)r * p.rows_pad) * DH) + c);
            acc.x += wgt * v.x; acc.y += wgt * v.y; acc.z += wgt * v.z; acc.w += wgt * v.w;
        }
        const float den = dens[q];
        const float inv = den > 0.f ? 1.f / den : 0.f;
        const int i = q / p.r, h = g * p.r + (q - i * p.r);
        const long long row = ((long long)b * p.n + i) * p.H + h;
        reinterpret_cast<float4 *>(p.out + row * DH)[c] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        if (c == 0 && p.lse) p.lse[row] = den > 0.f ? (mxs[q] + log2f(den)) * LN2 : -INFINITY;
    }
}

// ---------------------------------------------------------------------------- //
// host side
// ---------------------------------------------------------------------------- //
// M = 64 when the group's chunk rows fit (n r <= 64), else 128 for d_h = 64; the rest
// stays with the mma.sync kernel.
inline int prefill_tc_m(const gva_dims *d, int n) {
    if (d->cache_dtype != GVA_BF16) return 0;
    if (d->d_h != 64 && d->d_h != 128) return 0;
    if (d->d_r != 0 && d->d_r != 8 && d->d_r != 16 && d->d_r != 24 && d->d_r != 32) return 0;
    const int rows = n * (d->H / d->G);
    if (rows <= 64) return 64;
    if (rows <= 128 && d->d_h == 64) return 128;
    return 0;
}

template <int DH, int DR, int M>
inline int prefill_tc_smem(int ns) {
    using SM = PtSmem<DH, DR, M>;
    return 1024 + SM::fixed + ns * SM::STAGE + (2 * ns + 9) * 8 + 16;
}

template <int DH, int DR, int M>
inline int prefill_tc_stages() {
    int ns = PT_MAX_STAGES;
    while (ns >= 2 && prefill_tc_smem<DH, DR, M>(ns) > MMA_SMEM_LIMIT) --ns;
    return ns;
}

// 2D maps: value rows [rows][G d_h] box {64, ch}, 128-byte swizzle; positional rows
// [rows][d_r] box {16, ch} with the 32-byte swizzle (d_r <= 16) or {32, ch} with the 64-byte
// one (the columns past d_r are outside the tensor and arrive as zeros).
inline bool prefill_tc_maps(CUtensorMap *tv, CUtensorMap *tk, const void *V, const void *Kr,
                            long long rows, int width, int d_r, int ch) {
    if (!rk_make_map(tv, V, rows, width, ch)) return false;
    if (d_r == 0) {
        *tk = *tv;
        return true;
    }
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)d_r, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t strides[1] = {(cuuint64_t)d_r * 2};
    const bool narrow = d_r <= 16;
    cuuint32_t box[2] = {narrow ? 16u : 32u, (cuuint32_t)ch};
    cuuint32_t estr[2] = {1, 1};
    return enc(tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(Kr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               narrow ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DH, int DR, int M>
inline cudaError_t prefill_tc_launch_t(void *stream, PrefillTcParams &tp, const CUtensorMap &tv,
                                       const CUtensorMap &tk) {
    tp.nstages = prefill_tc_stages<DH, DR, M>();
    if (tp.nstages < 2) return cudaErrorInvalidValue;
    tp.smem_bytes = prefill_tc_smem<DH, DR, M>(tp.nstages);
    // the in-kernel merge stages every range's (max, sum) of the group's rows in the P
    // buffers: beyond their size the merge kernel runs instead
    using SM = PtSmem<DH, DR, M>;
    const long long nrows = (long long)tp.p.n * tp.p.r;
    if (tp.tickets && (2 * nrows * tp.p.splits + 2 * nrows) * 4 > (long long)SM::PB * 2 * SM::PPART)
        tp.tickets = nullptr;
    const dim3 grid(tp.p.splits, tp.p.G, tp.p.B);
    cudaError_t e = tp.by_length
                        ? launch(prefill_tc_kernel<DH, DR, M, true>, grid, dim3(PT_THREADS),
                                 (size_t)tp.smem_bytes, stream, tv, tk, tp)
                        : launch(prefill_tc_kernel<DH, DR, M, false>, grid, dim3(PT_THREADS),
                                 (size_t)tp.smem_bytes, stream, tv, tk, tp);
    if (e != cudaSuccess || tp.tickets != nullptr) return e;
    const long long rows = (long long)tp.p.B * tp.p.n * tp.p.H;
    const dim3 cg((unsigned)((rows + PF_COMBINE_WARPS - 1) / PF_COMBINE_WARPS));
    return launch(prefill_combine_kernel<DH>, cg, dim3(PF_COMBINE_WARPS * 32), 0, stream, tp.p);
}

template <int DH, int M>
inline cudaError_t prefill_tc_launch_dr(void *stream, int d_r, PrefillTcParams &tp,
                                        const CUtensorMap &tv, const CUtensorMap &tk) {
    switch (d_r) {
    case 0: return prefill_tc_launch_t<DH, 0, M>(stream, tp, tv, tk);
    case 8: return prefill_tc_launch_t<DH, 8, M>(stream, tp, tv, tk);
    case 16: return prefill_tc_launch_t<DH, 16, M>(stream, tp, tv, tk);
    case 24: return prefill_tc_launch_t<DH, 24, M>(stream, tp, tv, tk);
    default: return prefill_tc_launch_t<DH, 32, M>(stream, tp, tv, tk);
    }
}

inline cudaError_t prefill_tc_launch(void *stream, int d_h, int d_r, int M, PrefillTcParams &tp,
                                     const CUtensorMap &tv, const CUtensorMap &tk) {
    if (M == 64)
        return d_h == 64 ? prefill_tc_launch_dr<64, 64>(stream, d_r, tp, tv, tk)
                         : prefill_tc_launch_dr<128, 64>(stream, d_r, tp, tv, tk);
    return prefill_tc_launch_dr<64, 128>(stream, d_r, tp, tv, tk);
}

template <int DH, int M>
inline cudaError_t prefill_tc_opt_in_dm() {
    const void *ks[] = {
        (const void *)prefill_tc_kernel<DH, 0, M, false>, (const void *)prefill_tc_kernel<DH, 8, M, false>,
        (const void *)prefill_tc_kernel<DH, 16, M, false>, (const void *)prefill_tc_kernel<DH, 24, M, false>,
        (const void *)prefill_tc_kernel<DH, 32, M, false>, (const void *)prefill_tc_kernel<DH, 0, M, true>,
        (const void *)prefill_tc_kernel<DH, 8, M, true>, (const void *)prefill_tc_kernel<DH, 16, M, true>,
        (const void *)prefill_tc_kernel<DH, 24, M, true>, (const void *)prefill_tc_kernel<DH, 32, M, true>};
    for (const void *k : ks) {
        const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, MMA_SMEM_LIMIT);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

inline cudaError_t prefill_tc_opt_in_all() {
    cudaError_t e = prefill_tc_opt_in_dm<64, 64>();
    if (e == cudaSuccess) e = prefill_tc_opt_in_dm<128, 64>();
    if (e == cudaSuccess) e = prefill_tc_opt_in_dm<64, 128>();
    return e;
}

}  // namespace gva
