// decode_rope_keys.cuh -- decode for the GVA variant that applies ordinary RoPE to the
// reconstructed key itself (the scale-matched row of the agihunt summary, results
// discussion; the analysis page, 关键技巧二, on why M_h can then no longer be folded into
// the query: the relative rotation sits between q and M_h^T).
//
// Definition (the reading the oracle takes): for head h of group g = h / r,
//   K_h[j] = v_{j,g} M_h (width d_n), rotated by its own position j;
//   Q = Rot(t) q_h, t = L - 1;  z_j = scale Q . Rot(j) K_h[j];  out = softmax(z) V_g.
//
// Reformulation used here (exact up to rounding).  For rotation pair p, with
// (c, s) = (cos, sin)(j th_p),
//   Q_p . Rot(j) K_p = c (Q_{2p} K_{2p} + Q_{2p+1} K_{2p+1}) + s (Q_{2p+1} K_{2p} - Q_{2p} K_{2p+1}).
// Both brackets are linear in v_j, so [X_0 Y_0 X_1 Y_1 ...] = v_j W_bh with
//   W_bh[i][2p]   = scale (M_h[i][2p] Q_{2p}   + M_h[i][2p+1] Q_{2p+1}),
//   W_bh[i][2p+1] = scale (M_h[i][2p] Q_{2p+1} - M_h[i][2p+1] Q_{2p}),
// built once per (sequence, head), and z_j = sum_k (v_j W_bh)[k] T_j[k] where T_j is the
// (cos, sin) table row of position j.  The product v_j W_bh is a dense contraction (d_h
// d_n multiply-adds per token and head, about d_n / 2 per cache byte for r = 4): it runs
// on the tensor cores, with W_bh split into bf16 high and low parts so that the products
// keep about 16 bits of the fp32 weights, accumulated in fp32 in tensor memory.
//
// Kernels (chained with programmatic dependent launch):
//   rk_prep_kernel   -- W_bh as hi / lo bf16 images in the 128-byte-swizzled K-major
//                       layout the tensor cores read; validated lengths and the prefix of
//                       work units.
//   rk_decode_kernel -- one CTA per SM over an equal share of the work units
//                       (sequence, value group, head slice, 128-token tile):
//                       warp 8  TMA producer: value tiles, weight images;
//                       warp 9  tcgen05.mma issuer (one thread) into two tensor-memory
//                               accumulators of 128 tokens x (heads x d_n) columns;
//                       warps 0-7 epilogue: tcgen05.ld, the per-token dot product with the
//                               rotation of its position, online softmax, the value sum on
//                               CUDA cores from the staged tile, partials per segment.
//   rk_merge_kernel  -- log-sum-exp merge of the partials of each (sequence, head).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "decode_mma.cuh"

namespace gva {

constexpr int RK_TILE = 128;          // tokens per work unit (the MMA's M)
constexpr int RK_EPI_WARPS = 8;       // two per tensor-memory lane quarter
constexpr int RK_EPI_T = RK_EPI_WARPS * 32;
constexpr int RK_THREADS = (RK_EPI_WARPS + 2) * 32;
constexpr int RK_PREP_THREADS = 128;   // >= d_n
constexpr int RK_MERGE_THREADS = 128;
constexpr int RK_MAX_STAGES = 6;
constexpr float RK_RESCALE_TH = 8.f;  // log2 units

struct RkParams {
    int B, H, G, r, d_h, d_n;
    int hc, nhs;             // heads per slice (1, 2 or 4) and slices per group, r = hc nhs
    const int *seq_len;
    RowsDev R;
    const void *q;           // [B][H][d_n]
    int q_f32;
    const float *M;          // [H][d_h][d_n]
    const float *tab;        // [tab_rows][d_n / 2][2] (cos, sin)
    int tab_rows;
    float scale_log2;        // softmax scale times log2(e)
    unsigned char *img;      // per stream (b, g, slice): hi then lo image, d_h x N bf16 each
    int *Ls;                 // [B] validated lengths
    int *pre;                // [B + 1] exclusive prefix of work units
    float *part_o;           // [slots][hc][d_h]
    float *part_ml;          // [slots][hc][2] (max in log2 units, sum)
    float *out;              // [B][H][d_h]
    float *lse;              // [B][H] or null
    int n_ctas;
    int ch;                  // cache rows per TMA box (64, or 16 / 32 for small pages)
    int nstages, nbuf;       // value-tile ring depth, weight-image buffers
    int smem_bytes;
};

__host__ __device__ inline int rk_img_bytes(int d_h, int N) { return 2 * d_h * N * 2; }

// ---------------------------------------------------------------------------------- //
// Prep: weight images and the unit prefix
// ---------------------------------------------------------------------------------- //
__device__ __forceinline__ float rk_ld_q(const void *q, int f32, long long i) {
    return f32 ? static_cast<const float *>(q)[i]
               : __bfloat162float(static_cast<const __nv_bfloat16 *>(q)[i]);
}

__device__ __forceinline__ bool rk_len_ok(const RkParams &p, int b, int L) {
    return length_ok(p.R, b, L) && L <= p.tab_rows;
}

// Blocks [0, B H d_h / 8): for (sequence b, head h, value rows 8 ic .. 8 ic + 7), thread k
// writes image row hh d_n + k of those rows (one 16-byte chunk of the high and of the low
// image).  The last block: lengths and the unit prefix (units of sequence b:
// ceil(L_b / 128) tiles x G x nhs streams).
__global__ void __launch_bounds__(RK_PREP_THREADS) rk_prep_kernel(const RkParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int dn = p.d_n, dh = p.d_h, nic = dh / 8;
    const int blk = blockIdx.x;
    if (blk == p.B * p.H * nic) {
        for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
            int L = p.seq_len[b];
            if (!rk_len_ok(p, b, L)) {
                dev_report(length_ok(p.R, b, L) ? GVA_DEV_BAD_POSITION : GVA_DEV_BAD_LENGTH);
                L = 0;
            }
            p.Ls[b] = L;
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x, Gn = p.G * p.nhs;
            const int per = (p.B + 31) / 32;
            const int lo = lane * per, hi = min(lo + per, p.B);
            int sum = 0;
            for (int b = lo; b < hi; ++b) sum += (p.Ls[b] + RK_TILE - 1) / RK_TILE * Gn;
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            int run = incl - sum;
            for (int b = lo; b < hi; ++b) {
                p.pre[b] = run;
                run += (p.Ls[b] + RK_TILE - 1) / RK_TILE * Gn;
            }
            if (lane == 31) p.pre[p.B] = incl;
        }
        return;
    }
    const int k = threadIdx.x;
    if (k >= dn) return;
    const int ic = blk % nic, bh = blk / nic, b = bh / p.H, h = bh % p.H;
    const int L = p.seq_len[b];
    const int t = (rk_len_ok(p, b, L) && L > 0) ? L - 1 : 0;
    // this thread's rotation pair of Q = scale log2(e) Rot(t) q_bh
    const int pp = k >> 1;
    const long long qb = (long long)bh * dn;
    const float q0 = rk_ld_q(p.q, p.q_f32, qb + 2 * pp);
    const float q1 = rk_ld_q(p.q, p.q_f32, qb + 2 * pp + 1);
    const float2 cs = reinterpret_cast<const float2 *>(p.tab)[(long long)t * (dn / 2) + pp];
    const float Q0 = (q0 * cs.x - q1 * cs.y) * p.scale_log2;
    const float Q1 = (q0 * cs.y + q1 * cs.x) * p.scale_log2;
    const int g = h / p.r, hl = h % p.r, hs = hl / p.hc, hh = hl % p.hc;
    const int N = p.hc * dn;
    const long long stream = ((long long)b * p.G + g) * p.nhs + hs;
    unsigned char *img = p.img + stream * rk_img_bytes(dh, N);
    const float2 *Mp = reinterpret_cast<const float2 *>(p.M + (long long)h * dh * dn) + pp;
    float x[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float2 m = Mp[(long long)(ic * 8 + e) * (dn / 2)];
        x[e] = (k & 1) ? (m.x * Q1 - m.y * Q0) : (m.x * Q0 + m.y * Q1);
    }
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        const __nv_bfloat16 h0 = __float2bfloat16_rn(x[e]), h1 = __float2bfloat16_rn(x[e + 1]);
        const __nv_bfloat16 l0 = __float2bfloat16_rn(x[e] - __bfloat162float(h0));
        const __nv_bfloat16 l1 = __float2bfloat16_rn(x[e + 1] - __bfloat162float(h1));
        hw[e / 2] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
        lw[e / 2] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
    }
    const int n = hh * dn + k;
    const size_t off = (size_t)(ic >> 3) * N * 128 + (size_t)n * 128 + (size_t)(((ic & 7) ^ (n & 7)) << 4);
    *reinterpret_cast<uint4 *>(img + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4 *>(img + (size_t)dh * N * 2 + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

// ---------------------------------------------------------------------------------- //
// tcgen05 wrappers
// ---------------------------------------------------------------------------------- //
// Shared-memory matrix descriptor of a K-major operand in the 128-byte swizzle: rows of
// 128 B (64 bf16), groups of 8 rows 1024 B apart.
__device__ __forceinline__ uint64_t rk_sdesc(uint32_t addr) {
    uint64_t d = (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)1 << 16;              // leading byte offset (unused by this layout)
    d |= (uint64_t)(1024 >> 4) << 32;    // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;              // descriptor version
    d |= (uint64_t)2 << 61;              // 128-byte swizzle
    return d;
}
// Instruction descriptor: bf16 A and B (both K-major), fp32 D, M x N.
__host__ __device__ constexpr uint32_t rk_idesc(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// Arrive once on the mbarrier when every tcgen05 operation this thread issued before
// has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tc_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Bounded poll that ignores the abort flag: used to let copies and products already in
// flight land before the CTA leaves (its shared and tensor memory are then released).
__device__ __forceinline__ void rk_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > WAIT_LIMIT_NS) return;
}

// Walk over work units u = (sequence b, stream-in-sequence sidx, tile), b-major, over the
// unit prefix and validated lengths the prep kernel wrote.
struct RkIter {
    const int *pre;
    const int *Ls;
    int B, Gn;
    int b, nt, sidx, tile, L;
    __device__ __forceinline__ void begin(long long u) {
        b = seq_of_slab(pre, B, u);
        const int w = (int)(u - pre[b]);
        nt = (pre[b + 1] - pre[b]) / Gn;
        sidx = w / nt;
        tile = w - sidx * nt;
        L = Ls[b];
    }
    __device__ __forceinline__ void next() {
        if (++tile < nt) return;
        tile = 0;
        if (++sidx < Gn) return;
        sidx = 0;
        do {
            ++b;
        } while (b < B && pre[b + 1] == pre[b]);
        if (b < B) {
            nt = (pre[b + 1] - pre[b]) / Gn;
            L = Ls[b];
        }
    }
    __device__ __forceinline__ int stream() const { return b * Gn + sidx; }
};

// ---------------------------------------------------------------------------------- //
// Decode
// ---------------------------------------------------------------------------------- //
template <int DH, int DN, int HC>
struct RkSmem {   // the small buffers after the weight images and the value ring
    static constexpr int ZX = 2 * 4 * 2 * HC * 32 * 4;  // z halves [buf][quarter][half][hc][32]
    static constexpr int RED = 4 * HC * DH * 4;         // segment value sums [quarter][hc][d_h]
    static constexpr int ML = 4 * HC * 2 * 4;           // segment (max, sum) [quarter][hc]
    static constexpr int TR = RK_MAX_STAGES * DN * 4;   // table row of each stage's tile
    static constexpr int PW = RK_EPI_WARPS * 32 * HC * 4;  // per-warp probabilities [warp][32][hc]
    static constexpr int total = ZX + RED + ML + TR + PW;
};

// barriers, then the tensor-memory address and the abort flag
__host__ __device__ inline int rk_bar_bytes(int ns, int nbuf) {
    return (2 * ns + 2 * nbuf + 5) * 8 + 16;
}

// Epilogue layout: warp w < 8 reads tensor-memory lane quarter q = w & 3 (tokens 32 q ..
// 32 q + 31 of the tile) and handles half hf = w >> 2 of the rotation pairs and of the value
// columns.  The two warps of a quarter exchange their partial scores through shared memory
// (a 64-thread barrier); each quarter keeps its own running maximum, so the quarters run
// unsynchronised and are merged at the end of each segment.
template <int DH, int DN, int HC>
__global__ void __launch_bounds__(RK_THREADS, 1)
    rk_decode_kernel(const __grid_constant__ CUtensorMap tm_v, const RkParams p) {
    constexpr int N = HC * DN;                  // accumulator columns per tile
    // columns per MMA instruction: all of them (M = 128 takes N up to 256), so that each
    // 16-column slice of the value tile is read from shared memory once per k-step; at
    // N = 128 the two operands' reads alone would fill the shared-memory bandwidth
    constexpr int NCH = N;
    constexpr int TCOLS = 2 * N;                // two accumulators (64 <= N <= 256)
    constexpr int KB = DH / 64;                 // 64-column blocks of a value row
    constexpr int STAGE = RK_TILE * DH * 2;
    constexpr int IMG = 2 * DH * N * 2;
    constexpr int IMG_LO = DH * N * 2;
    constexpr int PH = DN / 4;                  // rotation pairs per epilogue thread
    constexpr int DGW = DH / 16;                // 8-column groups per warp (half the row)
    constexpr int NS = 32 / DGW;                // token subsets per warp
    constexpr int TS = 32 / NS;                 // tokens per subset
    static_assert(RK_EPI_WARPS == 8, "two epilogue warps per lane quarter");
    static_assert(N >= 64 && N <= 256 && (N % NCH) == 0, "accumulator width");
    static_assert(PH % 8 == 0, "pairs per thread");
    using SM = RkSmem<DH, DN, HC>;

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    unsigned char *sm = smem_raw + (base - raw_u32);
    const int ns = p.nstages, nbuf = p.nbuf;
    const uint32_t img_s = base;
    const uint32_t stage_s = img_s + (uint32_t)(nbuf * IMG);
    unsigned char *small = sm + nbuf * IMG + ns * STAGE;
    float *zx = reinterpret_cast<float *>(small);
    float *red = reinterpret_cast<float *>(small + SM::ZX);
    float *mls = reinterpret_cast<float *>(small + SM::ZX + SM::RED);
    float *trow_s = reinterpret_cast<float *>(small + SM::ZX + SM::RED + SM::ML);
    float *pws = reinterpret_cast<float *>(small + SM::ZX + SM::RED + SM::ML + SM::TR);
    const uint32_t bars = smem_u32(small + SM::total);
    const uint32_t bar_full = bars, bar_empty = bars + 8 * ns;
    const uint32_t bar_bfull = bar_empty + 8 * ns, bar_bempty = bar_bfull + 8 * nbuf;
    const uint32_t bar_tfull = bar_bempty + 8 * nbuf, bar_tempty = bar_tfull + 16;
    const uint32_t bar_done = bar_tempty + 16;
    unsigned char *tail = small + SM::total + (2 * ns + 2 * nbuf + 5) * 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tail);
    volatile int *abort = reinterpret_cast<volatile int *>(tail + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) GVA_TRACE_AT(0);
    if (tid == 0) {
        for (int s = 0; s < ns; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, RK_EPI_WARPS);
        }
        for (int s = 0; s < nbuf; ++s) {
            mbar_init(bar_bfull + 8 * s, 1);
            mbar_init(bar_bempty + 8 * s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar_tfull + 8 * s, 1);
            mbar_init(bar_tempty + 8 * s, RK_EPI_WARPS);
        }
        mbar_init(bar_done, 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == RK_EPI_WARPS) prefetch_tmap(&tm_v);

    // the epilogue thread's in-tile rotations (cos, sin)(tau th_p) for its pairs: the
    // table's rows 0..127 (an input, readable before the preceding grid completes)
    const int q = warp & 3, hf = (warp >> 2) & 1, tau = 32 * q + lane;
    float ct[PH], st[PH];
    if (warp < RK_EPI_WARPS) {
        const float2 *row = reinterpret_cast<const float2 *>(p.tab) + (long long)tau * (DN / 2) + hf * PH;
#pragma unroll
        for (int i = 0; i < PH; ++i) {
            const float2 cs = __ldg(row + i);
            ct[i] = cs.x;
            st[i] = cs.y;
        }
    }
    pdl_wait();
    pdl_launch_dependents();
    if (tid == 0) GVA_TRACE_AT(1);
    const long long U = p.pre[p.B];
    const Part part{U, p.n_ctas};
    const int cta = blockIdx.x;
    if (cta >= part.neff()) return;             // uniform: no work for this CTA
    const long long u0 = part.start(cta), u1 = part.start(cta + 1);

    if (warp == RK_EPI_WARPS + 1) {
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
    const int Gn = p.G * p.nhs;
    if (tid == 0) GVA_TRACE_AT(2);

    if (warp == RK_EPI_WARPS) {
        // ------------------------------ producer ------------------------------ //
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();   // the cache and the images
            uint64_t pol_keep;                              // the table rows, reused by all CTAs
            asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_keep));
            const int nbox = RK_TILE / p.ch;
            // value tile and table row of unit k (stage k % ns, which is free)
            auto issue_v = [&](const RkIter &it, long long k) {
                const int sl = (int)(k % ns);
                const int L = it.L;
                const int j0 = it.tile * RK_TILE, nv = min(RK_TILE, L - j0);
                const int g = it.sidx / p.nhs;
                long long rows[RK_TILE / 16];
                int nl = 0;
                for (int c = 0; c < nbox; ++c) {
                    rows[c] = -2;
                    if (c * p.ch < nv) {
                        rows[c] = row_of(p.R, it.b, j0 + c * p.ch);
                        if (rows[c] == -1) dev_report(GVA_DEV_BAD_PAGE);
                        if (rows[c] >= 0) ++nl;
                    }
                }
                const uint32_t fb = bar_full + 8 * sl;
                mbar_expect_tx(fb, (uint32_t)(nl * p.ch * 128 * KB + DN * 4));
                // (cos, sin)(j0 th_p) of the tile start, for the epilogue's rotations
                bulk_load(smem_u32(trow_s + sl * DN), p.tab + (long long)j0 * DN, DN * 4, fb, pol_keep);
                const uint32_t dst = stage_s + sl * STAGE;
                for (int c = 0; c < nbox; ++c) {
                    if (rows[c] < 0) continue;
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb)
                        tma_load_2d(dst + kb * (RK_TILE * 128) + c * p.ch * 128, &tm_v,
                                    g * DH + kb * 64, (int)rows[c], fb, pol);
                }
                GVA_TRACE_AT(200 + (int)k);
            };
            RkIter it{p.pre, p.Ls, p.B, Gn};
            it.begin(u0);
            int cur = -1, nimg = 0;
            long long k = 0;
            for (long long u = u0; u < u1; ++u, it.next(), ++k) {
                const int s = it.stream();
                if (s != cur) {
                    const int bb = nimg % nbuf;
                    if (nimg >= nbuf && !mbar_wait(bar_bempty + 8 * bb, ((nimg / nbuf) - 1) & 1, abort))
                        break;
                    mbar_expect_tx(bar_bfull + 8 * bb, IMG);
                    const unsigned char *src = p.img + (size_t)s * IMG;
                    for (int o = 0; o < IMG; o += 32768)
                        bulk_load(img_s + bb * IMG + o, src + o, min(32768, IMG - o),
                                  bar_bfull + 8 * bb, pol);
                    ++nimg;
                    cur = s;
                }
                const int sl = (int)(k % ns);
                if (k >= ns && !mbar_wait(bar_empty + 8 * sl, (uint32_t)((k / ns) - 1) & 1u, abort))
                    break;
                issue_v(it, k);
            }
            // let the copies in flight land before the CTA can leave
            for (long long i = (k > ns ? k - ns : 0); i < k; ++i)
                rk_drain(bar_full + 8 * (int)(i % ns), (uint32_t)(i / ns) & 1u);
            if (nimg > 0) {
                const int last = nimg - 1;
                rk_drain(bar_bfull + 8 * (last % nbuf), (uint32_t)(last / nbuf) & 1u);
            }
        }
    } else if (warp == RK_EPI_WARPS + 1) {
        // ------------------------------ MMA issuer ------------------------------ //
        if (lane == 0) {
            constexpr uint32_t idesc = rk_idesc(128, NCH);
            RkIter it{p.pre, p.Ls, p.B, Gn};
            it.begin(u0);
            int cur = -1, nimg = 0, bb = 0;
            long long k = 0;
            for (long long u = u0; u < u1; ++u, it.next()) {
                const int s = it.stream();
                if (s != cur) {
                    bb = nimg % nbuf;
                    if (!mbar_wait(bar_bfull + 8 * bb, (uint32_t)(nimg / nbuf) & 1u, abort)) break;
                    ++nimg;
                    cur = s;
                }
                const int sl = (int)(k % ns);
                GVA_TRACE_AT(10 + 3 * (int)k);
                if (!mbar_wait(bar_full + 8 * sl, (uint32_t)(k / ns) & 1u, abort)) break;
                const int tb = (int)(k & 1);
                if (k >= 2 && !mbar_wait(bar_tempty + 8 * tb, (uint32_t)((k >> 1) - 1) & 1u, abort))
                    break;
                tc_fence_after();
                GVA_TRACE_AT(11 + 3 * (int)k);
                const uint32_t a0 = stage_s + sl * STAGE, b0 = img_s + bb * IMG;
#pragma unroll
                for (int kb = 0; kb < KB; ++kb)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                        for (int part_ = 0; part_ < 2; ++part_)
#pragma unroll
                            for (int nh = 0; nh < N / NCH; ++nh) {
                                const uint64_t ad = rk_sdesc(a0 + kb * (RK_TILE * 128) + kk * 32);
                                const uint64_t bd = rk_sdesc(b0 + part_ * IMG_LO + kb * (N * 128) +
                                                             nh * (NCH * 128) + kk * 32);
                                tc_mma(tmem + tb * N + nh * NCH, ad, bd, idesc,
                                       (kb | kk | part_) != 0 ? 1u : 0u);
                            }
                tc_commit(bar_tfull + 8 * tb);
                GVA_TRACE_AT(12 + 3 * (int)k);
                if (it.tile == it.nt - 1 || u + 1 == u1) tc_commit(bar_bempty + 8 * bb);
                ++k;
            }
            // every product issued has completed before the tensor memory is freed
            tc_commit(bar_done);
            rk_drain(bar_done, 0);
        }
    } else {
        // ------------------------------ epilogue ------------------------------ //
        // paired fp32 arithmetic (two lanes per instruction) for the dot products and the
        // value sum: acc[hh][e] holds value columns d0 + 2 e, d0 + 2 e + 1
        float m[HC], lrun[HC];
        float2 acc[HC][4];
#pragma unroll
        for (int hh = 0; hh < HC; ++hh) {
            m[hh] = -INFINITY;
            lrun[hh] = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[hh][e] = make_float2(0.f, 0.f);
        }
        const int lg = lane % DGW, ls = lane / DGW;
        const int d0 = hf * (DH / 2) + 8 * lg, vkb = d0 >> 6, vch = (d0 & 63) >> 3;
        const uint32_t tbase0 = tmem + ((uint32_t)(32 * q) << 16) + hf * (2 * PH);
        RkIter it{p.pre, p.Ls, p.B, Gn};
        it.begin(u0);
        bool ok = true;
        long long k = 0;
        for (long long u = u0; u < u1; ++u, it.next(), ++k) {
            const int L = it.L;
            const int j0 = it.tile * RK_TILE, nv = min(RK_TILE, L - j0);
            const int tb = (int)(k & 1), buf = tb, sl = (int)(k % ns);
            ok = ok && mbar_wait(bar_tfull + 8 * tb, (uint32_t)(k >> 1) & 1u, abort);
            // the staged value tile and table row are published by the stage's own barrier
            ok = ok && mbar_wait(bar_full + 8 * sl, (uint32_t)(k / ns) & 1u, abort);
            ok = __all_sync(0xffffffffu, ok);
            if (tid == 0) GVA_TRACE_AT(100 + 3 * (int)k);
            float z[HC];
            float2 zz[HC][2];
#pragma unroll
            for (int hh = 0; hh < HC; ++hh) zz[hh][0] = zz[hh][1] = make_float2(0.f, 0.f);
            if (ok) {
                tc_fence_after();
                const float4 *trow = reinterpret_cast<const float4 *>(trow_s + sl * DN + hf * PH * 2);
                const uint32_t tbase = tbase0 + tb * N;
#pragma unroll
                for (int c = 0; c < PH / 8; ++c) {
                    // at most two heads' columns in flight (register budget); the first
                    // group's loads are issued before the rotations, which hide their latency
                    constexpr int NH = HC < 2 ? HC : 2;
                    uint32_t v[NH][16];
#pragma unroll
                    for (int w = 0; w < NH; ++w) tc_ld16(tbase + w * DN + c * 16, v[w]);
                    float2 cs[8];   // (cos, sin)(j th_p), j = j0 + tau, of the chunk's pairs
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const float4 x = trow[c * 4 + q4];   // (c0, s0) of two pairs
                        const int i = 2 * q4, a = c * 8 + i;
                        cs[i] = make_float2(x.x * ct[a] - x.y * st[a], x.y * ct[a] + x.x * st[a]);
                        cs[i + 1] = make_float2(x.z * ct[a + 1] - x.w * st[a + 1],
                                                x.w * ct[a + 1] + x.z * st[a + 1]);
                    }
#pragma unroll
                    for (int h0 = 0; h0 < HC; h0 += 2) {
                        if (h0 > 0) {
#pragma unroll
                            for (int w = 0; w < NH; ++w) tc_ld16(tbase + (h0 + w) * DN + c * 16, v[w]);
                        }
                        tc_wait_ld();
#pragma unroll
                        for (int w = 0; w < NH; ++w)
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                zz[h0 + w][i & 1] = __ffma2_rn(
                                    make_float2(__uint_as_float(v[w][2 * i]), __uint_as_float(v[w][2 * i + 1])),
                                    cs[i], zz[h0 + w][i & 1]);
                    }
                }
                tc_fence_before();
            }
#pragma unroll
            for (int hh = 0; hh < HC; ++hh) z[hh] = (zz[hh][0].x + zz[hh][1].x) + (zz[hh][0].y + zz[hh][1].y);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_tempty + 8 * tb);
            // the partner warp's half of the pairs
            float *zmine = zx + (((buf * 4 + q) * 2 + hf) * HC) * 32;
            const float *zother = zx + (((buf * 4 + q) * 2 + (hf ^ 1)) * HC) * 32;
#pragma unroll
            for (int hh = 0; hh < HC; ++hh) zmine[hh * 32 + lane] = z[hh];
            named_sync(2 + q, 64);
            if (tid == 0) GVA_TRACE_AT(101 + 3 * (int)k);
            const bool valid = tau < nv;
            float pz[HC], alpha[HC];
#pragma unroll
            for (int hh = 0; hh < HC; ++hh) {
                const float zt = valid ? z[hh] + zother[hh * 32 + lane] : -INFINITY;
                alpha[hh] = 1.f;
                // the exact maximum is needed only when a score passes the running one by
                // more than the rescale threshold (first tile of a segment, rare later)
                if (__any_sync(0xffffffffu, zt > m[hh] + RK_RESCALE_TH)) {
                    float mx = zt;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    alpha[hh] = exp2f(m[hh] - mx);
                    m[hh] = mx;
                }
                pz[hh] = valid ? exp2f(zt - m[hh]) : 0.f;
                lrun[hh] = lrun[hh] * alpha[hh] + pz[hh];
            }
            // this warp's copy of the probabilities [token][hc], read back per token below
            float *pw = pws + warp * (32 * HC);
            __syncwarp();
#pragma unroll
            for (int hh = 0; hh < HC; ++hh) pw[lane * HC + hh] = pz[hh];
            __syncwarp();
            // value sum over this warp's columns d0 .. d0 + 7 (lane group lg) and tokens
            // ls * TS .. ls * TS + TS - 1 of the quarter; probabilities from their lanes
#pragma unroll
            for (int hh = 0; hh < HC; ++hh)
                if (alpha[hh] != 1.f) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[hh][e] = __fmul2_rn(acc[hh][e], make_float2(alpha[hh], alpha[hh]));
                }
            const unsigned char *vt = sm + nbuf * IMG + sl * STAGE + vkb * (RK_TILE * 128);
#pragma unroll
            for (int i = 0; i < TS; ++i) {
                const int tl = ls * TS + i, tk = 32 * q + tl;
                if (tk < nv) {
                    float ph[HC];
#pragma unroll
                    for (int hh = 0; hh < HC; ++hh) ph[hh] = pw[tl * HC + hh];
                    const uint4 vv = *reinterpret_cast<const uint4 *>(vt + tk * 128 + ((vch ^ (tk & 7)) << 4));
                    float2 v[4];
                    v[0] = make_float2(__uint_as_float(vv.x << 16), __uint_as_float(vv.x & 0xffff0000u));
                    v[1] = make_float2(__uint_as_float(vv.y << 16), __uint_as_float(vv.y & 0xffff0000u));
                    v[2] = make_float2(__uint_as_float(vv.z << 16), __uint_as_float(vv.z & 0xffff0000u));
                    v[3] = make_float2(__uint_as_float(vv.w << 16), __uint_as_float(vv.w & 0xffff0000u));
#pragma unroll
                    for (int hh = 0; hh < HC; ++hh) {
                        const float2 p2 = make_float2(ph[hh], ph[hh]);
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[hh][e] = __ffma2_rn(p2, v[e], acc[hh][e]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * sl);
            if (tid == 0) GVA_TRACE_AT(102 + 3 * (int)k);
            if (it.tile == it.nt - 1 || u + 1 == u1) {
                // end of this CTA's segment of the stream: merge the quarters, write the partial
                const long long slot = (long long)it.stream() + cta;
#pragma unroll
                for (int o = DGW; o < 32; o <<= 1)
#pragma unroll
                    for (int hh = 0; hh < HC; ++hh)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            acc[hh][e].x += __shfl_xor_sync(0xffffffffu, acc[hh][e].x, o);
                            acc[hh][e].y += __shfl_xor_sync(0xffffffffu, acc[hh][e].y, o);
                        }
                if (lane < DGW) {
#pragma unroll
                    for (int hh = 0; hh < HC; ++hh) {
                        float4 *dst = reinterpret_cast<float4 *>(red + (q * HC + hh) * DH + d0);
                        dst[0] = make_float4(acc[hh][0].x, acc[hh][0].y, acc[hh][1].x, acc[hh][1].y);
                        dst[1] = make_float4(acc[hh][2].x, acc[hh][2].y, acc[hh][3].x, acc[hh][3].y);
                    }
                }
#pragma unroll
                for (int hh = 0; hh < HC; ++hh) {
                    float lw = lrun[hh];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
                    if (hf == 0 && lane == 0) {
                        mls[(q * HC + hh) * 2] = m[hh];
                        mls[(q * HC + hh) * 2 + 1] = lw;
                    }
                }
                named_sync(1, RK_EPI_T);
                for (int o = tid; o < HC * DH; o += RK_EPI_T) {
                    const int hh = o / DH;
                    float M = mls[hh * 2];
#pragma unroll
                    for (int w = 1; w < 4; ++w) M = fmaxf(M, mls[(w * HC + hh) * 2]);
                    float sum = 0.f;
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const float mw = mls[(w * HC + hh) * 2];
                        if (mw != -INFINITY) sum += red[w * HC * DH + o] * exp2f(mw - M);
                    }
                    p.part_o[slot * HC * DH + o] = sum;
                }
                if (tid < HC) {
                    float M = mls[tid * 2];
#pragma unroll
                    for (int w = 1; w < 4; ++w) M = fmaxf(M, mls[(w * HC + tid) * 2]);
                    float l = 0.f;
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const float mw = mls[(w * HC + tid) * 2];
                        if (mw != -INFINITY) l += mls[(w * HC + tid) * 2 + 1] * exp2f(mw - M);
                    }
                    p.part_ml[(slot * HC + tid) * 2] = M;
                    p.part_ml[(slot * HC + tid) * 2 + 1] = l;
                }
                named_sync(1, RK_EPI_T);
#pragma unroll
                for (int hh = 0; hh < HC; ++hh) {
                    m[hh] = -INFINITY;
                    lrun[hh] = 0.f;
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[hh][e] = make_float2(0.f, 0.f);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        GVA_TRACE_AT(300);
        GVA_TRACE_FLUSH(0, 320);
    }
    if (warp == RK_EPI_WARPS + 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TCOLS)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------------- //
// Merge
// ---------------------------------------------------------------------------------- //
constexpr int RK_MAX_PARTS = 1024;   // partials of one (sequence, head): at most the grid + 1

// One block per (sequence b, head h): weights of the parts (one thread each), then every
// output column sums its parts' values with all loads independent.
__global__ void __launch_bounds__(RK_MERGE_THREADS) rk_merge_kernel(const RkParams p) {
    __shared__ float wts[RK_MAX_PARTS];
    __shared__ float red[RK_MERGE_THREADS / 32];
    pdl_wait();
    const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
    const int g = h / p.r, hl = h % p.r, hs = hl / p.hc, hh = hl % p.hc;
    const int Gn = p.G * p.nhs, sidx = g * p.nhs + hs;
    const long long s = (long long)b * Gn + sidx;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float *o = p.out + (long long)bh * p.d_h;
    const long long U = p.pre[p.B];
    const int nt = (p.pre[b + 1] - p.pre[b]) / Gn;
    if (U == 0 || nt == 0) {
        for (int dd = tid; dd < p.d_h; dd += blockDim.x) o[dd] = 0.f;
        if (p.lse && tid == 0) p.lse[bh] = -INFINITY;
        return;
    }
    const long long uf = p.pre[b] + (long long)sidx * nt, ul = uf + nt - 1;
    const Part part{U, p.n_ctas};
    const int c0 = part.cta_of(uf), np = part.cta_of(ul) - c0 + 1;
    // slot of part i: s + c0 + i
    const float *ml = p.part_ml + ((s + c0) * p.hc + hh) * 2;
    float mx = -INFINITY;
    for (int i = tid; i < np; i += blockDim.x) mx = fmaxf(mx, ml[(long long)i * p.hc * 2]);
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, k));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    float M = red[0];
    for (int w = 1; w < RK_MERGE_THREADS / 32; ++w) M = fmaxf(M, red[w]);
    __syncthreads();
    float den = 0.f;
    for (int i = tid; i < np; i += blockDim.x) {
        const float w = exp2f(ml[(long long)i * p.hc * 2] - M);
        wts[i] = w;
        den += w * ml[(long long)i * p.hc * 2 + 1];
    }
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) den += __shfl_xor_sync(0xffffffffu, den, k);
    if (lane == 0) red[warp] = den;
    __syncthreads();
    den = 0.f;
    for (int w = 0; w < RK_MERGE_THREADS / 32; ++w) den += red[w];
    const float inv = 1.f / den;
    const float *po = p.part_o + ((s + c0) * p.hc + hh) * p.d_h;
    const long long pstride = (long long)p.hc * p.d_h;
    for (int dd = tid; dd < p.d_h; dd += blockDim.x) {
        float num0 = 0.f, num1 = 0.f;
        int i = 0;
        for (; i + 1 < np; i += 2) {
            num0 += wts[i] * po[i * pstride + dd];
            num1 += wts[i + 1] * po[(i + 1) * pstride + dd];
        }
        if (i < np) num0 += wts[i] * po[i * pstride + dd];
        o[dd] = (num0 + num1) * inv;
    }
    if (p.lse && tid == 0) p.lse[bh] = (M + log2f(den)) * 0.69314718055994531f;
}

// ---------------------------------------------------------------------------------- //
// Host side
// ---------------------------------------------------------------------------------- //
inline int rk_hc(int r, int d_n) {
    for (int hc = 4; hc > 1; hc >>= 1)
        if (r % hc == 0 && hc * d_n <= 256) return hc;
    return 1;
}

inline bool rk_supported(const gva_dims *d) {
    if (d->cache_dtype != GVA_BF16) return false;
    if (d->d_h != 64 && d->d_h != 128) return false;
    if (d->d_n != 64 && d->d_n != 128) return false;
    return true;
}

template <int DH, int DN, int HC>
inline int rk_smem_plan(RkParams &p, int limit) {
    constexpr int N = HC * DN;
    constexpr int IMG = 2 * DH * N * 2, STAGE = RK_TILE * DH * 2;
    const int fixed = 1024 + RkSmem<DH, DN, HC>::total;
    for (int nbuf = 2; nbuf >= 1; --nbuf) {
        int ns = RK_MAX_STAGES;
        while (ns >= 2 && fixed + nbuf * IMG + ns * STAGE + rk_bar_bytes(ns, nbuf) > limit) --ns;
        if (ns >= (nbuf == 2 ? 3 : 2)) {
            p.nbuf = nbuf;
            p.nstages = ns;
            p.smem_bytes = fixed + nbuf * IMG + ns * STAGE + rk_bar_bytes(ns, nbuf);
            return 0;
        }
    }
    return -1;
}

template <int DH, int DN, int HC>
inline cudaError_t rk_opt_in() {
    return cudaFuncSetAttribute(rk_decode_kernel<DH, DN, HC>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, MMA_SMEM_LIMIT);
}

inline cudaError_t rk_opt_in_all() {
    cudaError_t e = cudaSuccess;
#define RK_OPT(DH, DN, HC) \
    if (e == cudaSuccess) e = rk_opt_in<DH, DN, HC>();
    RK_OPT(64, 64, 1) RK_OPT(64, 64, 2) RK_OPT(64, 64, 4)
    RK_OPT(64, 128, 1) RK_OPT(64, 128, 2)
    RK_OPT(128, 64, 1) RK_OPT(128, 64, 2) RK_OPT(128, 64, 4)
    RK_OPT(128, 128, 1) RK_OPT(128, 128, 2)
#undef RK_OPT
    if (e == cudaSuccess) e = cudaFuncSetAttribute(rk_prep_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                                   (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(rk_merge_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                                   (int)cudaSharedmemCarveoutMaxShared);
    return e;
}

// 2D map over the value rows [num_rows][G d_h] (bf16), box {64, ch}, 128-byte swizzle.
inline bool rk_make_map(CUtensorMap *m, const void *V, long long rows, int width, int ch) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t strides[1] = {(cuuint64_t)width * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)ch};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(V), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DH, int DN, int HC>
inline int rk_launch_t(void *stream, RkParams &p, const CUtensorMap &tv) {
    if (rk_smem_plan<DH, DN, HC>(p, MMA_SMEM_LIMIT) != 0) return GVA_ERR_UNSUPPORTED;
    return cuda_status(launch(rk_decode_kernel<DH, DN, HC>, dim3(p.n_ctas), dim3(RK_THREADS),
                              (size_t)p.smem_bytes, stream, tv, p));
}

inline int rk_launch_decode(void *stream, RkParams &p, const CUtensorMap &tv) {
#define RK_CASE(DH_, DN_, HC_) \
    if (p.d_h == DH_ && p.d_n == DN_ && p.hc == HC_) return rk_launch_t<DH_, DN_, HC_>(stream, p, tv);
    RK_CASE(64, 64, 1) RK_CASE(64, 64, 2) RK_CASE(64, 64, 4)
    RK_CASE(64, 128, 1) RK_CASE(64, 128, 2)
    RK_CASE(128, 64, 1) RK_CASE(128, 64, 2) RK_CASE(128, 64, 4)
    RK_CASE(128, 128, 1) RK_CASE(128, 128, 2)
#undef RK_CASE
    return GVA_ERR_UNSUPPORTED;
}

}  // namespace gva
