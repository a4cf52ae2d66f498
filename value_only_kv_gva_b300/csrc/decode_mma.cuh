// decode_mma.cuh -- split-K GVA decode on the tensor cores for bf16 caches.
//
// Per CTA (one per SM): one producer warp streams 16-token slabs of the cache into a
// ring of shared-memory stages with TMA tensor copies (cp.async.bulk.tensor, 128-byte
// swizzle, mbarrier completion); consumer warps, each bound to one value group, score
// and accumulate with bf16 mma.sync (m16n8k16, fp32 accumulate):
//
//   S^T[16 x 8 tok]  = Q[16 x d_h] . V_g^T[d_h x 8 tok] (+ Q_r[16 x d_r] . K_rope^T)
//   O[16 x d_h]     += P[16 x 16 tok] . V_g[16 tok x d_h]
//
// The 16 rows hold the group's r <= 8 heads twice: row h carries the bf16 "hi" part
// of the fp32 query / probability and row h + 8 its "lo" remainder (x - hi), so the
// products keep about 16 mantissa bits; the two rows are summed in fp32 afterwards.
// The V tile serves as the B operand of both products: plain ldmatrix for scores,
// ldmatrix.trans for the weighted sum.  Each cache byte is read from HBM once.
//
// Online softmax in log2 units with a lazy rescale: the running maximum is raised
// only when a slab's maximum exceeds it by more than 8, so probabilities stay below
// 2^8 and the accumulator rescale (a multiply of every O register) is rare.
//
// Every wait on an mbarrier is bounded by a wall-clock limit; on expiry the kernel
// sets GVA_DEV_TIMEOUT, stops issuing work, waits (bounded) for the copies it has in
// flight and returns.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "decode_simt.cuh"
#include "launch.cuh"

namespace gva {

constexpr int MMA_CONSUMERS = 8;                      // consumer warps per CTA (G * warps per group)
constexpr int MMA_THREADS = (MMA_CONSUMERS + 1) * 32; // + one producer warp
constexpr int MMA_MAX_STAGES = 24;
constexpr float MMA_RESCALE_TH = 8.f;                 // log2 units
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;

struct MmaParams {
    DecodeParams d;
    int nstages;
    int stage_bytes;   // multiple of 1024
    int off_k;         // GQA key slab within a stage
    int off_r;         // positional-key slab within a stage
    int tx_bytes;      // bytes the TMA writes per stage
    int wpg;           // consumer warps per value group
    int ncons;         // G * wpg consumer warps
    int off_bar;       // barriers, from the aligned dynamic smem base
    int off_f;         // Ls[B], F[B+1]
    int off_merge;     // group-merge buffer
    int v3d;           // 1: one 3D TMA box per slab covers every value column
    int early;         // 1: the preceding kernel only writes the queries, so the cache
                       //    may be streamed before the grid dependency resolves
};

// Optional timeline of a few CTAs (compiled in only with -DGVA_TRACE; a debugging aid
// for measuring where a CTA spends its cycles, read back by gva_debug_trace_read).
#ifdef GVA_TRACE
constexpr int TRACE_CTAS = 4, TRACE_SLOTS = 512;
__device__ long long g_trace[TRACE_CTAS * TRACE_SLOTS];
#define GVA_TRACE_AT(slot)                                                          \
    do {                                                                            \
        if (blockIdx.x < TRACE_CTAS && (slot) < TRACE_SLOTS)                        \
            g_trace[blockIdx.x * TRACE_SLOTS + (slot)] = clock64();                 \
    } while (0)
#else
#define GVA_TRACE_AT(slot) \
    do {                   \
    } while (0)
#endif

// ---------------------------------------------------------------------------- //
// PTX wrappers
// ---------------------------------------------------------------------------- //
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t a, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t a, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t a) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t a, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for the phase with the given parity.  Gives up (returns false) when
// another warp raised `abort` or after WAIT_LIMIT_NS, raising abort and the status.
__device__ __forceinline__ bool mbar_wait(uint32_t a, uint32_t parity, volatile int *abort) {
    if (mbar_try_wait(a, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(a, parity)) return true;
        if (*abort) return false;
        if (global_ns() - t0 > WAIT_LIMIT_NS) {
            *abort = 1;
            dev_report(GVA_DEV_TIMEOUT);
            return false;
        }
    }
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *tm, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *tm, int x, int y,
                                            int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t a, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t a, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(a));
}
__device__ __forceinline__ void ldsm_x2(uint32_t a, uint32_t &r0, uint32_t &r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(a));
}
__device__ __forceinline__ void mma16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma1688(float c[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(b0));
}
__device__ __forceinline__ void named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ uint32_t pack_bf16(float lo_half, float hi_half) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo_half, hi_half);
    return *reinterpret_cast<uint32_t *>(&v);
}
// (x0, x1) -> bf16 pair hi = rn(x) and remainder lo = rn(x - hi)
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// Byte address of the 16-byte chunk c (8 bf16 along d) of token row t of group g's
// tile within a stage: one TMA box of 16 rows x 128 bytes per 64 columns, swizzled
// by XOR-ing the chunk index with (row mod 8).
template <int DH>
__device__ __forceinline__ uint32_t vtile_addr(uint32_t base, int g, int t, int c) {
    const int box = g * (DH / 64) + (c >> 3);
    return base + box * 2048 + t * 128 + (((c & 7) ^ (t & 7)) << 4);
}

// ---------------------------------------------------------------------------- //
// the kernel
// ---------------------------------------------------------------------------- //
template <int DH, int DR, bool GQA>
__global__ void __launch_bounds__(MMA_THREADS, 1)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_r, const MmaParams mp) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const DecodeParams &p = mp.d;
    // 1024-byte aligned base for the swizzled stages
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
    unsigned char *base = smem_raw + (base_u32 - raw_u32);
    const int NS = mp.nstages;
    const uint32_t bar_full = base_u32 + mp.off_bar;          // NS x 8 bytes
    const uint32_t bar_empty = bar_full + 8 * NS;             // NS x 8 bytes
    volatile int *abort = reinterpret_cast<volatile int *>(base + mp.off_bar + 16 * NS);
    int *Ls = reinterpret_cast<int *>(base + mp.off_f);
    int *F = Ls + p.B;
    float *merge = reinterpret_cast<float *>(base + mp.off_merge);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.G, r = p.r, B = p.B, H = p.H;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, (uint32_t)G);
        }
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == mp.ncons && lane == 0) {
        prefetch_tmap(&tm_v);
        if (GQA) prefetch_tmap(&tm_k);
        if (DR > 0) prefetch_tmap(&tm_r);
    }
    if (threadIdx.x == 0) GVA_TRACE_AT(0);
    // Lengths, row maps and the cache are final before the preceding grid (the query
    // absorption) was allowed to start, so with `early` they are read at once and the
    // cache streams while that grid still runs; the queries are read after the wait.
    if (!mp.early) pdl_wait();
    pdl_launch_dependents();
    build_prefix(p.seq_len, p.R, B, Ls, F, blockIdx.x == 0);   // includes __syncthreads
    if (threadIdx.x == 0) GVA_TRACE_AT(1);
    const Part P{F[B], p.n_ctas};
    if (P.S == 0) return;
    const int c = blockIdx.x;
    const long long s0 = P.start(c), s1 = P.start(c + 1);
    if (s0 >= s1) return;

    // ============================= producer warp ============================= //
    if (warp == mp.ncons) {
        if (lane == 0) {
            unsigned int last_phase_mask = 0, issued_mask = 0;  // per stage (NS <= 32)
            int b = seq_of_slab(F, B, s0);
            int stage = 0;
            uint32_t round = 0;                 // times the ring has wrapped
            const int nbox = G * (DH / 64);
            const int nslab = (int)(s1 - s0);
            for (int i = 0; i < nslab; ++i) {
                const long long s = s0 + i;
                while (F[b + 1] <= s) ++b;
                if (round > 0 && !mbar_wait(bar_empty + 8 * stage, (round - 1) & 1u, abort)) break;
                const long long j0 = (long long)(s - F[b]) * SLAB;
                long long row = row_of(p.R, b, j0);
                if (row < 0) row = 0;  // consumers mask a slab behind a bad page id
                const int y = (int)row;
                const uint32_t st = base_u32 + stage * mp.stage_bytes;
                const uint32_t fb = bar_full + 8 * stage;
                mbar_expect_tx(fb, (uint32_t)mp.tx_bytes);
                if (mp.v3d) {
                    tma_load_3d(st, &tm_v, 0, y, 0, fb);
                    if (GQA) tma_load_3d(st + mp.off_k, &tm_k, 0, y, 0, fb);
                } else {
                    for (int bx = 0; bx < nbox; ++bx) {
                        tma_load_2d(st + bx * 2048, &tm_v, bx * 64, y, fb);
                        if (GQA) tma_load_2d(st + mp.off_k + bx * 2048, &tm_k, bx * 64, y, fb);
                    }
                }
                if (DR > 0) tma_load_2d(st + mp.off_r, &tm_r, 0, y, fb);
                issued_mask |= 1u << stage;
                last_phase_mask = (last_phase_mask & ~(1u << stage)) | ((round & 1u) << stage);
                if (i == 0) GVA_TRACE_AT(2);
                if (++stage == NS) {
                    stage = 0;
                    ++round;
                }
            }
            GVA_TRACE_AT(3);
            // never leave with copies in flight: wait (bounded) for each stage's last load
            for (int s = 0; s < NS; ++s) {
                if (!(issued_mask & (1u << s))) continue;
                const uint32_t par = (last_phase_mask >> s) & 1u;
                const unsigned long long t0 = global_ns();
                while (!mbar_try_wait(bar_full + 8 * s, par)) {
                    if (global_ns() - t0 > WAIT_LIMIT_NS) {
                        dev_report(GVA_DEV_TIMEOUT);
                        break;
                    }
                }
            }
        }
        return;
    }

    // ============================= consumer warps ============================ //
    if (warp > mp.ncons) return;      // spare warps when G does not divide the consumer count
    const int g = warp % G;           // value group of this warp
    const int w = warp / G;           // rank among the group's warps
    const int wpg = mp.wpg;
    const int gid = lane >> 2, tig = lane & 3;
    const bool real_row = gid < r;    // lanes whose row (gid) is a real head of the group
    const int h = g * r + gid;        // head of this lane's rows (when real_row)

    // ldmatrix lane roles
    const int lm_mat = lane >> 3, lm_row = lane & 7;

    if (mp.early) pdl_wait();         // the absorbed queries come from the preceding grid
    int b = seq_of_slab(F, B, s0);
    int stage = 0, wsel = 0;          // ring stage and slab-owner counter of the next slab
    uint32_t phase = 0;
    int tslab = 0;                    // trace index
    long long s = s0;
    bool alive = true;
    while (s < s1) {
        while (F[b + 1] <= s) ++b;
        const long long seg_end = min(s1, (long long)F[b + 1]);
        const int Lb = Ls[b];

        // ---- query fragments for (b, g): hi part in row gid, lo part in row gid + 8 ----
        uint32_t qa[DH / 16][4];
        {
            const long long qoff = ((long long)b * H + h) * DH;
#pragma unroll
            for (int kk = 0; kk < DH / 16; ++kk) {
                float x[4] = {0.f, 0.f, 0.f, 0.f};
                if (real_row) {
                    const int d0 = kk * 16 + tig * 2;
                    if (p.qc_f32) {
                        const float *qf = reinterpret_cast<const float *>(p.qc) + qoff;
                        x[0] = qf[d0]; x[1] = qf[d0 + 1]; x[2] = qf[d0 + 8]; x[3] = qf[d0 + 9];
                    } else {
                        const __nv_bfloat16 *qb = reinterpret_cast<const __nv_bfloat16 *>(p.qc) + qoff;
                        x[0] = __bfloat162float(qb[d0]); x[1] = __bfloat162float(qb[d0 + 1]);
                        x[2] = __bfloat162float(qb[d0 + 8]); x[3] = __bfloat162float(qb[d0 + 9]);
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) x[e] *= p.qc_scale;
                }
                split_bf16(x[0], x[1], qa[kk][0], qa[kk][1]);
                split_bf16(x[2], x[3], qa[kk][2], qa[kk][3]);
            }
        }
        constexpr int DRK16 = DR / 16;          // full k16 steps over the positional slice
        constexpr bool DR_K8 = (DR % 16) == 8;  // one trailing k8 step
        uint32_t ra[DRK16 > 0 ? DRK16 : 1][4];
        uint32_t ra8[2];
        if (DR > 0) {
            const float *qr = p.qr + ((long long)b * H + h) * DR;
#pragma unroll
            for (int kk = 0; kk < DRK16; ++kk) {
                float x[4] = {0.f, 0.f, 0.f, 0.f};
                if (real_row) {
                    const int d0 = kk * 16 + tig * 2;
                    x[0] = qr[d0]; x[1] = qr[d0 + 1]; x[2] = qr[d0 + 8]; x[3] = qr[d0 + 9];
                }
                split_bf16(x[0], x[1], ra[kk][0], ra[kk][1]);
                split_bf16(x[2], x[3], ra[kk][2], ra[kk][3]);
            }
            if (DR_K8) {
                float x0 = 0.f, x1 = 0.f;
                if (real_row) {
                    const int d0 = DRK16 * 16 + tig * 2;
                    x0 = qr[d0]; x1 = qr[d0 + 1];
                }
                split_bf16(x0, x1, ra8[0], ra8[1]);
            }
        }

        float oacc[DH / 8][4];
#pragma unroll
        for (int nd = 0; nd < DH / 8; ++nd)
            oacc[nd][0] = oacc[nd][1] = oacc[nd][2] = oacc[nd][3] = 0.f;
        float m_run = -INFINITY, l_run = 0.f;

        if (w == 0 && g == 0 && lane == 0) GVA_TRACE_AT(4);
        for (; s < seg_end; ++s) {
            const int my_stage = stage;
            const uint32_t my_phase = phase;
            const bool mine = wsel == w;
            if (++stage == NS) { stage = 0; phase ^= 1u; }
            if (++wsel == wpg) wsel = 0;
            if (!mine || !alive) continue;
            if (!mbar_wait(bar_full + 8 * my_stage, my_phase, abort)) {
                alive = false;
                continue;
            }
            if (w == 0 && g == 0 && lane == 0) GVA_TRACE_AT(8 + 2 * tslab);
            const long long j0 = (long long)(s - F[b]) * SLAB;
            int nv = (int)min((long long)SLAB, (long long)Lb - j0);
            if (row_of(p.R, b, j0) < 0) {
                if (lane == 0 && g == 0) dev_report(GVA_DEV_BAD_PAGE);
                nv = 0;
            }
            const uint32_t st = base_u32 + my_stage * mp.stage_bytes;
            const uint32_t kst = GQA ? st + mp.off_k : st;

            // ---- scores S^T = Q . K^T for tokens 8nt .. 8nt+7 ----
            float sc[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
                for (int kp = 0; kp < DH / 32; ++kp) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(vtile_addr<DH>(kst, g, nt * 8 + lm_row, kp * 4 + lm_mat), b0, b1, b2, b3);
                    mma16816(sc[nt], qa[2 * kp], b0, b1);
                    mma16816(sc[nt], qa[2 * kp + 1], b2, b3);
                }
            }
            if (DR > 0) {
                const uint32_t rbase = st + mp.off_r;
#pragma unroll
                for (int kk = 0; kk < DRK16; ++kk) {
                    // matrices: (nt0, chunk 2kk), (nt0, 2kk+1), (nt1, 2kk), (nt1, 2kk+1)
                    const int t = (lm_mat >> 1) * 8 + lm_row;
                    const int ch = 2 * kk + (lm_mat & 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(rbase + t * (DR * 2) + ch * 16, b0, b1, b2, b3);
                    mma16816(sc[0], ra[kk], b0, b1);
                    mma16816(sc[1], ra[kk], b2, b3);
                }
                if (DR_K8) {
                    const int t = (lm_mat & 1) * 8 + lm_row;
                    uint32_t b0, b1;
                    ldsm_x2(rbase + t * (DR * 2) + DRK16 * 32, b0, b1);
                    mma1688(sc[0], ra8[0], ra8[1], b0);
                    mma1688(sc[1], ra8[0], ra8[1], b1);
                }
            }
            // ---- hi + lo rows -> one score per (head gid, token) ----
            // lane holds tokens 8nt + 2tig + {0,1}
            float z[2][2];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                z[nt][0] = sc[nt][0] + sc[nt][2];
                z[nt][1] = sc[nt][1] + sc[nt][3];
            }
            if (nv < SLAB) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        if (nt * 8 + 2 * tig + e >= nv) z[nt][e] = -INFINITY;
            }
            float mloc = fmaxf(fmaxf(z[0][0], z[0][1]), fmaxf(z[1][0], z[1][1]));
            mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 1));
            mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 2));
            const bool raise = mloc > m_run + MMA_RESCALE_TH;
            if (__any_sync(0xffffffffu, raise)) {
                const float alpha = raise ? exp2f(m_run - mloc) : 1.f;  // 0 when m_run = -inf
                if (raise) m_run = mloc;
                l_run *= alpha;
#pragma unroll
                for (int nd = 0; nd < DH / 8; ++nd) {
                    oacc[nd][0] *= alpha; oacc[nd][1] *= alpha;
                    oacc[nd][2] *= alpha; oacc[nd][3] *= alpha;
                }
            }
            float pr[2][2];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float v = exp2f(z[nt][e] - m_run);
                    pr[nt][e] = (z[nt][e] == -INFINITY) ? 0.f : v;
                }
            l_run += (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
            // ---- P as the A operand: rows gid (hi) / gid + 8 (lo), k = token ----
            uint32_t pa[4];
            split_bf16(pr[0][0], pr[0][1], pa[0], pa[1]);
            split_bf16(pr[1][0], pr[1][1], pa[2], pa[3]);
            // ---- O += P . V ----
#pragma unroll
            for (int np = 0; np < DH / 16; ++np) {
                // matrices: (tok 0-7, chunk 2np), (tok 8-15, 2np), (tok 0-7, 2np+1), (tok 8-15, 2np+1)
                const int t = (lm_mat & 1) * 8 + lm_row;
                const int ch = 2 * np + (lm_mat >> 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vtile_addr<DH>(st, g, t, ch), b0, b1, b2, b3);
                if (nv < SLAB) {
                    // zero the values of tokens past the end (they may hold NaN)
                    const int ta = 2 * tig, tb = 8 + 2 * tig;
                    const uint32_t ma = (ta >= nv ? 0u : 0xffffu) | (ta + 1 >= nv ? 0u : 0xffff0000u);
                    const uint32_t mb = (tb >= nv ? 0u : 0xffffu) | (tb + 1 >= nv ? 0u : 0xffff0000u);
                    b0 &= ma; b1 &= mb; b2 &= ma; b3 &= mb;
                }
                mma16816(oacc[2 * np], pa, b0, b1);
                mma16816(oacc[2 * np + 1], pa, b2, b3);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * my_stage);
            if (w == 0 && g == 0 && lane == 0) GVA_TRACE_AT(9 + 2 * tslab);
            ++tslab;
        }

        // ---- segment end: fold hi/lo rows, reduce l over the quad, merge the group's warps ----
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
        float o2[DH / 8][2];
#pragma unroll
        for (int nd = 0; nd < DH / 8; ++nd) {
            o2[nd][0] = oacc[nd][0] + oacc[nd][2];
            o2[nd][1] = oacc[nd][1] + oacc[nd][3];
        }
        if (wpg > 1) {
            // slot per (extra warp, group): 8 heads x (DH + 2) floats
            const int stride = 8 * (DH + 2);
            if (w > 0) {
                float *mb = merge + ((w - 1) * G + g) * stride + gid * (DH + 2);
#pragma unroll
                for (int nd = 0; nd < DH / 8; ++nd) {
                    mb[nd * 8 + 2 * tig] = o2[nd][0];
                    mb[nd * 8 + 2 * tig + 1] = o2[nd][1];
                }
                if (tig == 0) { mb[DH] = m_run; mb[DH + 1] = l_run; }
            }
            named_bar(1 + g, wpg * 32);
            if (w == 0) {
                for (int ww = 1; ww < wpg; ++ww) {
                    const float *mb = merge + ((ww - 1) * G + g) * stride + gid * (DH + 2);
                    const float m2 = mb[DH], l2 = mb[DH + 1];
                    const float mn = fmaxf(m_run, m2);
                    const float a1 = (m_run == -INFINITY) ? 0.f : exp2f(m_run - mn);
                    const float a2 = (m2 == -INFINITY) ? 0.f : exp2f(m2 - mn);
#pragma unroll
                    for (int nd = 0; nd < DH / 8; ++nd) {
                        o2[nd][0] = o2[nd][0] * a1 + mb[nd * 8 + 2 * tig] * a2;
                        o2[nd][1] = o2[nd][1] * a1 + mb[nd * 8 + 2 * tig + 1] * a2;
                    }
                    l_run = l_run * a1 + l2 * a2;
                    m_run = mn;
                }
            }
            named_bar(1 + g, wpg * 32);
        }
        if (w == 0 && g == 0 && lane == 0) GVA_TRACE_AT(5);
        if (w == 0 && real_row) {
            const bool whole = F[b] >= s0 && F[b + 1] <= s1;
            if (whole) {
                const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
                float *o = p.out + ((long long)b * H + h) * DH;
#pragma unroll
                for (int nd = 0; nd < DH / 8; ++nd)
                    *reinterpret_cast<float2 *>(o + nd * 8 + 2 * tig) =
                        make_float2(o2[nd][0] * inv, o2[nd][1] * inv);
                if (tig == 0 && p.lse)
                    p.lse[(long long)b * H + h] = l_run > 0.f ? (m_run + log2f(l_run)) * LN2 : -INFINITY;
            } else {
                const long long slot = (long long)c + b;
                float *o = p.part_o + (slot * H + h) * DH;
#pragma unroll
                for (int nd = 0; nd < DH / 8; ++nd)
                    *reinterpret_cast<float2 *>(o + nd * 8 + 2 * tig) = make_float2(o2[nd][0], o2[nd][1]);
                if (tig == 0) {
                    p.part_ml[(slot * H + h) * 2] = m_run;
                    p.part_ml[(slot * H + h) * 2 + 1] = l_run;
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------- //
// host side
// ---------------------------------------------------------------------------- //
inline bool mma_supported(const gva_dims *d) {
    if (d->cache_dtype != GVA_BF16) return false;
    if (d->d_h != 64 && d->d_h != 128) return false;
    if (d->G > MMA_CONSUMERS || d->H / d->G > 8) return false;
    if (d->d_r != 0 && d->d_r != 8 && d->d_r != 16 && d->d_r != 24 && d->d_r != 32) return false;
    return true;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// 2D bf16 map over `rows` rows of `width` elements; box = box_w x 16 rows.
inline bool make_map(CUtensorMap *m, const void *ptr, long long rows, int width, int box_w,
                     bool swizzle128) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)width * 2};
    cuuint32_t box[2] = {(cuuint32_t)box_w, (cuuint32_t)SLAB};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3D bf16 map viewing each row of `width` elements as width/64 chunks of 64: dims
// {64, rows, width/64}, strides {row pitch, 128 B}; one box {64, 16, width/64} lands
// in shared memory chunk-major ([chunk][16 rows][64]), each chunk 128-byte swizzled.
inline bool make_map3(CUtensorMap *m, const void *ptr, long long rows, int width) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(width / 64)};
    cuuint64_t strides[2] = {(cuuint64_t)width * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)SLAB, (cuuint32_t)(width / 64)};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int MMA_SMEM_LIMIT = 227 * 1024;

inline bool plan_mma(MmaParams &mp, int DH, int DR, bool gqa) {
    const DecodeParams &d = mp.d;
    const int vbytes = d.G * DH * SLAB * 2;
    mp.off_k = vbytes;
    mp.off_r = vbytes * (gqa ? 2 : 1);
    const int rbytes = DR * SLAB * 2;
    mp.tx_bytes = mp.off_r + rbytes;
    mp.stage_bytes = (int)align_up((size_t)mp.tx_bytes, 1024);
    mp.wpg = MMA_CONSUMERS / d.G;
    if (mp.wpg < 1) mp.wpg = 1;
    mp.ncons = d.G * mp.wpg;
    const int merge_bytes = (mp.wpg - 1) * d.G * 8 * (DH + 2) * 4;
    const int fixed = 1024 /* alignment slack */ + (int)align_up(sizeof(int) * (2 * d.B + 1), 16) +
                      merge_bytes + 16 * MMA_MAX_STAGES + 16;
    int ns = (MMA_SMEM_LIMIT - fixed) / mp.stage_bytes;
    if (ns > MMA_MAX_STAGES) ns = MMA_MAX_STAGES;
    if (ns < 2) return false;
    mp.nstages = ns;
    mp.off_bar = ns * mp.stage_bytes;
    mp.off_f = mp.off_bar + (int)align_up(16 * ns + 16, 16);
    mp.off_merge = mp.off_f + (int)align_up(sizeof(int) * (2 * d.B + 1), 16);
    return true;
}

inline size_t mma_smem_bytes(const MmaParams &mp, int DH) {
    const int merge_bytes = (mp.wpg - 1) * mp.d.G * 8 * (DH + 2) * 4;
    return 1024 + (size_t)mp.off_merge + merge_bytes;
}

template <int DH, int DR, bool GQA>
inline int launch_mma_t(void *stream, MmaParams &mp, const CUtensorMap &tv, const CUtensorMap &tk,
                        const CUtensorMap &tr, int grid) {
    auto kern = decode_mma_kernel<DH, DR, GQA>;
    const size_t smem = mma_smem_bytes(mp, DH);
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(MMA_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_allowed(cfg.stream) ? 1 : 0;
    return cuda_status(cudaLaunchKernelEx(&cfg, kern, tv, tk, tr, mp));
}

// Shared-memory opt-in of every instantiation (once per device, before any launch).
inline cudaError_t mma_opt_in_all() {
    const void *ks[] = {
        (const void *)decode_mma_kernel<64, 0, false>, (const void *)decode_mma_kernel<64, 8, false>,
        (const void *)decode_mma_kernel<64, 16, false>, (const void *)decode_mma_kernel<64, 24, false>,
        (const void *)decode_mma_kernel<64, 32, false>, (const void *)decode_mma_kernel<64, 0, true>,
        (const void *)decode_mma_kernel<128, 0, false>, (const void *)decode_mma_kernel<128, 8, false>,
        (const void *)decode_mma_kernel<128, 16, false>, (const void *)decode_mma_kernel<128, 24, false>,
        (const void *)decode_mma_kernel<128, 32, false>, (const void *)decode_mma_kernel<128, 0, true>};
    for (const void *k : ks) {
        const cudaError_t e =
            cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, MMA_SMEM_LIMIT);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int DH>
inline int launch_mma_dr(void *stream, MmaParams &mp, const CUtensorMap &tv, const CUtensorMap &tk,
                         const CUtensorMap &tr, int grid, int DR, bool gqa) {
    if (gqa) return launch_mma_t<DH, 0, true>(stream, mp, tv, tk, tr, grid);
    switch (DR) {
    case 0: return launch_mma_t<DH, 0, false>(stream, mp, tv, tk, tr, grid);
    case 8: return launch_mma_t<DH, 8, false>(stream, mp, tv, tk, tr, grid);
    case 16: return launch_mma_t<DH, 16, false>(stream, mp, tv, tk, tr, grid);
    case 24: return launch_mma_t<DH, 24, false>(stream, mp, tv, tk, tr, grid);
    case 32: return launch_mma_t<DH, 32, false>(stream, mp, tv, tk, tr, grid);
    default: return GVA_ERR_UNSUPPORTED;
    }
}

// Sets dp.n_ctas and launches the tensor-core decode (one CTA per SM by default).
inline int run_mma(void *stream, DecodeParams &dp, const gva_rows &rows, int sms, int req_ctas,
                   bool gqa, bool early) {
    if (rows.num_rows > 0x7fffffffLL) return GVA_ERR_UNSUPPORTED;   // TMA row coordinate is int32
    MmaParams mp;
    mp.d = dp;
    const int DH = dp.d_h, DR = gqa ? 0 : dp.d_r;
    if (!plan_mma(mp, DH, DR, gqa)) return GVA_ERR_UNSUPPORTED;
    const long long nrows = rows.num_rows > 0 ? rows.num_rows : 1;
    CUtensorMap tv, tk, tr;
    mp.early = early ? 1 : 0;
    mp.v3d = make_map3(&tv, dp.Vc, nrows, dp.G * DH) &&
             (!gqa || make_map3(&tk, dp.Kc, nrows, dp.G * DH));
    if (!mp.v3d) {
        if (!make_map(&tv, dp.Vc, nrows, dp.G * DH, 64, true)) return GVA_ERR_CUDA;
        if (gqa && !make_map(&tk, dp.Kc, nrows, dp.G * DH, 64, true)) return GVA_ERR_CUDA;
    }
    if (!gqa) tk = tv;
    tr = tv;
    if (DR > 0 && !make_map(&tr, dp.Krope, nrows, DR, DR, false)) return GVA_ERR_CUDA;
    int grid = req_ctas > 0 ? req_ctas : sms;
    if (grid > sms * 8) grid = sms * 8;
    dp.n_ctas = grid;
    mp.d.n_ctas = grid;
    return DH == 64 ? launch_mma_dr<64>(stream, mp, tv, tk, tr, grid, DR, gqa)
                    : launch_mma_dr<128>(stream, mp, tv, tk, tr, grid, DR, gqa);
}

}  // namespace gva
