// decode_mma.cuh -- split-K GVA decode on the tensor cores for bf16 caches.
//
// Per CTA (one per SM): one producer warp streams 16-token slabs of the cache into a
// ring of shared-memory stages with TMA tensor copies (one 3D box per slab covering
// every value column, 128-byte swizzle, plus a bulk copy of the slab's positional keys;
// mbarrier completion); consumer warps, each bound to one value group, score and
// accumulate with bf16 mma.sync (m16n8k16, fp32 accumulate) with the slab's 16 tokens
// on the MMA rows and the group's heads on the columns:
//
//   S[16 tok x 8]    = V_g[16 tok x d_h] . Q^T[d_h x 8]   (+ K_rope . Q_r^T)
//   O^T[d_h x 8]    += V_g^T[d_h x 16 tok] . P^T[16 tok x 8]
//
// Each 8-column tile holds up to 4 heads twice: column 2i carries the bf16 "hi" part
// of head i's fp32 query / probability and column 2i + 1 its "lo" remainder (x - hi),
// so the products keep about 16 mantissa bits; the two columns are summed in fp32
// afterwards (r <= 4 heads per group: one tile, r <= 8: two).  The value tile is the A
// operand of both products: plain ldmatrix for the scores, ldmatrix.trans for the
// weighted sum.  Each cache byte is read from HBM once.
//
// Online softmax in log2 units with a lazy rescale: the running maximum moves only when
// a score exceeds it by more than 8 (2^8 in probability), so the accumulator rescale
// (a multiply of every O register) and the max reduction over the token lanes are rare.
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

// Warp roles: warp 0 is the producer, warps 1 .. ncons the consumers (G x warps per
// group, at most 8).  The launch bound caps a thread at 128 registers, so a CTA (at most
// 9 warps) leaves a third of the SM's register file, and some of its shared memory, to
// the small kernels around the decode: the query absorption before it and the
// log-sum-exp combine after it are resident beside it under programmatic dependent
// launch instead of waiting for the SM to drain.
#ifndef GVA_MMA_CONSUMERS
#define GVA_MMA_CONSUMERS 8
#endif
#ifndef GVA_MMA_THREADS
#define GVA_MMA_THREADS 512
#endif
constexpr int MMA_CONSUMERS = GVA_MMA_CONSUMERS;      // at most GVA_MMA_THREADS / 32 - 1
constexpr int MMA_TRIPLE_CONSUMERS = 4;               // consumer warps of the three-per-SM plan
constexpr int MMA_THREADS = GVA_MMA_THREADS;          // launch bound (512 -> <= 128 registers)
static_assert((MMA_CONSUMERS + 1) * 32 <= MMA_THREADS, "consumer warps exceed the launch bound");
constexpr float MMA_RESCALE_TH = 8.f;                 // log2 units
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;
constexpr int MMA_MAX_STAGES = 24;

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
    int off_f;         // Ls[B], F[B+1] (and Hs[B] with hold_pos)
    int off_merge;     // group-merge buffer
    int v3d;           // 1: one 3D TMA box per slab covers every value column
    int vg;            // value groups stored per row: G, or 1 when every group of heads
                       //    reads the same row (the latent rows of the MLA-shaped decode)
    int early;         // 1: the preceding kernel only writes the queries, so the cache
                       //    may be streamed before the grid dependency resolves
    const int *hold_pos;  // with early: the preceding kernel also writes row hold_pos[b] of
                          //    each sequence b, so the producer waits on the grid dependency
                          //    before it copies the slab holding that row (Hs after F)
};

// Optional timeline of a few CTAs (compiled in only with -DGVA_TRACE; a debugging aid
// for measuring where a CTA spends its cycles, read back by gva_debug_trace_read).
#ifdef GVA_TRACE
constexpr int TRACE_CTAS = 4, TRACE_SLOTS = 512;
__device__ long long g_trace[TRACE_CTAS * TRACE_SLOTS];
// stamps go to shared memory (a global store before an mbarrier arrive would delay the
// arrive until the store completes) and are copied out when the stamping thread exits
__shared__ long long s_trace[TRACE_SLOTS];
#define GVA_TRACE_DECL
#define GVA_TRACE_AT(slot)                                                          \
    do {                                                                            \
        if ((slot) < TRACE_SLOTS) s_trace[(slot)] = clock64();                      \
    } while (0)
#define GVA_TRACE_FLUSH(lo, hi)                                                     \
    do {                                                                            \
        if (blockIdx.x < TRACE_CTAS)                                                \
            for (int i_ = (lo); i_ < (hi) && i_ < TRACE_SLOTS; ++i_)               \
                g_trace[blockIdx.x * TRACE_SLOTS + i_] = s_trace[i_];               \
    } while (0)
#else
#define GVA_TRACE_DECL
#define GVA_TRACE_AT(slot) \
    do {                   \
    } while (0)
#define GVA_TRACE_FLUSH(lo, hi) \
    do {                        \
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
// Arrive without release semantics, for a consumer giving a stage back: every read of
// the stage has already returned its data (the values were consumed by the products),
// so there is nothing for a release to order.
__device__ __forceinline__ void mbar_arrive_relaxed(uint32_t a) {
    asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
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
// As mbar_try_wait, but the thread may be suspended in hardware for up to `ns`
// nanoseconds while the phase is incomplete, so waiting warps leave the issue slots
// to the warps that have work (the producer shares its scheduler with consumers).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t a, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(a), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}
constexpr uint32_t WAIT_SLEEP_NS = 1000000u;   // per try; the overall limit is WAIT_LIMIT_NS
// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint32_t a, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for the phase with the given parity.  Gives up (returns false) when
// another warp raised `abort` or after `limit_ns`, raising abort and the status.
__device__ __forceinline__ bool mbar_wait_for(uint32_t a, uint32_t parity, volatile int *abort,
                                              unsigned long long limit_ns) {
    if (mbar_test_wait(a, parity)) return true;
    const unsigned long long t0 = global_ns();
    const uint32_t sleep = limit_ns < WAIT_SLEEP_NS ? (uint32_t)limit_ns : WAIT_SLEEP_NS;
    for (;;) {
        if (mbar_try_wait_sleep(a, parity, sleep)) return true;
        if (*abort) return false;
        if (global_ns() - t0 > limit_ns) {
            *abort = 1;
            dev_report(GVA_DEV_TIMEOUT);
            return false;
        }
    }
}
__device__ __forceinline__ bool mbar_wait(uint32_t a, uint32_t parity, volatile int *abort) {
    return mbar_wait_for(a, parity, abort, WAIT_LIMIT_NS);
}
// The cache is streamed once per step: its loads carry an L2 evict-first policy, so
// that they do not push out of L2 what is reused (the kernels' code, the maps M, the
// queries and the split partials).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *tm, int x, int y,
                                            uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *tm, int x, int y,
                                            int z, uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(pol)
        : "memory");
}
// Plain (non-tensor) bulk copy of `bytes` contiguous bytes: 16-byte aligned addresses,
// a multiple of 16 bytes.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(pol)
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
// The MMA wrappers are not volatile: they only read their operands and accumulators, so
// the compiler may interleave independent products; the ldmatrix wrappers above stay
// volatile so that no shared-memory read moves above the barrier wait that guards it.
__device__ __forceinline__ void mma16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma1688(float c[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm(
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

// One part of the bf16 hi/lo split of (x0, x1), packed: the hi part rn(x), or the
// remainder rn(x - hi) when `lo` is set.
__device__ __forceinline__ uint32_t part_bf16x2(float x0, float x1, bool lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    if (!lo) return *reinterpret_cast<const uint32_t *>(&h);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    return *reinterpret_cast<const uint32_t *>(&l);
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
// consumer building blocks (shared by the tensor-core decode kernels)
// ---------------------------------------------------------------------------- //
// Products with a slab's 16 tokens on the MMA rows and the group's heads on the
// columns, two columns per head (the bf16 "hi" part of the query or probability and
// its "lo" remainder), so r <= 4 heads fill one 8-column tile with no padding:
//   S[16 tok x 8]    = V_g[16 tok x d_h] . Q^T[d_h x 8]  (+ K_rope . Q_r^T)
//   O^T[d_h x 8]    += V_g^T[d_h x 16 tok] . P^T[16 tok x 8]
// Lane (gid, tig) holds the scores of head 4nt + tig for tokens gid and gid + 8, and
// the output of the same head for dimensions 16mt + gid (+ 8).
template <int DH, int DR, int NT>
struct QFrags {
    static constexpr int KD = DH / 16;       // k16 steps over d_h
    static constexpr int DRK16 = DR / 16;    // full k16 steps over the positional slice
    uint32_t bq[KD][NT][2];
    uint32_t bqr[DRK16 > 0 ? DRK16 : 1][NT][2];
    uint32_t bqr8[NT];                       // the trailing k8 step when DR % 16 == 8
};

// Q^T fragments of value group g for sequence b: column gid of tile nt is head
// 4nt + gid/2 of the group, its hi part (gid even) or lo remainder (gid odd).  The
// content query comes from p.qc (fp32 or bf16, times p.qc_scale; read through L2 only
// when `cg`, for queries written by other CTAs of the same grid); the positional query
// is p.qr when given (already rotated and scaled), else q_rope rotated here by
// Rot(L_b - 1) and scaled by p.qr_scale.
template <int DH, int DR, int NT, bool CG>
__device__ __forceinline__ void load_q_frags(const DecodeParams &p, int b, int g, int Lb, int lane,
                                             QFrags<DH, DR, NT> &q) {
    constexpr int KD = DH / 16, DRK16 = DR / 16;
    constexpr bool DR_K8 = (DR % 16) == 8;
    const int gid = lane >> 2, tig = lane & 3;
    const bool lo_col = (gid & 1) != 0;
    const int r = p.r, H = p.H;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int hl = 4 * nt + (gid >> 1);
        const bool real = hl < r;
        const long long qoff = ((long long)b * H + g * r + hl) * DH;
        float x[KD][4];
#pragma unroll
        for (int kk = 0; kk < KD; ++kk) {
            x[kk][0] = x[kk][1] = x[kk][2] = x[kk][3] = 0.f;
            if (real) {
                const int d0 = kk * 16 + tig * 2;
                if (p.qc_f32) {
                    const float *qf = reinterpret_cast<const float *>(p.qc) + qoff;
                    const float2 u = CG ? __ldcg(reinterpret_cast<const float2 *>(qf + d0))
                                        : *reinterpret_cast<const float2 *>(qf + d0);
                    const float2 v = CG ? __ldcg(reinterpret_cast<const float2 *>(qf + d0 + 8))
                                        : *reinterpret_cast<const float2 *>(qf + d0 + 8);
                    x[kk][0] = u.x; x[kk][1] = u.y; x[kk][2] = v.x; x[kk][3] = v.y;
                } else {
                    const __nv_bfloat16 *qb = reinterpret_cast<const __nv_bfloat16 *>(p.qc) + qoff;
                    const float2 u = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(qb + d0));
                    const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(qb + d0 + 8));
                    x[kk][0] = u.x; x[kk][1] = u.y; x[kk][2] = v.x; x[kk][3] = v.y;
                }
            }
        }
        float xr[DRK16 > 0 ? DRK16 : 1][4], xr8[2] = {0.f, 0.f};
        if (DR > 0) {
            // this lane's positional query pairs (d0, d0+1), (d0+8, d0+9) are RoPE
            // pairs d0/2 and d0/2 + 4: either rotated by the absorption kernel
            // (p.qr), or rotated here by Rot(L_b - 1) from the raw q_rope
            const long long qo = ((long long)b * H + g * r + hl) * DR;
            int t = Lb - 1;
            if (t < 0) t = 0;
            if (t >= p.rope_max_pos) {
                if (p.qr == nullptr && real && tig == 0 && (gid & 1) == 0)
                    dev_report(GVA_DEV_BAD_POSITION);
                t = 0;
            }
            const float2 *cs = reinterpret_cast<const float2 *>(p.rope_tab) + (long long)t * (DR / 2);
            auto pair = [&](int d) -> float2 {   // rotated, scaled pair (d, d + 1)
                if (p.qr != nullptr) return *reinterpret_cast<const float2 *>(p.qr + qo + d);
                float2 x;
                if (p.qr_f32) {
                    x = *reinterpret_cast<const float2 *>(reinterpret_cast<const float *>(p.q_rope) + qo + d);
                } else {
                    x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(
                        reinterpret_cast<const __nv_bfloat16 *>(p.q_rope) + qo + d));
                }
                const float2 c = cs[d / 2];
                return make_float2(p.qr_scale * (x.x * c.x - x.y * c.y),
                                   p.qr_scale * (x.x * c.y + x.y * c.x));
            };
#pragma unroll
            for (int kk = 0; kk < DRK16; ++kk) {
                xr[kk][0] = xr[kk][1] = xr[kk][2] = xr[kk][3] = 0.f;
                if (real) {
                    const int d0 = kk * 16 + tig * 2;
                    const float2 u = pair(d0);
                    const float2 v = pair(d0 + 8);
                    xr[kk][0] = u.x; xr[kk][1] = u.y; xr[kk][2] = v.x; xr[kk][3] = v.y;
                }
            }
            if (DR_K8 && real) {
                const float2 u = pair(DRK16 * 16 + tig * 2);
                xr8[0] = u.x; xr8[1] = u.y;
            }
        }
#pragma unroll
        for (int kk = 0; kk < KD; ++kk) {
#pragma unroll
            for (int e = 0; e < 4; ++e) x[kk][e] *= p.qc_scale;
            q.bq[kk][nt][0] = part_bf16x2(x[kk][0], x[kk][1], lo_col);
            q.bq[kk][nt][1] = part_bf16x2(x[kk][2], x[kk][3], lo_col);
        }
        if (DR > 0) {
#pragma unroll
            for (int kk = 0; kk < DRK16; ++kk) {
                q.bqr[kk][nt][0] = part_bf16x2(xr[kk][0], xr[kk][1], lo_col);
                q.bqr[kk][nt][1] = part_bf16x2(xr[kk][2], xr[kk][3], lo_col);
            }
            if (DR_K8) q.bqr8[nt] = part_bf16x2(xr8[0], xr8[1], lo_col);
        }
    }
}

// Scores of one staged slab for value group g: sc[nt][a] accumulates the k16 steps of
// parity a (two independent chains), hi and lo columns still separate.  kst: the tile
// scored against the content query (the value tile, or the GQA key tile); rst: the
// positional keys (DR > 0).
template <int DH, int DR, int NT>
__device__ __forceinline__ void slab_scores(uint32_t kst, uint32_t rst, int g, int lane,
                                            const QFrags<DH, DR, NT> &q, float (&sc)[NT][2][4]) {
    constexpr int KD = DH / 16, DRK16 = DR / 16;
    constexpr bool DR_K8 = (DR % 16) == 8;
    const int lm_mat = lane >> 3, lm_row = lane & 7;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int a2 = 0; a2 < 2; ++a2)
            sc[nt][a2][0] = sc[nt][a2][1] = sc[nt][a2][2] = sc[nt][a2][3] = 0.f;
    // wide rows (d > 128) read each k-step's tile just before its products (registers)
    constexpr bool STAGED = KD > 8;
    uint32_t av[STAGED ? 1 : KD][4];
    if constexpr (!STAGED) {
#pragma unroll
        for (int kk = 0; kk < KD; ++kk)
            ldsm_x4(vtile_addr<DH>(kst, g, lm_row + 8 * (lm_mat & 1), 2 * kk + (lm_mat >> 1)),
                    av[kk][0], av[kk][1], av[kk][2], av[kk][3]);
    }
    uint32_t ar[DRK16 > 0 ? DRK16 : 1][4], ar8[2];
    if (DR > 0) {
#pragma unroll
        for (int kk = 0; kk < DRK16; ++kk)
            ldsm_x4(rst + (lm_row + 8 * (lm_mat & 1)) * (DR * 2) + (2 * kk + (lm_mat >> 1)) * 16,
                    ar[kk][0], ar[kk][1], ar[kk][2], ar[kk][3]);
        if (DR_K8)
            ldsm_x2(rst + (lm_row + 8 * (lm_mat & 1)) * (DR * 2) + DRK16 * 32, ar8[0], ar8[1]);
    }
    if constexpr (!STAGED) {
#pragma unroll
        for (int kk = 0; kk < KD; ++kk)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                mma16816(sc[nt][kk & 1], av[kk], q.bq[kk][nt][0], q.bq[kk][nt][1]);
    } else {
#pragma unroll
        for (int kk = 0; kk < KD; ++kk) {
            ldsm_x4(vtile_addr<DH>(kst, g, lm_row + 8 * (lm_mat & 1), 2 * kk + (lm_mat >> 1)),
                    av[0][0], av[0][1], av[0][2], av[0][3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                mma16816(sc[nt][kk & 1], av[0], q.bq[kk][nt][0], q.bq[kk][nt][1]);
        }
    }
    if (DR > 0) {
#pragma unroll
        for (int kk = 0; kk < DRK16; ++kk)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                mma16816(sc[nt][(KD + kk) & 1], ar[kk], q.bqr[kk][nt][0], q.bqr[kk][nt][1]);
        if (DR_K8) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                mma1688(sc[nt][(KD + DRK16) & 1], ar8[0], ar8[1], q.bqr8[nt]);
        }
    }
}

// Value tiles of group g as the A operand of O^T += V^T P^T (ldmatrix.trans).
template <int DH>
__device__ __forceinline__ void slab_value_tiles(uint32_t st, int g, int lane,
                                                 uint32_t (&apv)[DH / 16][4]) {
    const int lm_mat = lane >> 3, lm_row = lane & 7;
#pragma unroll
    for (int mt = 0; mt < DH / 16; ++mt)
        ldsm_x4_t(vtile_addr<DH>(st, g, lm_row + 8 * (lm_mat >> 1), 2 * mt + (lm_mat & 1)),
                  apv[mt][0], apv[mt][1], apv[mt][2], apv[mt][3]);
}

// Zero the value tiles of tokens at or past nv (a slot past a sequence's end may hold
// anything, including NaN, and 0 * NaN would poison the sum).
template <int DH>
__device__ __forceinline__ void mask_value_tiles(uint32_t (&apv)[DH / 16][4], int nv, int lane) {
    const int tig = lane & 3;
    const int ta = 2 * tig, tb = 8 + 2 * tig;
    const uint32_t ma = (ta >= nv ? 0u : 0xffffu) | (ta + 1 >= nv ? 0u : 0xffff0000u);
    const uint32_t mb = (tb >= nv ? 0u : 0xffffu) | (tb + 1 >= nv ? 0u : 0xffff0000u);
#pragma unroll
    for (int mt = 0; mt < DH / 16; ++mt) {
        apv[mt][0] &= ma; apv[mt][1] &= ma; apv[mt][2] &= mb; apv[mt][3] &= mb;
    }
}

// ---------------------------------------------------------------------------- //
// producer warp (shared by the tensor-core decode kernels)
// ---------------------------------------------------------------------------- //
// One step issues up to il = min(NS, 32) consecutive slabs, one per lane: lane j finds
// its slab's storage row (for a paged cache the block-table reads of the step are in
// flight together), waits until its ring stage is free, and issues the copies.  The
// stages of one step are distinct, so no lane waits on another lane's copy.  A short
// cache (the whole share fits in the ring) is issued in a single step.  Slab s0 + i of
// the share goes to stage i mod NS in round i / NS.
template <int DH, int DR, bool GQA>
__device__ __forceinline__ void mma_producer(const CUtensorMap *tm_v, const CUtensorMap *tm_k,
                                             const MmaParams &mp, const int *F, const int *Hs,
                                             long long s0, long long s1, uint32_t base_u32,
                                             uint32_t bar_full, uint32_t bar_empty,
                                             volatile int *abort, int *stage_bad, uint64_t pol) {
    const DecodeParams &p = mp.d;
    const int NS = mp.nstages, B = p.B;
    const int lane = threadIdx.x & 31;
    const int il = NS < 32 ? NS : 32;
    int stage = 0;                      // stage of the step's first slab
    uint32_t round = 0;                 // ring wraps before the step's first slab
    bool dead = false;
    long long n_tried = 0;              // slabs of the steps attempted
    int b = seq_of_slab(F, B, s0);      // sequence of the step's first slab
    bool held = Hs == nullptr;          // the grid dependency has resolved (or need not)
    if (lane == 0) GVA_TRACE_AT(6);
    if (lane == 0) GVA_TRACE_AT(200);
    for (long long sb = s0; sb < s1; sb += il) {
        const long long s = sb + lane;
        const bool act = lane < il && s < s1;
        int st = stage + lane;
        uint32_t rd = round;
        if (st >= NS) { st -= NS; ++rd; }
        bool ok = true;
        int bl = b;
        if (act)
            while (F[bl + 1] <= s) ++bl;
        // a slab holding a row the preceding grid appends is copied only after that grid
        // has completed (its writes are then visible); the whole warp waits once
        if (!held) {
            if (__any_sync(0xffffffffu, act && Hs[bl] == (int)(s - F[bl]))) {
                pdl_wait();
                held = true;
            }
        }
        if (act) {
            const long long row = row_of(p.R, bl, (s - F[bl]) * SLAB);
            const int yk = row < 0 ? 0 : (int)row;
            if (s == s0) GVA_TRACE_AT(201);
            if (rd > 0 && !mbar_wait(bar_empty + 8 * st, (rd - 1) & 1u, abort)) {
                ok = false;
            } else {
                const uint32_t stb = base_u32 + st * mp.stage_bytes;
                const uint32_t fb = bar_full + 8 * st;
                stage_bad[st] = row < 0;   // published by the arrive below
                // the positional keys of the slab are one contiguous run of rows;
                // rows past the end of the cache storage are not copied (their
                // tokens are past every sequence's end, and masked)
                int rrows = SLAB;
                if ((long long)yk + SLAB > p.R.num_rows) {
                    const long long left = p.R.num_rows - (long long)yk;
                    rrows = left < 0 ? 0 : (int)left;
                }
                const uint32_t rbytes = (uint32_t)rrows * (DR * 2);
                mbar_expect_tx(fb, (uint32_t)mp.off_r + rbytes);
                if (s == s0) GVA_TRACE_AT(202);
                if (mp.v3d) {
                    tma_load_3d(stb, tm_v, 0, yk, 0, fb, pol);
                    if (s == s0) GVA_TRACE_AT(203);
                    if (GQA) tma_load_3d(stb + mp.off_k, tm_k, 0, yk, 0, fb, pol);
                } else {
                    for (int bx = 0; bx < mp.vg * (DH / 64); ++bx) {
                        tma_load_2d(stb + bx * 2048, tm_v, bx * 64, yk, fb, pol);
                        if (GQA) tma_load_2d(stb + mp.off_k + bx * 2048, tm_k, bx * 64, yk, fb, pol);
                    }
                }
                if (DR > 0 && rbytes > 0)
                    bulk_load(stb + mp.off_r,
                              reinterpret_cast<const unsigned char *>(p.Krope) + (size_t)yk * (DR * 2),
                              rbytes, fb, pol);
                const int ti = (int)(s - s0);
                if (ti == 0) GVA_TRACE_AT(2);
                if (ti == 0) GVA_REC(3, 3);
                if (ti < 64) GVA_TRACE_AT(300 + ti);
            }
        }
        n_tried += min((long long)il, s1 - sb);
        dead = __any_sync(0xffffffffu, act && !ok);
        if (dead) break;
        {   // sequence of the next step's first slab
            const long long sn = sb + il;
            while (b < B - 1 && F[b + 1] <= sn) ++b;
        }
        stage += il;
        if (stage >= NS) { stage -= NS; ++round; }
    }
    if (lane == 0) {
        GVA_TRACE_AT(3);
        GVA_TRACE_FLUSH(2, 4);
        GVA_TRACE_FLUSH(6, 8);
        GVA_TRACE_FLUSH(300, 364);
        GVA_TRACE_FLUSH(200, 204);
        // Never leave with copies in flight: wait (bounded) for the last copy of each
        // stage used.  Slab i used stage i % NS in round i / NS.  After an abort a
        // stage's last slab may not have been issued: those waits are kept short.
        const unsigned long long limit = dead ? 1000000ull : WAIT_LIMIT_NS;
        for (int st = 0; st < NS && st < n_tried; ++st) {
            const uint32_t par = (uint32_t)((n_tried - 1 - st) / NS) & 1u;
            const unsigned long long t0 = global_ns();
            while (!mbar_try_wait(bar_full + 8 * st, par)) {
                if (global_ns() - t0 > limit) {
                    if (!dead) dev_report(GVA_DEV_TIMEOUT);
                    break;
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------- //
// the kernel
// ---------------------------------------------------------------------------- //
// MINB = 2 or 3: the instances that run two or three CTAs per SM (the registers of that
// many CTAs of the launched size within the SM's 64 K), each with a smaller ring; three
// per SM with MMA_TRIPLE_CONSUMERS consumer warps.
template <int DH, int DR, bool GQA, int NT, bool SV = false, int MINB = 1>
__global__ void __launch_bounds__(MINB == 1   ? MMA_THREADS
                                  : MINB == 2 ? (MMA_CONSUMERS + 1) * 32
                                              : (MMA_TRIPLE_CONSUMERS + 1) * 32,
                                  MINB)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_k, const MmaParams mp) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    GVA_TRACE_DECL;
    const DecodeParams &p = mp.d;
    // 1024-byte aligned base for the swizzled stages
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
    unsigned char *base = smem_raw + (base_u32 - raw_u32);
    const int NS = mp.nstages;
    const uint32_t bar_full = base_u32 + mp.off_bar;          // NS x 8 bytes
    const uint32_t bar_empty = bar_full + 8 * NS;             // NS x 8 bytes
    volatile int *abort = reinterpret_cast<volatile int *>(base + mp.off_bar + 16 * NS);
    // per stage: 1 when the slab's block-table entry was out of range (its tokens are skipped)
    int *stage_bad = reinterpret_cast<int *>(base + mp.off_bar + 16 * NS + 16);
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
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_v);
        if (GQA) prefetch_tmap(&tm_k);
    }
    // the cache loads' L2 policy, made while the lengths load (it takes a while)
    const uint64_t pol = warp == 0 ? l2_evict_first_policy() : 0ull;
    if (threadIdx.x == 0) GVA_TRACE_AT(0);
    if (threadIdx.x == 0) GVA_REC(3, 0);
    if (threadIdx.x == 0) GVA_KT(5);
    if (threadIdx.x == 0) GVA_CTA_T(0);
    // Lengths, row maps and the cache are final before the preceding grid (the query
    // absorption) was allowed to start, so with `early` they are read at once and the
    // cache streams while that grid still runs; the queries are read after the wait.
    if (!mp.early) pdl_wait();
    pdl_launch_dependents();
    int *Hs = mp.hold_pos ? F + B + 1 : nullptr;
    build_prefix(p.seq_len, p.R, B, Ls, F, blockIdx.x == 0,   // includes __syncthreads
                 blockIdx.x == 0 ? p.prefix_ws : nullptr, mp.hold_pos, Hs);
    if (threadIdx.x == 0) GVA_TRACE_AT(1);
    if (threadIdx.x == 0) GVA_REC(3, 5);
    const Part P{F[B], p.n_ctas};
    const int c = blockIdx.x;
    if (P.S == 0) return;
    const long long s0 = P.start(c), s1 = P.start(c + 1);
    if (s0 >= s1) return;

    // ============================= producer warp ============================= //
    if (warp == 0) {
        mma_producer<DH, DR, GQA>(&tm_v, &tm_k, mp, F, Hs, s0, s1, base_u32, bar_full,
                                  bar_empty, abort, stage_bad, pol);
        return;
    }

    // ============================= consumer warps ============================ //
    const int ci = warp - 1;          // consumer index
    if (ci >= mp.ncons) return;       // spare warps
    const int g = ci % G;             // value group of this warp
    const int w = ci / G;             // rank among the group's warps
    const int wpg = mp.wpg;
    const int gid = lane >> 2, tig = lane & 3;
    constexpr int KD = DH / 16;       // k16 steps over d_h (and 16-row tiles of O^T)
    // P^T exchange: the lanes holding tokens 2tig and 2tig+1 of this lane's column head
    const int srcA = (2 * tig) * 4 + (gid >> 1), srcB = (2 * tig + 1) * 4 + (gid >> 1);
    const bool lo_col = (gid & 1) != 0;

    if (mp.early) pdl_wait();         // the absorbed queries come from the preceding grid
    if (w == 0 && g == 0 && lane == 0) GVA_KT(6);
    if (w == 0 && g == 0 && lane == 0) GVA_REC(3, 1);
    if (w == 0 && g == 0 && lane == 0) GVA_CTA_T(1);
    // The slabs of the share go round-robin to the group's warps: this warp takes
    // s0 + w, s0 + w + wpg, ...; slab s0 + i sits in ring stage i mod NS, phase (i / NS) & 1.
    long long my_s = s0 + w;
    int my_stage = w % NS;
    uint32_t my_phase = (uint32_t)(w / NS) & 1u;
    int b = seq_of_slab(F, B, s0);
    int tslab = 0;                    // trace index
    long long s = s0;                 // start of the current segment (one sequence's slabs)
    bool alive = true;
    while (s < s1) {
        while (F[b + 1] <= s) ++b;
        const long long seg_end = min(s1, (long long)F[b + 1]);
        const int Lb = Ls[b];
        const int Fb = F[b];

        QFrags<DH, DR, NT> qf;
        load_q_frags<DH, DR, NT, false>(p, b, g, Lb, lane, qf);

        float oacc[KD][NT][4];
#pragma unroll
        for (int mt = 0; mt < KD; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                oacc[mt][nt][0] = oacc[mt][nt][1] = oacc[mt][nt][2] = oacc[mt][nt][3] = 0.f;
        float m_run[NT], l_run[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) { m_run[nt] = -INFINITY; l_run[nt] = 0.f; }

        if (w == 0 && g == 0 && lane == 0) GVA_TRACE_AT(4);
        while (my_s < seg_end && alive) {
            // one decision for the warp (the code below is warp-synchronous)
            const bool waited = __all_sync(0xffffffffu, mbar_wait(bar_full + 8 * my_stage, my_phase, abort));
            if (!waited) {
                alive = false;
                break;
            }
            if (w == 0 && g == 0 && lane == 0) GVA_TRACE_AT(8 + 2 * tslab);
            if (w == 0 && g == 0 && lane == 0 && tslab == 0) GVA_REC(3, 4);
            const int j0 = (int)(my_s - Fb) * SLAB;
            int nv = min(SLAB, Lb - j0);
            if (stage_bad[my_stage]) {
                if (lane == 0 && g == 0) dev_report(GVA_DEV_BAD_PAGE);
                nv = 0;
            }
            const uint32_t st = base_u32 + my_stage * mp.stage_bytes;

            // ---- scores: A = the key tile (tokens x d), B = Q^T ----
            float sc[NT][2][4];
            slab_scores<DH, DR, NT>(GQA ? st + mp.off_k : st, st + mp.off_r, SV ? 0 : g, lane,
                                    qf, sc);
            if (w == 0 && g == 0 && lane == 0 && tslab < 8) GVA_TRACE_AT(100 + 10 * tslab);
            // value tiles for the weighted sum (V^T as the A operand), read while the
            // softmax below runs
            // (wide value rows: the value tiles are read per output tile below instead)
            constexpr bool STAGED = KD > 8;
            uint32_t apv[STAGED ? 1 : KD][4];
            if constexpr (!STAGED) slab_value_tiles<DH>(st, SV ? 0 : g, lane, apv);

            // ---- per head: hi + lo columns -> score of tokens gid, gid + 8 ----
            float z[NT][2];
            bool over = false;   // a score above the running maximum by more than the threshold
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                z[nt][0] = (sc[nt][0][0] + sc[nt][0][1]) + (sc[nt][1][0] + sc[nt][1][1]);
                z[nt][1] = (sc[nt][0][2] + sc[nt][0][3]) + (sc[nt][1][2] + sc[nt][1][3]);
                if (gid >= nv) z[nt][0] = -INFINITY;
                if (gid + 8 >= nv) z[nt][1] = -INFINITY;
                over |= fmaxf(z[nt][0], z[nt][1]) > m_run[nt] + MMA_RESCALE_TH;
            }
            // Lazy rescale: the running maximum moves only when a score exceeds it by
            // more than the threshold (always on a head's first valid token); otherwise
            // the probabilities are taken against the stale maximum (at most 2^threshold)
            // and the max reduction over the token lanes is skipped.
            if (w == 0 && g == 0 && lane == 0 && tslab < 8) GVA_TRACE_AT(101 + 10 * tslab);
            if (__any_sync(0xffffffffu, over)) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float m = fmaxf(z[nt][0], z[nt][1]);
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                    const bool raise = m > m_run[nt] + MMA_RESCALE_TH;
                    const float alpha = raise ? exp2f(m_run[nt] - m) : 1.f;  // 0 when m_run = -inf
                    if (raise) m_run[nt] = m;
                    l_run[nt] *= alpha;
#pragma unroll
                    for (int mt = 0; mt < KD; ++mt) {
                        oacc[mt][nt][0] *= alpha; oacc[mt][nt][1] *= alpha;
                        oacc[mt][nt][2] *= alpha; oacc[mt][nt][3] *= alpha;
                    }
                }
            }
            // ---- probabilities, then P^T as the B operand (column gid: head 4nt + gid/2) ----
            uint32_t bp[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float p0 = z[nt][0] == -INFINITY ? 0.f : exp2f(z[nt][0] - m_run[nt]);
                const float p1 = z[nt][1] == -INFINITY ? 0.f : exp2f(z[nt][1] - m_run[nt]);
                l_run[nt] += p0 + p1;
                const float a0 = __shfl_sync(0xffffffffu, p0, srcA);   // token 2tig
                const float a1 = __shfl_sync(0xffffffffu, p1, srcA);   // token 2tig + 8
                const float b0 = __shfl_sync(0xffffffffu, p0, srcB);   // token 2tig + 1
                const float b1 = __shfl_sync(0xffffffffu, p1, srcB);   // token 2tig + 9
                bp[nt][0] = part_bf16x2(a0, b0, lo_col);
                bp[nt][1] = part_bf16x2(a1, b1, lo_col);
            }
            // ---- O^T += V^T . P^T ----
            if (w == 0 && g == 0 && lane == 0 && tslab < 8) GVA_TRACE_AT(102 + 10 * tslab);
            if constexpr (!STAGED) {
                if (nv < SLAB) mask_value_tiles<DH>(apv, nv, lane);
#pragma unroll
                for (int mt = 0; mt < KD; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma16816(oacc[mt][nt], apv[mt], bp[nt][0], bp[nt][1]);
            } else {
                const int lm_mat = lane >> 3, lm_row = lane & 7;
                const int ta = 2 * tig, tb = 8 + 2 * tig;
                const uint32_t ma = (ta >= nv ? 0u : 0xffffu) | (ta + 1 >= nv ? 0u : 0xffff0000u);
                const uint32_t mb = (tb >= nv ? 0u : 0xffffu) | (tb + 1 >= nv ? 0u : 0xffff0000u);
#pragma unroll
                for (int mt = 0; mt < KD; ++mt) {
                    uint32_t a[4];
                    ldsm_x4_t(vtile_addr<DH>(st, SV ? 0 : g, lm_row + 8 * (lm_mat >> 1), 2 * mt + (lm_mat & 1)),
                              a[0], a[1], a[2], a[3]);
                    if (nv < SLAB) { a[0] &= ma; a[1] &= ma; a[2] &= mb; a[3] &= mb; }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma16816(oacc[mt][nt], a, bp[nt][0], bp[nt][1]);
                }
            }
            // the products above consumed every tile register, so all of the warp's
            // shared-memory reads of the stage are complete: release it to the producer
            if (w == 0 && g == 0 && lane == 0 && tslab < 8) GVA_TRACE_AT(103 + 10 * tslab);
            __syncwarp();
            if (lane == 0) mbar_arrive_relaxed(bar_empty + 8 * my_stage);
            if (w == 0 && g == 0 && lane == 0) GVA_TRACE_AT(9 + 2 * tslab);
            ++tslab;
            my_s += wpg;
            my_stage += wpg;
            while (my_stage >= NS) { my_stage -= NS; my_phase ^= 1u; }
        }
        s = seg_end;

        // ---- segment end: fold hi/lo columns, reduce l over the 8 token lanes, merge
        //      the group's warps ----
        float o2[KD][NT][2];   // O[head 4nt + tig][16mt + gid (+8)]
#pragma unroll
        for (int mt = 0; mt < KD; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                o2[mt][nt][0] = oacc[mt][nt][0] + oacc[mt][nt][1];
                o2[mt][nt][1] = oacc[mt][nt][2] + oacc[mt][nt][3];
            }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], 4);
            l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], 8);
            l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], 16);
        }
        if (wpg > 1) {
            // slot per (extra warp, group): 4 NT heads x (DH + 2) floats
            const int stride = 4 * NT * (DH + 2);
            if (w > 0) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float *mb = merge + ((w - 1) * G + g) * stride + (4 * nt + tig) * (DH + 2);
#pragma unroll
                    for (int mt = 0; mt < KD; ++mt) {
                        mb[16 * mt + gid] = o2[mt][nt][0];
                        mb[16 * mt + gid + 8] = o2[mt][nt][1];
                    }
                    if (gid == 0) { mb[DH] = m_run[nt]; mb[DH + 1] = l_run[nt]; }
                }
            }
            named_bar(1 + g, wpg * 32);
            if (w == 0) {
                for (int ww = 1; ww < wpg; ++ww) {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const float *mb = merge + ((ww - 1) * G + g) * stride + (4 * nt + tig) * (DH + 2);
                        const float m2 = mb[DH], l2 = mb[DH + 1];
                        const float mn = fmaxf(m_run[nt], m2);
                        const float a1 = (m_run[nt] == -INFINITY) ? 0.f : exp2f(m_run[nt] - mn);
                        const float a2 = (m2 == -INFINITY) ? 0.f : exp2f(m2 - mn);
#pragma unroll
                        for (int mt = 0; mt < KD; ++mt) {
                            o2[mt][nt][0] = o2[mt][nt][0] * a1 + mb[16 * mt + gid] * a2;
                            o2[mt][nt][1] = o2[mt][nt][1] * a1 + mb[16 * mt + gid + 8] * a2;
                        }
                        l_run[nt] = l_run[nt] * a1 + l2 * a2;
                        m_run[nt] = mn;
                    }
                }
            }
            named_bar(1 + g, wpg * 32);
        }
        if (w == 0 && g == 0 && lane == 0) GVA_TRACE_AT(5);
        if (w == 0) {
            const bool whole = Fb >= s0 && F[b + 1] <= s1;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int hl = 4 * nt + tig;
                if (hl >= r) continue;
                const int h = g * r + hl;
                if (whole) {
                    const float inv = l_run[nt] > 0.f ? 1.f / l_run[nt] : 0.f;
                    float *o = p.out + ((long long)b * H + h) * DH;
#pragma unroll
                    for (int mt = 0; mt < KD; ++mt) {
                        o[16 * mt + gid] = o2[mt][nt][0] * inv;
                        o[16 * mt + gid + 8] = o2[mt][nt][1] * inv;
                    }
                    if (gid == 0 && p.lse)
                        p.lse[(long long)b * H + h] =
                            l_run[nt] > 0.f ? (m_run[nt] + log2f(l_run[nt])) * LN2 : -INFINITY;
                } else {
                    const long long slot = (long long)c + b;
                    float *o = p.part_o + (slot * H + h) * DH;
#pragma unroll
                    for (int mt = 0; mt < KD; ++mt) {
                        o[16 * mt + gid] = o2[mt][nt][0];
                        o[16 * mt + gid + 8] = o2[mt][nt][1];
                    }
                    if (gid == 0) {
                        p.part_ml[(slot * H + h) * 2] = m_run[nt];
                        p.part_ml[(slot * H + h) * 2 + 1] = l_run[nt];
                    }
                }
            }
        }
    }
    if (w == 0 && g == 0 && lane == 0) {
        GVA_REC(3, 2);
        GVA_KT(7);
        GVA_CTA_T(2);
        GVA_TRACE_FLUSH(0, 2);
        GVA_TRACE_FLUSH(4, 6);
        GVA_TRACE_FLUSH(8, 8 + 2 * tslab);
        GVA_TRACE_FLUSH(100, 180);
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

#ifdef GVA_TRACE
constexpr int MMA_SMEM_LIMIT = 227 * 1024 - TRACE_SLOTS * 8;   // the trace buffer is static
#else
constexpr int MMA_SMEM_LIMIT = 227 * 1024;
#endif
// The stage ring is sized to leave room on the SM for the query-absorption grid that
// precedes the decode: with programmatic dependent launch the decode's CTAs start
// while that grid's CTAs are still resident, and stream the cache meanwhile.
constexpr int MMA_SMEM_TARGET = 196 * 1024;
// Two CTAs per SM: each within half of the SM's 228 KB (less the per-CTA reservation).
// Taken when the cache's capacity gives each of the 2 x SMs CTAs at least
// MMA_PAIR_MIN_SLABS slabs and the half-size ring still holds MMA_PAIR_MIN_STAGES: a long
// share streams while the other CTA of its SM starts or ends, and an SM's time is the
// sum of two shares, so the spread of CTA ends shrinks.  Measured on the ragged batch
// (d_h = 64, about 30 slabs per CTA): 26.6 against 29.8 µs per decode op; on the 350M
// layer (7 slabs per CTA) it is slower, 14.3 against 13.8 µs.
constexpr int MMA_SMEM_PAIR = 108 * 1024;
constexpr int MMA_PAIR_MIN_SLABS = 16;
constexpr int MMA_PAIR_MIN_STAGES = 6;
// Three CTAs per SM, each with one consumer warp per value group (G <= 4) and a third of
// the SM's shared memory, under the same rules: ragged batch 24.8 against 26.5 µs per
// decode op with two CTAs per SM.
constexpr int MMA_SMEM_TRIPLE = 72 * 1024;

inline int bar_region_bytes(int ns) { return (int)align_up(16 * ns + 16 + 4 * ns, 16); }

// Merge buffer of the group's extra warps: per (extra warp, group) 4 NT heads x (DH + 2).
inline int merge_bytes_of(int wpg, int G, int DH, int NT) {
    return (wpg - 1) * G * 4 * NT * (DH + 2) * 4;
}

// `target`: the shared memory the ring is sized for; with `strict` the plan keeps to it
// (no fallback to the per-CTA maximum).
inline bool plan_mma(MmaParams &mp, int DH, int DR, bool gqa, int NT,
                     int target = MMA_SMEM_TARGET, bool strict = false,
                     int consumers = MMA_CONSUMERS) {
    const DecodeParams &d = mp.d;
    const int vbytes = mp.vg * DH * SLAB * 2;
    mp.off_k = vbytes;
    mp.off_r = vbytes * (gqa ? 2 : 1);
    const int rbytes = DR * SLAB * 2;
    mp.tx_bytes = mp.off_r + rbytes;
    mp.stage_bytes = (int)align_up((size_t)mp.tx_bytes, 1024);
    mp.wpg = consumers / d.G;
    if (mp.wpg < 1) mp.wpg = 1;
    mp.ncons = d.G * mp.wpg;
    const int merge_bytes = merge_bytes_of(mp.wpg, d.G, DH, NT);
    // Ls, F (and Hs) in shared memory.  The several-CTAs-per-SM plans (strict) reserve Hs
    // whether or not it is used: their choice, which sets the grid and so the order of
    // the sums, is then the same for a decode call and the decode step's call.
    const int narr = ((mp.hold_pos || strict) ? 3 : 2) * d.B + 1;
    const int fixed = 1024 /* alignment slack */ + (int)align_up(sizeof(int) * narr, 16) +
                      merge_bytes + bar_region_bytes(MMA_MAX_STAGES);
    int ns = (target - fixed) / mp.stage_bytes;
    if (ns < 4 && !strict) ns = (MMA_SMEM_LIMIT - fixed) / mp.stage_bytes;
    if (ns > MMA_MAX_STAGES) ns = MMA_MAX_STAGES;
    // Warp w of a group takes the share's slabs w, w + wpg, ... and slab i sits in stage
    // i mod ns, so with ns a multiple of wpg every round of a stage goes to the same
    // warp of each group: a warp waits for round R of a stage only after it consumed
    // round R - 1 of that stage itself, so the stage's full barrier is then in phase R
    // or past it, and the parity wait is exact.  With any other ns, a warp can reach
    // round R while another warp's round R - 1 copy into that stage is still in flight;
    // the barrier's current phase (R - 1) then has the other parity, the parity test
    // passes at once, and the warp reads a half-written stage and gives back a stage
    // whose round has not begun (the empty barrier's phases then drift from the rounds).
    ns -= ns % mp.wpg;
    if (ns < 2) return false;
    mp.nstages = ns;
    mp.off_bar = ns * mp.stage_bytes;
    mp.off_f = mp.off_bar + bar_region_bytes(ns);
    mp.off_merge = mp.off_f + (int)align_up(sizeof(int) * narr, 16);
    return true;
}

inline size_t mma_smem_bytes(const MmaParams &mp, int DH, int NT) {
    return 1024 + (size_t)mp.off_merge + merge_bytes_of(mp.wpg, mp.d.G, DH, NT);
}

template <int DH, int DR, bool GQA, int NT, bool SV = false, int MINB = 1>
inline int launch_mma_t(void *stream, MmaParams &mp, const CUtensorMap &tv, const CUtensorMap &tk,
                        int grid) {
    auto kern = decode_mma_kernel<DH, DR, GQA, NT, SV, MINB>;
    const size_t smem = mma_smem_bytes(mp, DH, NT);
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3((mp.ncons + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    int na = 0;
    if (pdl_allowed(cfg.stream)) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cuda_status(cudaLaunchKernelEx(&cfg, kern, tv, tk, mp));
}

// Shared-memory opt-in of every instantiation (once per device, before any launch).
template <int DH, int NT>
inline cudaError_t mma_opt_in_dh() {
    const void *ks[] = {
        (const void *)decode_mma_kernel<DH, 0, false, NT>, (const void *)decode_mma_kernel<DH, 8, false, NT>,
        (const void *)decode_mma_kernel<DH, 16, false, NT>, (const void *)decode_mma_kernel<DH, 24, false, NT>,
        (const void *)decode_mma_kernel<DH, 32, false, NT>, (const void *)decode_mma_kernel<DH, 0, true, NT>};
    for (const void *k : ks) {
        const cudaError_t e =
            cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, MMA_SMEM_LIMIT);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}
template <int DH>
inline cudaError_t mma_opt_in_sv() {
    const void *ks[] = {(const void *)decode_mma_kernel<DH, 0, false, 1, true>,
                        (const void *)decode_mma_kernel<DH, 8, false, 1, true>,
                        (const void *)decode_mma_kernel<DH, 16, false, 1, true>,
                        (const void *)decode_mma_kernel<DH, 24, false, 1, true>,
                        (const void *)decode_mma_kernel<DH, 32, false, 1, true>};
    for (const void *k : ks) {
        const cudaError_t e =
            cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, MMA_SMEM_LIMIT);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}
inline cudaError_t mma_opt_in_pair() {
    const void *ks[] = {(const void *)decode_mma_kernel<64, 0, false, 1, false, 2>,
                        (const void *)decode_mma_kernel<64, 8, false, 1, false, 2>,
                        (const void *)decode_mma_kernel<64, 16, false, 1, false, 2>,
                        (const void *)decode_mma_kernel<64, 24, false, 1, false, 2>,
                        (const void *)decode_mma_kernel<64, 32, false, 1, false, 2>,
                        (const void *)decode_mma_kernel<64, 0, true, 1, false, 2>};
    for (const void *k : ks) {
        const cudaError_t e =
            cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, MMA_SMEM_PAIR);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}
inline cudaError_t mma_opt_in_triple() {
    const void *ks[] = {(const void *)decode_mma_kernel<64, 0, false, 1, false, 3>,
                        (const void *)decode_mma_kernel<64, 8, false, 1, false, 3>,
                        (const void *)decode_mma_kernel<64, 16, false, 1, false, 3>,
                        (const void *)decode_mma_kernel<64, 24, false, 1, false, 3>,
                        (const void *)decode_mma_kernel<64, 32, false, 1, false, 3>,
                        (const void *)decode_mma_kernel<64, 0, true, 1, false, 3>};
    for (const void *k : ks) {
        const cudaError_t e =
            cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, MMA_SMEM_TRIPLE);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}
inline cudaError_t mma_opt_in_all() {
    cudaError_t e = mma_opt_in_pair();
    if (e == cudaSuccess) e = mma_opt_in_triple();
    if (e == cudaSuccess) e = mma_opt_in_sv<128>();
    if (e == cudaSuccess) e = mma_opt_in_sv<256>();
    if (e == cudaSuccess) e = mma_opt_in_dh<64, 1>();
    if (e == cudaSuccess) e = mma_opt_in_dh<64, 2>();
    if (e == cudaSuccess) e = mma_opt_in_dh<128, 1>();
    if (e == cudaSuccess) e = mma_opt_in_dh<128, 2>();
    return e;
}

template <int DH, int NT, int MINB = 1>
inline int launch_mma_dr(void *stream, MmaParams &mp, const CUtensorMap &tv, const CUtensorMap &tk,
                         int grid, int DR, bool gqa) {
    if (gqa) return launch_mma_t<DH, 0, true, NT, false, MINB>(stream, mp, tv, tk, grid);
    switch (DR) {
    case 0: return launch_mma_t<DH, 0, false, NT, false, MINB>(stream, mp, tv, tk, grid);
    case 8: return launch_mma_t<DH, 8, false, NT, false, MINB>(stream, mp, tv, tk, grid);
    case 16: return launch_mma_t<DH, 16, false, NT, false, MINB>(stream, mp, tv, tk, grid);
    case 24: return launch_mma_t<DH, 24, false, NT, false, MINB>(stream, mp, tv, tk, grid);
    case 32: return launch_mma_t<DH, 32, false, NT, false, MINB>(stream, mp, tv, tk, grid);
    default: return GVA_ERR_UNSUPPORTED;
    }
}

template <int DH>
inline int launch_mma_sv(void *stream, MmaParams &mp, const CUtensorMap &tv, int grid, int DR) {
    switch (DR) {
    case 0: return launch_mma_t<DH, 0, false, 1, true>(stream, mp, tv, tv, grid);
    case 8: return launch_mma_t<DH, 8, false, 1, true>(stream, mp, tv, tv, grid);
    case 16: return launch_mma_t<DH, 16, false, 1, true>(stream, mp, tv, tv, grid);
    case 24: return launch_mma_t<DH, 24, false, 1, true>(stream, mp, tv, tv, grid);
    case 32: return launch_mma_t<DH, 32, false, 1, true>(stream, mp, tv, tv, grid);
    default: return GVA_ERR_UNSUPPORTED;
    }
}

// Sets dp.n_ctas and launches the tensor-core decode (one CTA per SM by default).  With
// `shared_v` every one of the dp.G groups of dp.r <= 4 heads reads the same value row of
// width dp.d_h in {128, 256} (the latent rows of the MLA-shaped decode).
// With hold_pos (and early), the preceding grid also appends row hold_pos[b] of each
// sequence b: the cache streams early except for the slabs holding those rows.
inline int run_mma(void *stream, DecodeParams &dp, const gva_rows &rows, int sms, int req_ctas,
                   bool gqa, bool early, bool shared_v = false, const int *hold_pos = nullptr) {
    if (rows.num_rows > 0x7fffffffLL) return GVA_ERR_UNSUPPORTED;   // TMA row coordinate is int32
    MmaParams mp;
    mp.d = dp;
    mp.hold_pos = early ? hold_pos : nullptr;
    const int DH = dp.d_h, DR = gqa ? 0 : dp.d_r;
    const int NT = dp.r <= 4 ? 1 : 2;   // 8-column tiles holding the group's heads (hi, lo)
    if (shared_v && (gqa || NT != 1 || (DH != 128 && DH != 256))) return GVA_ERR_UNSUPPORTED;
    mp.vg = shared_v ? 1 : dp.G;
    // three, else two CTAs per SM for long caches (the row capacity bounds the slabs from
    // above): the first plan whose ring still holds MMA_PAIR_MIN_STAGES
    int per_sm = 1;
    const long long cap_slabs = rows.num_rows / SLAB;
    if (!shared_v && DH == 64 && NT == 1 && req_ctas == 0) {
        struct Cand { int n, smem, consumers; };
        const Cand cands[2] = {{3, MMA_SMEM_TRIPLE, MMA_TRIPLE_CONSUMERS},
                               {2, MMA_SMEM_PAIR, MMA_CONSUMERS}};
        for (const Cand &cd : cands) {
            if (cd.consumers < dp.G || cap_slabs < (long long)cd.n * sms * MMA_PAIR_MIN_SLABS)
                continue;
            MmaParams m2 = mp;
            if (plan_mma(m2, DH, DR, gqa, NT, cd.smem, true, cd.consumers) &&
                m2.nstages >= MMA_PAIR_MIN_STAGES && mma_smem_bytes(m2, DH, NT) <= (size_t)cd.smem) {
                mp = m2;
                per_sm = cd.n;
                break;
            }
        }
    }
    if (per_sm == 1 && !plan_mma(mp, DH, DR, gqa, NT)) return GVA_ERR_UNSUPPORTED;
    const long long nrows = rows.num_rows > 0 ? rows.num_rows : 1;
    CUtensorMap tv, tk;
    mp.early = early ? 1 : 0;
    mp.v3d = make_map3(&tv, dp.Vc, nrows, mp.vg * DH) &&
             (!gqa || make_map3(&tk, dp.Kc, nrows, mp.vg * DH));
    if (!mp.v3d) {
        if (!make_map(&tv, dp.Vc, nrows, mp.vg * DH, 64, true)) return GVA_ERR_CUDA;
        if (gqa && !make_map(&tk, dp.Kc, nrows, mp.vg * DH, 64, true)) return GVA_ERR_CUDA;
    }
    if (!gqa) tk = tv;
    int grid = per_sm > 1 ? per_sm * sms : req_ctas > 0 ? req_ctas : sms;
    if (grid > sms * 8) grid = sms * 8;
    dp.n_ctas = grid;
    mp.d.n_ctas = grid;
    if (per_sm == 3) return launch_mma_dr<64, 1, 3>(stream, mp, tv, tk, grid, DR, gqa);
    if (per_sm == 2) return launch_mma_dr<64, 1, 2>(stream, mp, tv, tk, grid, DR, gqa);
    if (shared_v)
        return DH == 128 ? launch_mma_sv<128>(stream, mp, tv, grid, DR)
                         : launch_mma_sv<256>(stream, mp, tv, grid, DR);
    if (DH == 64)
        return NT == 1 ? launch_mma_dr<64, 1>(stream, mp, tv, tk, grid, DR, gqa)
                       : launch_mma_dr<64, 2>(stream, mp, tv, tk, grid, DR, gqa);
    return NT == 1 ? launch_mma_dr<128, 1>(stream, mp, tv, tk, grid, DR, gqa)
                   : launch_mma_dr<128, 2>(stream, mp, tv, tk, grid, DR, gqa);
}

}  // namespace gva
