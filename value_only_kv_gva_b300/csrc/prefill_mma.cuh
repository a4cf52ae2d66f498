// prefill_mma.cuh -- causal chunked prefill on the tensor cores.
//
// Every new token of a chunk attends to the cached history and to the chunk up to and
// including itself (MQA/GQA page §1; GVA analysis page, 关键技巧一/二 for the scores:
// z = q~_h . v_{j,g(h)} + q^_h . k_rope_j).  The prompt's tokens enter together and a
// group's query heads share its cached rows without copying them (MQA/GQA page §6.1).
// Unlike a decode, all n queries of a sequence read the same rows, so a CTA loads each
// 16-token slab of the rows once and scores it against every query row it holds: the
// chunk's (query, head) pairs of one value group are the MMA rows (16 per warp), the
// slab's tokens the columns.
//
// Per slab and warp: S[16 x 16] = Q~ V_g^T (+ Q^ K_rope^T), a causal mask (token j is
// visible to the query at position p when j <= p), an online softmax in log2 units,
// O[16 x d_h] += P V_g.  The fp32 queries and probabilities are split into bf16 hi and
// lo parts (about 16 mantissa bits, as in the decode kernel).  The history of each
// sequence is cut into `splits` ranges of slabs, one per CTA, and a second kernel merges
// the ranges by log-sum-exp.
//
// Slabs stream through a ring of shared-memory stages filled with 16-byte cp.async
// copies (zero-filled past the sequence's end); no wait in this file spins on a flag.
#pragma once

#include "common.cuh"
#include "decode_mma.cuh"
#include "launch.cuh"

namespace gva {

constexpr int PF_STAGES = 6;
constexpr int PF_SMEM_LIMIT = 227 * 1024;

struct PrefillMmaParams {
    int B, n, H, G, r;
    const int *L0;          // [B] tokens cached before the chunk
    RowsDev R;              // the caller's rows (contiguous or paged)
    const void *V;          // bf16 rows [G][d_h]
    const void *Kr;         // bf16 rows [d_r]
    const float *qt;        // [B*n][H][d_h] absorbed content queries, x scale * log2(e)
    const float *qh;        // [B*n][H][d_r] positional queries rotated by L0+i, x scale * log2(e)
    float *part_o;          // [B][splits][rows_pad][d_h] unnormalised partial outputs
    float *part_ml;         // [B][splits][rows_pad][2] (running max, sum) in log2 units
    float *out;             // [B][n][H][d_h]
    float *lse;             // [B][n][H] or null
    int splits;             // slab ranges per sequence
    int wpg;                // 16-row tiles per value group: ceil(n r / 16)
    int rows_pad;           // G * wpg * 16
    int vpitch;             // bytes per value row in shared memory (G d_h 2 + 16)
    int stage_bytes;        // one ring stage: 16 value rows then 16 positional-key rows
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Row layout of the partials: group g's rows first (wpg * 16 of them, query-major: row
// q = i * r + (h mod r)), padded rows never read.
template <int DH, int DR, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, 1) prefill_mma_kernel(const PrefillMmaParams p) {
    extern __shared__ __align__(128) unsigned char pf_smem[];
    pdl_wait();
    pdl_launch_dependents();
    const int split = blockIdx.x, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int GDH = p.G * DH;
    const long long l0 = p.L0[b];
    // tokens once the chunk is appended; the append skipped those past the capacity,
    // and their queries see nothing (out 0, lse -inf), as in a decode of a bad length
    const long long cap = min(seq_capacity(p.R, b), 0x7fffffffLL);
    const bool l0_ok = l0 >= 0 && l0 <= cap;
    const long long Lt = l0_ok ? min(l0 + p.n, cap) : 0;
    if ((!l0_ok || l0 + p.n > cap) && split == 0 && blockIdx.y == 0 && threadIdx.x == 0)
        dev_report(GVA_DEV_BAD_LENGTH);
    const long long nslab = (Lt + SLAB - 1) / SLAB;
    const long long per = (nslab + p.splits - 1) / p.splits;
    const long long s_begin = min(nslab, (long long)split * per);
    const int ns = (int)(min(nslab, s_begin + per) - s_begin);

    // this warp's 16 rows: group g, rows q = wt * 16 + 0..15 of the group's n * r
    const int wglob = blockIdx.y * WARPS + warp;
    const int g = wglob / p.wpg, wt = wglob - g * p.wpg;
    const bool active = g < p.G;
    const int nr = p.n * p.r;
    const int qA = wt * 16 + gid, qB = qA + 8;   // the two rows this thread holds
    const bool vA = active && qA < nr, vB = active && qB < nr;
    const int iA = vA ? qA / p.r : 0, iB = vB ? qB / p.r : 0;
    const int hA = g * p.r + (vA ? qA - iA * p.r : 0), hB = g * p.r + (vB ? qB - iB * p.r : 0);
    // last visible position of each row (the query's own), -1 for padding rows and
    // for queries past the capacity
    const long long limA = vA && l0 + iA < Lt ? l0 + iA : -1;
    const long long limB = vB && l0 + iB < Lt ? l0 + iB : -1;
    const int qlast = min(nr - 1, wt * 16 + 15);
    const long long wlim = active ? min(l0 + qlast / p.r, Lt - 1) : -1;

    // query fragments (A operands, bf16 hi/lo): a[0] rows A, cols 2tig; a[1] rows B;
    // a[2] rows A, cols 8 + 2tig; a[3] rows B, cols 8 + 2tig
    uint32_t qhi[DH / 16][4], qlo[DH / 16][4];
    {
        const float *rA = p.qt + (((long long)b * p.n + iA) * p.H + hA) * DH;
        const float *rB = p.qt + (((long long)b * p.n + iB) * p.H + hB) * DH;
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int c = kk * 16 + half * 8 + 2 * tig;
                const float2 xa = vA ? *reinterpret_cast<const float2 *>(rA + c) : make_float2(0.f, 0.f);
                const float2 xb = vB ? *reinterpret_cast<const float2 *>(rB + c) : make_float2(0.f, 0.f);
                split_bf16(xa.x, xa.y, qhi[kk][half * 2], qlo[kk][half * 2]);
                split_bf16(xb.x, xb.y, qhi[kk][half * 2 + 1], qlo[kk][half * 2 + 1]);
            }
        }
    }
    constexpr int KR16 = DR / 16, KR8 = (DR % 16) / 8;
    uint32_t rhi[KR16 > 0 ? KR16 : 1][4], rlo[KR16 > 0 ? KR16 : 1][4];
    uint32_t r8hi[2], r8lo[2];
    if (DR > 0) {
        const float *rA = p.qh + (((long long)b * p.n + iA) * p.H + hA) * DR;
        const float *rB = p.qh + (((long long)b * p.n + iB) * p.H + hB) * DR;
#pragma unroll
        for (int kk = 0; kk < KR16; ++kk) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int c = kk * 16 + half * 8 + 2 * tig;
                const float2 xa = vA ? *reinterpret_cast<const float2 *>(rA + c) : make_float2(0.f, 0.f);
                const float2 xb = vB ? *reinterpret_cast<const float2 *>(rB + c) : make_float2(0.f, 0.f);
                split_bf16(xa.x, xa.y, rhi[kk][half * 2], rlo[kk][half * 2]);
                split_bf16(xb.x, xb.y, rhi[kk][half * 2 + 1], rlo[kk][half * 2 + 1]);
            }
        }
        if (KR8) {
            const int c = KR16 * 16 + 2 * tig;
            const float2 xa = vA ? *reinterpret_cast<const float2 *>(rA + c) : make_float2(0.f, 0.f);
            const float2 xb = vB ? *reinterpret_cast<const float2 *>(rB + c) : make_float2(0.f, 0.f);
            split_bf16(xa.x, xa.y, r8hi[0], r8lo[0]);
            split_bf16(xb.x, xb.y, r8hi[1], r8lo[1]);
        }
    }

    const uint32_t sbase = smem_u32(pf_smem);
    auto load_slab = [&](int k, int st) {
        const long long j0 = (s_begin + k) * SLAB;
        const long long row0 = row_of(p.R, b, j0);
        if (row0 < 0 && threadIdx.x == 0) dev_report(GVA_DEV_BAD_PAGE);
        const int valid = row0 < 0 ? 0 : (int)min((long long)SLAB, Lt - j0);
        const uint32_t sv = sbase + st * p.stage_bytes;
        const int vch = GDH / 8;   // 16-byte chunks per value row
        for (int c = threadIdx.x; c < SLAB * vch; c += WARPS * 32) {
            const int t = c / vch, cc = c - t * vch;
            const bool ok = t < valid;
            const void *src = ok ? static_cast<const void *>(
                                       static_cast<const __nv_bfloat16 *>(p.V) +
                                       (row0 + t) * GDH + cc * 8)
                                 : p.V;
            cp_async16(sv + t * p.vpitch + cc * 16, src, ok ? 16 : 0);
        }
        if (DR > 0) {
            const uint32_t sk = sv + SLAB * p.vpitch;
            constexpr int kch = DR > 0 ? DR / 8 : 1;
            for (int c = threadIdx.x; c < SLAB * kch; c += WARPS * 32) {
                const int t = c / kch, cc = c - t * kch;
                const bool ok = t < valid;
                const void *src = ok ? static_cast<const void *>(
                                           static_cast<const __nv_bfloat16 *>(p.Kr) +
                                           (row0 + t) * DR + cc * 8)
                                     : p.Kr;
                cp_async16(sk + t * (DR * 2) + cc * 16, src, ok ? 16 : 0);
            }
        }
    };

#pragma unroll
    for (int k = 0; k < PF_STAGES - 1; ++k) {
        if (k < ns) load_slab(k, k);
        cp_async_commit();
    }
    float o[DH / 8][4];
#pragma unroll
    for (int nt = 0; nt < DH / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
    const int mi = lane >> 3, rr = lane & 7;

    for (int k = 0; k < ns; ++k) {
        cp_async_wait<PF_STAGES - 2>();
        __syncthreads();
        {
            const int kn = k + PF_STAGES - 1;
            if (kn < ns) load_slab(kn, kn % PF_STAGES);
            cp_async_commit();
        }
        const long long j0 = (s_begin + k) * SLAB;
        if (j0 > wlim) continue;   // no row of this warp sees any token of the slab
        const uint32_t sv = sbase + (k % PF_STAGES) * p.stage_bytes;
        // the hi and lo query parts accumulate separately (two independent MMA chains
        // per score tile), summed before the mask
        float s[2][4], sl[2][4];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
            sl[t][0] = sl[t][1] = sl[t][2] = sl[t][3] = 0.f;
        }
        // S = Q~ V_g^T: matrices (tokens 0-7 | 8-15) x (dims lo | hi) of a 16-dim step
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
            const int tok = (mi >> 1) * 8 + rr, dim = kk * 16 + (mi & 1) * 8;
            uint32_t b0, b1, b2, b3;
            ldsm_x4(sv + tok * p.vpitch + (g * DH + dim) * 2, b0, b1, b2, b3);
            mma16816(s[0], qhi[kk], b0, b1);
            mma16816(sl[0], qlo[kk], b0, b1);
            mma16816(s[1], qhi[kk], b2, b3);
            mma16816(sl[1], qlo[kk], b2, b3);
        }
        if (DR > 0) {
            const uint32_t sk = sv + SLAB * p.vpitch;
#pragma unroll
            for (int kk = 0; kk < KR16; ++kk) {
                const int tok = (mi >> 1) * 8 + rr, dim = kk * 16 + (mi & 1) * 8;
                uint32_t b0, b1, b2, b3;
                ldsm_x4(sk + tok * (DR * 2) + dim * 2, b0, b1, b2, b3);
                mma16816(s[0], rhi[kk], b0, b1);
                mma16816(sl[0], rlo[kk], b0, b1);
                mma16816(s[1], rhi[kk], b2, b3);
                mma16816(sl[1], rlo[kk], b2, b3);
            }
            if (KR8) {
                const int tok = (mi & 1) * 8 + rr;
                uint32_t b0, b1;
                ldsm_x2(sk + tok * (DR * 2) + KR16 * 16 * 2, b0, b1);
                mma1688(s[0], r8hi[0], r8hi[1], b0);
                mma1688(sl[0], r8lo[0], r8lo[1], b0);
                mma1688(s[1], r8hi[0], r8hi[1], b1);
                mma1688(sl[1], r8lo[0], r8lo[1], b1);
            }
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            s[t][0] += sl[t][0];
            s[t][1] += sl[t][1];
            s[t][2] += sl[t][2];
            s[t][3] += sl[t][3];
        }
        // causal mask: column (tile t, pair element e) is token j0 + 8t + 2tig + e
#pragma unroll
        for (int t = 0; t < 2; ++t) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const long long j = j0 + t * 8 + 2 * tig + e;
                if (j > limA) s[t][e] = -INFINITY;
                if (j > limB) s[t][2 + e] = -INFINITY;
            }
        }
        float xA = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
        float xB = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
        xA = fmaxf(xA, __shfl_xor_sync(0xffffffffu, xA, 1));
        xB = fmaxf(xB, __shfl_xor_sync(0xffffffffu, xB, 1));
        xA = fmaxf(xA, __shfl_xor_sync(0xffffffffu, xA, 2));
        xB = fmaxf(xB, __shfl_xor_sync(0xffffffffu, xB, 2));
        const float nA = fmaxf(mA, xA), nB = fmaxf(mB, xB);
        // a row that has seen no visible token keeps max -inf; 0 stands in as reference
        const float refA = nA == -INFINITY ? 0.f : nA, refB = nB == -INFINITY ? 0.f : nB;
        const float aA = exp2f(mA - refA), aB = exp2f(mB - refB);
        mA = nA;
        mB = nB;
        float pr[2][4];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            pr[t][0] = exp2f(s[t][0] - refA);
            pr[t][1] = exp2f(s[t][1] - refA);
            pr[t][2] = exp2f(s[t][2] - refB);
            pr[t][3] = exp2f(s[t][3] - refB);
        }
        lA = lA * aA + (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
        lB = lB * aB + (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
#pragma unroll
        for (int nt = 0; nt < DH / 8; ++nt) {
            o[nt][0] *= aA;
            o[nt][1] *= aA;
            o[nt][2] *= aB;
            o[nt][3] *= aB;
        }
        // P as the A operand of P V: the score tiles' accumulator layout is the A layout
        uint32_t ph[4], pl[4];
        split_bf16(pr[0][0], pr[0][1], ph[0], pl[0]);
        split_bf16(pr[0][2], pr[0][3], ph[1], pl[1]);
        split_bf16(pr[1][0], pr[1][1], ph[2], pl[2]);
        split_bf16(pr[1][2], pr[1][3], ph[3], pl[3]);
        // O += P V_g: matrices (tokens 0-7 | 8-15) x (dims lo | hi) of a 16-dim pair of
        // output tiles, transposed on load
#pragma unroll
        for (int np = 0; np < DH / 16; ++np) {
            const int tok = (mi & 1) * 8 + rr, dim = np * 16 + (mi >> 1) * 8;
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(sv + tok * p.vpitch + (g * DH + dim) * 2, b0, b1, b2, b3);
            mma16816(o[2 * np], ph, b0, b1);
            mma16816(o[2 * np], pl, b0, b1);
            mma16816(o[2 * np + 1], ph, b2, b3);
            mma16816(o[2 * np + 1], pl, b2, b3);
        }
    }
    cp_async_wait<0>();
    if (!active) return;
    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    const long long base = ((long long)b * p.splits + split) * p.rows_pad + (long long)g * p.wpg * 16;
    float *oA = p.part_o + (base + qA) * DH, *oB = p.part_o + (base + qB) * DH;
#pragma unroll
    for (int nt = 0; nt < DH / 8; ++nt) {
        *reinterpret_cast<float2 *>(oA + nt * 8 + 2 * tig) = make_float2(o[nt][0], o[nt][1]);
        *reinterpret_cast<float2 *>(oB + nt * 8 + 2 * tig) = make_float2(o[nt][2], o[nt][3]);
    }
    if (tig == 0) {
        *reinterpret_cast<float2 *>(p.part_ml + (base + qA) * 2) = make_float2(mA, lA);
        *reinterpret_cast<float2 *>(p.part_ml + (base + qB) * 2) = make_float2(mB, lB);
    }
}

// Log-sum-exp merge of the slab ranges: one warp per (b, i, h).  The lanes read the
// ranges' (max, sum) 32 at a time, so every load of a row is independent of the others.
constexpr int PF_COMBINE_WARPS = 8;

template <int DH>
__global__ void __launch_bounds__(PF_COMBINE_WARPS * 32)
    prefill_combine_kernel(const PrefillMmaParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * PF_COMBINE_WARPS + warp;   // (b, i, h)
    if (row >= (long long)p.B * p.n * p.H) return;
    const int h = (int)(row % p.H);
    const long long bi = row / p.H;
    const int i = (int)(bi % p.n), b = (int)(bi / p.n);
    const int g = h / p.r;
    const long long prow = (long long)g * p.wpg * 16 + (long long)i * p.r + (h - g * p.r);
    const long long at0 = (long long)b * p.splits * p.rows_pad + prow;   // range 0's row
    float M = -INFINITY;
    for (int s0 = 0; s0 < p.splits; s0 += 32) {
        const int s = s0 + lane;
        if (s < p.splits) M = fmaxf(M, p.part_ml[(at0 + (long long)s * p.rows_pad) * 2]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float acc[DH / 32];
#pragma unroll
    for (int u = 0; u < DH / 32; ++u) acc[u] = 0.f;
    float den = 0.f;
    if (M != -INFINITY) {
        for (int s0 = 0; s0 < p.splits; s0 += 32) {
            const int s = s0 + lane;
            float w = 0.f;
            if (s < p.splits) {
                const float2 ml =
                    *reinterpret_cast<const float2 *>(p.part_ml + (at0 + (long long)s * p.rows_pad) * 2);
                w = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
                den += w * ml.y;
            }
            const int cnt = min(32, p.splits - s0);
#pragma unroll 4
            for (int k = 0; k < cnt; ++k) {
                // a range whose rows saw nothing wrote zeros, so its weight 0 adds 0
                const float wk = __shfl_sync(0xffffffffu, w, k);
                const float *src = p.part_o + (at0 + (long long)(s0 + k) * p.rows_pad) * DH;
#pragma unroll
                for (int u = 0; u < DH / 32; ++u) acc[u] += wk * src[lane + 32 * u];
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    float *dst = p.out + row * DH;
#pragma unroll
    for (int u = 0; u < DH / 32; ++u) dst[lane + 32 * u] = den > 0.f ? acc[u] / den : 0.f;
    if (p.lse && lane == 0) p.lse[row] = den > 0.f ? (M + log2f(den)) * LN2 : -INFINITY;
}

// ---------------------------------------------------------------------------- //
// host side
// ---------------------------------------------------------------------------- //
struct PrefillMmaPlan {
    int warps, wpg, tiles, splits, rows_pad, vpitch, stage_bytes;
    size_t smem, part_o_bytes, part_ml_bytes;
};

inline int prefill_warps(int d_h) { return d_h == 64 ? 16 : 8; }

// bf16 cache, d_h 64 or 128, d_r in {0, 8, 16, 24, 32}, and a ring that fits.
inline bool prefill_mma_plan(const gva_dims *d, int n, int sms, PrefillMmaPlan *pl) {
    if (d->cache_dtype != GVA_BF16 || (d->d_h != 64 && d->d_h != 128)) return false;
    if (d->d_r != 0 && d->d_r != 8 && d->d_r != 16 && d->d_r != 24 && d->d_r != 32) return false;
    const int r = d->H / d->G;
    pl->warps = prefill_warps(d->d_h);
    pl->wpg = (n * r + 15) / 16;
    pl->rows_pad = d->G * pl->wpg * 16;
    pl->tiles = (d->G * pl->wpg + pl->warps - 1) / pl->warps;
    // one CTA per SM (the kernel's registers allow one): as many slab ranges per
    // sequence as keep the grid within a single wave
    const long long ctas = (long long)d->B * pl->tiles;
    const long long sp = ctas >= sms ? 1 : sms / ctas;
    pl->splits = (int)sp;
    pl->vpitch = d->G * d->d_h * 2 + 16;
    pl->stage_bytes = (int)align_up((size_t)SLAB * pl->vpitch + (size_t)SLAB * d->d_r * 2, 128);
    pl->smem = (size_t)PF_STAGES * pl->stage_bytes;
    if (pl->smem > (size_t)PF_SMEM_LIMIT) return false;
    if (pl->tiles > 65535) return false;
    const size_t rows = (size_t)d->B * pl->splits * pl->rows_pad;
    pl->part_o_bytes = align_up(rows * d->d_h * sizeof(float), 256);
    pl->part_ml_bytes = align_up(rows * 2 * sizeof(float), 256);
    return true;
}

template <int DH, int DR>
inline cudaError_t prefill_launch_dr(void *stream, const PrefillMmaPlan &pl, const PrefillMmaParams &p) {
    constexpr int W = DH == 64 ? 16 : 8;
    const dim3 grid(pl.splits, pl.tiles, p.B);
    cudaError_t e = launch(prefill_mma_kernel<DH, DR, W>, grid, dim3(W * 32), pl.smem, stream, p);
    if (e != cudaSuccess) return e;
    const long long rows = (long long)p.B * p.n * p.H;
    const dim3 cg((unsigned)((rows + PF_COMBINE_WARPS - 1) / PF_COMBINE_WARPS));
    return launch(prefill_combine_kernel<DH>, cg, dim3(PF_COMBINE_WARPS * 32), 0, stream, p);
}

template <int DH>
inline cudaError_t prefill_launch_dh(void *stream, int d_r, const PrefillMmaPlan &pl,
                                     const PrefillMmaParams &p) {
    switch (d_r) {
    case 0: return prefill_launch_dr<DH, 0>(stream, pl, p);
    case 8: return prefill_launch_dr<DH, 8>(stream, pl, p);
    case 16: return prefill_launch_dr<DH, 16>(stream, pl, p);
    case 24: return prefill_launch_dr<DH, 24>(stream, pl, p);
    default: return prefill_launch_dr<DH, 32>(stream, pl, p);
    }
}

template <int DH>
inline cudaError_t prefill_opt_in_dh() {
    constexpr int W = DH == 64 ? 16 : 8;
    const int lim = PF_SMEM_LIMIT;
    cudaError_t e = cudaFuncSetAttribute(prefill_mma_kernel<DH, 0, W>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(prefill_mma_kernel<DH, 8, W>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(prefill_mma_kernel<DH, 16, W>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(prefill_mma_kernel<DH, 24, W>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(prefill_mma_kernel<DH, 32, W>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    return e;
}

inline cudaError_t prefill_opt_in_all() {
    cudaError_t e = prefill_opt_in_dh<64>();
    return e == cudaSuccess ? prefill_opt_in_dh<128>() : e;
}

}  // namespace gva
