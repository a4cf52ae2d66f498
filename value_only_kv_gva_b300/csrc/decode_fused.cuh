// decode_fused.cuh -- split-K GVA decode on the tensor cores for bf16 caches with the
// log-sum-exp merge of the splits in the same kernel.
//
// Work is split over (value group g, sequence b) pairs.  The unit of the split-K
// partition is one 16-token slab of one group; the units are ordered group-major,
// u = g * S + s (s the flat slab index over the batch, S the slab count), and every CTA
// (one per SM) takes one contiguous, equal share of them, so a CTA touches one or a few
// pairs.  The absorbed queries q~_h = q_h^nope M_h^T and the rotated positional queries
// (GVA analysis page, 关键技巧一 / 关键技巧二) come from the absorption kernel that
// precedes this one; the cache is streamed before that grid has finished.
//
// Streaming: the producer warp copies chunks of up to KC consecutive slabs of one pair
// (KC * 16 tokens x d_h values, plus the matching positional-key rows) into a ring of
// shared-memory stages, one mbarrier per stage.  The value copy is a tensor copy through
// a 4D view of the cache whose fourth dimension steps 16 rows at a time, so a single
// TMA instruction moves up to 16 slabs; chunk sizes are issued as powers of two.  A
// chunk holds only whole slabs of one sequence, so every row it reads is inside the
// cache storage; a sequence's last, partial slab is a chunk of its own, read through
// the bounds-checked row dimension (rows past the storage are zero-filled).
//
// Consumers: 8 warps take the slabs of each chunk round-robin and score / accumulate
// with bf16 mma.sync (tokens on the MMA rows, the group's heads on the columns, bf16
// hi + lo parts of the fp32 query and probabilities), online softmax in log2 units
// with a lazy rescale.  At the end of a pair the 8 warps' partial (m, l, O) are merged
// in shared memory.  A pair served by one CTA is written out directly; otherwise each
// CTA stores its partial and the last of them to finish (an atomic ticket per pair)
// merges all of them and writes the output and the log-sum-exp.
//
// Every wait on an mbarrier is bounded; on expiry the kernel sets GVA_DEV_TIMEOUT,
// stops consuming, keeps the pair-end barriers and tickets balanced, waits (bounded)
// for its copies in flight and returns.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "decode_mma.cuh"

namespace gva {

constexpr int FU_NC = 8;                          // consumer warps
constexpr int FU_THREADS = (FU_NC + 1) * 32;
constexpr int FU_NQ = 4;                          // pairs whose queries are staged at once
constexpr int FU_MAX_STAGES = 32;
constexpr int FU_MAX_KC = 16;                     // slabs per chunk (TMA box depth)

struct FusedParams {
    int B, H, G, r, d_r;
    const int *seq_len;
    RowsDev R;
    const void *Krope;        // [rows][d_r] bf16
    const float *qt;          // absorbed content queries [B][H][d_h], log2-scaled
    const float *qh;          // rotated positional queries [B][H][d_r], log2-scaled
    float *out;               // [B][H][d_h]
    float *lse;               // [B][H] or null
    float *part_o;            // [slots][r][d_h]
    float *part_ml;           // [slots][r][2]
    int *ticket;              // [G * B], zero between calls
    int n_ctas;
    int early;                // 1: lengths, row maps and cache are final before the
                              //    preceding grid (the absorption) started
    // ring and shared-memory plan
    int kc;                   // slabs per chunk (power of two, <= 16)
    int nss;                  // ring stages
    int off_kr;               // positional-key ring
    int off_bar;              // full[nss], empty[nss], abort, chunk_bad[nss]
    int off_ls;               // Ls[B], F[B + 1]
    int off_qt;               // content queries of the staged pairs [FU_NQ][4 NT][d_h]
    int off_qh;               // positional queries [FU_NQ][4 NT][d_r]
    int off_mg;               // warp merge [FU_NC][4 NT][d_h + 2] fp32
    int off_flag;             // last-arriver flag
};

// The chunks of a CTA's share, in order.  A chunk is a run of consecutive slabs of one
// pair: it ends at a multiple of kc (sequence-relative), at the sequence's first
// partial slab (which is a chunk of its own), at the end of the sequence and at the end
// of the share.
struct ChunkIter {
    long long u, u1;   // next unit, end of the share
    long long S;       // slabs per group
    long long s;       // flat slab of unit u (u - g * S)
    int g, b;          // pair of unit u
    __device__ void init(long long u0, long long u1_, long long S_, const int *F, int B) {
        u = u0;
        u1 = u1_;
        S = S_;
        g = S > 0 ? (int)(u0 / S) : 0;
        s = u0 - (long long)g * S;
        b = (u0 < u1 && S > 0) ? seq_of_slab(F, B, s) : 0;
    }
    // Next chunk: pair (cg, cb), first sequence-relative slab k0, slab count kc.
    __device__ __forceinline__ bool next(const int *F, const int *Ls, int kcap, int &cg, int &cb,
                                         int &k0, int &kc) {
        if (u >= u1) return false;
        while (F[b + 1] <= s) ++b;   // skips empty sequences; s < S keeps b < B
        cg = g;
        cb = b;
        k0 = (int)(s - F[b]);
        const int nf = Ls[b] / SLAB;   // whole slabs
        int c;
        if (k0 >= nf) {
            c = 1;
        } else {
            c = kcap - (k0 & (kcap - 1));
            if (c > nf - k0) c = nf - k0;
        }
        if ((long long)c > u1 - u) c = (int)(u1 - u);
        kc = c;
        u += c;
        s += c;
        if (s >= S) {
            s -= S;
            ++g;
            b = 0;
        }
        return true;
    }
};

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *tm, int x, int y,
                                            int z, int w, uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar), "l"(pol)
        : "memory");
}

// The five value maps: box depth 1, 2, 4, 8, 16 slabs.
struct FusedMaps {
    CUtensorMap m[5];
};

// Byte address of the 16-byte chunk c (8 bf16 along d) of token row t within one slab
// of one group: DH / 64 boxes of 16 rows x 128 bytes, 128-byte swizzled.
__device__ __forceinline__ uint32_t slab_addr(uint32_t slab_base, int t, int c) {
    return slab_base + (c >> 3) * 2048 + t * 128 + (((c & 7) ^ (t & 7)) << 4);
}

// Stage the queries of up to FU_NQ pairs in shared memory (all consumer threads; ends
// with a consumer-wide barrier): slot sl[j] <- pair (gs[j], bs[j]), heads hl < r from
// the absorbed queries in global memory, heads r .. 4 NT - 1 zero.
template <int DH, int DR, int NT>
__device__ void fused_load_queries(const FusedParams &p, unsigned char *base, const int *sl,
                                   const int *gs, const int *bs, int np, int ct) {
    constexpr int NH = 4 * NT;
    const int r = p.r;
    float *qt = reinterpret_cast<float *>(base + p.off_qt);
    float *qh = reinterpret_cast<float *>(base + p.off_qh);
    const int NCT = FU_NC * 32;
    for (int e = ct; e < np * NH * (DH / 4); e += NCT) {
        const int j = e / (NH * (DH / 4)), rem = e % (NH * (DH / 4));
        const int hl = rem / (DH / 4), i4 = rem % (DH / 4);
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (hl < r)
            v = *(reinterpret_cast<const float4 *>(
                      p.qt + ((long long)bs[j] * p.H + gs[j] * r + hl) * DH) + i4);
        *reinterpret_cast<float4 *>(qt + (sl[j] * NH + hl) * DH + 4 * i4) = v;
    }
    if (DR > 0) {
        constexpr int DR4 = DR > 0 ? DR / 4 : 1;
        for (int e = ct; e < np * NH * DR4; e += NCT) {
            const int j = e / (NH * DR4), rem = e % (NH * DR4);
            const int hl = rem / DR4, i4 = rem % DR4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (hl < r)
                v = *(reinterpret_cast<const float4 *>(
                          p.qh + ((long long)bs[j] * p.H + gs[j] * r + hl) * DR) + i4);
            *reinterpret_cast<float4 *>(qh + (sl[j] * NH + hl) * DR + 4 * i4) = v;
        }
    }
    named_bar(1, NCT);
}

template <int DH, int DR, int NT>
__global__ void __launch_bounds__(FU_THREADS, 1)
    decode_fused_kernel(const __grid_constant__ FusedMaps maps, const FusedParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    GVA_TRACE_DECL;
    constexpr int NH = 4 * NT;
    constexpr int KD = DH / 16;
    constexpr int SLABV = SLAB * DH * 2;          // bytes of one slab of one group
    constexpr int SLABR = SLAB * DR * 2;
    constexpr int DRK16 = DR / 16;
    constexpr bool DR_K8 = (DR % 16) == 8;
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
    unsigned char *base = smem_raw + (base_u32 - raw_u32);
    const int NSS = p.nss, KC = p.kc;
    const uint32_t bar_full = base_u32 + p.off_bar;
    const uint32_t bar_empty = bar_full + 8 * NSS;
    volatile int *abort = reinterpret_cast<volatile int *>(base + p.off_bar + 16 * NSS);
    int *chunk_bad = reinterpret_cast<int *>(base + p.off_bar + 16 * NSS + 16);
    int *Ls = reinterpret_cast<int *>(base + p.off_ls);
    int *F = Ls + p.B;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int B = p.B, G = p.G, r = p.r;

    if (warp == 0) {
        for (int s = lane; s < NSS; s += 32) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, FU_NC);
        }
        if (lane == 0) *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (lane == 0)
            for (int k = 0; k < 5; ++k) prefetch_tmap(&maps.m[k]);
    }
    if (threadIdx.x == 0) GVA_CTA_T(0);
    if (threadIdx.x == 0) GVA_KT(5);
    if (threadIdx.x == 0) GVA_TRACE_AT(0);
    // With `early`, lengths, row maps and the cache were final before the preceding
    // grid (the absorption) was allowed to start: they are read at once and the cache
    // streams while that grid still runs; the queries are read after the wait.
    if (!p.early) pdl_wait();
    if (threadIdx.x == 0) GVA_TRACE_AT(1);
    pdl_launch_dependents();
    build_prefix(p.seq_len, p.R, B, Ls, F, blockIdx.x == 0);   // includes __syncthreads
    if (threadIdx.x == 0) GVA_TRACE_AT(2);
    const long long S = F[B];
    const Part P{(long long)G * S, p.n_ctas};
    const int c = blockIdx.x;
    const long long u0 = S > 0 ? P.start(c) : 0, u1 = S > 0 ? P.start(c + 1) : 0;
    // sequences with no tokens: zero output, -inf log-sum-exp (CTA 0, one warp per
    // sequence, after the wait: the preceding kernels may read the outputs)
    if (c == 0 && warp > 0) {
        if (p.early) pdl_wait();
        for (int b = warp - 1; b < B; b += FU_NC) {
            if (Ls[b] != 0) continue;
            float *ob = p.out + (long long)b * p.H * DH;
            for (int e = lane; e < p.H * DH; e += 32) ob[e] = 0.f;
            if (p.lse)
                for (int h = lane; h < p.H; h += 32) p.lse[(long long)b * p.H + h] = -INFINITY;
        }
    }
    if (u0 >= u1) return;

    // ============================= producer warp ============================= //
    // One step takes up to min(NSS, 32) chunks, one per lane: the lanes enumerate the
    // chunks together, find their rows (block-table reads in flight together), wait for
    // their ring stages and issue the copies.
    if (warp == 0) {
        const int il = NSS < 32 ? NSS : 32;
        const uint64_t pol = l2_evict_first_policy();
        ChunkIter it;
        it.init(u0, u1, S, F, B);
        long long ci0 = 0;     // ring index of the step's first chunk
        bool dead = false;
        for (;;) {
            const int lim = il;
            int mg = 0, mb = 0, mk0 = 0, mkc = 0, n = 0;
            for (; n < lim; ++n) {
                int cg, cb, k0, kc;
                if (!it.next(F, Ls, KC, cg, cb, k0, kc)) break;
                if (lane == n) { mg = cg; mb = cb; mk0 = k0; mkc = kc; }
            }
            if (n == 0) break;
            bool ok = true;
            if (lane < n) {
                const long long ci = ci0 + lane;
                const int ss = (int)(ci % NSS);
                const uint32_t rd = (uint32_t)(ci / NSS);
                const long long row = row_of(p.R, mb, (long long)mk0 * SLAB);
                if (rd > 0 && !mbar_wait(bar_empty + 8 * ss, (rd - 1) & 1u, abort)) {
                    ok = false;
                } else {
                    const uint32_t fb = bar_full + 8 * ss;
                    chunk_bad[ss] = row < 0;
                    if (row < 0) {
                        mbar_arrive(fb);   // nothing to copy: complete the phase
                    } else {
                        const int y = (int)row;
                        // positional-key rows: whole slabs, the last clamped to the storage
                        long long rrows = (long long)SLAB * mkc;
                        if (row + rrows > p.R.num_rows) rrows = p.R.num_rows - row;
                        if (rrows < 0) rrows = 0;
                        const uint32_t rbytes = DR > 0 ? (uint32_t)rrows * (DR * 2) : 0u;
                        mbar_expect_tx(fb, (uint32_t)(mkc * SLABV) + rbytes);
                        const uint32_t vdst = base_u32 + (uint32_t)ss * (uint32_t)(KC * SLABV);
                        int off = 0;
#pragma unroll
                        for (int lg = 4; lg >= 0; --lg) {
                            if (mkc & (1 << lg)) {
                                tma_load_4d(vdst + off * SLABV, &maps.m[lg], 0, y + SLAB * off,
                                            mg * (DH / 64), 0, fb, pol);
                                off += 1 << lg;
                            }
                        }
                        if (DR > 0 && rbytes > 0)
                            bulk_load(base_u32 + p.off_kr + (uint32_t)ss * (uint32_t)(KC * SLABR),
                                      reinterpret_cast<const unsigned char *>(p.Krope) +
                                          (size_t)row * (DR * 2),
                                      rbytes, fb, pol);
                    }
                }
            }
            dead = __any_sync(0xffffffffu, lane < n && !ok);
            ci0 += n;
            if (dead || n < lim) break;
        }
        if (lane == 0) {
            GVA_KT(8);
            GVA_TRACE_AT(22);
            GVA_TRACE_FLUSH(22, 23);
            // Never leave with copies in flight: wait (bounded) for the last use of each
            // stage (chunk i used stage i % NSS in round i / NSS).
            const unsigned long long limit = dead ? 1000000ull : WAIT_LIMIT_NS;
            for (int ss = 0; ss < NSS && ss < ci0; ++ss) {
                const uint32_t par = (uint32_t)((ci0 - 1 - ss) / NSS) & 1u;
                const unsigned long long t0 = global_ns();
                while (!mbar_try_wait(bar_full + 8 * ss, par)) {
                    if (global_ns() - t0 > limit) {
                        if (!dead) dev_report(GVA_DEV_TIMEOUT);
                        break;
                    }
                }
            }
        }
        return;
    }

    // ============================= consumer warps ============================ //
    const int w = warp - 1;              // consumer index
    const int ct = threadIdx.x - 32;     // consumer thread index
    const int gid = lane >> 2, tig = lane & 3;
    const int lm_mat = lane >> 3, lm_row = lane & 7;
    const int srcA = (2 * tig) * 4 + (gid >> 1), srcB = (2 * tig + 1) * 4 + (gid >> 1);
    const bool lo_col = (gid & 1) != 0;
    const float *qt_s = reinterpret_cast<const float *>(base + p.off_qt);
    const float *qh_s = reinterpret_cast<const float *>(base + p.off_qh);
    float *mg_s = reinterpret_cast<float *>(base + p.off_mg);
    volatile int *flag = reinterpret_cast<volatile int *>(base + p.off_flag);

    // Stage the queries of the share's first pairs (they come from the preceding grid).
    {
        int sl[FU_NQ], pg[FU_NQ], pb[FU_NQ], np = 0;
        for (long long u = u0; np < FU_NQ && u < u1;) {
            const int g = (int)(u / S);
            const int b = seq_of_slab(F, B, u - (long long)g * S);
#pragma unroll
            for (int j = 0; j < FU_NQ; ++j)
                if (j == np) { sl[j] = j; pg[j] = g; pb[j] = b; }
            ++np;
            u = (long long)g * S + F[b + 1];   // first unit of the next pair
        }
        if (w == 0 && lane == 0) GVA_TRACE_AT(3);
        if (p.early && c != 0) pdl_wait();   // (CTA 0 waited above)
        fused_load_queries<DH, DR, NT>(p, base, sl, pg, pb, np, ct);
    }
    if (w == 0 && lane == 0) {
        GVA_TRACE_AT(6);
        GVA_CTA_T(1);
        GVA_KT(6);
    }

    ChunkIter it;
    it.init(u0, u1, S, F, B);
    long long ci = 0;          // ring index of the chunk
    long long js = 0;          // slab index within the share (round-robin owner: js % FU_NC)
    int cur_p = -1, cur_g = 0, cur_b = 0, seg = -1;
    bool alive = true;
    uint32_t bq[KD][NT][2];
    uint32_t bqr[DRK16 > 0 ? DRK16 : 1][NT][2];
    uint32_t bqr8[NT];
    float oacc[KD][NT][4];
    float m_run[NT], l_run[NT];

    // Ends pair (cur_g, cur_b): merge the warps' partials, then write the output or this
    // CTA's partial and take a ticket.  Every consumer warp calls it the same number of
    // times (the named barriers inside it are consumer-wide).
    auto finish_pair = [&]() {
        // fold hi/lo columns, reduce l over the 8 token lanes, stage in shared memory
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], 4);
            l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], 8);
            l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], 16);
            float *mb = mg_s + (w * NH + 4 * nt + tig) * (DH + 2);
#pragma unroll
            for (int mt = 0; mt < KD; ++mt) {
                mb[16 * mt + gid] = oacc[mt][nt][0] + oacc[mt][nt][1];
                mb[16 * mt + gid + 8] = oacc[mt][nt][2] + oacc[mt][nt][3];
            }
            if (gid == 0) { mb[DH] = m_run[nt]; mb[DH + 1] = l_run[nt]; }
        }
        named_bar(1, FU_NC * 32);
        const int b = cur_b, g = cur_g;
        const long long first = (long long)g * S + F[b];
        const int nb = F[b + 1] - F[b];
        const int c_lo = P.cta_of(first), c_hi = P.cta_of(first + nb - 1);
        const int pp = g * B + b;
        const long long slot = (long long)c + pp;
        // thread ct merges outputs (hl, i) = ct, ct + 256, ...
        for (int o = ct; o < r * DH; o += FU_NC * 32) {
            const int hl = o / DH, i = o % DH;
            float mx = -INFINITY;
#pragma unroll
            for (int ww = 0; ww < FU_NC; ++ww) mx = fmaxf(mx, mg_s[(ww * NH + hl) * (DH + 2) + DH]);
            float L = 0.f, O = 0.f;
#pragma unroll
            for (int ww = 0; ww < FU_NC; ++ww) {
                const float *mb = mg_s + (ww * NH + hl) * (DH + 2);
                const float a = mb[DH] == -INFINITY ? 0.f : exp2f(mb[DH] - mx);
                L += a * mb[DH + 1];
                O += a * mb[i];
            }
            const int h = g * r + hl;
            if (c_lo == c_hi) {
                p.out[((long long)b * p.H + h) * DH + i] = L > 0.f ? O / L : 0.f;
                if (i == 0 && p.lse)
                    p.lse[(long long)b * p.H + h] = L > 0.f ? (mx + log2f(L)) * LN2 : -INFINITY;
            } else {
                p.part_o[(slot * r + hl) * DH + i] = O;
                if (i == 0) {
                    p.part_ml[(slot * r + hl) * 2] = mx;
                    p.part_ml[(slot * r + hl) * 2 + 1] = L;
                }
            }
        }
        if (c_lo != c_hi) {
            // publish the partial, take a ticket; the last CTA of the pair merges
            __threadfence();
            named_bar(1, FU_NC * 32);
            if (ct == 0) {
                const int old = atomicAdd(&p.ticket[pp], 1);
                const bool last = old == c_hi - c_lo;
                if (last) {
                    __threadfence();
                    p.ticket[pp] = 0;   // ready for the next call
                }
                *flag = last ? 1 : 0;
            }
            named_bar(1, FU_NC * 32);
            if (*flag) {
                for (int o = ct; o < r * DH; o += FU_NC * 32) {
                    const int hl = o / DH, i = o % DH;
                    float mx = -INFINITY;
                    for (int cc = c_lo; cc <= c_hi; ++cc)
                        mx = fmaxf(mx, __ldcg(p.part_ml + (((long long)cc + pp) * r + hl) * 2));
                    float L = 0.f, O = 0.f;
                    for (int cc = c_lo; cc <= c_hi; ++cc) {
                        const long long sl = (long long)cc + pp;
                        const float m = __ldcg(p.part_ml + (sl * r + hl) * 2);
                        const float a = m == -INFINITY ? 0.f : exp2f(m - mx);
                        L += a * __ldcg(p.part_ml + (sl * r + hl) * 2 + 1);
                        O += a * __ldcg(p.part_o + (sl * r + hl) * DH + i);
                    }
                    const int h = g * r + hl;
                    p.out[((long long)b * p.H + h) * DH + i] = L > 0.f ? O / L : 0.f;
                    if (i == 0 && p.lse)
                        p.lse[(long long)b * p.H + h] = L > 0.f ? (mx + log2f(L)) * LN2 : -INFINITY;
                }
            }
        }
        // the merge buffer and the flag are reused by the next pair
        named_bar(1, FU_NC * 32);
    };

    int cg, cb, k0, kc;
    while (it.next(F, Ls, KC, cg, cb, k0, kc)) {
        const int pp = cg * B + cb;
        if (pp != cur_p) {
            if (cur_p >= 0) finish_pair();
            cur_p = pp;
            cur_g = cg;
            cur_b = cb;
            ++seg;
            int slot = seg;
            if (seg >= FU_NQ) {
                // staged on demand: the slot's previous pair is finished by every warp
                slot = seg % FU_NQ;
                int sl[FU_NQ], gg[FU_NQ], bb[FU_NQ];
                sl[0] = slot;
                gg[0] = cg;
                bb[0] = cb;
                fused_load_queries<DH, DR, NT>(p, base, sl, gg, bb, 1, ct);
            }
            // ---- Q^T fragments: column gid = head 4nt + gid/2, hi (gid even) or lo part ----
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int hl = 4 * nt + (gid >> 1);
                const float *qrow = qt_s + (slot * NH + hl) * DH;
#pragma unroll
                for (int kk = 0; kk < KD; ++kk) {
                    const int d0 = kk * 16 + tig * 2;
                    bq[kk][nt][0] = part_bf16x2(qrow[d0], qrow[d0 + 1], lo_col);
                    bq[kk][nt][1] = part_bf16x2(qrow[d0 + 8], qrow[d0 + 9], lo_col);
                }
                if (DR > 0) {
                    const float *hrow = qh_s + (slot * NH + hl) * DR;
#pragma unroll
                    for (int kk = 0; kk < DRK16; ++kk) {
                        const int d0 = kk * 16 + tig * 2;
                        bqr[kk][nt][0] = part_bf16x2(hrow[d0], hrow[d0 + 1], lo_col);
                        bqr[kk][nt][1] = part_bf16x2(hrow[d0 + 8], hrow[d0 + 9], lo_col);
                    }
                    if (DR_K8) {
                        const int d0 = DRK16 * 16 + tig * 2;
                        bqr8[nt] = part_bf16x2(hrow[d0], hrow[d0 + 1], lo_col);
                    }
                }
#pragma unroll
                for (int mt = 0; mt < KD; ++mt)
                    oacc[mt][nt][0] = oacc[mt][nt][1] = oacc[mt][nt][2] = oacc[mt][nt][3] = 0.f;
                m_run[nt] = -INFINITY;
                l_run[nt] = 0.f;
            }
        }
        const int ss = (int)(ci % NSS);
        const uint32_t par = (uint32_t)(ci / NSS) & 1u;
        ++ci;
        if (alive) alive = __all_sync(0xffffffffu, mbar_wait(bar_full + 8 * ss, par, abort));
        if (w == 0 && lane == 0 && ci <= 64) GVA_TRACE_AT(100 + (int)ci);
        const bool bad = alive && chunk_bad[ss] != 0;
        if (bad && w == 0 && lane == 0) dev_report(GVA_DEV_BAD_PAGE);
        const int Lb = Ls[cb];
        // this warp's slabs of the chunk: j = first, first + FU_NC, ...
        int j = (int)((w - js % FU_NC + FU_NC) % FU_NC);
        js += kc;
        for (; alive && j < kc; j += FU_NC) {
            const int kk_slab = k0 + j;
            int nv = min(SLAB, Lb - kk_slab * SLAB);
            if (bad) nv = 0;
            const uint32_t st = base_u32 + (uint32_t)ss * (uint32_t)(KC * SLABV) + (uint32_t)(j * SLABV);
            const uint32_t rt = base_u32 + p.off_kr + (uint32_t)ss * (uint32_t)(KC * SLABR) + (uint32_t)(j * SLABR);

            // ---- scores: A = the value tile (tokens x d), B = Q^T ----
            float sc[NT][2][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int a2 = 0; a2 < 2; ++a2)
                    sc[nt][a2][0] = sc[nt][a2][1] = sc[nt][a2][2] = sc[nt][a2][3] = 0.f;
            {
                uint32_t av[KD][4];
#pragma unroll
                for (int kk = 0; kk < KD; ++kk)
                    ldsm_x4(slab_addr(st, lm_row + 8 * (lm_mat & 1), 2 * kk + (lm_mat >> 1)),
                            av[kk][0], av[kk][1], av[kk][2], av[kk][3]);
                uint32_t ar[DRK16 > 0 ? DRK16 : 1][4], ar8[2];
                if (DR > 0) {
#pragma unroll
                    for (int kk = 0; kk < DRK16; ++kk)
                        ldsm_x4(rt + (lm_row + 8 * (lm_mat & 1)) * (DR * 2) + (2 * kk + (lm_mat >> 1)) * 16,
                                ar[kk][0], ar[kk][1], ar[kk][2], ar[kk][3]);
                    if (DR_K8)
                        ldsm_x2(rt + (lm_row + 8 * (lm_mat & 1)) * (DR * 2) + DRK16 * 32, ar8[0], ar8[1]);
                }
#pragma unroll
                for (int kk = 0; kk < KD; ++kk)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma16816(sc[nt][kk & 1], av[kk], bq[kk][nt][0], bq[kk][nt][1]);
                if (DR > 0) {
#pragma unroll
                    for (int kk = 0; kk < DRK16; ++kk)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma16816(sc[nt][(KD + kk) & 1], ar[kk], bqr[kk][nt][0], bqr[kk][nt][1]);
                    if (DR_K8) {
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma1688(sc[nt][(KD + DRK16) & 1], ar8[0], ar8[1], bqr8[nt]);
                    }
                }
            }
            // value tiles for the weighted sum (V^T as the A operand)
            uint32_t apv[KD][4];
#pragma unroll
            for (int mt = 0; mt < KD; ++mt)
                ldsm_x4_t(slab_addr(st, lm_row + 8 * (lm_mat >> 1), 2 * mt + (lm_mat & 1)),
                          apv[mt][0], apv[mt][1], apv[mt][2], apv[mt][3]);

            // ---- per head: hi + lo columns -> score of tokens gid, gid + 8 ----
            float z[NT][2];
            bool over = false;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                z[nt][0] = (sc[nt][0][0] + sc[nt][0][1]) + (sc[nt][1][0] + sc[nt][1][1]);
                z[nt][1] = (sc[nt][0][2] + sc[nt][0][3]) + (sc[nt][1][2] + sc[nt][1][3]);
                if (gid >= nv) z[nt][0] = -INFINITY;
                if (gid + 8 >= nv) z[nt][1] = -INFINITY;
                over |= fmaxf(z[nt][0], z[nt][1]) > m_run[nt] + MMA_RESCALE_TH;
            }
            // lazy rescale: the running maximum moves only when a score exceeds it by
            // more than the threshold (always on a head's first valid token)
            if (__any_sync(0xffffffffu, over)) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float m = fmaxf(z[nt][0], z[nt][1]);
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                    const bool raise = m > m_run[nt] + MMA_RESCALE_TH;
                    const float alpha = raise ? exp2f(m_run[nt] - m) : 1.f;
                    if (raise) m_run[nt] = m;
                    l_run[nt] *= alpha;
#pragma unroll
                    for (int mt = 0; mt < KD; ++mt) {
                        oacc[mt][nt][0] *= alpha; oacc[mt][nt][1] *= alpha;
                        oacc[mt][nt][2] *= alpha; oacc[mt][nt][3] *= alpha;
                    }
                }
            }
            // ---- probabilities, then P^T as the B operand ----
            uint32_t bp[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float p0 = z[nt][0] == -INFINITY ? 0.f : exp2f(z[nt][0] - m_run[nt]);
                const float p1 = z[nt][1] == -INFINITY ? 0.f : exp2f(z[nt][1] - m_run[nt]);
                l_run[nt] += p0 + p1;
                const float a0 = __shfl_sync(0xffffffffu, p0, srcA);
                const float a1 = __shfl_sync(0xffffffffu, p1, srcA);
                const float b0 = __shfl_sync(0xffffffffu, p0, srcB);
                const float b1 = __shfl_sync(0xffffffffu, p1, srcB);
                bp[nt][0] = part_bf16x2(a0, b0, lo_col);
                bp[nt][1] = part_bf16x2(a1, b1, lo_col);
            }
            // ---- O^T += V^T . P^T ----
            if (nv < SLAB) {
                const int ta = 2 * tig, tb = 8 + 2 * tig;
                const uint32_t ma = (ta >= nv ? 0u : 0xffffu) | (ta + 1 >= nv ? 0u : 0xffff0000u);
                const uint32_t mb = (tb >= nv ? 0u : 0xffffu) | (tb + 1 >= nv ? 0u : 0xffff0000u);
#pragma unroll
                for (int mt = 0; mt < KD; ++mt) {
                    apv[mt][0] &= ma; apv[mt][1] &= ma; apv[mt][2] &= mb; apv[mt][3] &= mb;
                }
            }
#pragma unroll
            for (int mt = 0; mt < KD; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma16816(oacc[mt][nt], apv[mt], bp[nt][0], bp[nt][1]);
        }
        // every warp gives every chunk back once: the products above consumed the
        // tile registers, so its shared-memory reads of the stage are complete
        __syncwarp();
        if (lane == 0) mbar_arrive_relaxed(bar_empty + 8 * ss);
    }
    if (w == 0 && lane == 0) GVA_KT(7);
    if (w == 0 && lane == 0) GVA_TRACE_AT(8);
    if (cur_p >= 0) finish_pair();
    if (w == 0 && lane == 0) GVA_CTA_T(2);
    if (w == 0 && lane == 0) {
        GVA_KT(9);
        GVA_TRACE_AT(9);
        GVA_TRACE_FLUSH(0, 16);
        GVA_TRACE_FLUSH(100, 166);
    }
}

// ---------------------------------------------------------------------------- //
// host side
// ---------------------------------------------------------------------------- //
inline bool fused_supported(const gva_dims *d, const gva_rows &rows) {
    if (d->cache_dtype != GVA_BF16) return false;
    if (d->d_h != 64 && d->d_h != 128) return false;
    if (d->H / d->G > 8) return false;
    if (d->d_r != 0 && d->d_r != 8 && d->d_r != 16 && d->d_r != 24 && d->d_r != 32) return false;
    if (rows.num_rows > 0x7fffffffLL) return false;   // TMA row coordinate is int32
    if (rows.layout == GVA_LAYOUT_PAGED && rows.page_size % SLAB != 0) return false;
    return true;
}

#ifdef GVA_TRACE
constexpr int FU_SMEM_LIMIT = 227 * 1024 - TRACE_SLOTS * 8;
#else
constexpr int FU_SMEM_LIMIT = 227 * 1024;
#endif

// Shared-memory plan; false when even one-slab chunks leave fewer than 2 stages.
inline bool plan_fused(FusedParams &p, int DH, int DR, int NT, const gva_rows &rows) {
    const int NH = 4 * NT;
    size_t o = 0;
    // fixed regions after the ring: barriers, lengths, staging, merge, flag
    const size_t bar = align_up(16 * FU_MAX_STAGES + 16 + 4 * FU_MAX_STAGES, 16);
    const size_t ls = align_up(sizeof(int) * (2 * (size_t)p.B + 1), 16);
    const size_t qt = align_up((size_t)FU_NQ * NH * DH * 4, 16);
    const size_t qh = align_up((size_t)FU_NQ * NH * (DR > 0 ? DR : 1) * 4, 16);
    const size_t mg = align_up((size_t)FU_NC * NH * (DH + 2) * 4, 16);
    const size_t fixed = 1024 /* alignment slack */ + bar + ls + qt + qh + mg + 16;
    if (fixed >= (size_t)FU_SMEM_LIMIT) return false;
    const size_t ring = (size_t)FU_SMEM_LIMIT - fixed;
    const int slab_bytes = SLAB * DH * 2 + SLAB * DR * 2;
    // chunk depth: the deepest power of two (<= 16, and dividing the slabs per page of a
    // paged cache) that still leaves at least 4 ring stages
    int kcap = FU_MAX_KC;
    if (rows.layout == GVA_LAYOUT_PAGED) {
        const int spp = rows.page_size / SLAB;
        while (kcap > 1 && spp % kcap != 0) kcap >>= 1;
    }
    int kc = kcap;
    while (kc > 1 && ring / ((size_t)kc * slab_bytes) < 4) kc >>= 1;
    int nss = (int)(ring / ((size_t)kc * slab_bytes));
    if (nss > FU_MAX_STAGES) nss = FU_MAX_STAGES;
    if (nss < 2) return false;
    p.kc = kc;
    p.nss = nss;
    o = (size_t)nss * kc * SLAB * DH * 2;                     // value ring (1024-multiple)
    p.off_kr = (int)o;
    o = align_up(o + (size_t)nss * kc * SLAB * DR * 2, 16);
    p.off_bar = (int)o;
    o += bar;
    p.off_ls = (int)o;
    o += ls;
    p.off_qt = (int)o;
    o += qt;
    p.off_qh = (int)o;
    o += qh;
    p.off_mg = (int)o;
    o += mg;
    p.off_flag = (int)o;
    o += 16;
    return o + 1024 <= (size_t)FU_SMEM_LIMIT;
}

inline size_t fused_smem_bytes(const FusedParams &p) { return 1024 + (size_t)p.off_flag + 16; }

// 4D bf16 view of the value cache for group tiles of `k` slabs: dims {64, rows,
// G*d_h/64, 16}, strides {row pitch, 128 B, 16 row pitches}; box {64, 16, d_h/64, k}.
// The fourth dimension overlaps the second: coordinate (0, y, z, 0) with box depth k
// reads rows y .. y + 16k - 1, of which only the first 16 are bounds-checked (callers
// keep the rest inside the storage).  The box lands slab-major, each slab
// [d_h/64][16 rows][128 B], 128-byte swizzled.
inline bool make_map4(CUtensorMap *m, const void *ptr, long long rows, int width, int dh, int k) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {64, (cuuint64_t)rows, (cuuint64_t)(width / 64), (cuuint64_t)FU_MAX_KC};
    cuuint64_t strides[3] = {(cuuint64_t)width * 2, 128, (cuuint64_t)width * 2 * SLAB};
    cuuint32_t box[4] = {64, (cuuint32_t)SLAB, (cuuint32_t)(dh / 64), (cuuint32_t)k};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DH, int DR, int NT>
inline int launch_fused_t(void *stream, const FusedParams &p, const FusedMaps &maps, int grid) {
    auto kern = decode_fused_kernel<DH, DR, NT>;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(FU_THREADS);
    cfg.dynamicSmemBytes = fused_smem_bytes(p);
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
    return cuda_status(cudaLaunchKernelEx(&cfg, kern, maps, p));
}

template <int DH, int NT>
inline cudaError_t fused_opt_in_dh() {
    const void *ks[] = {(const void *)decode_fused_kernel<DH, 0, NT>, (const void *)decode_fused_kernel<DH, 8, NT>,
                        (const void *)decode_fused_kernel<DH, 16, NT>, (const void *)decode_fused_kernel<DH, 24, NT>,
                        (const void *)decode_fused_kernel<DH, 32, NT>};
    for (const void *k : ks) {
        const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, FU_SMEM_LIMIT);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}
inline cudaError_t fused_opt_in_all() {
    cudaError_t e = fused_opt_in_dh<64, 1>();
    if (e == cudaSuccess) e = fused_opt_in_dh<64, 2>();
    if (e == cudaSuccess) e = fused_opt_in_dh<128, 1>();
    if (e == cudaSuccess) e = fused_opt_in_dh<128, 2>();
    return e;
}

template <int DH, int NT>
inline int launch_fused_dr(void *stream, const FusedParams &p, const FusedMaps &maps, int grid, int DR) {
    switch (DR) {
    case 0: return launch_fused_t<DH, 0, NT>(stream, p, maps, grid);
    case 8: return launch_fused_t<DH, 8, NT>(stream, p, maps, grid);
    case 16: return launch_fused_t<DH, 16, NT>(stream, p, maps, grid);
    case 24: return launch_fused_t<DH, 24, NT>(stream, p, maps, grid);
    case 32: return launch_fused_t<DH, 32, NT>(stream, p, maps, grid);
    default: return GVA_ERR_UNSUPPORTED;
    }
}

// Plans, encodes the maps and launches the fused decode (one CTA per SM by default).
inline int run_fused(void *stream, FusedParams &p, const void *V, const gva_rows &rows, int d_h,
                     int sms, int req_ctas) {
    const int DH = d_h, DR = p.d_r;
    const int NT = p.r <= 4 ? 1 : 2;
    if (!plan_fused(p, DH, DR, NT, rows)) return GVA_ERR_UNSUPPORTED;
    const long long nrows = rows.num_rows > 0 ? rows.num_rows : 1;
    FusedMaps maps;
    for (int k = 0; k < 5; ++k)
        if (!make_map4(&maps.m[k], V, nrows, p.G * DH, DH, 1 << k)) return GVA_ERR_CUDA;
    int grid = req_ctas > 0 ? req_ctas : sms;
    if (grid > sms * 8) grid = sms * 8;
    p.n_ctas = grid;
    if (DH == 64)
        return NT == 1 ? launch_fused_dr<64, 1>(stream, p, maps, grid, DR)
                       : launch_fused_dr<64, 2>(stream, p, maps, grid, DR);
    return NT == 1 ? launch_fused_dr<128, 1>(stream, p, maps, grid, DR)
                   : launch_fused_dr<128, 2>(stream, p, maps, grid, DR);
}

}  // namespace gva
