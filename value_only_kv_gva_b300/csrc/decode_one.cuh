// decode_one.cuh -- the whole GVA decode of one layer in a single tensor-core kernel:
// query absorption, split-K partial decode over the cache, and the log-sum-exp merge
// of the splits (GVA analysis page, 关键技巧一: absorb once per step; MQA/GQA page §1:
// the softmax over every cached position).
//
// Grid: at most one CTA per SM, all resident together.  Each CTA:
//   1. (consumer warps) absorbs a slice of the batch's (head, sequence) pairs,
//      q~[b,h,:] = scale log2(e) M_h q_nope[b,h,:], writes it to the workspace and
//      counts it in ready[b] (release);  meanwhile the producer warp reads the lengths,
//      builds the slab prefix and starts streaming its share of the cache through the
//      TMA ring exactly as the separate-kernel decode does;
//   2. (consumer warps) for each sequence of its share, waits until all H heads of
//      that sequence are absorbed (acquire on ready[b]), then scores two slabs per
//      iteration with bf16 mma.sync (the same products as the separate kernel) and
//      keeps an online softmax;
//   3. at the end of a sequence's segment: a sequence wholly inside the share is
//      finished in place; otherwise the partial (o, m, l) is written, the CTA takes a
//      ticket for the sequence, and the CTA that takes the last ticket merges every
//      partial of that sequence (one pass over the parts' (m, l, o)).
// The last reader of each counter clears it, so the workspace's counters are zero
// again after every completed call.  Every wait is bounded: on expiry the kernel
// raises GVA_DEV_TIMEOUT and stops issuing work.
#pragma once

#include "decode_mma.cuh"

namespace gva {

struct OneParams {
    MmaParams m;             // ring plan and decode arguments (m.d.qc: the absorbed queries
                             // for GVA, the query for the GQA comparator)
    const void *q_nope;      // GVA: content query [B][H][d_n] (fp32 or bf16)
    const float *M;          // GVA: [H][d_h][d_n]
    int d_n;
    int q_f32;               // q_nope is fp32 (else bf16)
    float prescale;          // scale * log2(e), applied to the absorbed query
    float *qt;               // GVA: absorbed queries [B][H][d_h] (workspace; = m.d.qc)
    int *ready;              // GVA: [B] absorbed heads per sequence, zero between calls
    int *ticket;             // [B] finished parts per split sequence, zero between calls
    int off_w;               // merge weights: ncons x ONE_MAX_PARTS floats, from the aligned base
    int qnorm;               // 1: RMSNorm of each head's content query before the absorption
    const float *qn_gain;    //    per-dimension gain [d_n] or null (ones)
    float qn_eps;
};

constexpr int ONE_MAX_CTAS = 160;          // grid cap: a sequence has at most this many parts
constexpr int ONE_MAX_PARTS = ONE_MAX_CTAS;
constexpr int ONE_BAR_ALL = 9;             // named barrier of the consumer warps
constexpr int ONE_BAR_PREFIX = 10;         // producer -> consumers: lengths and prefix ready
constexpr int ONE_BAR_ABSORBED = 11;       // consumers -> producer: absorption slice published
constexpr unsigned ONE_POLL_NS = 128;

// ld.acquire at GPU scope: later loads of this thread see what the releasing thread
// wrote before its release.
__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ void named_arrive(int id, int n) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Bounded wait (every lane of the warp) until *p >= target; false when another warp
// raised `abort` or after WAIT_LIMIT_NS (raising abort and GVA_DEV_TIMEOUT).
__device__ __forceinline__ bool wait_count(const int *p, int target, volatile int *abort) {
    const unsigned long long t0 = global_ns();
    bool ok = true;
    for (;;) {
        if (ld_acquire_gpu(p) >= target) break;
        if (*abort) { ok = false; break; }
        if (global_ns() - t0 > WAIT_LIMIT_NS) {
            *abort = 1;
            dev_report(GVA_DEV_TIMEOUT);
            ok = false;
            break;
        }
        __nanosleep(ONE_POLL_NS);
    }
    return __all_sync(0xffffffffu, ok);
}

// One warp: validated lengths into Ls[0..B), exclusive slab prefix into F[0..B] (the
// rule of build_prefix: an unusable length counts as 0 and, with `report`, sets
// GVA_DEV_BAD_LENGTH).
__device__ __forceinline__ void warp_prefix(const int *seq_len, const RowsDev &R, int B, int *Ls,
                                            int *F, bool report) {
    const int lane = threadIdx.x & 31;
    const int per = (B + 31) / 32;
    const int lo = lane * per, hi = min(lo + per, B);
    int sum = 0;
    for (int b = lo; b < hi; ++b) {
        int L = seq_len[b];
        if (!length_ok(R, b, L)) {
            if (report) dev_report(GVA_DEV_BAD_LENGTH);
            L = 0;
        }
        Ls[b] = L;
        sum += (L + SLAB - 1) / SLAB;
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int b = lo; b < hi; ++b) {
        F[b] = run;
        run += (Ls[b] + SLAB - 1) / SLAB;
    }
    if (lane == 31) F[B] = incl;
}

// The absorption slice of CTA c: pairs e in [e0, e1) of the h-major order (head e / B,
// sequence e % B), taken as runs of up to two sequences of one head.  Four threads share
// an output row i, each a quarter of the d_n products (summed by two shuffles); a thread
// loads its quarter of M_h row i once per run and the matching quarters of the run's
// queries, every load of a 16-element chunk issued before the first product, so a slice
// costs one memory round trip per chunk.  With the query RMSNorm (the scale-matched +
// query RMSNorm variant) the lanes also sum the squares of their query quarters:
// q~ = (1 / sqrt(mean q^2 + eps)) M_h (gain * q).
constexpr int ABS_RUN = 2;
template <int DH>
__device__ __forceinline__ void absorb_slice(const OneParams &op, int B, int H, long long e0,
                                             long long e1, int ct, int nthr) {
    const int dn = op.d_n, part = dn / 4;   // d_n is a multiple of 8: part is even
    for (long long e = e0; e < e1;) {
        const int h = (int)(e / B), b0 = (int)(e % B);
        long long left = e1 - e;
        if (left > B - b0) left = B - b0;
        const int nb = left < ABS_RUN ? (int)left : ABS_RUN;   // sequences b0 .. b0 + nb - 1
        const float *Mh = op.M + (long long)h * DH * dn;
        for (int idx = ct; idx < DH * 4; idx += nthr) {
            const int i = idx >> 2, k0 = (idx & 3) * part;
            const float *mrow = Mh + (long long)i * dn + k0;
            float acc[ABS_RUN], ss[ABS_RUN];
#pragma unroll
            for (int u = 0; u < ABS_RUN; ++u) acc[u] = ss[u] = 0.f;
            for (int kc = 0; kc < part; kc += 16) {
                float2 mv[8], qv[ABS_RUN][8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int k = kc + 2 * u;
                    mv[u] = k < part ? __ldg(reinterpret_cast<const float2 *>(mrow + k))
                                     : make_float2(0.f, 0.f);
                }
#pragma unroll
                for (int bi = 0; bi < ABS_RUN; ++bi) {
                    const long long qo = ((long long)(b0 + bi) * H + h) * dn + k0;
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int k = kc + 2 * u;
                        float2 x = make_float2(0.f, 0.f);
                        if (bi < nb && k < part) {
                            if (op.q_f32)
                                x = __ldg(reinterpret_cast<const float2 *>(
                                    reinterpret_cast<const float *>(op.q_nope) + qo + k));
                            else
                                x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(
                                    reinterpret_cast<const __nv_bfloat16 *>(op.q_nope) + qo + k));
                        }
                        qv[bi][u] = x;
                    }
                }
#pragma unroll
                for (int bi = 0; bi < ABS_RUN; ++bi)
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int k = kc + 2 * u;
                        float2 x = qv[bi][u];
                        if (op.qnorm) {
                            ss[bi] = fmaf(x.x, x.x, fmaf(x.y, x.y, ss[bi]));
                            if (op.qn_gain && k < part) {   // scalar loads: 4-byte alignment
                                x.x *= __ldg(op.qn_gain + k0 + k);
                                x.y *= __ldg(op.qn_gain + k0 + k + 1);
                            }
                        }
                        acc[bi] = fmaf(x.x, mv[u].x, fmaf(x.y, mv[u].y, acc[bi]));
                    }
            }
#pragma unroll
            for (int bi = 0; bi < ABS_RUN; ++bi) {
                float a = acc[bi];
                a += __shfl_xor_sync(0xffffffffu, a, 1);
                a += __shfl_xor_sync(0xffffffffu, a, 2);
                if (op.qnorm) {
                    float q2 = ss[bi];
                    q2 += __shfl_xor_sync(0xffffffffu, q2, 1);
                    q2 += __shfl_xor_sync(0xffffffffu, q2, 2);
                    a *= 1.f / sqrtf(q2 / (float)dn + op.qn_eps);
                }
                if ((idx & 3) == 0 && bi < nb)
                    op.qt[((long long)(b0 + bi) * H + h) * DH + i] = op.prescale * a;
            }
        }
        e += nb;
    }
}

// Merge of every part of sequence b by the CTA that finished it last.  The consumer
// threads take (head, 4-dimension chunk) pairs; each loads the (m, l, o) of all n parts
// in batches of ONE_MERGE_BATCH (all in flight together) and folds them with an online
// log-sum-exp, so the merge costs about ceil(n / batch) L2 round trips.
constexpr int ONE_MERGE_BATCH = 12;
template <int DH>
__device__ __forceinline__ void merge_seq(const DecodeParams &p, int b, int c_lo, int n, int ct,
                                          int nthr) {
    constexpr int DQ = DH / 4;
    const int H = p.H;
    const long long ostep = (long long)H * DH, mstep = (long long)H * 2;   // next slot
    for (int e = ct; e < H * DQ; e += nthr) {
        const int h = e / DQ, dq = e % DQ;
        const long long slot0 = (long long)c_lo + b;
        const float *po = p.part_o + (slot0 * H + h) * DH + 4 * dq;
        const float *pm = p.part_ml + (slot0 * H + h) * 2;
        float m = -INFINITY, l = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k0 = 0; k0 < n; k0 += ONE_MERGE_BATCH) {
            float2 ml[ONE_MERGE_BATCH];
            float4 o[ONE_MERGE_BATCH];
#pragma unroll
            for (int u = 0; u < ONE_MERGE_BATCH; ++u) {
                ml[u] = make_float2(-INFINITY, 0.f);
                if (k0 + u < n) {
                    ml[u] = __ldcg(reinterpret_cast<const float2 *>(pm + (k0 + u) * mstep));
                    o[u] = __ldcg(reinterpret_cast<const float4 *>(po + (k0 + u) * ostep));
                }
            }
#pragma unroll
            for (int u = 0; u < ONE_MERGE_BATCH; ++u) {
                if (ml[u].x == -INFINITY) continue;   // no part, or a part with no valid token
                const float mn = fmaxf(m, ml[u].x);
                const float a = exp2f(m - mn);        // 0 while m = -inf
                const float wgt = exp2f(ml[u].x - mn);
                acc.x = fmaf(acc.x, a, wgt * o[u].x);
                acc.y = fmaf(acc.y, a, wgt * o[u].y);
                acc.z = fmaf(acc.z, a, wgt * o[u].z);
                acc.w = fmaf(acc.w, a, wgt * o[u].w);
                l = fmaf(l, a, wgt * ml[u].y);
                m = mn;
            }
        }
        const float inv = l > 0.f ? 1.f / l : 0.f;
        *(reinterpret_cast<float4 *>(p.out + ((long long)b * H + h) * DH) + dq) =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        if (dq == 0 && p.lse)
            p.lse[(long long)b * H + h] = l > 0.f ? (m + log2f(l)) * LN2 : -INFINITY;
    }
}

template <int DH, int DR, bool GQA, int NT>
__global__ void __launch_bounds__(MMA_THREADS, 1)
    decode_one_kernel(const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_k, const OneParams op) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const MmaParams &mp = op.m;
    const DecodeParams &p = mp.d;
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
    unsigned char *base = smem_raw + (base_u32 - raw_u32);
    const int NS = mp.nstages;
    const uint32_t bar_full = base_u32 + mp.off_bar;          // NS x 8 bytes
    const uint32_t bar_empty = bar_full + 8 * NS;             // NS x 8 bytes
    volatile int *abort = reinterpret_cast<volatile int *>(base + mp.off_bar + 16 * NS);
    volatile int *last_flag = abort + 1;                      // [2]: first / last sequence
    int *stage_bad = reinterpret_cast<int *>(base + mp.off_bar + 16 * NS + 16);
    int *Ls = reinterpret_cast<int *>(base + mp.off_f);
    int *F = Ls + p.B;
    float *merge = reinterpret_cast<float *>(base + mp.off_merge);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.G, r = p.r, B = p.B, H = p.H;
    const int c = blockIdx.x, nct = p.n_ctas;
    const int nthr = mp.ncons * 32;                           // consumer threads

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, (uint32_t)G);
        }
        *abort = 0;
        last_flag[0] = last_flag[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_v);
        if (GQA) prefetch_tmap(&tm_k);
    }
    __syncthreads();
    if (threadIdx.x == 0) GVA_ONE_T(0);
    if (threadIdx.x == 0) GVA_REC(5, 0);
    if (threadIdx.x == 0) GVA_TRACE_AT(0);
    // everything read below (lengths, queries, maps, cache) may come from the preceding grid
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x == 0) GVA_ONE_T(1);
    if (threadIdx.x == 0) GVA_REC(5, 1);

    // ============================= producer warp ============================= //
    if (warp == 0) {
        const uint64_t pol = l2_evict_first_policy();   // made while the lengths load
        warp_prefix(p.seq_len, p.R, B, Ls, F, c == 0);
        __syncwarp();
        if (lane == 0) GVA_ONE_T(2);
        if (lane == 0) GVA_TRACE_AT(1);
        named_arrive(ONE_BAR_PREFIX, 32 + nthr);
        // the stream starts once this CTA's absorption slice is published: its stores and
        // fence do not queue behind the CTA's own cache copies
        if (!GQA) named_bar(ONE_BAR_ABSORBED, 32 + nthr);
        const Part P{F[B], nct};
        const long long s0 = P.start(c), s1 = P.start(c + 1);
        if (s0 < s1)
            mma_producer<DH, DR, GQA>(&tm_v, &tm_k, mp, F, s0, s1, base_u32, bar_full, bar_empty,
                                      abort, stage_bad, pol);
        return;
    }
    const int ci = warp - 1;          // consumer index
    if (ci >= mp.ncons) return;       // spare warps
    const int ct = ci * 32 + lane;

    // ---- absorption slice (GVA): independent of the lengths, overlaps the prefix ----
    if (!GQA) {
        const long long items = (long long)B * H;
        const long long e0 = items * c / nct, e1 = items * (c + 1) / nct;
        absorb_slice<DH>(op, B, H, e0, e1, ct, nthr);
        // every thread's rows are stored and ordered before the counts are raised
        fence_acq_rel_gpu();
        named_bar(ONE_BAR_ALL, nthr);
        if (ci == 0)
            for (long long e = e0 + lane; e < e1; e += 32) atomicAdd(op.ready + (int)(e % B), 1);
        if (ct == 0) GVA_ONE_T(3);
        named_arrive(ONE_BAR_ABSORBED, 32 + nthr);
    }
    named_bar(ONE_BAR_PREFIX, 32 + nthr);   // lengths and prefix from the producer
    const Part P{F[B], nct};
    const long long s0 = P.start(c), s1 = P.start(c + 1);

    {
        const int g = ci % G;             // value group of this warp
        const int w = ci / G;             // rank among the group's warps
        const int wpg = mp.wpg;
        const int gid = lane >> 2, tig = lane & 3;
        constexpr int KD = DH / 16;
        const int srcA = (2 * tig) * 4 + (gid >> 1), srcB = (2 * tig + 1) * 4 + (gid >> 1);
        const bool lo_col = (gid & 1) != 0;
        // two slabs per iteration where the ring has room for them (no deadlock needs NS > wpg)
        const bool pairs = NT == 1 && NS > wpg;

        long long my_s = s0 + w;
        int my_stage = w % NS;
        uint32_t my_phase = (uint32_t)(w / NS) & 1u;
        int b = s0 < s1 ? seq_of_slab(F, B, s0) : 0;
        long long s = s0;
        bool alive = true;
        int tslab = 0;                    // trace index (debug builds)
        (void)tslab;
        while (s < s1) {
            while (F[b + 1] <= s) ++b;
            const long long seg_end = min(s1, (long long)F[b + 1]);
            const int Lb = Ls[b];
            const int Fb = F[b];

            // the sequence's absorbed queries: written by CTAs of this grid
            if (!GQA && alive && !wait_count(op.ready + b, H, abort)) alive = false;
            if (ct == 0 && s == s0) GVA_ONE_T(4);
            if (ct == 0 && s == s0) GVA_TRACE_AT(4);
            QFrags<DH, DR, NT> qf;
            load_q_frags<DH, DR, NT, !GQA>(p, b, g, Lb, lane, qf);

            float oacc[KD][NT][4];
    #pragma unroll
            for (int mt = 0; mt < KD; ++mt)
    #pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    oacc[mt][nt][0] = oacc[mt][nt][1] = oacc[mt][nt][2] = oacc[mt][nt][3] = 0.f;
            float m_run[NT], l_run[NT];
    #pragma unroll
            for (int nt = 0; nt < NT; ++nt) { m_run[nt] = -INFINITY; l_run[nt] = 0.f; }

            while (my_s < seg_end && alive) {
                const bool two = pairs && my_s + wpg < seg_end;
                int stg1 = my_stage + wpg;
                uint32_t ph1 = my_phase;
                while (stg1 >= NS) { stg1 -= NS; ph1 ^= 1u; }
                bool okw = mbar_wait(bar_full + 8 * my_stage, my_phase, abort);
                if (two && okw) okw = mbar_wait(bar_full + 8 * stg1, ph1, abort);
                if (!__all_sync(0xffffffffu, okw)) {
                    alive = false;
                    break;
                }
                if (ct == 0) GVA_TRACE_AT(8 + 2 * tslab);
                int nv0 = min(SLAB, Lb - (int)(my_s - Fb) * SLAB);
                int nv1 = two ? min(SLAB, Lb - (int)(my_s + wpg - Fb) * SLAB) : 0;
                if (stage_bad[my_stage]) {
                    if (lane == 0 && g == 0) dev_report(GVA_DEV_BAD_PAGE);
                    nv0 = 0;
                }
                if (two && stage_bad[stg1]) {
                    if (lane == 0 && g == 0) dev_report(GVA_DEV_BAD_PAGE);
                    nv1 = 0;
                }
                const uint32_t st0 = base_u32 + my_stage * mp.stage_bytes;
                const uint32_t st1 = base_u32 + stg1 * mp.stage_bytes;

                // ---- scores of both slabs (independent product chains) ----
                float sc0[NT][2][4], sc1[NT][2][4];
                slab_scores<DH, DR, NT>(GQA ? st0 + mp.off_k : st0, st0 + mp.off_r, g, lane, qf, sc0);
                if (two) slab_scores<DH, DR, NT>(GQA ? st1 + mp.off_k : st1, st1 + mp.off_r, g, lane, qf, sc1);
                uint32_t apv[KD][4];
                slab_value_tiles<DH>(st0, g, lane, apv);

                // ---- hi + lo columns -> scores of tokens gid, gid + 8 of each slab ----
                float z0[NT][2], z1[NT][2];
                bool over = false;
    #pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    z0[nt][0] = (sc0[nt][0][0] + sc0[nt][0][1]) + (sc0[nt][1][0] + sc0[nt][1][1]);
                    z0[nt][1] = (sc0[nt][0][2] + sc0[nt][0][3]) + (sc0[nt][1][2] + sc0[nt][1][3]);
                    if (gid >= nv0) z0[nt][0] = -INFINITY;
                    if (gid + 8 >= nv0) z0[nt][1] = -INFINITY;
                    z1[nt][0] = z1[nt][1] = -INFINITY;
                    if (two) {
                        z1[nt][0] = (sc1[nt][0][0] + sc1[nt][0][1]) + (sc1[nt][1][0] + sc1[nt][1][1]);
                        z1[nt][1] = (sc1[nt][0][2] + sc1[nt][0][3]) + (sc1[nt][1][2] + sc1[nt][1][3]);
                        if (gid >= nv1) z1[nt][0] = -INFINITY;
                        if (gid + 8 >= nv1) z1[nt][1] = -INFINITY;
                    }
                    const float zm = fmaxf(fmaxf(z0[nt][0], z0[nt][1]), fmaxf(z1[nt][0], z1[nt][1]));
                    over |= zm > m_run[nt] + MMA_RESCALE_TH;
                }
                // lazy rescale, as in the separate-kernel decode, over both slabs at once
                if (__any_sync(0xffffffffu, over)) {
    #pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        float m = fmaxf(fmaxf(z0[nt][0], z0[nt][1]), fmaxf(z1[nt][0], z1[nt][1]));
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
                // ---- probabilities -> P^T fragments (column gid: head 4nt + gid/2) ----
                uint32_t bp0[NT][2], bp1[NT][2];
    #pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    {
                        const float p0 = z0[nt][0] == -INFINITY ? 0.f : exp2f(z0[nt][0] - m_run[nt]);
                        const float p1 = z0[nt][1] == -INFINITY ? 0.f : exp2f(z0[nt][1] - m_run[nt]);
                        l_run[nt] += p0 + p1;
                        const float a0 = __shfl_sync(0xffffffffu, p0, srcA);
                        const float a1 = __shfl_sync(0xffffffffu, p1, srcA);
                        const float b0 = __shfl_sync(0xffffffffu, p0, srcB);
                        const float b1 = __shfl_sync(0xffffffffu, p1, srcB);
                        bp0[nt][0] = part_bf16x2(a0, b0, lo_col);
                        bp0[nt][1] = part_bf16x2(a1, b1, lo_col);
                    }
                    if (two) {
                        const float p0 = z1[nt][0] == -INFINITY ? 0.f : exp2f(z1[nt][0] - m_run[nt]);
                        const float p1 = z1[nt][1] == -INFINITY ? 0.f : exp2f(z1[nt][1] - m_run[nt]);
                        l_run[nt] += p0 + p1;
                        const float a0 = __shfl_sync(0xffffffffu, p0, srcA);
                        const float a1 = __shfl_sync(0xffffffffu, p1, srcA);
                        const float b0 = __shfl_sync(0xffffffffu, p0, srcB);
                        const float b1 = __shfl_sync(0xffffffffu, p1, srcB);
                        bp1[nt][0] = part_bf16x2(a0, b0, lo_col);
                        bp1[nt][1] = part_bf16x2(a1, b1, lo_col);
                    }
                }
                // ---- O^T += V^T . P^T, slab by slab ----
                if (nv0 < SLAB) mask_value_tiles<DH>(apv, nv0, lane);
    #pragma unroll
                for (int mt = 0; mt < KD; ++mt)
    #pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma16816(oacc[mt][nt], apv[mt], bp0[nt][0], bp0[nt][1]);
                if (two) {
                    slab_value_tiles<DH>(st1, g, lane, apv);
                    if (nv1 < SLAB) mask_value_tiles<DH>(apv, nv1, lane);
    #pragma unroll
                    for (int mt = 0; mt < KD; ++mt)
    #pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma16816(oacc[mt][nt], apv[mt], bp1[nt][0], bp1[nt][1]);
                }
                // every tile register was consumed by the products: release the stages
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_relaxed(bar_empty + 8 * my_stage);
                    if (two) mbar_arrive_relaxed(bar_empty + 8 * stg1);
                }
                if (ct == 0) GVA_TRACE_AT(9 + 2 * tslab);
                ++tslab;
                const int adv = two ? 2 * wpg : wpg;
                my_s += adv;
                my_stage += adv;
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
            const bool whole = Fb >= s0 && F[b + 1] <= s1;
            if (w == 0) {
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

        // ---- the sequences this CTA shares with others (at most the share's first and last):
        //      one ticket each, all taken together after the last slab; the CTA that takes a
        //      sequence's last ticket merges its parts ----
        if (ct == 0) {
            GVA_TRACE_AT(5);
            GVA_TRACE_FLUSH(4, 6);
            GVA_TRACE_FLUSH(8, 8 + 2 * tslab);
        }
    }
    if (ct == 0) GVA_ONE_T(5);
    if (ct == 0) GVA_TRACE_FLUSH(0, 2);
    if (s0 < s1) {
        if (ci < G) fence_acq_rel_gpu();   // this CTA's partials are stored before its tickets
        named_bar(ONE_BAR_ALL, nthr);
        const int bf = seq_of_slab(F, B, s0), bl = seq_of_slab(F, B, s1 - 1);
        if (ci == 0 && lane < 2) {
            const int bb = lane == 0 ? bf : bl;
            const bool split = !(F[bb] >= s0 && F[bb + 1] <= s1);
            int last = 0;
            if (split && (lane == 0 || bl != bf) && !*abort) {
                const int c_lo = P.cta_of(F[bb]), c_hi = P.cta_of((long long)F[bb + 1] - 1);
                last = atomicAdd(op.ticket + bb, 1) == c_hi - c_lo;
                if (last) fence_acq_rel_gpu();   // the other parts' stores are visible
            }
            last_flag[lane] = last;
        }
        named_bar(ONE_BAR_ALL, nthr);
        if (ct == 0) GVA_ONE_T(6);
        // the non-empty sequences wholly inside the share had this CTA as their only
        // reader of the absorbed-head count (every consumer warp is past its wait): clear
        // them (empty ones are cleared by CTA 0 below)
        if (!GQA && !*abort)
            for (int bb = bf + ct; bb <= bl; bb += nthr)
                if (Ls[bb] > 0 && F[bb] >= s0 && F[bb + 1] <= s1) op.ready[bb] = 0;
        for (int i = 0; i < 2; ++i) {
            if (!last_flag[i]) continue;
            const int bb = i == 0 ? bf : bl;
            const int c_lo = P.cta_of(F[bb]), c_hi = P.cta_of((long long)F[bb + 1] - 1);
            merge_seq<DH>(p, bb, c_lo, c_hi - c_lo + 1, ct, nthr);
            // every reader of this sequence's counters has passed them: clear them
            if (ct == 0) {
                op.ticket[bb] = 0;
                if (!GQA) op.ready[bb] = 0;
            }
        }
    }

    if (ct == 0) GVA_ONE_T(7);
    if (ct == 0) GVA_REC(5, 2);
    // ---- empty sequences (CTA 0): out = 0, lse = -inf; their counts are cleared once
    //      their absorption (which does not look at the lengths) has been counted ----
    if (c == 0) {
        for (int bb = ci; bb < B; bb += mp.ncons) {
            if (Ls[bb] != 0) continue;
            if (!GQA && !wait_count(op.ready + bb, H, abort)) break;
            for (int e = lane; e < H * DH; e += 32) p.out[(long long)bb * H * DH + e] = 0.f;
            if (p.lse)
                for (int h = lane; h < H; h += 32) p.lse[(long long)bb * H + h] = -INFINITY;
            __syncwarp();
            if (!GQA && lane == 0) op.ready[bb] = 0;
        }
    }
}

// ---------------------------------------------------------------------------- //
// host side
// ---------------------------------------------------------------------------- //
inline bool one_supported(const gva_dims *d) { return mma_supported(d); }

// The ring plan of the separate-kernel decode, with the whole shared memory of the SM
// (nothing else has to be resident beside this grid) and the merge weights added.
inline bool plan_one(OneParams &op, int DH, int DR, bool gqa, int NT) {
    MmaParams &mp = op.m;
    const DecodeParams &d = mp.d;
    mp.vg = d.G;
    const int vbytes = d.G * DH * SLAB * 2;
    mp.off_k = vbytes;
    mp.off_r = vbytes * (gqa ? 2 : 1);
    const int rbytes = DR * SLAB * 2;
    mp.tx_bytes = mp.off_r + rbytes;
    mp.stage_bytes = (int)align_up((size_t)mp.tx_bytes, 1024);
    mp.wpg = MMA_CONSUMERS / d.G;
    if (mp.wpg < 1) mp.wpg = 1;
    mp.ncons = d.G * mp.wpg;
    const int merge_bytes = merge_bytes_of(mp.wpg, d.G, DH, NT);
    const int wbytes = mp.ncons * ONE_MAX_PARTS * 4;
    const int fbytes = (int)align_up(sizeof(int) * (2 * d.B + 1), 16);
    const int fixed = 1024 + fbytes + merge_bytes + wbytes + bar_region_bytes(MMA_MAX_STAGES);
    int ns = (MMA_SMEM_LIMIT - fixed) / mp.stage_bytes;
    if (ns > MMA_MAX_STAGES) ns = MMA_MAX_STAGES;
    if (ns < 2) return false;
    mp.nstages = ns;
    mp.off_bar = ns * mp.stage_bytes;
    mp.off_f = mp.off_bar + bar_region_bytes(ns);
    mp.off_merge = mp.off_f + fbytes;
    op.off_w = mp.off_merge + merge_bytes;
    return true;
}

inline size_t one_smem_bytes(const OneParams &op) {
    return 1024 + (size_t)op.off_w + (size_t)op.m.ncons * ONE_MAX_PARTS * 4;
}

template <int DH, int DR, bool GQA, int NT>
inline int launch_one_t(void *stream, const OneParams &op, const CUtensorMap &tv,
                        const CUtensorMap &tk, int grid) {
    auto kern = decode_one_kernel<DH, DR, GQA, NT>;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3((op.m.ncons + 1) * 32);
    cfg.dynamicSmemBytes = one_smem_bytes(op);
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
    return cuda_status(cudaLaunchKernelEx(&cfg, kern, tv, tk, op));
}

template <int DH, int NT>
inline cudaError_t one_opt_in_dh() {
    const void *ks[] = {
        (const void *)decode_one_kernel<DH, 0, false, NT>, (const void *)decode_one_kernel<DH, 8, false, NT>,
        (const void *)decode_one_kernel<DH, 16, false, NT>, (const void *)decode_one_kernel<DH, 24, false, NT>,
        (const void *)decode_one_kernel<DH, 32, false, NT>, (const void *)decode_one_kernel<DH, 0, true, NT>};
    for (const void *k : ks) {
        const cudaError_t e =
            cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, MMA_SMEM_LIMIT);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}
inline cudaError_t one_opt_in_all() {
    cudaError_t e = one_opt_in_dh<64, 1>();
    if (e == cudaSuccess) e = one_opt_in_dh<64, 2>();
    if (e == cudaSuccess) e = one_opt_in_dh<128, 1>();
    if (e == cudaSuccess) e = one_opt_in_dh<128, 2>();
    return e;
}

template <int DH, int NT>
inline int launch_one_dr(void *stream, const OneParams &op, const CUtensorMap &tv,
                         const CUtensorMap &tk, int grid, int DR, bool gqa) {
    if (gqa) return launch_one_t<DH, 0, true, NT>(stream, op, tv, tk, grid);
    switch (DR) {
    case 0: return launch_one_t<DH, 0, false, NT>(stream, op, tv, tk, grid);
    case 8: return launch_one_t<DH, 8, false, NT>(stream, op, tv, tk, grid);
    case 16: return launch_one_t<DH, 16, false, NT>(stream, op, tv, tk, grid);
    case 24: return launch_one_t<DH, 24, false, NT>(stream, op, tv, tk, grid);
    case 32: return launch_one_t<DH, 32, false, NT>(stream, op, tv, tk, grid);
    default: return GVA_ERR_UNSUPPORTED;
    }
}

// Grid: one CTA per SM at most (every CTA must be resident for the absorbed queries and
// the tickets), at most ONE_MAX_CTAS; sets op.m.d.n_ctas.
inline int run_one(void *stream, OneParams &op, const gva_rows &rows, int sms, int req_ctas,
                   bool gqa) {
    if (rows.num_rows > 0x7fffffffLL) return GVA_ERR_UNSUPPORTED;   // TMA row coordinate is int32
    DecodeParams &dp = op.m.d;
    const int DH = dp.d_h, DR = gqa ? 0 : dp.d_r;
    const int NT = dp.r <= 4 ? 1 : 2;
    if (!plan_one(op, DH, DR, gqa, NT)) return GVA_ERR_UNSUPPORTED;
    const long long nrows = rows.num_rows > 0 ? rows.num_rows : 1;
    CUtensorMap tv, tk;
    op.m.early = 0;
    op.m.v3d = make_map3(&tv, dp.Vc, nrows, dp.G * DH) &&
               (!gqa || make_map3(&tk, dp.Kc, nrows, dp.G * DH));
    if (!op.m.v3d) {
        if (!make_map(&tv, dp.Vc, nrows, dp.G * DH, 64, true)) return GVA_ERR_CUDA;
        if (gqa && !make_map(&tk, dp.Kc, nrows, dp.G * DH, 64, true)) return GVA_ERR_CUDA;
    }
    if (!gqa) tk = tv;
    int grid = req_ctas > 0 ? req_ctas : sms;
    if (grid > sms) grid = sms;
    if (grid > ONE_MAX_CTAS) grid = ONE_MAX_CTAS;
    dp.n_ctas = grid;
    if (DH == 64)
        return NT == 1 ? launch_one_dr<64, 1>(stream, op, tv, tk, grid, DR, gqa)
                       : launch_one_dr<64, 2>(stream, op, tv, tk, grid, DR, gqa);
    return NT == 1 ? launch_one_dr<128, 1>(stream, op, tv, tk, grid, DR, gqa)
                   : launch_one_dr<128, 2>(stream, op, tv, tk, grid, DR, gqa);
}

}  // namespace gva
