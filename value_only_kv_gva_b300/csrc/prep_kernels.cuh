// prep_kernels.cuh -- the per-step small kernels: cache append and query absorption.
#pragma once

#include "common.cuh"

namespace gva {

// --------------------------------------------------------------------------- //
// Append  (Grouped Value Attention summary page: the positional key is cached
// already rotated; MQA/GQA page §1: the current token is appended before attending)
// --------------------------------------------------------------------------- //
struct AppendParams {
    int B, G, d_h, d_r;
    const float *v_new;     // [B][G][d_h]
    const float *k_new;     // [B][d_r], unrotated
    const int *pos;         // [B]
    int *seq_len_out;       // [B] or null; may alias pos
    const int *L0;          // chunk mode (chunk_n > 0): entry v is token v % chunk_n of a
    int chunk_n;            //   chunk appended to sequence v / chunk_n after its L0 tokens
    int *zero;              // nzero words set to 0 (the counters of the kernel that follows
    int nzero;              //   in the same call), or null
    RowsDev R;
    void *V;                // rows [G][d_h]
    void *Kr;               // rows [d_r]
    const float *rope_tab;  // [rope_max_pos][d_r/2][2]
    int rope_max_pos;
};

// Position of chunk entry v (token v % n of sequence v / n): L0[b] + v % n, or -1 when the
// history is negative or the position leaves the int range (reported as a bad position).
__device__ __forceinline__ int chunk_pos(const int *L0, int n, int v) {
    const long long l0 = L0[v / n];
    const long long e = l0 + v % n;
    return (l0 >= 0 && e < 0x7fffffffLL) ? (int)e : -1;
}

// One CTA per sequence (per chunk entry in chunk mode).  V gets the new value rounded once; K_rope gets
// Rot(pos) k_new computed in fp32 in the fixed order y0 = (x0*c) - (x1*s),
// y1 = (x0*s) + (x1*c) with every product and sum rounded separately (no FMA), then
// rounded once to the cache dtype, so the stored bytes are reproducible.
// The work of entry b, for a CTA of NTHR threads (the block's first NTHR threads; nblk
// CTAs share the zeroing).
template <typename CT, int NTHR>
__device__ __forceinline__ void append_body(const AppendParams &p, int b, int nblk) {
    const int sb = p.chunk_n > 0 ? b / p.chunk_n : b;        // sequence of its rows
    for (int e = b * NTHR + (int)threadIdx.x; e < p.nzero; e += nblk * NTHR) p.zero[e] = 0;
    const int W = p.G * p.d_h;
    // Loads that do not depend on the position are issued with it: the new value (up
    // to VPT elements per thread), the unrotated key pair, the position.  The table entry
    // and, for a paged cache, the block-table entry follow: two memory round trips.
    constexpr int VPT = 1024 / NTHR;
    const float *vn = p.v_new + (long long)b * W;
    float vv[VPT];
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
        const int e = threadIdx.x + u * NTHR;
        vv[u] = e < W ? vn[e] : 0.f;
    }
    const int half = p.d_r / 2;
    const bool kthr = (int)threadIdx.x < half;
    float x0 = 0.f, x1 = 0.f;
    if (kthr) {
        const float *kn = p.k_new + (long long)b * p.d_r;
        x0 = kn[2 * threadIdx.x];
        x1 = kn[2 * threadIdx.x + 1];
    }
    const int pos = p.chunk_n > 0 ? chunk_pos(p.L0, p.chunk_n, b) : p.pos[b];
    __syncthreads();  // every thread has read pos[b] before seq_len_out (may alias) is written
    bool ok = pos >= 0 && (long long)pos < seq_capacity(p.R, sb) && (p.d_r == 0 || pos < p.rope_max_pos);
    float c = 0.f, sn = 0.f;
    if (ok && kthr) {
        const float *cs = p.rope_tab + (long long)pos * p.d_r;  // (d_r/2) (cos, sin) pairs
        c = cs[2 * threadIdx.x];
        sn = cs[2 * threadIdx.x + 1];
    }
    long long row = ok ? row_of(p.R, sb, pos) : -1;
    if (p.R.layout == GVA_LAYOUT_RAGGED && row >= p.R.num_rows) row = -1;
    if (row < 0) {
        if (threadIdx.x == 0) dev_report(ok ? GVA_DEV_BAD_PAGE : GVA_DEV_BAD_POSITION);
        return;
    }
    CT *V = reinterpret_cast<CT *>(p.V) + row * W;
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
        const int e = threadIdx.x + u * NTHR;
        if (e < W) V[e] = from_f<CT>(vv[u]);
    }
    for (int e = threadIdx.x + VPT * NTHR; e < W; e += NTHR) V[e] = from_f<CT>(vn[e]);
    if (kthr) {
        CT *K = reinterpret_cast<CT *>(p.Kr) + row * p.d_r;
        const float y0 = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, sn));
        const float y1 = __fadd_rn(__fmul_rn(x0, sn), __fmul_rn(x1, c));
        K[2 * threadIdx.x] = from_f<CT>(y0);
        K[2 * threadIdx.x + 1] = from_f<CT>(y1);
    }
    __syncthreads();
    if (threadIdx.x == 0 && p.seq_len_out) p.seq_len_out[b] = pos + 1;
}

template <typename CT>
__global__ void __launch_bounds__(128) append_kernel(const AppendParams p) {
    if (threadIdx.x == 0) GVA_KT(0);
    if (threadIdx.x == 0) GVA_REC(1, 0);
    pdl_wait();
    if (threadIdx.x == 0) GVA_REC(1, 1);
    pdl_launch_dependents();
    append_body<CT, 128>(p, blockIdx.x, gridDim.x);
    if (threadIdx.x == 0) GVA_KT(1);
    if (threadIdx.x == 0) GVA_REC(1, 2);
}

// --------------------------------------------------------------------------- //
// Chunked-prefill view  (MQA/GQA page §1: each new token attends to the cached history
// and to the chunk up to and including itself)
// --------------------------------------------------------------------------- //
// Query i of sequence b becomes entry v = b*n + i of a decode batch: a sequence of
// length L0[b] + i + 1 stored in sequence b's rows.  The append then writes the token
// at position L0[b] + i and the decode of entry v attends over positions 0..L0[b]+i,
// which is the causal mask.  Every entry reads b's rows through its own copy of b's
// block-table row; a contiguous cache is read as pages of T_cap rows (page b holds
// sequence b), so the view is a paged one for both layouts.
struct PrefillViewParams {
    int B, n;
    const int *L0;            // [B] tokens cached before the chunk
    const int *block_table;   // paged: the caller's [B][max_pages]; contiguous: null
    int max_pages;            // columns of both tables (1 for a contiguous cache)
    int *bt;                  // [B*n][max_pages] block table of the view
    int *pos;                 // [B*n] append position of entry v: L0[b] + i, or -1
    int *len;                 // [B*n] decode length of entry v: L0[b] + i + 1, or -1
};
constexpr int PV_ROWS = 32;   // chunk queries per CTA (grid: B x ceil(n / PV_ROWS))

__global__ void __launch_bounds__(128) prefill_view_kernel(const PrefillViewParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int b = blockIdx.x;
    const int i0 = blockIdx.y * PV_ROWS;
    const int i1 = min(p.n, i0 + PV_ROWS);
    const long long l0 = p.L0[b];
    // a negative history or a position past the int range is marked -1: the append
    // reports a bad position and the decode a bad length for that entry
    for (int i = i0 + (int)threadIdx.x; i < i1; i += blockDim.x) {
        const long long v = (long long)b * p.n + i;
        const long long end = l0 + i + 1;
        const bool ok = l0 >= 0 && end <= 0x7fffffffLL;
        p.pos[v] = ok ? (int)(end - 1) : -1;
        p.len[v] = ok ? (int)end : -1;
    }
    const long long W = (long long)(i1 - i0) * p.max_pages;
    for (long long e = threadIdx.x; e < W; e += blockDim.x) {
        const long long v = (long long)b * p.n + i0 + e / p.max_pages;
        const long long col = e % p.max_pages;
        p.bt[v * p.max_pages + col] =
            p.block_table ? p.block_table[(long long)b * p.max_pages + col] : b;
    }
}

// --------------------------------------------------------------------------- //
// Absorb  (GVA analysis page, 关键技巧一: q_h k_{j,h}^T = (q_h M_h^T) v_{j,g(h)}^T)
// --------------------------------------------------------------------------- //
struct AbsorbParams {
    int B, H, d_h, d_n, d_r, bpb;  // bpb: sequences per CTA
    const void *q_nope;            // [B][H][d_n]
    const void *q_rope;            // [B][H][d_r]
    const float *M;                // [H][d_h][d_n]
    const int *seq_len;            // [B]; in chunk mode null, and the length of entry v
    const int *L0;                 //   is L0[v / chunk_n] + v % chunk_n + 1 (-1 when out of
    int chunk_n;                   //   range), its rows those of sequence v / chunk_n
    const float *rope_tab;
    int rope_max_pos;
    float prescale;                // multiplies both outputs
    float *q_tilde;                // [B][H][d_h]
    float *q_hat;                  // [B][H][d_r]
    int check_rows;                // 1: a length the cache cannot hold is skipped silently
    RowsDev R;                     //    (the decode kernel reports it); used when check_rows
    int skip_rope;                 // 1: q_hat is not computed (the decode rotates q_rope)
    int qnorm;                     // 1: RMSNorm of each head's content query first
    const float *qn_gain;          //    per-dimension gain [d_n] or null (ones)
    float qn_eps;
};

// Grid (H, ceil(B / bpb), d_h / 32), 256 threads, bpb <= 32 sequences per CTA.
//
// Warp w owns rows i0 + 4w .. i0 + 4w + 3 of M_h; lane (o = lane / 8, kl = lane % 8)
// holds the kl-th contiguous chunk of cs = d_n / 8 entries of its row in registers for
// the whole CTA.  The CTA's query rows are staged in shared memory as fp32 in the same
// chunking, each chunk padded to cst floats (a multiple of 4 with cst / 4 odd), so that
// the 8 lanes of a row read their chunks with conflict-free 16-byte loads, each one
// broadcast to the 4 rows of the warp: one shared-memory wavefront feeds 128 FMAs.
// The 8 chunk partials of a row are combined for 8 sequences at a time by a
// reduce-scatter over the 8 lanes (7 shuffles), after which lane kl holds sequence kl.
// Every global load of the CTA (its M rows, its query rows, the positional inputs) is
// issued in one unrolled batch before the first use: one memory round trip.
constexpr int ABSORB_THREADS = 256;
constexpr int ABSORB_CSMAX = 32;   // d_n <= 256
constexpr int ABSORB_QVEC = 4;     // 16-byte query vectors per thread (bpb is sized to fit)
constexpr int ABSORB_BPB_MAX = 32;

__host__ __device__ constexpr int absorb_cst(int d_n) {
    // chunk stride: cs rounded up to 4, plus 4 when that leaves an even number of float4
    return (((d_n / 8 + 3) / 4) & 1) ? ((d_n / 8 + 3) / 4) * 4 : ((d_n / 8 + 3) / 4) * 4 + 4;
}
// sequences per CTA the query staging allows for one query row of d_n elements of qsize bytes
__host__ __device__ constexpr int absorb_bpb_limit(int d_n, int qsize) {
    return (ABSORB_QVEC * ABSORB_THREADS) / (d_n * qsize / 16) < ABSORB_BPB_MAX
               ? (ABSORB_QVEC * ABSORB_THREADS) / (d_n * qsize / 16) : ABSORB_BPB_MAX;
}
__host__ __device__ constexpr int absorb_smem_bytes(int d_n, int bpb) {
    return ((bpb + 7) / 8) * 8 * 8 * absorb_cst(d_n) * 4;
}

// Element t of a 16-byte vector of query values, widened exactly to fp32.
template <typename QT> __device__ __forceinline__ float vec_elem(const uint4 &v, int t);
template <> __device__ __forceinline__ float vec_elem<float>(const uint4 &v, int t) {
    const unsigned w = t == 0 ? v.x : t == 1 ? v.y : t == 2 ? v.z : v.w;
    return __uint_as_float(w);
}
template <> __device__ __forceinline__ float vec_elem<__nv_bfloat16>(const uint4 &v, int t) {
    const unsigned w = (t >> 1) == 0 ? v.x : (t >> 1) == 1 ? v.y : (t >> 1) == 2 ? v.z : v.w;
    return __uint_as_float((t & 1) ? (w & 0xffff0000u) : (w << 16));   // bf16 = high half of fp32
}

// CSF: the chunk size d_n / 8 when it is fixed at compile time (8, 16, 32), 0 otherwise.
// The work of CTA (h, by, bz) of the grid above, staging in sm_abs.
template <typename QT, int CSF>
__device__ __forceinline__ void absorb_body(const AbsorbParams &p, int h, int by, int bz,
                                            float *sm_abs) {
    const int b0 = by * p.bpb;
    const int nb = min(p.bpb, p.B - b0);
    const int i0 = bz * 32;
    const int d_n = p.d_n, d_h = p.d_h;
    const int cs = CSF > 0 ? CSF : d_n / 8, cst = absorb_cst(8 * cs);
    constexpr int CSMAX = CSF > 0 ? CSF : ABSORB_CSMAX;
    const int lane = threadIdx.x & 31, kl = lane & 7;
    const int o = (threadIdx.x >> 5) * 4 + (lane >> 3);   // row within the CTA's 32
    const int rows = min(32, d_h - i0);
    const int nbr = (nb + 7) & ~7;                        // staged rows (zero past nb)

    // Positional slice: one (sequence, pair) per thread and pass, two passes at most
    // (bpb * d_r / 2 <= 32 * 16).  Its inputs are loaded with the rest; the rotation
    // table entries, which depend on the lengths, right after.
    const int half = p.d_r / 2;
    const bool rope = p.d_r > 0 && !p.skip_rope && bz == 0;
    constexpr int RPT = 2;
    int rL[RPT];
    float rx0[RPT], rx1[RPT];
#pragma unroll
    for (int u = 0; u < RPT; ++u) {
        const int e = threadIdx.x + u * ABSORB_THREADS;
        if (rope && e < nb * half) {
            const int rb = b0 + e / half, ri = e % half;
            const QT *qr = reinterpret_cast<const QT *>(p.q_rope) + ((long long)rb * p.H + h) * p.d_r;
            if (p.chunk_n > 0) {
                const int cp = chunk_pos(p.L0, p.chunk_n, rb);
                rL[u] = cp < 0 ? -1 : cp + 1;
            } else {
                rL[u] = p.seq_len[rb];
            }
            rx0[u] = to_f<QT>(qr[2 * ri]);
            rx1[u] = to_f<QT>(qr[2 * ri + 1]);
        }
    }

    // 1. this thread's chunk of M row i0 + o
    float mr[CSMAX];
    {
        const float *mrow = p.M + ((long long)h * d_h + i0 + o) * d_n + kl * cs;
        const bool own = o < rows;
        if ((cs & 3) == 0) {
#pragma unroll
            for (int u = 0; u < CSMAX / 4; ++u) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (own && 4 * u < cs) v = __ldg(reinterpret_cast<const float4 *>(mrow) + u);
                mr[4 * u] = v.x; mr[4 * u + 1] = v.y; mr[4 * u + 2] = v.z; mr[4 * u + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < CSMAX; ++j) mr[j] = (own && j < cs) ? __ldg(mrow + j) : 0.f;
        }
    }
    // 2. the query rows of the CTA's sequences, as raw 16-byte vectors
    constexpr int EPV = 16 / (int)sizeof(QT);   // elements per vector
    const int vrow = d_n / EPV;                 // vectors per query row
    uint4 qv[ABSORB_QVEC];
#pragma unroll
    for (int u = 0; u < ABSORB_QVEC; ++u) {
        const int e = threadIdx.x + u * ABSORB_THREADS;
        if (e < nb * vrow) {
            const int r = e / vrow, vi = e % vrow;
            const uint4 *src = reinterpret_cast<const uint4 *>(
                reinterpret_cast<const QT *>(p.q_nope) + ((long long)(b0 + r) * p.H + h) * d_n);
            qv[u] = __ldg(src + vi);
        }
    }
    // 3. stage: zero what the dot products read but no query fills (the rows past nb
    // and, for a chunk size that is not a multiple of 4, the chunk tails), then scatter
    {
        float4 *z = reinterpret_cast<float4 *>(sm_abs);
        for (int e = nb * 2 * cst + threadIdx.x; e < nbr * 2 * cst; e += ABSORB_THREADS)
            z[e] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (cs & 3) {
            const int pad = 4 - (cs & 3);
            for (int e = threadIdx.x; e < nb * 8 * pad; e += ABSORB_THREADS)
                sm_abs[(e / pad) * cst + cs + e % pad] = 0.f;
        }
    }
#pragma unroll
    for (int u = 0; u < ABSORB_QVEC; ++u) {
        const int e = threadIdx.x + u * ABSORB_THREADS;
        if (e < nb * vrow) {
            const int r = e / vrow, k0 = (e % vrow) * EPV;
            if (cs % EPV == 0) {
                // the vector lies in one chunk: EPV / 4 aligned 16-byte stores
                float *dst = sm_abs + (r * 8 + k0 / cs) * cst + k0 % cs;
#pragma unroll
                for (int t = 0; t < EPV; t += 4)
                    *reinterpret_cast<float4 *>(dst + t) =
                        make_float4(vec_elem<QT>(qv[u], t), vec_elem<QT>(qv[u], t + 1),
                                    vec_elem<QT>(qv[u], t + 2), vec_elem<QT>(qv[u], t + 3));
            } else {
#pragma unroll
                for (int t = 0; t < EPV; ++t) {
                    const int k = k0 + t;
                    sm_abs[(r * 8 + k / cs) * cst + k % cs] = vec_elem<QT>(qv[u], t);
                }
            }
        }
    }
    __syncthreads();
    // 3b. query RMSNorm (the scale-matched + query RMSNorm variant): one warp per staged
    //     row, y = gain * x / sqrt(mean(x^2) + eps) over the row's d_n values
    if (p.qnorm) {
        const int wq = threadIdx.x >> 5, lq = threadIdx.x & 31;
        for (int r = wq; r < nb; r += ABSORB_THREADS / 32) {
            float ss = 0.f;
            for (int k = lq; k < d_n; k += 32) {
                const float x = sm_abs[(r * 8 + k / cs) * cst + k % cs];
                ss = fmaf(x, x, ss);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float inv = 1.f / sqrtf(ss / (float)d_n + p.qn_eps);
            for (int k = lq; k < d_n; k += 32) {
                float *xp = sm_abs + (r * 8 + k / cs) * cst + k % cs;
                *xp = *xp * inv * (p.qn_gain ? __ldg(p.qn_gain + k) : 1.f);
            }
        }
        __syncthreads();
    }
    // 4. eight sequences at a time: chunk dot products, then the reduce-scatter
    for (int g0 = 0; g0 < nb; g0 += 8) {
        float acc[8];
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const float4 *qc = reinterpret_cast<const float4 *>(sm_abs + ((g0 + s) * 8 + kl) * cst);
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int u = 0; u < CSMAX / 4; ++u) {
                if (4 * u < cs) {
                    const float4 q = qc[u];
                    a0 = fmaf(q.x, mr[4 * u], a0);
                    a1 = fmaf(q.y, mr[4 * u + 1], a1);
                    a0 = fmaf(q.z, mr[4 * u + 2], a0);
                    a1 = fmaf(q.w, mr[4 * u + 3], a1);
                }
            }
            acc[s] = a0 + a1;
        }
        // lanes kl and kl ^ 4 swap halves: each keeps 4 sequences, then 2, then 1
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const bool up = kl & 4;
            const float send = up ? acc[i] : acc[i + 4];
            const float keep = up ? acc[i + 4] : acc[i];
            acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const bool up = kl & 2;
            const float send = up ? acc[i] : acc[i + 2];
            const float keep = up ? acc[i + 2] : acc[i];
            acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
        }
        {
            const bool up = kl & 1;
            const float send = up ? acc[0] : acc[1];
            const float keep = up ? acc[1] : acc[0];
            acc[0] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
        }
        const int s = g0 + kl;   // the sequence this lane now holds
        if (o < rows && s < nb)
            p.q_tilde[((long long)(b0 + s) * p.H + h) * d_h + i0 + o] = p.prescale * acc[0];
    }
    // 5. the positional queries: Rot(t) q_rope with t = L_b - 1
#pragma unroll
    for (int u = 0; u < RPT; ++u) {
        const int e = threadIdx.x + u * ABSORB_THREADS;
        if (rope && e < nb * half) {
            const int rb = b0 + e / half, ri = e % half;
            int t = rL[u] - 1;
            if (t < 0) t = 0;
            if (t >= p.rope_max_pos) {
                if (!p.check_rows || length_ok(p.R, p.chunk_n > 0 ? rb / p.chunk_n : rb, rL[u]))
                    dev_report(GVA_DEV_BAD_POSITION);
                t = 0;
            }
            const float rc = p.rope_tab[((long long)t * half + ri) * 2];
            const float rs = p.rope_tab[((long long)t * half + ri) * 2 + 1];
            float *qh = p.q_hat + ((long long)rb * p.H + h) * p.d_r;
            qh[2 * ri] = p.prescale * (rx0[u] * rc - rx1[u] * rs);
            qh[2 * ri + 1] = p.prescale * (rx0[u] * rs + rx1[u] * rc);
        }
    }
}

template <typename QT, int CSF>
__global__ void __launch_bounds__(ABSORB_THREADS, 2) absorb_kernel(const AbsorbParams p) {
    extern __shared__ __align__(16) float sm_abs[];
    if (threadIdx.x == 0) GVA_KT(2);
    if (threadIdx.x == 0) GVA_REC(2, 0);
    pdl_wait();
    if (threadIdx.x == 0) GVA_KT(3);
    if (threadIdx.x == 0) GVA_REC(2, 1);
    pdl_launch_dependents();
    absorb_body<QT, CSF>(p, blockIdx.x, blockIdx.y, blockIdx.z, sm_abs);
    if (threadIdx.x == 0) GVA_KT(4);
    if (threadIdx.x == 0) GVA_REC(2, 2);
}

// --------------------------------------------------------------------------- //
// Absorption and append of one decode step in one grid.  The two read disjoint inputs
// and write disjoint outputs (the absorbed queries; the new cache rows), so they need
// not be ordered: the first na CTAs (a linear form of the absorption's grid, H x ny x
// nz) absorb, the next B append one entry each.  A decode grid that follows reads the
// cache only after its grid dependency resolves.
// --------------------------------------------------------------------------- //
template <typename QT, int CSF, typename CT>
__global__ void __launch_bounds__(ABSORB_THREADS, 2)
    prep_step_kernel(const AbsorbParams a, const AppendParams ap, int ny, int nz) {
    extern __shared__ __align__(16) float sm_abs[];
    pdl_wait();
    pdl_launch_dependents();
    const int na = a.H * ny * nz;
    const int bid = blockIdx.x;
    if (bid < na) {
        absorb_body<QT, CSF>(a, bid % a.H, (bid / a.H) % ny, bid / (a.H * ny), sm_abs);
    } else {
        append_body<CT, ABSORB_THREADS>(ap, bid - na, gridDim.x - na);
    }
}

// --------------------------------------------------------------------------- //
// MLA-shaped decode: per-head up-projection of the latent attention output
// (KV-cache compression survey, MLA sections: the value of head h is c_j W^UV_h, so
// sum_j p_j (c_j W^UV_h) = (sum_j p_j c_j) W^UV_h)
// --------------------------------------------------------------------------- //
struct UpProjParams {
    int B, H, d_c, d_h;
    const float *o_lat;     // [B][H][d_c]  softmax-weighted latent rows
    const float *Wuv;       // [H][d_c][d_h]
    float *out;             // [B][H][d_h]
};
constexpr int UP_THREADS = 256;
constexpr int UP_SEQ = 8;      // sequences per CTA (one map read serves all of them)
constexpr int UP_UNROLL = 16;  // map loads in flight per thread

// Grid (H, ceil(B / UP_SEQ)).  The CTA's threads are (c-quarter, output column d) pairs:
// each sums UP_SEQ dot products over its quarter of the latent width with UP_UNROLL map
// loads in flight, then the quarters are added through shared memory.
__global__ void __launch_bounds__(UP_THREADS) mla_up_kernel(const UpProjParams p) {
    extern __shared__ float s_up[];           // o rows [UP_SEQ][d_c], then partial sums
    pdl_wait();
    pdl_launch_dependents();
    const int h = blockIdx.x, b0 = blockIdx.y * UP_SEQ;
    const int nb = min(UP_SEQ, p.B - b0);
    float *so = s_up;
    float *sp = s_up + UP_SEQ * p.d_c;        // [UP_THREADS][UP_SEQ]
    for (int e = threadIdx.x; e < UP_SEQ * p.d_c; e += UP_THREADS) {
        const int bi = e / p.d_c, c = e % p.d_c;
        so[e] = bi < nb ? p.o_lat[((long long)(b0 + bi) * p.H + h) * p.d_c + c] : 0.f;
    }
    __syncthreads();
    const int splits = UP_THREADS / p.d_h;    // d_h divides UP_THREADS
    const int d = threadIdx.x % p.d_h, part = threadIdx.x / p.d_h;
    const int c_per = p.d_c / splits, c0 = part * c_per;
    const float *w = p.Wuv + ((long long)h * p.d_c + c0) * p.d_h + d;
    float acc[UP_SEQ];
#pragma unroll
    for (int bi = 0; bi < UP_SEQ; ++bi) acc[bi] = 0.f;
    for (int cc = 0; cc < c_per; cc += UP_UNROLL) {   // c_per is a multiple of UP_UNROLL
        float wv[UP_UNROLL];
#pragma unroll
        for (int u = 0; u < UP_UNROLL; ++u) wv[u] = __ldg(w + (long long)(cc + u) * p.d_h);
#pragma unroll
        for (int u = 0; u < UP_UNROLL; ++u)
#pragma unroll
            for (int bi = 0; bi < UP_SEQ; ++bi)
                acc[bi] = fmaf(so[bi * p.d_c + c0 + cc + u], wv[u], acc[bi]);
    }
#pragma unroll
    for (int bi = 0; bi < UP_SEQ; ++bi) sp[threadIdx.x * UP_SEQ + bi] = acc[bi];
    __syncthreads();
    if (threadIdx.x < p.d_h) {
        for (int bi = 0; bi < nb; ++bi) {
            float v = 0.f;
            for (int k = 0; k < splits; ++k) v += sp[(k * p.d_h + d) * UP_SEQ + bi];
            p.out[((long long)(b0 + bi) * p.H + h) * p.d_h + d] = v;
        }
    }
}
inline size_t mla_up_smem_bytes(int d_c) {
    return sizeof(float) * ((size_t)UP_SEQ * d_c + (size_t)UP_THREADS * UP_SEQ);
}

}  // namespace gva
