// decode_simt.cuh -- split-K decode on CUDA cores (fp32 FMA), for every supported
// shape and both cache dtypes, plus the log-sum-exp combine shared by all decode paths.
#pragma once

#include "common.cuh"

namespace gva {

// Parameters of one decode launch (GVA, or the GQA comparator when Kc != Vc).
struct DecodeParams {
    int B, H, G, r, d_h, d_r;
    const int *seq_len;
    RowsDev R;
    const void *Kc;         // rows scored against the content query: V (GVA) or K (GQA)
    const void *Vc;         // value rows [G][d_h]
    const void *Krope;      // positional key rows [d_r] (GVA, d_r > 0)
    const void *qc;         // content query [B][H][d_h]
    int qc_f32;             // 1: fp32, 0: bf16
    float qc_scale;         // multiplies qc when loaded (softmax scale in log2 units)
    const float *qr;        // positional query [B][H][d_r], already rotated and scaled (GVA)
    // the raw positional query, rotated in the tensor-core decode when qr is null
    const void *q_rope;     // [B][H][d_r], q_dtype
    int qr_f32;             // 1: q_rope fp32, 0: bf16
    const float *rope_tab;  // [rope_max_pos][d_r/2][2] (cos, sin)
    int rope_max_pos;
    float qr_scale;         // multiplies the rotated q_rope (softmax scale in log2 units)
    float *out;             // [B][H][d_h]
    float *lse;             // [B][H] or null
    float *part_o;          // [slots][H][d_h]
    float *part_ml;         // [slots][H][2]  (running max in log2 units, sum)
    int n_ctas;
    int *prefix_ws;         // [B + 1] slab offsets, written by CTA 0 (or null)
};

constexpr int SIMT_THREADS = 256;
constexpr int SIMT_MAXQ = 16;   // (H * d_h) / SIMT_THREADS outputs per thread, at most

// Shared-memory plan of the SIMT kernel (bytes), padded rows for conflict-free reads.
struct SimtSmem {
    size_t ls, f, qc, qr, s, m, l, a, tk, tv, tr, total;
    int rs_k, rs_r;  // row strides of the key/value tile and the positional tile, 4-byte words
};

__host__ __device__ inline SimtSmem simt_smem(int B, int H, int G, int d_h, int d_r,
                                              int elem, bool gqa) {
    SimtSmem s;
    size_t o = 0;
    s.ls = o; o += sizeof(int) * B;
    s.f = o; o += sizeof(int) * (B + 1);
    o = align_up(o, 16);
    s.qc = o; o += sizeof(float) * H * d_h;
    s.qr = o; o += sizeof(float) * H * (d_r > 0 ? d_r : 1);
    s.s = o; o += sizeof(float) * H * SLAB;
    s.m = o; o += sizeof(float) * H;
    s.l = o; o += sizeof(float) * H;
    s.a = o; o += sizeof(float) * H;
    o = align_up(o, 16);
    s.rs_k = (G * d_h * elem) / 4 + 1;
    s.rs_r = (d_r * elem) / 4 + 1;
    s.tk = o; o += sizeof(int) * SLAB * s.rs_k;
    s.tv = s.tk;
    if (gqa) { s.tv = o; o += sizeof(int) * SLAB * s.rs_k; }
    s.tr = o; o += sizeof(int) * SLAB * (d_r > 0 ? s.rs_r : 1);
    s.total = align_up(o, 16);
    return s;
}

// Copy `nv` contiguous rows of `row_words` 4-byte words from global memory into a
// tile with row stride `rs` words; rows nv..SLAB-1 are zeroed (a cache slot past a
// sequence's end may hold anything, including NaN).
__device__ __forceinline__ void load_rows(uint32_t *dst, const uint32_t *src, int nv,
                                          int row_words, int rs) {
    const int n4 = row_words / 4;  // 16-byte vectors per row
    for (int e = threadIdx.x; e < SLAB * n4; e += blockDim.x) {
        const int t = e / n4, c = e % n4;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (t < nv) v = reinterpret_cast<const uint4 *>(src + (long long)t * row_words)[c];
        uint32_t *d = dst + t * rs + 4 * c;
        d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
    }
}

template <typename CT>
__device__ __forceinline__ float tile_elem(const uint32_t *tile, int rs, int t, int e) {
    return to_f<CT>(reinterpret_cast<const CT *>(tile + t * rs)[e]);
}

// One CTA walks its share [c*S/n, (c+1)*S/n) of the batch's slabs.  For each slab:
// scores for all (head, token) pairs, an online-softmax update per head, then the
// probability-weighted value sum per (head, dimension).  A sequence entirely inside
// the CTA's share is finished here; otherwise its (o, m, l) partial goes to slot c+b.
template <typename CT, bool GQA>
__global__ void __launch_bounds__(SIMT_THREADS) decode_simt_kernel(const DecodeParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    pdl_wait();
    pdl_launch_dependents();
    const int B = p.B, H = p.H, d_h = p.d_h, r = p.r;
    const int d_r = GQA ? 0 : p.d_r;
    const int W = p.G * d_h;
    const SimtSmem L = simt_smem(B, H, p.G, d_h, d_r, (int)sizeof(CT), GQA);
    int *Ls = reinterpret_cast<int *>(smem + L.ls);
    int *F = reinterpret_cast<int *>(smem + L.f);
    float *qc_s = reinterpret_cast<float *>(smem + L.qc);
    float *qr_s = reinterpret_cast<float *>(smem + L.qr);
    float *S = reinterpret_cast<float *>(smem + L.s);
    float *m_s = reinterpret_cast<float *>(smem + L.m);
    float *l_s = reinterpret_cast<float *>(smem + L.l);
    float *a_s = reinterpret_cast<float *>(smem + L.a);
    uint32_t *tk = reinterpret_cast<uint32_t *>(smem + L.tk);
    uint32_t *tv = reinterpret_cast<uint32_t *>(smem + L.tv);
    uint32_t *tr = reinterpret_cast<uint32_t *>(smem + L.tr);

    build_prefix(p.seq_len, p.R, B, Ls, F, blockIdx.x == 0, blockIdx.x == 0 ? p.prefix_ws : nullptr);
    const Part P{F[B], p.n_ctas};
    if (P.S == 0) return;
    const int c = blockIdx.x;
    const long long s0 = P.start(c), s1 = P.start(c + 1);
    if (s0 >= s1) return;

    const int tid = threadIdx.x, nthr = blockDim.x;
    const int nq = (H * d_h + nthr - 1) / nthr;
    const int row_words = W * (int)sizeof(CT) / 4;
    const int rrow_words = d_r * (int)sizeof(CT) / 4;
    const CT *Kg = reinterpret_cast<const CT *>(p.Kc);
    const CT *Vg = reinterpret_cast<const CT *>(p.Vc);
    const CT *Rg = reinterpret_cast<const CT *>(p.Krope);

    int b = seq_of_slab(F, B, s0);
    long long s = s0;
    while (s < s1) {
        while (F[b + 1] <= s) ++b;
        const long long seg_end = min(s1, (long long)F[b + 1]);
        const int Lb = Ls[b];
        // ---- per-sequence state ----
        for (int e = tid; e < H * d_h; e += nthr) {
            const long long q = (long long)b * H * d_h + e;
            qc_s[e] = p.qc_scale * (p.qc_f32 ? reinterpret_cast<const float *>(p.qc)[q]
                                             : __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p.qc)[q]));
        }
        for (int e = tid; e < H * d_r; e += nthr) qr_s[e] = p.qr[(long long)b * H * d_r + e];
        for (int h = tid; h < H; h += nthr) { m_s[h] = -INFINITY; l_s[h] = 0.f; }
        float o[SIMT_MAXQ];
#pragma unroll
        for (int u = 0; u < SIMT_MAXQ; ++u) o[u] = 0.f;
        __syncthreads();

        for (; s < seg_end; ++s) {
            const long long j0 = (long long)(s - F[b]) * SLAB;
            int nv = (int)min((long long)SLAB, (long long)Lb - j0);
            const long long row0 = row_of(p.R, b, j0);
            if (row0 < 0) {  // corrupt block-table entry: skip the slab's tokens
                if (tid == 0) dev_report(GVA_DEV_BAD_PAGE);
                nv = 0;
            }
            const long long rr = row0 < 0 ? 0 : row0;
            load_rows(tk, reinterpret_cast<const uint32_t *>(Kg + rr * W), nv, row_words, L.rs_k);
            if (GQA) load_rows(tv, reinterpret_cast<const uint32_t *>(Vg + rr * W), nv, row_words, L.rs_k);
            if (d_r > 0) load_rows(tr, reinterpret_cast<const uint32_t *>(Rg + rr * d_r), nv, rrow_words, L.rs_r);
            __syncthreads();
            // scores, log2 units
            for (int e = tid; e < H * SLAB; e += nthr) {
                const int h = e / SLAB, t = e % SLAB, g = h / r;
                float z = -INFINITY;
                if (t < nv) {
                    float acc = 0.f;
                    const float *q = qc_s + h * d_h;
                    for (int i = 0; i < d_h; ++i) acc = fmaf(q[i], tile_elem<CT>(tk, L.rs_k, t, g * d_h + i), acc);
                    const float *qr = qr_s + h * d_r;
                    for (int i = 0; i < d_r; ++i) acc = fmaf(qr[i], tile_elem<CT>(tr, L.rs_r, t, i), acc);
                    z = acc;
                }
                S[e] = z;
            }
            __syncthreads();
            // online softmax, one thread per head
            for (int h = tid; h < H; h += nthr) {
                float mx = -INFINITY;
                for (int t = 0; t < SLAB; ++t) mx = fmaxf(mx, S[h * SLAB + t]);
                const float m_old = m_s[h];
                const float m_new = fmaxf(m_old, mx);
                const float alpha = (m_old == -INFINITY) ? 0.f : exp2f(m_old - m_new);
                float sum = 0.f;
                for (int t = 0; t < SLAB; ++t) {
                    const float zz = S[h * SLAB + t];
                    const float pr = (zz == -INFINITY) ? 0.f : exp2f(zz - m_new);
                    S[h * SLAB + t] = pr;
                    sum += pr;
                }
                l_s[h] = l_s[h] * alpha + sum;
                m_s[h] = m_new;
                a_s[h] = alpha;
            }
            __syncthreads();
            // probability-weighted values
#pragma unroll
            for (int u = 0; u < SIMT_MAXQ; ++u) {
                if (u < nq) {
                    const int e = tid + u * nthr;
                    if (e < H * d_h) {
                        const int h = e / d_h, i = e % d_h, g = h / r;
                        float acc = o[u] * a_s[h];
                        for (int t = 0; t < nv; ++t)
                            acc = fmaf(S[h * SLAB + t], tile_elem<CT>(tv, L.rs_k, t, g * d_h + i), acc);
                        o[u] = acc;
                    }
                }
            }
            __syncthreads();
        }
        // ---- segment end ----
        const bool whole = F[b] >= s0 && F[b + 1] <= s1;
        const long long slot = (long long)c + b;
#pragma unroll
        for (int u = 0; u < SIMT_MAXQ; ++u) {
            if (u < nq) {
                const int e = tid + u * nthr;
                if (e < H * d_h) {
                    const int h = e / d_h;
                    if (whole) {
                        const float l = l_s[h];
                        p.out[(long long)b * H * d_h + e] = l > 0.f ? o[u] / l : 0.f;
                    } else {
                        p.part_o[slot * H * d_h + e] = o[u];
                    }
                }
            }
        }
        for (int h = tid; h < H; h += nthr) {
            if (whole) {
                const float l = l_s[h];
                if (p.lse) p.lse[(long long)b * H + h] = l > 0.f ? (m_s[h] + log2f(l)) * LN2 : -INFINITY;
            } else {
                p.part_ml[(slot * H + h) * 2] = m_s[h];
                p.part_ml[(slot * H + h) * 2 + 1] = l_s[h];
            }
        }
        __syncthreads();
    }
}

// --------------------------------------------------------------------------- //
// Log-sum-exp combine of split-K partials (flash-decoding):
//   m* = max_s m_s,  o = sum_s 2^(m_s - m*) o_s / sum_s 2^(m_s - m*) l_s,
//   lse = (m* + log2 sum_s 2^(m_s - m*) l_s) ln 2.
// Grid (B*H, ceil(d_h/32)), 128 threads = 4 part lanes x 32 dimensions.  Two memory
// round trips after the grid dependency: the lengths (final before the decode call,
// so they are read while the decode kernel still runs), then every part's (m, l) and
// o slice at once; the weights are applied in registers.  Sequences owned by a single
// CTA were finished by the decode kernel; empty ones get out = 0, lse = -inf.
// --------------------------------------------------------------------------- //
struct CombineParams {
    int B, H, d_h;
    const int *seq_len;
    RowsDev R;
    const float *part_o;
    const float *part_ml;
    float *out;
    float *lse;
    int n_ctas;
    const int *prefix_ws;   // [B + 1] slab offsets from the decode grid (large batches)
};

constexpr int COMBINE_THREADS = 128;
// Above this batch the combine reads its sequence's slab offsets from the decode
// grid's copy (after the grid wait) instead of scanning every length in every CTA.
constexpr int COMBINE_SCAN_MAX = 256;
constexpr int COMBINE_BATCH = 16;         // o loads in flight per thread

// Dynamic shared memory: 2 x n_ctas floats (a sequence spans at most n_ctas parts).  It
// is kept small so that the combine's CTAs fit beside the decode's on an SM and start
// (then wait on the grid dependency) while the decode still runs.
inline size_t combine_smem_bytes(int n_ctas) { return sizeof(float) * 2 * (size_t)n_ctas; }

__global__ void __launch_bounds__(COMBINE_THREADS) combine_kernel(const CombineParams p) {
    extern __shared__ float comb_dyn[];
    float *w_s = comb_dyn;                 // part weight 2^(m - m*), 0 for no part
    float *l_s = comb_dyn + p.n_ctas;
    __shared__ long long red_ll[2][COMBINE_THREADS / 32];
    __shared__ float red_f[COMBINE_THREADS / 32];
    __shared__ float acc_s[4][32];
    if (threadIdx.x == 0) GVA_KT(8);
    if (threadIdx.x == 0 && blockIdx.y == 0) GVA_REC(4, 0);
    pdl_launch_dependents();
    const int b = blockIdx.x / p.H, h = blockIdx.x % p.H;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    // ---- F_b and S: the validated slab counts (same rule as build_prefix) ----
    const bool scan = p.B <= COMBINE_SCAN_MAX || p.prefix_ws == nullptr;
    long long before = 0, total = 0;
    for (int bb = tid; scan && bb < p.B; bb += COMBINE_THREADS) {
        int L = p.seq_len[bb];
        if (!length_ok(p.R, bb, L)) L = 0;
        const long long n = (L + SLAB - 1) / SLAB;
        total += n;
        if (bb < b) before += n;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        before += __shfl_xor_sync(0xffffffffu, before, o);
        total += __shfl_xor_sync(0xffffffffu, total, o);
    }
    if (lane == 0) { red_ll[0][wid] = before; red_ll[1][wid] = total; }
    __syncthreads();
    long long Fb = 0, S = 0;
#pragma unroll
    for (int w = 0; w < COMBINE_THREADS / 32; ++w) { Fb += red_ll[0][w]; S += red_ll[1][w]; }
    int Lb = p.seq_len[b];
    if (!length_ok(p.R, b, Lb)) Lb = 0;
    long long nb = (Lb + SLAB - 1) / SLAB;
    const int d0 = blockIdx.y * 32;
    float *out = p.out + ((long long)b * p.H + h) * p.d_h;
    // the parts of the sequence depend on the lengths only: found before the wait
    // (large batches: from the decode grid's prefix, after the wait)
    Part P{S, p.n_ctas};
    int c_lo = nb > 0 ? P.cta_of(Fb) : 0, c_hi = nb > 0 ? P.cta_of(Fb + nb - 1) : 0;
    // the partials (and the outputs the decode kernel writes) come from the preceding grid
    pdl_wait();
    if (!scan) {
        Fb = p.prefix_ws[b];
        nb = p.prefix_ws[b + 1] - Fb;
        S = p.prefix_ws[p.B];
        P = Part{S, p.n_ctas};
        c_lo = nb > 0 ? P.cta_of(Fb) : 0;
        c_hi = nb > 0 ? P.cta_of(Fb + nb - 1) : 0;
    }
    if (threadIdx.x == 0) GVA_KT(9);
    if (threadIdx.x == 0 && blockIdx.y == 0) GVA_REC(4, 1);
    if (nb == 0) {
        if (tid < 32 && d0 + tid < p.d_h) out[d0 + tid] = 0.f;
        if (tid == 0 && blockIdx.y == 0 && p.lse) p.lse[(long long)b * p.H + h] = -INFINITY;
        return;
    }
    if (c_lo == c_hi) return;
    const int n = c_hi - c_lo + 1;
    const int i = d0 + lane;
    const long long step = (long long)p.H * p.d_h;   // next slot (c + 1 + b)
    const float *po = p.part_o + (((long long)c_lo + b) * p.H + h) * p.d_h + i;
    // ---- every part's (m, l), and this thread's first batch of o values, in one trip ----
    float ov[COMBINE_BATCH];
#pragma unroll
    for (int u = 0; u < COMBINE_BATCH; ++u) {
        const int k = wid + 4 * u;
        ov[u] = (k < n && i < p.d_h) ? po[(long long)k * step] : 0.f;
    }
    float mloc = -INFINITY;
    for (int k = tid; k < n; k += COMBINE_THREADS) {
        // a CTA with an empty share (more CTAs than slabs) wrote no partial: weight 0
        float m = -INFINITY, l = 0.f;
        if (P.start(c_lo + k) != P.start(c_lo + k + 1)) {
            const float2 ml = *reinterpret_cast<const float2 *>(
                p.part_ml + (((long long)c_lo + k + b) * p.H + h) * 2);
            m = ml.x;
            l = ml.y;
        }
        w_s[k] = m;
        l_s[k] = l;
        mloc = fmaxf(mloc, m);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
    if (lane == 0) red_f[wid] = mloc;
    __syncthreads();
    float mstar = -INFINITY;
#pragma unroll
    for (int w = 0; w < COMBINE_THREADS / 32; ++w) mstar = fmaxf(mstar, red_f[w]);
    __syncthreads();
    float dloc = 0.f;
    for (int k = tid; k < n; k += COMBINE_THREADS) {
        const float m = w_s[k];
        const float wgt = (m == -INFINITY) ? 0.f : exp2f(m - mstar);
        w_s[k] = wgt;
        dloc += wgt * l_s[k];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dloc += __shfl_xor_sync(0xffffffffu, dloc, o);
    if (lane == 0) red_f[wid] = dloc;
    __syncthreads();
    float den = 0.f;
#pragma unroll
    for (int w = 0; w < COMBINE_THREADS / 32; ++w) den += red_f[w];
    // ---- weighted sum of this CTA's 32-dimension slice: part lane wid, dimension lane ----
    float acc = 0.f;
#pragma unroll
    for (int u = 0; u < COMBINE_BATCH; ++u) {
        const int k = wid + 4 * u;
        if (k < n && w_s[k] != 0.f) acc += w_s[k] * ov[u];
    }
    for (int k0 = wid + 4 * COMBINE_BATCH; k0 < n; k0 += 4 * COMBINE_BATCH) {
#pragma unroll
        for (int u = 0; u < COMBINE_BATCH; ++u) {
            const int k = k0 + 4 * u;
            ov[u] = (k < n && i < p.d_h) ? po[(long long)k * step] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < COMBINE_BATCH; ++u) {
            const int k = k0 + 4 * u;
            if (k < n && w_s[k] != 0.f) acc += w_s[k] * ov[u];
        }
    }
    acc_s[wid][lane] = acc;
    __syncthreads();
    if (wid == 0 && i < p.d_h) {
        const float a = acc_s[0][lane] + acc_s[1][lane] + acc_s[2][lane] + acc_s[3][lane];
        out[i] = den > 0.f ? a / den : 0.f;
    }
    if (tid == 0 && blockIdx.y == 0 && p.lse)
        p.lse[(long long)b * p.H + h] = den > 0.f ? (mstar + log2f(den)) * LN2 : -INFINITY;
    if (tid == 0) GVA_KT(10);
    if (tid == 0 && blockIdx.y == 0) GVA_REC(4, 2);
}

}  // namespace gva
