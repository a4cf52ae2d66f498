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
    RowsDev R;
    void *V;                // rows [G][d_h]
    void *Kr;               // rows [d_r]
    const float *rope_tab;  // [rope_max_pos][d_r/2][2]
    int rope_max_pos;
};

// One CTA per sequence.  V gets the new value rounded once; K_rope gets
// Rot(pos) k_new computed in fp32 in the fixed order y0 = (x0*c) - (x1*s),
// y1 = (x0*s) + (x1*c) with every product and sum rounded separately (no FMA), then
// rounded once to the cache dtype, so the stored bytes are reproducible.
template <typename CT>
__global__ void __launch_bounds__(128) append_kernel(const AppendParams p) {
    if (threadIdx.x == 0) GVA_KT(0);
    pdl_wait();
    pdl_launch_dependents();
    const int b = blockIdx.x;
    const int W = p.G * p.d_h;
    // Loads that do not depend on the position are issued with it: the new value (up
    // to 8 elements per thread), the unrotated key pair, the position.  The table entry
    // and, for a paged cache, the block-table entry follow: two memory round trips.
    constexpr int VPT = 8;
    const float *vn = p.v_new + (long long)b * W;
    float vv[VPT];
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
        const int e = threadIdx.x + u * 128;
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
    const int pos = p.pos[b];
    __syncthreads();  // every thread has read pos[b] before seq_len_out (may alias) is written
    bool ok = pos >= 0 && (long long)pos < seq_capacity(p.R, b) && (p.d_r == 0 || pos < p.rope_max_pos);
    float c = 0.f, sn = 0.f;
    if (ok && kthr) {
        const float *cs = p.rope_tab + (long long)pos * p.d_r;  // (d_r/2) (cos, sin) pairs
        c = cs[2 * threadIdx.x];
        sn = cs[2 * threadIdx.x + 1];
    }
    long long row = ok ? row_of(p.R, b, pos) : -1;
    if (p.R.layout == GVA_LAYOUT_RAGGED && row >= p.R.num_rows) row = -1;
    if (row < 0) {
        if (threadIdx.x == 0) dev_report(ok ? GVA_DEV_BAD_PAGE : GVA_DEV_BAD_POSITION);
        return;
    }
    CT *V = reinterpret_cast<CT *>(p.V) + row * W;
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
        const int e = threadIdx.x + u * 128;
        if (e < W) V[e] = from_f<CT>(vv[u]);
    }
    for (int e = threadIdx.x + VPT * 128; e < W; e += 128) V[e] = from_f<CT>(vn[e]);
    if (kthr) {
        CT *K = reinterpret_cast<CT *>(p.Kr) + row * p.d_r;
        const float y0 = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, sn));
        const float y1 = __fadd_rn(__fmul_rn(x0, sn), __fmul_rn(x1, c));
        K[2 * threadIdx.x] = from_f<CT>(y0);
        K[2 * threadIdx.x + 1] = from_f<CT>(y1);
    }
    __syncthreads();
    if (threadIdx.x == 0 && p.seq_len_out) p.seq_len_out[b] = pos + 1;
    if (threadIdx.x == 0) GVA_KT(1);
}

// --------------------------------------------------------------------------- //
// Absorb  (GVA analysis page, 关键技巧一: q_h k_{j,h}^T = (q_h M_h^T) v_{j,g(h)}^T)
// --------------------------------------------------------------------------- //
struct AbsorbParams {
    int B, H, d_h, d_n, d_r, bpb;  // bpb: sequences per CTA
    const void *q_nope;            // [B][H][d_n]
    const void *q_rope;            // [B][H][d_r]
    const float *M;                // [H][d_h][d_n]
    const int *seq_len;            // [B]
    const float *rope_tab;
    int rope_max_pos;
    float prescale;                // multiplies both outputs
    float *q_tilde;                // [B][H][d_h]
    float *q_hat;                  // [B][H][d_r]
    int check_rows;                // 1: a length the cache cannot hold is skipped silently
    RowsDev R;                     //    (the decode kernel reports it); used when check_rows
    int skip_rope;                 // 1: q_hat is not computed (the decode rotates q_rope)
};

// Grid (H, ceil(B / bpb), d_h / 32), 256 threads.  A CTA owns 32 rows of M_h (at most
// 32 x 256 fp32 = 32 KB) and issues all of its 16-byte loads of them at once (one
// memory round trip, even while the decode streams the cache); each output row is
// split over 8 threads (k strided by 8) and reduced with shuffles.
constexpr int ABSORB_THREADS = 256;

template <typename QT>
__global__ void __launch_bounds__(ABSORB_THREADS) absorb_kernel(const AbsorbParams p) {
    extern __shared__ __align__(16) float sm_abs[];
    if (threadIdx.x == 0) GVA_KT(2);
    pdl_wait();
    if (threadIdx.x == 0) GVA_KT(3);
    pdl_launch_dependents();
    const int h = blockIdx.x;
    const int b0 = blockIdx.y * p.bpb;
    const int nb = min(p.bpb, p.B - b0);
    const int i0 = blockIdx.z * 32;
    const int d_n = p.d_n, d_h = p.d_h;
    const int ldm = d_n + 4;                 // padded row (16-byte aligned)
    float *Ms = sm_abs;                      // [32][d_n + 4]
    float *qs = Ms + 32 * ldm;               // [bpb][d_n]
    // Positional slice: one (sequence, pair) per thread (bpb * d_r / 2 <= 8 * 16 threads).
    // Its inputs are read together with M and q_nope, and the rotation table entry right
    // after, so the whole CTA costs two memory round trips.
    const int half = p.d_r / 2;
    const bool rot = p.d_r > 0 && !p.skip_rope && blockIdx.z == 0 && (int)threadIdx.x < nb * half;
    int rb = 0, ri = 0, rL = 0;
    float rx0 = 0.f, rx1 = 0.f;
    long long qoff_r = 0;
    if (rot) {
        rb = b0 + threadIdx.x / half;
        ri = threadIdx.x % half;
        rL = p.seq_len[rb];
        qoff_r = ((long long)rb * p.H + h) * p.d_r;
        const QT *qr = reinterpret_cast<const QT *>(p.q_rope);
        rx0 = to_f<QT>(qr[qoff_r + 2 * ri]);
        rx1 = to_f<QT>(qr[qoff_r + 2 * ri + 1]);
    }
    const float *Mh = p.M + ((long long)h * d_h + i0) * d_n;
    const int rows = min(32, d_h - i0);
    const int n4 = rows * d_n / 4;
    for (int e = threadIdx.x; e < n4; e += ABSORB_THREADS) {
        const float4 v = reinterpret_cast<const float4 *>(Mh)[e];
        const int i = (4 * e) / d_n, k = (4 * e) % d_n;
        *reinterpret_cast<float4 *>(Ms + i * ldm + k) = v;
    }
    const QT *qn = reinterpret_cast<const QT *>(p.q_nope);
    for (int e = threadIdx.x; e < nb * d_n; e += ABSORB_THREADS) {
        const int bl = e / d_n, k = e % d_n;
        qs[e] = to_f<QT>(qn[((long long)(b0 + bl) * p.H + h) * d_n + k]);
    }
    float rc = 1.f, rs = 0.f;
    if (rot) {
        int t = rL - 1;
        if (t < 0) t = 0;
        if (t >= p.rope_max_pos) {
            if (!p.check_rows || length_ok(p.R, rb, rL)) dev_report(GVA_DEV_BAD_POSITION);
            t = 0;
        }
        rc = p.rope_tab[((long long)t * half + ri) * 2];
        rs = p.rope_tab[((long long)t * half + ri) * 2 + 1];
    }
    __syncthreads();
    const int o = threadIdx.x >> 3, kl = threadIdx.x & 7;   // output row, k lane
    for (int bl = 0; bl < nb; ++bl) {
        float acc = 0.f;
        if (o < rows) {
            const float *mrow = Ms + o * ldm;
            const float *q = qs + bl * d_n;
            for (int k = kl; k < d_n; k += 8) acc = fmaf(q[k], mrow[k], acc);
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        if (kl == 0 && o < rows)
            p.q_tilde[((long long)(b0 + bl) * p.H + h) * d_h + i0 + o] = p.prescale * acc;
    }
    if (rot) {
        p.q_hat[qoff_r + 2 * ri] = p.prescale * (rx0 * rc - rx1 * rs);
        p.q_hat[qoff_r + 2 * ri + 1] = p.prescale * (rx0 * rs + rx1 * rc);
    }
    if (threadIdx.x == 0) GVA_KT(4);
}

}  // namespace gva
