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
    pdl_wait();
    pdl_launch_dependents();
    const int b = blockIdx.x;
    const int pos = p.pos[b];
    __syncthreads();  // every thread has read pos[b] before seq_len_out (may alias) is written
    bool ok = pos >= 0 && (long long)pos < seq_capacity(p.R, b) && (p.d_r == 0 || pos < p.rope_max_pos);
    long long row = ok ? row_of(p.R, b, pos) : -1;
    if (p.R.layout == GVA_LAYOUT_RAGGED && row >= p.R.num_rows) row = -1;
    if (row < 0) {
        if (threadIdx.x == 0) dev_report(ok ? GVA_DEV_BAD_PAGE : GVA_DEV_BAD_POSITION);
        return;
    }
    const int W = p.G * p.d_h;
    CT *V = reinterpret_cast<CT *>(p.V) + row * W;
    const float *vn = p.v_new + (long long)b * W;
    for (int e = threadIdx.x; e < W; e += blockDim.x) V[e] = from_f<CT>(vn[e]);
    if (p.d_r > 0) {
        CT *K = reinterpret_cast<CT *>(p.Kr) + row * p.d_r;
        const float *kn = p.k_new + (long long)b * p.d_r;
        const float *cs = p.rope_tab + (long long)pos * p.d_r;  // (d_r/2) (cos, sin) pairs
        for (int i = threadIdx.x; i < p.d_r / 2; i += blockDim.x) {
            const float x0 = kn[2 * i], x1 = kn[2 * i + 1];
            const float c = cs[2 * i], s = cs[2 * i + 1];
            const float y0 = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
            const float y1 = __fadd_rn(__fmul_rn(x0, s), __fmul_rn(x1, c));
            K[2 * i] = from_f<CT>(y0);
            K[2 * i + 1] = from_f<CT>(y1);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && p.seq_len_out) p.seq_len_out[b] = pos + 1;
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
};

// Grid (H, ceil(B / bpb), d_h / 32), 256 threads.  A CTA owns 32 rows of M_h (at most
// 32 x 256 fp32 = 32 KB) and issues all of its 16-byte loads of them at once (one
// memory round trip, even while the decode streams the cache); each output row is
// split over 8 threads (k strided by 8) and reduced with shuffles.
constexpr int ABSORB_THREADS = 256;

template <typename QT>
__global__ void __launch_bounds__(ABSORB_THREADS) absorb_kernel(const AbsorbParams p) {
    extern __shared__ __align__(16) float sm_abs[];
    pdl_wait();
    pdl_launch_dependents();
    const int h = blockIdx.x;
    const int b0 = blockIdx.y * p.bpb;
    const int nb = min(p.bpb, p.B - b0);
    const int i0 = blockIdx.z * 32;
    const int d_n = p.d_n, d_h = p.d_h;
    const int ldm = d_n + 4;                 // padded row (16-byte aligned)
    float *Ms = sm_abs;                      // [32][d_n + 4]
    float *qs = Ms + 32 * ldm;               // [bpb][d_n]
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
    if (p.d_r > 0 && blockIdx.z == 0) {
        const QT *qr = reinterpret_cast<const QT *>(p.q_rope);
        const int half = p.d_r / 2;
        for (int e = threadIdx.x; e < nb * half; e += ABSORB_THREADS) {
            const int bl = e / half, i = e % half, b = b0 + bl;
            const int L = p.seq_len[b];
            int t = L - 1;
            if (t < 0) t = 0;
            if (t >= p.rope_max_pos) {
                if (!p.check_rows || length_ok(p.R, b, L)) dev_report(GVA_DEV_BAD_POSITION);
                t = 0;
            }
            const long long qoff = ((long long)b * p.H + h) * p.d_r;
            const float x0 = to_f<QT>(qr[qoff + 2 * i]), x1 = to_f<QT>(qr[qoff + 2 * i + 1]);
            const float c = p.rope_tab[((long long)t * half + i) * 2];
            const float s = p.rope_tab[((long long)t * half + i) * 2 + 1];
            p.q_hat[qoff + 2 * i] = p.prescale * (x0 * c - x1 * s);
            p.q_hat[qoff + 2 * i + 1] = p.prescale * (x0 * s + x1 * c);
        }
    }
}

}  // namespace gva
