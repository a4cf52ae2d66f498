// common.cuh -- device helpers shared by the GVA decode kernels (one translation unit).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gva.h"

namespace gva {

constexpr int SLAB = 16;              // tokens per slab: unit of the split-K partition
constexpr int MAX_B = 4096;           // largest batch the in-kernel prefix scan handles
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// First device-side check code (gva_device_check), 0 when none tripped.
__device__ int g_status;

__device__ __forceinline__ void dev_report(int code) { atomicCAS(&g_status, 0, code); }

// Optional kernel timeline (compiled in only with -DGVA_TRACE, a debugging aid): the
// earliest (g_kt_min) and latest (g_kt_max) global-timer reading of thread 0 of any CTA
// at marked points of each kernel.
#ifdef GVA_TRACE
__device__ unsigned long long g_kt_min[16];
__device__ unsigned long long g_kt_max[16];
__device__ __forceinline__ unsigned long long kt_now() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ unsigned long long g_cta_t[4096][4];   // decode CTA: start, queries ready, end, SM
__device__ __forceinline__ unsigned smid() {
    unsigned r;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
    return r;
}
#define GVA_CTA_T(k)                                                          \
    do {                                                                      \
        if (blockIdx.x < 4096) g_cta_t[blockIdx.x][(k)] = kt_now();           \
        if ((k) == 2 && blockIdx.x < 4096) g_cta_t[blockIdx.x][3] = smid();  \
    } while (0)
// kernel event log: (kind << 56 | event << 48 | blockIdx.x, global time) per record
__device__ unsigned long long g_rec[1 << 16][2];
__device__ unsigned int g_rec_n;
#define GVA_REC(kind, ev)                                                          \
    do {                                                                           \
        const unsigned i_ = atomicAdd(&g_rec_n, 1u);                               \
        if (i_ < (1u << 16)) {                                                     \
            g_rec[i_][0] = ((unsigned long long)(kind) << 56) |                    \
                           ((unsigned long long)(ev) << 48) | blockIdx.x;          \
            g_rec[i_][1] = kt_now();                                               \
        }                                                                          \
    } while (0)
#define GVA_KT(slot)                                   \
    do {                                               \
        const unsigned long long t_ = kt_now();        \
        atomicMin(&g_kt_min[(slot)], t_);              \
        atomicMax(&g_kt_max[(slot)], t_);              \
    } while (0)
#else
#define GVA_KT(slot) \
    do {             \
    } while (0)
#define GVA_CTA_T(k) \
    do {             \
    } while (0)
#define GVA_REC(kind, ev) \
    do {                  \
    } while (0)
#endif

// Programmatic dependent launch: wait until the preceding grid in the stream has
// completed and its writes are visible; then let the next grid start its prologue.
// Every kernel waits before its first global read, so a grid is only ever released
// once everything before it has finished.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Where logical token j of sequence b lives (mirror of gva_rows plus the page count).
struct RowsDev {
    int layout;
    long long num_rows;
    long long T_cap;
    const int *offsets;
    const int *block_table;
    int max_pages;
    int page_size;
    int num_pages;
};

__device__ __forceinline__ long long seq_capacity(const RowsDev &R, int b) {
    if (R.layout == GVA_LAYOUT_CONTIGUOUS) return R.T_cap;
    if (R.layout == GVA_LAYOUT_RAGGED) return (long long)R.offsets[b + 1] - R.offsets[b];
    return (long long)R.max_pages * R.page_size;
}

// A length is usable when it fits the sequence's capacity and its rows exist.
__device__ __forceinline__ bool length_ok(const RowsDev &R, int b, long long L) {
    if (L < 0 || L > seq_capacity(R, b)) return false;
    if (R.layout == GVA_LAYOUT_RAGGED)
        return R.offsets[b] >= 0 && (long long)R.offsets[b] + L <= R.num_rows;
    return true;
}

// Storage row of token j (0 <= j < capacity) of sequence b, or -1 when the page id
// read from the block table is out of range.
__device__ __forceinline__ long long row_of(const RowsDev &R, int b, long long j) {
    if (R.layout == GVA_LAYOUT_CONTIGUOUS) return (long long)b * R.T_cap + j;
    if (R.layout == GVA_LAYOUT_RAGGED) return (long long)R.offsets[b] + j;
    const int jj = (int)j;   // positions are below 2^31 (lengths are int): 32-bit division
    const int page = R.block_table[(long long)b * R.max_pages + jj / R.page_size];
    if (page < 0 || page >= R.num_pages) return -1;
    return (long long)page * R.page_size + jj % R.page_size;
}

// Flat split-K partition over slabs.  Sequence b has n_b = ceil(L_b / 16) slabs
// starting at flat index F[b] (exclusive prefix); S = F[B].  The first
// neff = min(n, S) CTAs of the grid share the slabs: CTA c < neff owns flat slabs
// [floor(c*S/neff), floor((c+1)*S/neff)), at least one each, equal shares of the
// whole batch's cache whatever the length mix; CTAs c >= neff own none.  Partials of
// (CTA c, sequence b) go to slot c + b, which is unique along the monotone walk of
// (c, b) pairs.
//
// The shares are computed with 32-bit divisions only (S < 2^31, c <= neff < 2^12):
// floor(c*S/neff) = c*floor(S/neff) + floor(c*(S mod neff)/neff), c*(S mod neff) < 2^23.
struct Part {
    long long S;
    int n;
    __device__ __forceinline__ int neff() const { return S < (long long)n ? (int)S : n; }
    __device__ __forceinline__ long long start(int c) const {
        const int ne = neff();
        if (c >= ne) return S;
        const unsigned su = (unsigned)S, nu = (unsigned)ne, cu = (unsigned)c;
        const unsigned q = su / nu, r = su - q * nu;
        return (long long)cu * q + (long long)((cu * r) / nu);
    }
    // the CTA that owns flat slab s (0 <= s < S): the largest c with start(c) <= s,
    // i.e. floor(((s + 1) neff - 1) / S).  The quotient is below neff < 2^12, so a
    // single-precision estimate is within one of it and two integer checks make it
    // exact (FP64 arithmetic is slow on this GPU).
    __device__ __forceinline__ int cta_of(long long s) const {
        const long long a = (s + 1) * (long long)neff() - 1;
        long long q = (long long)__fdiv_rn((float)a, (float)S);
        while (q > 0 && q * S > a) --q;
        while ((q + 1) * S <= a) ++q;
        return (int)q;
    }
};

// Block-wide: validated lengths into Ls[0..B), exclusive slab prefix into F[0..B].
// Invalid lengths count as 0 and set GVA_DEV_BAD_LENGTH when `report` is set.
// When `prefix_out` is given, the CTA also stores F[0..B] there (one CTA of the grid
// does, for the combine kernel's large-batch path).
// With `hold_pos` (and Hs[B]), Hs[b] is the slab of sequence b that holds position
// hold_pos[b] when 0 <= hold_pos[b] < L_b, else -1 (loaded with the lengths).
__device__ void build_prefix(const int *seq_len, const RowsDev &R, int B, int *Ls, int *F,
                             bool report, int *prefix_out = nullptr,
                             const int *hold_pos = nullptr, int *Hs = nullptr) {
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        int L = seq_len[b];
        const int hp = hold_pos ? hold_pos[b] : -1;
        if (!length_ok(R, b, L)) {
            if (report) dev_report(GVA_DEV_BAD_LENGTH);
            L = 0;
        }
        Ls[b] = L;
        if (hold_pos) Hs[b] = (hp >= 0 && hp < L) ? hp / SLAB : -1;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int per = (B + 31) / 32;
        const int lo = lane * per, hi = min(lo + per, B);
        int sum = 0;
        for (int b = lo; b < hi; ++b) sum += (Ls[b] + SLAB - 1) / SLAB;
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
    __syncthreads();
    if (prefix_out)
        for (int b = threadIdx.x; b <= B; b += blockDim.x) prefix_out[b] = F[b];
}

// Largest b with F[b] <= s (F non-decreasing, F[0] = 0 <= s < F[B]); that sequence
// is non-empty and contains flat slab s.
__device__ __forceinline__ int seq_of_slab(const int *F, int B, long long s) {
    int lo = 0, hi = B;  // invariant: F[lo] <= s < F[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (F[mid] <= s) lo = mid; else hi = mid;
    }
    return lo;
}

__host__ __device__ __forceinline__ size_t align_up(size_t x, size_t a) {
    return (x + a - 1) / a * a;
}

}  // namespace gva
