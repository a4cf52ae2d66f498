// gva_api.cu -- the C ABI of libgva.so (declared in include/gva.h): host-side
// validation, workspace planning and kernel launches.  One translation unit holds
// every kernel so that they share the device status word.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

#include "gva.h"
#include "common.cuh"
#include "launch.cuh"
#include "prep_kernels.cuh"
#include "decode_simt.cuh"
#include "decode_mma.cuh"
#include "prefill_mma.cuh"
#include "decode_rope_keys.cuh"
#include "prefill_tc.cuh"

using namespace gva;

namespace {

constexpr int MAX_DEVICES = 64;
constexpr int CTAS_PER_SM_CAP = 8;   // the workspace is sized for this many CTAs per SM


bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Make the stream's device current for this library's runtime (the caller's runtime
// may be another copy of cudart).
cudaError_t bind_stream_device(void *stream) {
    if (stream == nullptr) return cudaSuccess;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cs);
    if (e != cudaSuccess) return e;
    // a capturing stream belongs to the device current at capture; device queries on it
    // are not needed (and not all are permitted while capturing)
    if (cs != cudaStreamCaptureStatusNone) return cudaSuccess;
    int dev = -1;
    e = cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &dev);
    if (e != cudaSuccess) return e;
    int cur = -1;
    e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return e;
    return cur == dev ? cudaSuccess : cudaSetDevice(dev);
}

int bind_or_fail(void *stream) {
    const cudaError_t e = bind_stream_device(stream);
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return GVA_ERR_CUDA;
    }
    return GVA_OK;
}

// Once per device, on the first call that reaches it: the SM count, the shared-memory
// opt-in of every kernel that may use more than 48 KB, and the register counts the
// CUDA-core grid is sized from.  Later calls (including calls made during stream
// capture) only read these values.
struct DevState {
    int ready;
    int sms;
    int simt_regs[4];   // decode_simt_kernel <f32,gva> <bf16,gva> <f32,gqa> <bf16,gqa>
};
DevState g_dev[MAX_DEVICES];
std::mutex g_dev_mu;

template <typename Kern>
cudaError_t opt_in_smem(Kern k) {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, MMA_SMEM_LIMIT);
}

// The small kernels chained with the decode (append, absorption, combine, prefill view
// and merge) prefer the largest shared-memory carveout, the one the decode kernels need:
// an SM holds CTAs of one L1 / shared-memory split at a time, so a small kernel running
// under a small carveout would keep the next decode grid off that SM until it drains,
// instead of the decode's CTAs starting (and streaming the cache) beside it.
template <typename Kern>
cudaError_t max_carveout(Kern k) {
    return cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                (int)cudaSharedmemCarveoutMaxShared);
}

template <typename Kern>
int kernel_regs(Kern k) {
    cudaFuncAttributes a;
    return cudaFuncGetAttributes(&a, k) == cudaSuccess ? a.numRegs : 255;
}

const DevState *device_state() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        if (e != cudaSuccess) g_last_cuda_error = (int)e;
        return nullptr;
    }
    if (g_dev[dev].ready) return &g_dev[dev];
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevState &d = g_dev[dev];
    if (d.ready) return &d;
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = opt_in_smem(absorb_kernel<float, 0>);
    if (e == cudaSuccess) e = opt_in_smem(absorb_kernel<__nv_bfloat16, 0>);
    if (e == cudaSuccess) e = opt_in_smem(decode_simt_kernel<float, false>);
    if (e == cudaSuccess) e = opt_in_smem(decode_simt_kernel<__nv_bfloat16, false>);
    if (e == cudaSuccess) e = opt_in_smem(decode_simt_kernel<float, true>);
    if (e == cudaSuccess) e = opt_in_smem(decode_simt_kernel<__nv_bfloat16, true>);
    if (e == cudaSuccess) e = mma_opt_in_all();
    if (e == cudaSuccess) e = prefill_opt_in_all();
    if (e == cudaSuccess) e = rk_opt_in_all();
    if (e == cudaSuccess) e = prefill_tc_opt_in_all();
    if (e == cudaSuccess) e = max_carveout(append_kernel<float>);
    if (e == cudaSuccess) e = max_carveout(append_kernel<__nv_bfloat16>);
    if (e == cudaSuccess) e = max_carveout(combine_kernel);
    if (e == cudaSuccess) e = max_carveout(mla_up_kernel);
    if (e == cudaSuccess) e = max_carveout(prefill_view_kernel);
    if (e == cudaSuccess) e = max_carveout(prefill_combine_kernel<64>);
    if (e == cudaSuccess) e = max_carveout(prefill_combine_kernel<128>);
    for (int q = 0; q < 2 && e == cudaSuccess; ++q) {
        const bool f = q == 0;
        if (e == cudaSuccess) e = f ? max_carveout(absorb_kernel<float, 0>) : max_carveout(absorb_kernel<__nv_bfloat16, 0>);
        if (e == cudaSuccess) e = f ? max_carveout(absorb_kernel<float, 8>) : max_carveout(absorb_kernel<__nv_bfloat16, 8>);
        if (e == cudaSuccess) e = f ? max_carveout(absorb_kernel<float, 16>) : max_carveout(absorb_kernel<__nv_bfloat16, 16>);
        if (e == cudaSuccess) e = f ? max_carveout(absorb_kernel<float, 32>) : max_carveout(absorb_kernel<__nv_bfloat16, 32>);
    }
    if (e == cudaSuccess && !encode_fn()) e = cudaErrorSymbolNotFound;
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        cudaGetLastError();
        return nullptr;
    }
    d.simt_regs[0] = kernel_regs(decode_simt_kernel<float, false>);
    d.simt_regs[1] = kernel_regs(decode_simt_kernel<__nv_bfloat16, false>);
    d.simt_regs[2] = kernel_regs(decode_simt_kernel<float, true>);
    d.simt_regs[3] = kernel_regs(decode_simt_kernel<__nv_bfloat16, true>);
    d.sms = n;
    d.ready = 1;
    return &d;
}

int num_sms_current() {
    const DevState *d = device_state();
    return d ? d->sms : 0;
}

bool dims_ok(const gva_dims *d, bool gva_shape) {
    if (!d) return false;
    if (d->B < 1 || d->B > MAX_B || d->H < 1 || d->G < 1 || d->H % d->G != 0) return false;
    const int r = d->H / d->G;
    if (r > 8) return false;
    if (d->d_h != 32 && d->d_h != 64 && d->d_h != 128) return false;
    if (d->cache_dtype != GVA_F32 && d->cache_dtype != GVA_BF16) return false;
    if (d->q_dtype != GVA_F32 && d->q_dtype != GVA_BF16) return false;
    if (d->H * d->d_h > SIMT_THREADS * SIMT_MAXQ) return false;
    if (gva_shape) {
        if (d->d_n < 8 || d->d_n > 256 || d->d_n % 8 != 0) return false;
        if (d->d_r < 0 || d->d_r > 32 || d->d_r % 8 != 0) return false;
    }
    return true;
}

bool rows_ok(const gva_rows *R, int B) {
    if (!R || R->num_rows < 0) return false;
    switch (R->layout) {
    case GVA_LAYOUT_CONTIGUOUS:
        return R->T_cap >= 0 && (long long)B * R->T_cap <= R->num_rows;
    case GVA_LAYOUT_RAGGED:
        return R->offsets != nullptr;
    case GVA_LAYOUT_PAGED:
        return R->block_table != nullptr && R->page_size > 0 && R->page_size % SLAB == 0 &&
               R->max_pages >= 1 && R->num_rows % R->page_size == 0;
    default:
        return false;
    }
}

RowsDev to_dev(const gva_rows &R) {
    RowsDev d;
    d.layout = R.layout;
    d.num_rows = R.num_rows;
    d.T_cap = R.T_cap;
    d.offsets = R.offsets;
    d.block_table = R.block_table;
    d.max_pages = R.max_pages;
    d.page_size = R.page_size;
    d.num_pages = R.layout == GVA_LAYOUT_PAGED ? (int)(R.num_rows / R.page_size) : 0;
    return d;
}

// Workspace: [q_tilde B*H*d_h][q_hat B*H*d_r][part_o slots*H*d_h][part_ml slots*H*2]
struct WsPlan {
    size_t qt, qh, po, pm, pf, total;
    long long slots;
};

WsPlan plan_ws(const gva_dims *d, int sms) {
    WsPlan w;
    w.slots = (long long)sms * CTAS_PER_SM_CAP + d->B;
    size_t o = 0;
    w.qt = o; o = align_up(o + sizeof(float) * d->B * d->H * d->d_h, 256);
    w.qh = o; o = align_up(o + sizeof(float) * d->B * d->H * (d->d_r > 0 ? d->d_r : 1), 256);
    w.po = o; o = align_up(o + sizeof(float) * w.slots * d->H * d->d_h, 256);
    w.pm = o; o = align_up(o + sizeof(float) * w.slots * d->H * 2, 256);
    w.pf = o; o = align_up(o + sizeof(int) * ((size_t)d->B + 1), 256);   // slab offsets
    w.total = o;
    return w;
}

// Grid of the SIMT decode kernel: resident CTAs per SM (shared memory, registers,
// threads; B300 SM: 228 KB shared memory, 64K registers, 2048 threads) x SMs, capped.
int simt_grid(int regs, size_t smem, int sms, int req) {
    if (req > 0) return req < sms * CTAS_PER_SM_CAP ? req : sms * CTAS_PER_SM_CAP;
    const int by_smem = (int)((228 * 1024) / (smem + 1024));
    const int regs_warp = ((regs * 32 + 255) / 256) * 256;
    const int by_regs = 65536 / (regs_warp * (SIMT_THREADS / 32));
    int per = by_smem < by_regs ? by_smem : by_regs;
    if (per > 2048 / SIMT_THREADS) per = 2048 / SIMT_THREADS;
    if (per > CTAS_PER_SM_CAP) per = CTAS_PER_SM_CAP;
    if (per < 1) per = 1;
    return sms * per;
}

int launch_combine(void *stream, const DecodeParams &dp, const gva_rows &rows) {
    CombineParams cp;
    cp.B = dp.B;
    cp.H = dp.H;
    cp.d_h = dp.d_h;
    cp.seq_len = dp.seq_len;
    cp.R = to_dev(rows);
    cp.part_o = dp.part_o;
    cp.part_ml = dp.part_ml;
    cp.out = dp.out;
    cp.prefix_ws = dp.prefix_ws;
    cp.lse = dp.lse;
    cp.n_ctas = dp.n_ctas;
    return cuda_status(launch(combine_kernel, dim3(dp.B * dp.H, (dp.d_h + 31) / 32),
                              dim3(COMBINE_THREADS), combine_smem_bytes(dp.n_ctas), stream, cp));
}

// Sets dp.n_ctas (the combine kernel re-derives the partition from it) and launches.
template <typename CT, bool GQA>
int run_simt(void *stream, DecodeParams &dp, int sms, int req_ctas) {
    const SimtSmem L = simt_smem(dp.B, dp.H, dp.G, dp.d_h, GQA ? 0 : dp.d_r, (int)sizeof(CT), GQA);
    auto kern = decode_simt_kernel<CT, GQA>;
    const DevState *ds = device_state();
    if (!ds) return GVA_ERR_CUDA;
    const int regs = ds->simt_regs[(sizeof(CT) == 2 ? 1 : 0) + (GQA ? 2 : 0)];
    dp.n_ctas = simt_grid(regs, L.total, sms, req_ctas);
    return cuda_status(launch(kern, dim3(dp.n_ctas), dim3(SIMT_THREADS), L.total, stream, dp));
}

// The absorption's parameters, grid and shared memory (arguments validated by the caller).
struct AbsorbLaunch {
    AbsorbParams p;
    dim3 grid;
    size_t smem;
};
AbsorbLaunch absorb_plan(const gva_dims *d, const void *q_nope, const void *q_rope,
                         const float *M, const int *seq_len, const float *rope_tab,
                         int rope_max_pos, float prescale, float *q_tilde, float *q_hat, int sms,
                         const gva_rows *rows, bool skip_rope, const gva_decode_opts *qn,
                         const int *L0, int chunk_n) {
    AbsorbLaunch A;
    AbsorbParams &p = A.p;
    p.skip_rope = skip_rope ? 1 : 0;
    p.L0 = L0;
    p.chunk_n = chunk_n;
    p.qnorm = qn && (qn->flags & GVA_FLAG_QUERY_RMSNORM) ? 1 : 0;
    p.qn_gain = p.qnorm ? qn->q_norm_gain : nullptr;
    p.qn_eps = p.qnorm ? qn->q_norm_eps : 0.f;
    p.check_rows = rows != nullptr;
    if (rows) p.R = to_dev(*rows);
    else memset(&p.R, 0, sizeof(p.R));
    p.B = d->B;
    p.H = d->H;
    p.d_h = d->d_h;
    p.d_n = d->d_n;
    p.d_r = d->d_r;
    // sequences per CTA: about one CTA per SM (the grid is resident at once and
    // leaves room beside it for the dependent decode grid to start), no more
    // sequences per CTA than the query staging holds
    const int zs = (d->d_h + 31) / 32;
    const long long per_b = (long long)d->H * zs;   // CTAs per sequence chunk
    const int qsize = d->q_dtype == GVA_F32 ? 4 : 2;
    long long nbc = (long long)(sms > 0 ? sms : 1) / per_b;
    if (nbc < 1) nbc = 1;
    if (nbc > d->B) nbc = d->B;
    int bpb = (int)((d->B + nbc - 1) / nbc);
    const int lim = absorb_bpb_limit(d->d_n, qsize);
    if (bpb > lim) bpb = lim;
    p.bpb = bpb;
    p.q_nope = q_nope;
    p.q_rope = q_rope;
    p.M = M;
    p.seq_len = seq_len;
    p.rope_tab = rope_tab;
    p.rope_max_pos = rope_max_pos;
    p.prescale = prescale;
    p.q_tilde = q_tilde;
    p.q_hat = q_hat;
    A.smem = (size_t)absorb_smem_bytes(d->d_n, bpb);
    A.grid = dim3(d->H, (d->B + bpb - 1) / bpb, zs);
    return A;
}

int absorb_run(void *stream, const gva_dims *d, const AbsorbLaunch &A) {
    const AbsorbParams &p = A.p;
    const dim3 grid = A.grid;
    const size_t smem = A.smem;
    cudaError_t e;
    const dim3 blk(ABSORB_THREADS);
    const bool f32 = d->q_dtype == GVA_F32;
    switch (d->d_n) {
    case 64:
        e = f32 ? launch(absorb_kernel<float, 8>, grid, blk, smem, stream, p)
                : launch(absorb_kernel<__nv_bfloat16, 8>, grid, blk, smem, stream, p);
        break;
    case 128:
        e = f32 ? launch(absorb_kernel<float, 16>, grid, blk, smem, stream, p)
                : launch(absorb_kernel<__nv_bfloat16, 16>, grid, blk, smem, stream, p);
        break;
    case 256:
        e = f32 ? launch(absorb_kernel<float, 32>, grid, blk, smem, stream, p)
                : launch(absorb_kernel<__nv_bfloat16, 32>, grid, blk, smem, stream, p);
        break;
    default:
        e = f32 ? launch(absorb_kernel<float, 0>, grid, blk, smem, stream, p)
                : launch(absorb_kernel<__nv_bfloat16, 0>, grid, blk, smem, stream, p);
    }
    return cuda_status(e);
}

int absorb_launch(void *stream, const gva_dims *d, const void *q_nope, const void *q_rope,
                  const float *M, const int *seq_len, const float *rope_tab, int rope_max_pos,
                  float prescale, float *q_tilde, float *q_hat, int sms,
                  const gva_rows *rows = nullptr, bool skip_rope = false,
                  const gva_decode_opts *qn = nullptr, const int *L0 = nullptr,
                  int chunk_n = 0) {
    return absorb_run(stream, d,
                      absorb_plan(d, q_nope, q_rope, M, seq_len, rope_tab, rope_max_pos,
                                  prescale, q_tilde, q_hat, sms, rows, skip_rope, qn, L0,
                                  chunk_n));
}

// The append's parameters (arguments validated by the caller).
AppendParams append_params(const gva_dims *d, const float *v_new, const float *k_new,
                           const int *pos, int *seq_len_out, const gva_rows &rows, void *V,
                           void *Kr, const float *rope_tab, int rope_max_pos, const int *L0,
                           int chunk_n, int *zero, int nzero) {
    AppendParams p;
    p.L0 = L0;
    p.chunk_n = chunk_n;
    p.zero = zero;
    p.nzero = nzero;
    p.B = d->B;
    p.G = d->G;
    p.d_h = d->d_h;
    p.d_r = d->d_r;
    p.v_new = v_new;
    p.k_new = k_new;
    p.pos = pos;
    p.seq_len_out = seq_len_out;
    p.R = to_dev(rows);
    p.V = V;
    p.Kr = Kr;
    p.rope_tab = rope_tab;
    p.rope_max_pos = rope_max_pos;
    return p;
}

// One CTA per entry of the batch d->B (arguments validated by the caller).
int append_launch(void *stream, const gva_dims *d, const float *v_new, const float *k_new,
                  const int *pos, int *seq_len_out, const gva_rows &rows, void *V, void *Kr,
                  const float *rope_tab, int rope_max_pos, const int *L0 = nullptr,
                  int chunk_n = 0, int *zero = nullptr, int nzero = 0) {
    const AppendParams p = append_params(d, v_new, k_new, pos, seq_len_out, rows, V, Kr,
                                         rope_tab, rope_max_pos, L0, chunk_n, zero, nzero);
    cudaError_t e = d->cache_dtype == GVA_F32
                        ? launch(append_kernel<float>, dim3(d->B), dim3(128), 0, stream, p)
                        : launch(append_kernel<__nv_bfloat16>, dim3(d->B), dim3(128), 0, stream, p);
    return cuda_status(e);
}

// The absorption and the append of one decode step as one grid: bf16 cache and a
// content-query width of 64 or 128 (the other shapes launch the two kernels).
bool prep_step_supported(const gva_dims *d) {
    return d->cache_dtype == GVA_BF16 && (d->d_n == 64 || d->d_n == 128);
}

int prep_step_launch(void *stream, const gva_dims *d, const AbsorbLaunch &A,
                     const AppendParams &ap) {
    const int ny = (int)A.grid.y, nz = (int)A.grid.z;
    const dim3 grid(A.grid.x * A.grid.y * A.grid.z + d->B), blk(ABSORB_THREADS);
    const bool f32 = d->q_dtype == GVA_F32;
    cudaError_t e;
    if (d->d_n == 64)
        e = f32 ? launch(prep_step_kernel<float, 8, __nv_bfloat16>, grid, blk, A.smem, stream,
                         A.p, ap, ny, nz)
                : launch(prep_step_kernel<__nv_bfloat16, 8, __nv_bfloat16>, grid, blk, A.smem,
                         stream, A.p, ap, ny, nz);
    else
        e = f32 ? launch(prep_step_kernel<float, 16, __nv_bfloat16>, grid, blk, A.smem, stream,
                         A.p, ap, ny, nz)
                : launch(prep_step_kernel<__nv_bfloat16, 16, __nv_bfloat16>, grid, blk, A.smem,
                         stream, A.p, ap, ny, nz);
    return cuda_status(e);
}

// Chunked prefill over n queries per sequence: the view's tables, the decode workspace
// of the B*n-entry batch (its absorbed-query regions also feed the tensor-core prefill
// kernel), then that kernel's split partials.
// Workspace: [view block table][positions][lengths][merge tickets][decode][prefill partials o][m, l].
struct PrefillPlan {
    size_t bt, pos, len, tk, dec, po, pml, total;
    int max_pages;
    gva_dims dv;        // the decode batch: B*n entries
    WsPlan dws;         // its workspace plan (offsets relative to dec)
    bool mq;            // the mma.sync prefill kernel takes this shape
    int tcm;            // rows per product of the tcgen05 prefill kernel (64 or 128), or 0
    int tc_splits;      // its history ranges per sequence
    PrefillMmaPlan mp;
};

// False when the chunk cannot be viewed as a decode batch of this library.
bool plan_prefill(const gva_dims *d, int n, const gva_rows &R, int sms, PrefillPlan *p) {
    if (n < 1 || (long long)d->B * n > MAX_B) return false;
    p->dv = *d;
    p->dv.B = d->B * n;
    p->max_pages = R.layout == GVA_LAYOUT_PAGED ? R.max_pages : 1;
    size_t o = 0;
    p->bt = o;  o = align_up(o + sizeof(int) * (size_t)p->dv.B * p->max_pages, 256);
    p->pos = o; o = align_up(o + sizeof(int) * (size_t)p->dv.B, 256);
    p->len = o; o = align_up(o + sizeof(int) * (size_t)p->dv.B, 256);
    p->tk = o;  o = align_up(o + sizeof(int) * (size_t)d->B * d->G, 256);   // merge tickets
    p->dws = plan_ws(&p->dv, sms);
    p->dec = o; o += p->dws.total;
    p->mq = prefill_mma_plan(d, n, sms, &p->mp);
    // the tcgen05 kernel: one CTA per (history range, value group, sequence), one wave
    p->tcm = p->mq ? prefill_tc_m(d, n) : 0;
    const long long gb = (long long)d->G * d->B;
    // one wave of CTAs, and at least two history ranges per (group, sequence), so that a
    // long sequence among short ones does not run alone at the end
    p->tc_splits = p->tcm ? (int)std::max<long long>(2, sms / gb) : 0;
    size_t po_bytes = p->mq ? p->mp.part_o_bytes : 0, pml_bytes = p->mq ? p->mp.part_ml_bytes : 0;
    if (p->tcm) {
        const size_t rows = (size_t)d->B * p->tc_splits * p->mp.rows_pad;
        po_bytes = std::max(po_bytes, align_up(rows * d->d_h * sizeof(float), 256));
        pml_bytes = std::max(pml_bytes, align_up(rows * 2 * sizeof(float), 256));
    }
    p->po = o;  o += po_bytes;
    p->pml = o; o += pml_bytes;
    p->total = o;
    return true;
}

// Layouts the view supports: paged, and contiguous with a capacity that is a
// multiple of the 16-token slab (read as one page per sequence).
bool prefill_layout_ok(const gva_rows &R) {
    if (R.layout == GVA_LAYOUT_PAGED) return true;
    return R.layout == GVA_LAYOUT_CONTIGUOUS && R.T_cap >= SLAB && R.T_cap % SLAB == 0 &&
           R.T_cap <= 0x7fffffffLL;
}

const gva_decode_opts kDefaultOpts = {GVA_PATH_AUTO, 0, 0, 0.f, nullptr};


// Option flags: only the query RMSNorm, with a finite eps >= 0.
bool flags_ok(const gva_decode_opts *o) {
    if ((o->flags & ~GVA_FLAG_QUERY_RMSNORM) != 0) return false;
    if (o->flags & GVA_FLAG_QUERY_RMSNORM)
        return o->q_norm_eps >= 0.f && o->q_norm_eps < INFINITY;
    return true;
}

}  // namespace

// Read-only streaming probe: every thread issues PROBE_UNROLL independent 16-byte
// non-allocating loads per trip and folds them into a XOR; one atomic per warp.
constexpr int PROBE_THREADS = 512, PROBE_UNROLL = 16;
__global__ void __launch_bounds__(PROBE_THREADS) read_probe_kernel(const uint4 *p, long long n16,
                                                                   unsigned *sink) {
    unsigned acc = 0;
    const long long stride = (long long)gridDim.x * PROBE_THREADS;
    long long i = (long long)blockIdx.x * PROBE_THREADS + threadIdx.x;
    for (; i + (PROBE_UNROLL - 1) * stride < n16; i += PROBE_UNROLL * stride) {
        uint4 v[PROBE_UNROLL];
#pragma unroll
        for (int u = 0; u < PROBE_UNROLL; ++u)
            asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(v[u].x), "=r"(v[u].y), "=r"(v[u].z), "=r"(v[u].w)
                         : "l"(p + i + u * stride));
#pragma unroll
        for (int u = 0; u < PROBE_UNROLL; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
    // the rest (a buffer smaller than one full trip of the grid, or the last part of a
    // larger one): up to PROBE_UNROLL predicated loads per thread, all in flight together
    if (i < n16) {
        uint4 v[PROBE_UNROLL];
#pragma unroll
        for (int u = 0; u < PROBE_UNROLL; ++u) {
            v[u] = make_uint4(0u, 0u, 0u, 0u);
            if (i + u * stride < n16)
                asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                             : "=r"(v[u].x), "=r"(v[u].y), "=r"(v[u].z), "=r"(v[u].w)
                             : "l"(p + i + u * stride));
        }
#pragma unroll
        for (int u = 0; u < PROBE_UNROLL; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
    // one atomic per CTA (same-address atomics serialise: one per warp would dominate a
    // small buffer's time)
    __shared__ unsigned warp_x[PROBE_THREADS / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) warp_x[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned x = 0;
#pragma unroll
        for (int k = 0; k < PROBE_THREADS / 32; ++k) x ^= warp_x[k];
        atomicXor(sink, x);
    }
}

// Self-test of the bounded waits: one warp waits on an mbarrier that nothing arrives on;
// the wait gives up after `limit_ns` and records GVA_DEV_TIMEOUT.
__global__ void wait_selftest_kernel(unsigned long long limit_ns) {
    __shared__ __align__(8) unsigned long long bar;
    __shared__ int abort;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait_for(smem_u32(&bar), 0, &abort, limit_ns);
}

// =========================================================================== //
// MLA-shaped decode helpers (the entry points are below).
namespace {

bool mla_dims_ok(const gva_mla_dims *d) {
    if (!d) return false;
    if (d->B < 1 || d->B > MAX_B || d->H < 4 || d->H % 4 != 0 || d->H / 4 > MMA_CONSUMERS)
        return false;
    if (d->d_c != 128 && d->d_c != 256) return false;
    if (d->d_n < 8 || d->d_n > 256 || d->d_n % 8 != 0) return false;
    if (d->d_r < 0 || d->d_r > 32 || d->d_r % 8 != 0) return false;
    if (d->d_h != 32 && d->d_h != 64 && d->d_h != 128 && d->d_h != 256) return false;
    if (d->q_dtype != GVA_F32 && d->q_dtype != GVA_BF16) return false;
    return d->cache_dtype == GVA_F32 || d->cache_dtype == GVA_BF16;
}

// The latent decode viewed as this library's decode: H/4 groups of 4 heads, every group
// reading the whole latent row of width d_c.
gva_dims mla_as_gva(const gva_mla_dims *d) {
    gva_dims g;
    g.B = d->B;
    g.H = d->H;
    g.G = d->H / 4;
    g.d_h = d->d_c;
    g.d_n = d->d_n;
    g.d_r = d->d_r;
    g.cache_dtype = d->cache_dtype;
    g.q_dtype = d->q_dtype;
    return g;
}

// Workspace: the decode's (queries, partials, slab offsets) for the latent width, then
// the latent outputs [B][H][d_c].
size_t mla_ws_bytes(const gva_mla_dims *d, int sms, size_t *off_lat) {
    const gva_dims g = mla_as_gva(d);
    const WsPlan w = plan_ws(&g, sms);
    *off_lat = w.total;
    return w.total + align_up(sizeof(float) * (size_t)d->B * d->H * d->d_c, 256);
}

}  // namespace

// =========================================================================== //
// Helpers of the decode with RoPE on the reconstructed key (entry points below).
namespace {

bool rk_dims_ok(const gva_dims *d) {
    if (!d) return false;
    if (d->B < 1 || d->B > MAX_B || d->H < 1 || d->G < 1 || d->H % d->G != 0) return false;
    if (d->d_r != 0) return false;                     // the query is d_n wide, no extra slice
    if (d->d_h < 8 || d->d_h > 256 || d->d_h % 8 != 0) return false;
    if (d->d_n < 2 || d->d_n > 256 || d->d_n % 2 != 0) return false;
    if (d->q_dtype != GVA_F32 && d->q_dtype != GVA_BF16) return false;
    return d->cache_dtype == GVA_F32 || d->cache_dtype == GVA_BF16;
}

// Workspace: [Ls B][pre B+1] | images [streams][hi, lo] | part_o [slots][hc][d_h] |
// part_ml [slots][hc][2]; streams = B G nhs, slots = streams + CTAs.
struct RkWs {
    size_t ls, pre, img, po, pm, total;
    int hc, nhs;
};

RkWs rk_plan(const gva_dims *d, int sms) {
    RkWs w;
    const int r = d->H / d->G;
    w.hc = rk_hc(r, d->d_n);
    w.nhs = r / w.hc;
    const long long streams = (long long)d->B * d->G * w.nhs;
    const long long slots = streams + (sms < RK_MAX_PARTS ? sms : RK_MAX_PARTS);
    size_t o = 0;
    w.ls = o;
    o += sizeof(int) * d->B;
    w.pre = o;
    o += sizeof(int) * (d->B + 1);
    o = align_up(o, 256);
    w.img = o;
    o += (size_t)streams * rk_img_bytes(d->d_h, w.hc * d->d_n);
    o = align_up(o, 256);
    w.po = o;
    o += sizeof(float) * (size_t)slots * w.hc * d->d_h;
    o = align_up(o, 256);
    w.pm = o;
    o += sizeof(float) * (size_t)slots * w.hc * 2;
    w.total = align_up(o, 256);
    return w;
}

int gcd_int(int a, int b) { return b == 0 ? a : gcd_int(b, a % b); }

}  // namespace

extern "C" {

const char *gva_status_string(int s) {
    switch (s) {
    case GVA_OK: return "GVA_OK";
    case GVA_ERR_ARG: return "GVA_ERR_ARG: invalid argument";
    case GVA_ERR_UNSUPPORTED: return "GVA_ERR_UNSUPPORTED: shape or dtype not supported";
    case GVA_ERR_CUDA: return "GVA_ERR_CUDA: CUDA runtime or launch failure";
    case GVA_ERR_WORKSPACE: return "GVA_ERR_WORKSPACE: workspace missing, too small or misaligned";
    case GVA_ERR_DEVICE_CHECK: return "GVA_ERR_DEVICE_CHECK: a device-side check tripped";
    case GVA_DEV_BAD_LENGTH: return "GVA_DEV_BAD_LENGTH: sequence length outside its capacity";
    case GVA_DEV_BAD_PAGE: return "GVA_DEV_BAD_PAGE: block-table entry out of range";
    case GVA_DEV_BAD_POSITION: return "GVA_DEV_BAD_POSITION: position outside capacity or RoPE table";
    case GVA_DEV_TIMEOUT: return "GVA_DEV_TIMEOUT: a bounded in-kernel wait gave up";
    default: return "unknown gva status";
    }
}

int gva_abi_version(void) { return GVA_ABI_VERSION; }

int gva_num_sms(void) { return num_sms_current(); }

int gva_selftest_bounded_wait(void *stream, unsigned limit_us) {
    if (limit_us < 1 || limit_us > 1000000) return GVA_ERR_ARG;
    if (bind_or_fail(stream) != GVA_OK) return GVA_ERR_CUDA;
    wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        (unsigned long long)limit_us * 1000ull);
    return cuda_status(cudaGetLastError());
}

int gva_read_probe(void *stream, const void *buf, size_t bytes, unsigned *sink) {
    if (!buf || !sink || bytes == 0 || bytes % 16 != 0 || !aligned16(buf)) return GVA_ERR_ARG;
    if (bind_or_fail(stream) != GVA_OK) return GVA_ERR_CUDA;
    const int sms = num_sms_current();
    if (sms <= 0) return GVA_ERR_CUDA;
    cudaError_t e = cudaMemsetAsync(sink, 0, sizeof(unsigned), static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) {
        // a plain launch: the probe starts only after the preceding work has finished
        read_probe_kernel<<<sms * (2048 / PROBE_THREADS), PROBE_THREADS, 0,
                            static_cast<cudaStream_t>(stream)>>>(
            reinterpret_cast<const uint4 *>(buf), (long long)(bytes / 16), sink);
        e = cudaGetLastError();
    }
    return cuda_status(e);
}

int gva_last_cuda_error(void) { return g_last_cuda_error; }

int gva_rope_table_fill(float *tab, int max_pos, int d_r, double base) {
    if (max_pos < 1 || d_r < 0 || d_r % 2 != 0 || !(base > 0.0)) return GVA_ERR_ARG;
    if (d_r == 0) return GVA_OK;
    if (!tab) return GVA_ERR_ARG;
    const int half = d_r / 2;
    for (long long p = 0; p < max_pos; ++p) {
        for (int i = 0; i < half; ++i) {
            const double theta = std::pow(base, -(2.0 * (double)i) / (double)d_r);
            const double ang = (double)p * theta;
            tab[(p * half + i) * 2 + 0] = (float)std::cos(ang);
            tab[(p * half + i) * 2 + 1] = (float)std::sin(ang);
        }
    }
    return GVA_OK;
}

int gva_absorb_query(void *stream, const gva_dims *d, const void *q_nope, const void *q_rope,
                     const float *M, const int *seq_len, const float *rope_tab, int rope_max_pos,
                     float scale, float *q_tilde, float *q_rope_rot) {
    return gva_absorb_query_ex(stream, d, q_nope, q_rope, M, seq_len, rope_tab, rope_max_pos,
                               scale, q_tilde, q_rope_rot, nullptr);
}

int gva_absorb_query_ex(void *stream, const gva_dims *d, const void *q_nope, const void *q_rope,
                        const float *M, const int *seq_len, const float *rope_tab,
                        int rope_max_pos, float scale, float *q_tilde, float *q_rope_rot,
                        const gva_decode_opts *opts) {
    const gva_decode_opts *o = opts ? opts : &kDefaultOpts;
    if (!flags_ok(o)) return GVA_ERR_ARG;
    if (!dims_ok(d, true)) return GVA_ERR_ARG;
    if (!q_nope || !M || !seq_len || !q_tilde || !aligned16(q_nope) || !aligned16(M) ||
        !aligned16(q_tilde))
        return GVA_ERR_ARG;
    if (d->d_r > 0 && (!q_rope || !rope_tab || !q_rope_rot || rope_max_pos < 1 ||
                       !aligned16(q_rope) || !aligned16(q_rope_rot) || !aligned16(rope_tab)))
        return GVA_ERR_ARG;
    if (bind_or_fail(stream) != GVA_OK) return GVA_ERR_CUDA;
    return absorb_launch(stream, d, q_nope, q_rope, M, seq_len, rope_tab, rope_max_pos, scale,
                         q_tilde, q_rope_rot, num_sms_current(), nullptr, false, o);
}

// Host-only checks of the append's arguments (no CUDA call).
static int append_arg_checks(const gva_dims *d, const float *v_new, const float *k_new,
                             const int *pos, const gva_cache *cache, const float *rope_tab,
                             int rope_max_pos) {
    if (!dims_ok(d, true) || !cache || !rows_ok(&cache->rows, d->B)) return GVA_ERR_ARG;
    if (!v_new || !pos || !cache->V || !aligned16(v_new) || !aligned16(cache->V)) return GVA_ERR_ARG;
    if (d->d_r > 0 && (!k_new || !cache->K_rope || !rope_tab || rope_max_pos < 1 ||
                       !aligned16(k_new) || !aligned16(cache->K_rope)))
        return GVA_ERR_ARG;
    return GVA_OK;
}

int gva_append_cache(void *stream, const gva_dims *d, const float *v_new, const float *k_new,
                     const int *pos, int *seq_len_out, const gva_cache *cache,
                     const float *rope_tab, int rope_max_pos) {
    const int ck = append_arg_checks(d, v_new, k_new, pos, cache, rope_tab, rope_max_pos);
    if (ck != GVA_OK) return ck;
    if (bind_or_fail(stream) != GVA_OK) return GVA_ERR_CUDA;
    if (!device_state()) return GVA_ERR_CUDA;
    return append_launch(stream, d, v_new, k_new, pos, seq_len_out, cache->rows, cache->V,
                         cache->K_rope, rope_tab, rope_max_pos);
}

size_t gva_decode_workspace_size(const gva_dims *d) {
    if (!dims_ok(d, false)) return 0;
    const int sms = num_sms_current();
    if (sms <= 0) return 0;
    return plan_ws(d, sms).total;
}

// Host-only checks shared by both decode entry points (no CUDA call).
static int decode_arg_checks(const gva_dims *d, const gva_rows *rows, float *out, float *lse,
                             const gva_decode_opts *o, bool gva_shape) {
    if (!dims_ok(d, gva_shape) || !rows_ok(rows, d->B)) return GVA_ERR_ARG;
    if (!out || !aligned16(out) || (lse && !aligned16(lse))) return GVA_ERR_ARG;
    if (!flags_ok(o) || o->path < GVA_PATH_AUTO || o->path > GVA_PATH_MMA || o->num_ctas < 0)
        return GVA_ERR_ARG;
    return GVA_OK;
}

// Device binding, SM count and the workspace check.
static int decode_device_checks(void *stream, const gva_dims *d, void *ws, size_t ws_bytes,
                                WsPlan *plan, int *sms) {
    if (bind_or_fail(stream) != GVA_OK) return GVA_ERR_CUDA;
    *sms = num_sms_current();
    if (*sms <= 0) return GVA_ERR_CUDA;
    *plan = plan_ws(d, *sms);
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < plan->total)
        return GVA_ERR_WORKSPACE;
    return GVA_OK;
}

// The new token of a decode step, appended by the same call (gva_decode_step).
struct StepAppend {
    const float *v_new, *k_new;
    const int *pos;
};

// One layer's decode, after the append of `app` when it is given: with the tensor-core
// decode and a shape the fused kernel takes, the append runs in the absorption's grid
// and the decode streams the cache meanwhile, except for the slab that holds each
// sequence's new row (copied once that grid has completed); otherwise the append kernel
// runs first.
static int decode_call(void *stream, const gva_dims *d, const void *q_nope, const void *q_rope,
                       const float *M, const int *seq_len, const gva_cache *cache,
                       const float *rope_tab, int rope_max_pos, float scale, float *out,
                       float *lse, void *ws, size_t ws_bytes, const gva_decode_opts *opts,
                       const StepAppend *app) {
    const gva_decode_opts *o = opts ? opts : &kDefaultOpts;
    if (!cache) return GVA_ERR_ARG;
    int st = decode_arg_checks(d, &cache->rows, out, lse, o, true);
    if (st != GVA_OK) return st;
    if (app) {
        st = append_arg_checks(d, app->v_new, app->k_new, app->pos, cache, rope_tab,
                               rope_max_pos);
        if (st != GVA_OK) return st;
    }
    if (!q_nope || !M || !seq_len || !cache->V || !aligned16(q_nope) || !aligned16(M) ||
        !aligned16(cache->V))
        return GVA_ERR_ARG;
    if (d->d_r > 0 && (!q_rope || !cache->K_rope || !rope_tab || rope_max_pos < 1 ||
                       !aligned16(q_rope) || !aligned16(cache->K_rope) || !aligned16(rope_tab)))
        return GVA_ERR_ARG;
    const bool mma_ok = mma_supported(d);
    if (o->path == GVA_PATH_MMA && !mma_ok) return GVA_ERR_UNSUPPORTED;
    WsPlan plan;
    int sms = 0;
    st = decode_device_checks(stream, d, ws, ws_bytes, &plan, &sms);
    if (st != GVA_OK) return st;
    char *w = static_cast<char *>(ws);
    const bool use_mma = o->path == GVA_PATH_MMA || (o->path == GVA_PATH_AUTO && mma_ok);

    float *qt = reinterpret_cast<float *>(w + plan.qt);
    float *qh = reinterpret_cast<float *>(w + plan.qh);
    // the tensor-core decode rotates the positional query itself (its inputs are final
    // before the call, so it overlaps the absorption), leaving the absorption a single
    // memory round trip
    const AbsorbLaunch A = absorb_plan(d, q_nope, q_rope, M, seq_len, rope_tab, rope_max_pos,
                                       scale * LOG2E, qt, qh, sms, &cache->rows, use_mma, o,
                                       nullptr, 0);
    const bool fused = app && use_mma && prep_step_supported(d);
    if (fused) {
        st = prep_step_launch(stream, d, A,
                              append_params(d, app->v_new, app->k_new, app->pos, nullptr,
                                            cache->rows, cache->V, cache->K_rope, rope_tab,
                                            rope_max_pos, nullptr, 0, nullptr, 0));
    } else {
        if (app) {
            if (!device_state()) return GVA_ERR_CUDA;
            st = append_launch(stream, d, app->v_new, app->k_new, app->pos, nullptr, cache->rows,
                               cache->V, cache->K_rope, rope_tab, rope_max_pos);
            if (st != GVA_OK) return st;
        }
        st = absorb_run(stream, d, A);
    }
    if (st != GVA_OK) return st;

    DecodeParams dp;
    dp.B = d->B;
    dp.H = d->H;
    dp.G = d->G;
    dp.r = d->H / d->G;
    dp.d_h = d->d_h;
    dp.d_r = d->d_r;
    dp.seq_len = seq_len;
    dp.R = to_dev(cache->rows);
    dp.Kc = cache->V;
    dp.Vc = cache->V;
    dp.Krope = cache->K_rope;
    dp.qc = qt;
    dp.qc_f32 = 1;
    dp.qc_scale = 1.f;
    dp.qr = use_mma ? nullptr : qh;
    dp.q_rope = q_rope;
    dp.qr_f32 = d->q_dtype == GVA_F32;
    dp.rope_tab = rope_tab;
    dp.rope_max_pos = rope_max_pos;
    dp.qr_scale = scale * LOG2E;
    dp.out = out;
    dp.lse = lse;
    dp.part_o = reinterpret_cast<float *>(w + plan.po);
    dp.part_ml = reinterpret_cast<float *>(w + plan.pm);
    dp.n_ctas = 0;
    dp.prefix_ws = reinterpret_cast<int *>(w + plan.pf);
    if (use_mma) {
        // the cache streams before the grid dependency resolves; after the fused grid,
        // which also appends, the slab holding each sequence's new row waits for it
        st = run_mma(stream, dp, cache->rows, sms, o->num_ctas, false, true, false,
                     fused ? app->pos : nullptr);
    } else if (d->cache_dtype == GVA_F32) {
        st = run_simt<float, false>(stream, dp, sms, o->num_ctas);
    } else {
        st = run_simt<__nv_bfloat16, false>(stream, dp, sms, o->num_ctas);
    }
    if (st != GVA_OK) return st;
    return launch_combine(stream, dp, cache->rows);
}

int gva_decode_attention_ex(void *stream, const gva_dims *d, const void *q_nope,
                            const void *q_rope, const float *M, const int *seq_len,
                            const gva_cache *cache, const float *rope_tab, int rope_max_pos,
                            float scale, float *out, float *lse, void *ws, size_t ws_bytes,
                            const gva_decode_opts *opts) {
    return decode_call(stream, d, q_nope, q_rope, M, seq_len, cache, rope_tab, rope_max_pos,
                       scale, out, lse, ws, ws_bytes, opts, nullptr);
}

int gva_decode_attention(void *stream, const gva_dims *d, const void *q_nope, const void *q_rope,
                         const float *M, const int *seq_len, const gva_cache *cache,
                         const float *rope_tab, int rope_max_pos, float scale, float *out,
                         float *lse, void *ws, size_t ws_bytes) {
    return gva_decode_attention_ex(stream, d, q_nope, q_rope, M, seq_len, cache, rope_tab,
                                   rope_max_pos, scale, out, lse, ws, ws_bytes, nullptr);
}

int gva_decode_step(void *stream, const gva_dims *d, int n_layers, const gva_layer_args *layers,
                    const int *pos, const int *seq_len, const float *rope_tab, int rope_max_pos,
                    float scale, void *ws, size_t ws_bytes, const gva_decode_opts *opts) {
    if (n_layers < 0 || (n_layers > 0 && !layers)) return GVA_ERR_ARG;
    for (int l = 0; l < n_layers; ++l) {
        const gva_layer_args &L = layers[l];
        const StepAppend app{L.v_new, L.k_rope_new, pos};
        const int st = decode_call(stream, d, L.q_nope, L.q_rope, L.M, seq_len, &L.cache,
                                   rope_tab, rope_max_pos, scale, L.out, L.lse, ws, ws_bytes,
                                   opts, L.v_new ? &app : nullptr);
        if (st != GVA_OK) return st;
    }
    return GVA_OK;
}

struct gva_step_plan {
    int device;
    cudaStream_t stream;      // private stream the step was recorded on
    cudaGraph_t graph;
    cudaGraphExec_t exec;
};

namespace {
void plan_release(gva_step_plan *p) {
    if (!p) return;
    if (p->exec) cudaGraphExecDestroy(p->exec);
    if (p->graph) cudaGraphDestroy(p->graph);
    if (p->stream) cudaStreamDestroy(p->stream);
    delete p;
}
}  // namespace

extern "C++" {
// Records the calls `issue` makes on a private stream into an instantiated graph.
template <typename Issue>
int plan_record(Issue &&issue, gva_step_plan **plan_out) {
    // the one-time set-up (kernel attributes, SM count) must not happen inside a capture
    if (!device_state()) return GVA_ERR_CUDA;
    gva_step_plan *p = new (std::nothrow) gva_step_plan{};
    if (!p) return GVA_ERR_CUDA;
    cudaError_t e = cudaGetDevice(&p->device);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->stream, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamBeginCapture(p->stream, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        plan_release(p);
        return GVA_ERR_CUDA;
    }
    const int st = issue(p->stream);
    e = cudaStreamEndCapture(p->stream, &p->graph);
    if (st != GVA_OK || e != cudaSuccess) {
        if (e != cudaSuccess) g_last_cuda_error = (int)e;
        cudaGetLastError();
        plan_release(p);
        return st != GVA_OK ? st : GVA_ERR_CUDA;
    }
    e = cudaGraphInstantiate(&p->exec, p->graph, 0);
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        plan_release(p);
        return GVA_ERR_CUDA;
    }
    *plan_out = p;
    return GVA_OK;
}
}  // extern "C++"

int gva_step_plan_create(const gva_dims *d, int n_layers, const gva_layer_args *layers,
                         const int *pos, const int *seq_len, const float *rope_tab,
                         int rope_max_pos, float scale, void *ws, size_t ws_bytes,
                         const gva_decode_opts *opts, gva_step_plan **plan_out) {
    if (!plan_out) return GVA_ERR_ARG;
    *plan_out = nullptr;
    if (n_layers < 1 || !layers) return GVA_ERR_ARG;
    return plan_record(
        [&](cudaStream_t s) {
            return gva_decode_step(s, d, n_layers, layers, pos, seq_len, rope_tab, rope_max_pos,
                                   scale, ws, ws_bytes, opts);
        },
        plan_out);
}

int gva_prefill_plan_create(const gva_dims *d, int n, int n_layers,
                            const gva_prefill_layer_args *layers, const int *L0,
                            const float *rope_tab, int rope_max_pos, float scale, void *ws,
                            size_t ws_bytes, const gva_decode_opts *opts,
                            gva_step_plan **plan_out) {
    if (!plan_out) return GVA_ERR_ARG;
    *plan_out = nullptr;
    if (n < 1 || n_layers < 1 || !layers) return GVA_ERR_ARG;
    return plan_record(
        [&](cudaStream_t s) {
            for (int l = 0; l < n_layers; ++l) {
                const gva_prefill_layer_args &L = layers[l];
                const int st = gva_prefill_attention(s, d, n, L.q_nope, L.q_rope, L.M, L0,
                                                     L.v_new, L.k_rope_new, &L.cache, rope_tab,
                                                     rope_max_pos, scale, L.out, L.lse, ws,
                                                     ws_bytes, opts);
                if (st != GVA_OK) return st;
            }
            return (int)GVA_OK;
        },
        plan_out);
}

int gva_step_plan_launch(gva_step_plan *p, void *stream) {
    if (!p) return GVA_ERR_ARG;
    int dev = -1;
    cudaError_t e = cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &dev);
    if (e == cudaSuccess && dev != p->device) e = cudaErrorInvalidDevice;
    if (e == cudaSuccess) e = cudaGraphLaunch(p->exec, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return GVA_ERR_CUDA;
    }
    return GVA_OK;
}

int gva_step_plan_destroy(gva_step_plan *p) {
    plan_release(p);
    return GVA_OK;
}

// A ragged cache has no view (its rows are not page-aligned): only the tcgen05 prefill,
// which reads the caller's rows, takes it.
bool prefill_takes_ragged(const gva_dims *d, const PrefillPlan &pp) {
    return d->cache_dtype == GVA_BF16 && pp.mq && pp.tcm > 0;
}

size_t gva_prefill_workspace_size(const gva_dims *d, int n, const gva_rows *rows) {
    if (!dims_ok(d, true) || !rows || !rows_ok(rows, d->B)) return 0;
    const bool ragged = rows->layout == GVA_LAYOUT_RAGGED;
    if (!ragged && !prefill_layout_ok(*rows)) return 0;
    const int sms = num_sms_current();
    if (sms <= 0) return 0;
    PrefillPlan pp;
    if (!plan_prefill(d, n, *rows, sms, &pp)) return 0;
    return ragged && !prefill_takes_ragged(d, pp) ? 0 : pp.total;
}

int gva_prefill_attention(void *stream, const gva_dims *d, int n, const void *q_nope,
                          const void *q_rope, const float *M, const int *L0,
                          const float *v_new, const float *k_new, const gva_cache *cache,
                          const float *rope_tab, int rope_max_pos, float scale, float *out,
                          float *lse, void *ws, size_t ws_bytes, const gva_decode_opts *opts) {
    const gva_decode_opts *o = opts ? opts : &kDefaultOpts;
    if (!cache || n < 1 || !dims_ok(d, true) || (long long)d->B * n > MAX_B) return GVA_ERR_ARG;
    if (!rows_ok(&cache->rows, d->B)) return GVA_ERR_ARG;
    if (!out || !aligned16(out) || (lse && !aligned16(lse))) return GVA_ERR_ARG;
    if (!flags_ok(o) || o->path < GVA_PATH_AUTO || o->path > GVA_PATH_MMA || o->num_ctas < 0)
        return GVA_ERR_ARG;
    if (!q_nope || !M || !L0 || !v_new || !cache->V || !aligned16(q_nope) || !aligned16(M) ||
        !aligned16(v_new) || !aligned16(cache->V))
        return GVA_ERR_ARG;
    if (d->d_r > 0 && (!q_rope || !k_new || !cache->K_rope || !rope_tab || rope_max_pos < 1 ||
                       !aligned16(q_rope) || !aligned16(k_new) || !aligned16(cache->K_rope) ||
                       !aligned16(rope_tab)))
        return GVA_ERR_ARG;
    const gva_rows &R = cache->rows;
    const bool ragged = R.layout == GVA_LAYOUT_RAGGED;
    if (!ragged && !prefill_layout_ok(R)) return GVA_ERR_UNSUPPORTED;
    if (ragged && o->path != GVA_PATH_AUTO) return GVA_ERR_UNSUPPORTED;   // the view paths
    if (bind_or_fail(stream) != GVA_OK) return GVA_ERR_CUDA;
    const int sms = num_sms_current();
    if (sms <= 0) return GVA_ERR_CUDA;
    PrefillPlan pp;
    if (!plan_prefill(d, n, R, sms, &pp)) return GVA_ERR_ARG;
    if (ragged && (o->path != GVA_PATH_AUTO || !prefill_takes_ragged(d, pp)))
        return GVA_ERR_UNSUPPORTED;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < pp.total)
        return GVA_ERR_WORKSPACE;
    char *w = static_cast<char *>(ws);
    PrefillViewParams vp;
    vp.B = d->B;
    vp.n = n;
    vp.L0 = L0;
    vp.block_table = R.layout == GVA_LAYOUT_PAGED ? R.block_table : nullptr;
    vp.max_pages = pp.max_pages;
    vp.bt = reinterpret_cast<int *>(w + pp.bt);
    vp.pos = reinterpret_cast<int *>(w + pp.pos);
    vp.len = reinterpret_cast<int *>(w + pp.len);
    gva_rows vr;
    memset(&vr, 0, sizeof(vr));
    vr.layout = GVA_LAYOUT_PAGED;
    vr.block_table = vp.bt;
    vr.max_pages = pp.max_pages;
    if (R.layout == GVA_LAYOUT_PAGED) {
        vr.page_size = R.page_size;
        vr.num_rows = R.num_rows;
    } else {
        vr.page_size = (int)R.T_cap;
        vr.num_rows = (long long)d->B * R.T_cap;
    }
    // a path that cannot run the chunk is refused before anything is appended
    if (o->path == GVA_PATH_MMA && !mma_supported(d)) return GVA_ERR_UNSUPPORTED;
    // The tcgen05 prefill kernel reads the caller's rows: the append and the absorption
    // take each chunk entry's position from L0 themselves, and no view is built.  The
    // other paths run on the view (a decode batch of B n entries).
    const bool tc_path = o->path == GVA_PATH_AUTO && pp.mq && pp.tcm;
    int st;
    if (tc_path) {
        // it also zeroes the prefill kernel's merge tickets
        st = append_launch(stream, &pp.dv, v_new, k_new, nullptr, nullptr, R, cache->V,
                           cache->K_rope, rope_tab, rope_max_pos, L0, n,
                           reinterpret_cast<int *>(w + pp.tk), d->B * d->G);
    } else {
        st = cuda_status(launch(prefill_view_kernel, dim3(d->B, (n + PV_ROWS - 1) / PV_ROWS),
                                dim3(128), 0, stream, vp));
        if (st != GVA_OK) return st;
        st = append_launch(stream, &pp.dv, v_new, k_new, vp.pos, nullptr, vr, cache->V,
                           cache->K_rope, rope_tab, rope_max_pos);
    }
    if (st != GVA_OK) return st;
    if (o->path == GVA_PATH_AUTO && pp.mq) {
        // tensor-core prefill: absorb every (query, head) of the chunk, then one pass
        // over each sequence's rows shared by all its queries, then the merge
        float *qt = reinterpret_cast<float *>(w + pp.dec + pp.dws.qt);
        float *qh = reinterpret_cast<float *>(w + pp.dec + pp.dws.qh);
        st = tc_path ? absorb_launch(stream, &pp.dv, q_nope, q_rope, M, nullptr, rope_tab,
                                     rope_max_pos, scale * LOG2E, qt, qh, sms, &R, false, o, L0, n)
                     : absorb_launch(stream, &pp.dv, q_nope, q_rope, M, vp.len, rope_tab,
                                     rope_max_pos, scale * LOG2E, qt, qh, sms, &vr, false, o);
        if (st != GVA_OK) return st;
        PrefillMmaParams mp;
        mp.B = d->B;
        mp.n = n;
        mp.H = d->H;
        mp.G = d->G;
        mp.r = d->H / d->G;
        mp.L0 = L0;
        mp.R = to_dev(R);
        mp.V = cache->V;
        mp.Kr = cache->K_rope;
        mp.qt = qt;
        mp.qh = qh;
        mp.part_o = reinterpret_cast<float *>(w + pp.po);
        mp.part_ml = reinterpret_cast<float *>(w + pp.pml);
        mp.out = out;
        mp.lse = lse;
        mp.splits = pp.mp.splits;
        mp.wpg = pp.mp.wpg;
        mp.rows_pad = pp.mp.rows_pad;
        mp.vpitch = pp.mp.vpitch;
        mp.stage_bytes = pp.mp.stage_bytes;
        if (pp.tcm) {
            // tcgen05 kernel: 128-token tiles of each sequence's rows through TMA
            PrefillTcParams tp;
            memset(&tp, 0, sizeof(tp));
            tp.p = mp;
            tp.p.splits = pp.tc_splits;
            tp.tickets = reinterpret_cast<int *>(w + pp.tk);   // zeroed by the append
            // the order matters only when the grid takes more than one wave (one CTA per
            // SM): then the longest sequences' ranges should start in the first
            tp.by_length = d->B > 1 && d->B <= PT_ORDER_MAX &&
                                   (long long)pp.tc_splits * d->G * d->B > sms
                               ? 1 : 0;
            tp.ch = R.layout == GVA_LAYOUT_PAGED ? gcd_int(R.page_size, 64) : 64;
            CUtensorMap tv, tk;
            if (!prefill_tc_maps(&tv, &tk, cache->V, cache->K_rope, R.num_rows, d->G * d->d_h,
                                 d->d_r, tp.ch))
                return GVA_ERR_CUDA;
            return cuda_status(prefill_tc_launch(stream, d->d_h, d->d_r, pp.tcm, tp, tv, tk));
        }
        const cudaError_t e = d->d_h == 64 ? prefill_launch_dh<64>(stream, d->d_r, pp.mp, mp)
                                           : prefill_launch_dh<128>(stream, d->d_r, pp.mp, mp);
        return cuda_status(e);
    }
    gva_cache vc;
    vc.rows = vr;
    vc.V = cache->V;
    vc.K_rope = cache->K_rope;
    return gva_decode_attention_ex(stream, &pp.dv, q_nope, q_rope, M, vp.len, &vc, rope_tab,
                                   rope_max_pos, scale, out, lse, w + pp.dec, ws_bytes - pp.dec,
                                   o);
}

int gva_gqa_decode_attention(void *stream, const gva_dims *d, const void *q, const int *seq_len,
                             const gva_kv_cache *cache, float scale, float *out, float *lse,
                             void *ws, size_t ws_bytes, const gva_decode_opts *opts) {
    const gva_decode_opts *o = opts ? opts : &kDefaultOpts;
    if (!cache) return GVA_ERR_ARG;
    int st = decode_arg_checks(d, &cache->rows, out, lse, o, false);
    if (st != GVA_OK) return st;
    if (!q || !seq_len || !cache->K || !cache->V || !aligned16(q) || !aligned16(cache->K) ||
        !aligned16(cache->V))
        return GVA_ERR_ARG;
    if (o->flags & GVA_FLAG_QUERY_RMSNORM) return GVA_ERR_UNSUPPORTED;   // GVA decode only
    gva_dims dg = *d;
    dg.d_r = 0;
    const bool mma_ok = mma_supported(&dg);
    if (o->path == GVA_PATH_MMA && !mma_ok) return GVA_ERR_UNSUPPORTED;
    WsPlan plan;
    int sms = 0;
    st = decode_device_checks(stream, d, ws, ws_bytes, &plan, &sms);
    if (st != GVA_OK) return st;
    // the same choice as the GVA decode, so that the comparator runs the same design
    const bool use_mma = o->path == GVA_PATH_MMA || (o->path == GVA_PATH_AUTO && mma_ok);
    char *w = static_cast<char *>(ws);
    DecodeParams dp;
    dp.B = d->B;
    dp.H = d->H;
    dp.G = d->G;
    dp.r = d->H / d->G;
    dp.d_h = d->d_h;
    dp.d_r = 0;
    dp.seq_len = seq_len;
    dp.R = to_dev(cache->rows);
    dp.Kc = cache->K;
    dp.Vc = cache->V;
    dp.Krope = nullptr;
    dp.qc = q;
    dp.qc_f32 = d->q_dtype == GVA_F32;
    dp.qc_scale = scale * LOG2E;
    dp.qr = nullptr;
    dp.q_rope = nullptr;
    dp.qr_f32 = 1;
    dp.rope_tab = nullptr;
    dp.rope_max_pos = 0;
    dp.qr_scale = 0.f;
    dp.out = out;
    dp.lse = lse;
    dp.part_o = reinterpret_cast<float *>(w + plan.po);
    dp.part_ml = reinterpret_cast<float *>(w + plan.pm);
    dp.n_ctas = 0;
    dp.prefix_ws = reinterpret_cast<int *>(w + plan.pf);
    if (use_mma) {
        st = run_mma(stream, dp, cache->rows, sms, o->num_ctas, true, false);
    } else if (d->cache_dtype == GVA_F32) {
        st = run_simt<float, true>(stream, dp, sms, o->num_ctas);
    } else {
        st = run_simt<__nv_bfloat16, true>(stream, dp, sms, o->num_ctas);
    }
    if (st != GVA_OK) return st;
    return launch_combine(stream, dp, cache->rows);
}

// ---------------------------------------------------------------------------- //
// MLA-shaped decode (the comparator with a latent cache)
// ---------------------------------------------------------------------------- //
size_t gva_mla_workspace_size(const gva_mla_dims *d) {
    if (!mla_dims_ok(d)) return 0;
    const int sms = num_sms_current();
    if (sms <= 0) return 0;
    size_t off = 0;
    return mla_ws_bytes(d, sms, &off);
}

int gva_mla_decode_attention(void *stream, const gva_mla_dims *d, const void *q_nope,
                             const void *q_rope, const float *W_uk, const float *W_uv,
                             const int *seq_len, const gva_cache *cache, const float *rope_tab,
                             int rope_max_pos, float scale, float *out, float *lse, void *ws,
                             size_t ws_bytes) {
    if (!mla_dims_ok(d) || !cache || !rows_ok(&cache->rows, d->B)) return GVA_ERR_ARG;
    if (!out || !aligned16(out) || (lse && !aligned16(lse))) return GVA_ERR_ARG;
    if (!q_nope || !W_uk || !W_uv || !seq_len || !cache->V || !aligned16(q_nope) ||
        !aligned16(W_uk) || !aligned16(W_uv) || !aligned16(cache->V))
        return GVA_ERR_ARG;
    if (d->d_r > 0 && (!q_rope || !cache->K_rope || !rope_tab || rope_max_pos < 1 ||
                       !aligned16(q_rope) || !aligned16(cache->K_rope) || !aligned16(rope_tab)))
        return GVA_ERR_ARG;
    if (d->cache_dtype != GVA_BF16) return GVA_ERR_UNSUPPORTED;   // tensor-core kernel only
    if (bind_or_fail(stream) != GVA_OK) return GVA_ERR_CUDA;
    const int sms = num_sms_current();
    if (sms <= 0) return GVA_ERR_CUDA;
    size_t off_lat = 0;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 ||
        ws_bytes < mla_ws_bytes(d, sms, &off_lat))
        return GVA_ERR_WORKSPACE;
    const gva_dims g = mla_as_gva(d);
    const WsPlan plan = plan_ws(&g, sms);
    char *w = static_cast<char *>(ws);
    float *qt = reinterpret_cast<float *>(w + plan.qt);
    float *qh = reinterpret_cast<float *>(w + plan.qh);
    float *o_lat = reinterpret_cast<float *>(w + off_lat);
    // 1. q~_h = scale log2(e) q_nope W_uk_h^T (width d_c); the decode rotates q_rope itself
    int st = absorb_launch(stream, &g, q_nope, q_rope, W_uk, seq_len, rope_tab, rope_max_pos,
                           scale * LOG2E, qt, qh, sms, &cache->rows, true, nullptr);
    if (st != GVA_OK) return st;
    // 2. split-K attention over the latent rows, 3. log-sum-exp merge into o_lat
    DecodeParams dp;
    memset(&dp, 0, sizeof(dp));
    dp.B = d->B;
    dp.H = d->H;
    dp.G = d->H / 4;
    dp.r = 4;
    dp.d_h = d->d_c;
    dp.d_r = d->d_r;
    dp.seq_len = seq_len;
    dp.R = to_dev(cache->rows);
    dp.Kc = cache->V;
    dp.Vc = cache->V;
    dp.Krope = cache->K_rope;
    dp.qc = qt;
    dp.qc_f32 = 1;
    dp.qc_scale = 1.f;
    dp.qr = nullptr;
    dp.q_rope = q_rope;
    dp.qr_f32 = d->q_dtype == GVA_F32;
    dp.rope_tab = rope_tab;
    dp.rope_max_pos = rope_max_pos;
    dp.qr_scale = scale * LOG2E;
    dp.out = o_lat;
    dp.lse = lse;
    dp.part_o = reinterpret_cast<float *>(w + plan.po);
    dp.part_ml = reinterpret_cast<float *>(w + plan.pm);
    dp.prefix_ws = reinterpret_cast<int *>(w + plan.pf);
    st = run_mma(stream, dp, cache->rows, sms, 0, false, true, true);
    if (st != GVA_OK) return st;
    st = launch_combine(stream, dp, cache->rows);
    if (st != GVA_OK) return st;
    // 4. out[b,h] = o_lat[b,h] W_uv_h
    UpProjParams up;
    up.B = d->B;
    up.H = d->H;
    up.d_c = d->d_c;
    up.d_h = d->d_h;
    up.o_lat = o_lat;
    up.Wuv = W_uv;
    up.out = out;
    return cuda_status(launch(mla_up_kernel, dim3(d->H, (d->B + UP_SEQ - 1) / UP_SEQ),
                              dim3(UP_THREADS), mla_up_smem_bytes(d->d_c), stream, up));
}

// ---------------------------------------------------------------------------- //
// Decode with ordinary RoPE on the reconstructed key (M_h not absorbable)
// ---------------------------------------------------------------------------- //
size_t gva_rope_keys_workspace_size(const gva_dims *d) {
    if (!rk_dims_ok(d)) return 0;
    const int sms = num_sms_current();
    if (sms <= 0) return 0;
    return rk_plan(d, sms).total;
}

int gva_rope_keys_decode_attention(void *stream, const gva_dims *d, const void *q, const float *M,
                                   const int *seq_len, const gva_cache *cache,
                                   const float *rope_tab, int rope_max_pos, float scale,
                                   float *out, float *lse, void *ws, size_t ws_bytes) {
    if (!rk_dims_ok(d) || !cache || !rows_ok(&cache->rows, d->B)) return GVA_ERR_ARG;
    if (!q || !M || !seq_len || !cache->V || !rope_tab || !out) return GVA_ERR_ARG;
    if (!aligned16(q) || !aligned16(M) || !aligned16(cache->V) || !aligned16(rope_tab) ||
        !aligned16(out) || (lse && !aligned16(lse)))
        return GVA_ERR_ARG;
    if (rope_max_pos < RK_TILE || !std::isfinite(scale)) return GVA_ERR_ARG;
    if (!rk_supported(d)) return GVA_ERR_UNSUPPORTED;
    if (bind_or_fail(stream) != GVA_OK) return GVA_ERR_CUDA;
    const int sms = num_sms_current();
    if (sms <= 0) return GVA_ERR_CUDA;
    const RkWs w = rk_plan(d, sms);
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < w.total)
        return GVA_ERR_WORKSPACE;
    char *wb = static_cast<char *>(ws);
    RkParams p;
    memset(&p, 0, sizeof(p));
    p.B = d->B;
    p.H = d->H;
    p.G = d->G;
    p.r = d->H / d->G;
    p.d_h = d->d_h;
    p.d_n = d->d_n;
    p.hc = w.hc;
    p.nhs = w.nhs;
    p.seq_len = seq_len;
    p.R = to_dev(cache->rows);
    p.q = q;
    p.q_f32 = d->q_dtype == GVA_F32;
    p.M = M;
    p.tab = rope_tab;
    p.tab_rows = rope_max_pos;
    p.scale_log2 = scale * LOG2E;
    p.img = reinterpret_cast<unsigned char *>(wb + w.img);
    p.Ls = reinterpret_cast<int *>(wb + w.ls);
    p.pre = reinterpret_cast<int *>(wb + w.pre);
    p.part_o = reinterpret_cast<float *>(wb + w.po);
    p.part_ml = reinterpret_cast<float *>(wb + w.pm);
    p.out = out;
    p.lse = lse;
    p.n_ctas = sms < RK_MAX_PARTS ? sms : RK_MAX_PARTS;
    p.ch = cache->rows.layout == GVA_LAYOUT_PAGED ? gcd_int(cache->rows.page_size, 64) : 64;
    CUtensorMap tv;
    if (!rk_make_map(&tv, cache->V, cache->rows.num_rows, d->G * d->d_h, p.ch)) return GVA_ERR_CUDA;
    int st = cuda_status(launch(rk_prep_kernel, dim3(d->B * d->H * (d->d_h / 8) + 1),
                                dim3(RK_PREP_THREADS), 0,
                                stream, p));
    if (st != GVA_OK) return st;
    st = rk_launch_decode(stream, p, tv);
    if (st != GVA_OK) return st;
    return cuda_status(launch(rk_merge_kernel, dim3(d->B * d->H), dim3(RK_MERGE_THREADS), 0,
                              stream, p));
}

// ---------------------------------------------------------------------------- //
// Decode without a caller-provided workspace.
//
// For callers that cannot allocate device memory at the point where they decode:
// plugins and embedded runtimes that are handed no allocator and no scratch buffer,
// engines whose device memory is planned once at start-up and may not grow, and
// latency-critical loops that forbid allocator calls because those can block or
// synchronise the device.  The scratch lives in one fixed-size array in device memory
// that every GPU loading this library holds until the process exits.
// ---------------------------------------------------------------------------- //
static __device__ __align__(256) unsigned char g_static_scratch[GVA_STATIC_SCRATCH_BYTES];

static void *g_static_scratch_ptr[MAX_DEVICES];   // device address, per device
static std::mutex g_static_scratch_mu;

// Resolve the array's device address once per device, with that device current.
// Host code must not hand `g_static_scratch` itself to a kernel: on the host the name
// is a stand-in, not a device address.
static void *static_scratch_for_device(int dev) {
    if (dev < 0 || dev >= MAX_DEVICES) return nullptr;
    std::lock_guard<std::mutex> lk(g_static_scratch_mu);
    if (!g_static_scratch_ptr[dev]) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess) {
            g_last_cuda_error = (int)e;
            cudaGetLastError();
            return nullptr;
        }
        g_static_scratch_ptr[dev] = ptr;
    }
    return g_static_scratch_ptr[dev];
}

int gva_decode_attention_static(void *stream, const gva_dims *d, const void *q_nope,
                                const void *q_rope, const float *M, const int *seq_len,
                                const gva_cache *cache, const float *rope_tab, int rope_max_pos,
                                float scale, float *out, float *lse) {
    if (!dims_ok(d, true)) return GVA_ERR_ARG;
    if (bind_or_fail(stream) != GVA_OK) return GVA_ERR_CUDA;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess && stream != nullptr) {
        // the scratch handed to the kernels must be the stream's device's own copy.  A
        // capturing stream cannot be asked for its device; the output buffer, which the
        // kernels write on that device, stands for it then.
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        e = cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cs);
        int sdev = -1;
        if (e == cudaSuccess && cs == cudaStreamCaptureStatusNone) {
            e = cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev);
        } else if (e == cudaSuccess) {
            cudaPointerAttributes pa;
            e = cudaPointerGetAttributes(&pa, out);
            if (e == cudaSuccess && pa.type != cudaMemoryTypeDevice) e = cudaErrorInvalidValue;
            sdev = pa.device;
        }
        if (e == cudaSuccess && sdev != dev) e = cudaErrorInvalidDevice;
    }
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        cudaGetLastError();
        return GVA_ERR_CUDA;
    }
    const size_t need = gva_decode_workspace_size(d);
    if (need == 0) return GVA_ERR_CUDA;
    if (need > (size_t)GVA_STATIC_SCRATCH_BYTES) return GVA_ERR_WORKSPACE;  // beyond the fixed maximum
    void *ws = static_scratch_for_device(dev);
    if (!ws) return GVA_ERR_CUDA;
    // The automatic path writes every scratch value it reads within the call, so nothing
    // in the array has to start at any particular value.
    return gva_decode_attention_ex(stream, d, q_nope, q_rope, M, seq_len, cache, rope_tab,
                                   rope_max_pos, scale, out, lse, ws,
                                   (size_t)GVA_STATIC_SCRATCH_BYTES, nullptr);
}

#ifdef GVA_TRACE
// Debug builds only: copy / clear the per-CTA cycle timeline of the tensor-core decode.
int gva_debug_trace_read(long long *host, int n) {
    if (n > TRACE_CTAS * TRACE_SLOTS) n = TRACE_CTAS * TRACE_SLOTS;
    return cudaMemcpyFromSymbol(host, g_trace, sizeof(long long) * n) == cudaSuccess ? GVA_OK
                                                                                    : GVA_ERR_CUDA;
}
int gva_debug_trace_clear(void) {
    static long long zeros[TRACE_CTAS * TRACE_SLOTS];
    unsigned long long lo[16], hi[16];
    for (int i = 0; i < 16; ++i) { lo[i] = ~0ull; hi[i] = 0ull; }
    const bool ok = cudaMemcpyToSymbol(g_trace, zeros, sizeof(zeros)) == cudaSuccess &&
                    cudaMemcpyToSymbol(g_kt_min, lo, sizeof(lo)) == cudaSuccess &&
                    cudaMemcpyToSymbol(g_kt_max, hi, sizeof(hi)) == cudaSuccess;
    return ok ? GVA_OK : GVA_ERR_CUDA;
}
int gva_debug_cta_read(unsigned long long *host, int n) {
    if (n > 4096) n = 4096;
    return cudaMemcpyFromSymbol(host, g_cta_t, sizeof(unsigned long long) * 4 * n) == cudaSuccess
               ? GVA_OK : GVA_ERR_CUDA;
}
// kernel event log: n records of (tag, time); returns the count written (capped)
int gva_debug_rec_read(unsigned long long *host, int n) {
    unsigned cnt = 0;
    if (cudaMemcpyFromSymbol(&cnt, g_rec_n, sizeof(cnt)) != cudaSuccess) return -1;
    if (cnt > (1u << 16)) cnt = 1u << 16;
    if ((int)cnt < n) n = (int)cnt;
    if (n > 0 && cudaMemcpyFromSymbol(host, g_rec, sizeof(unsigned long long) * 2 * n) != cudaSuccess)
        return -1;
    return n;
}
int gva_debug_rec_clear(void) {
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_rec_n, &zero, sizeof(zero)) == cudaSuccess ? GVA_OK : GVA_ERR_CUDA;
}
// [0..16) earliest, [16..32) latest global-timer reading per timeline slot
int gva_debug_kt_read(unsigned long long *host) {
    const bool ok = cudaMemcpyFromSymbol(host, g_kt_min, 16 * 8) == cudaSuccess &&
                    cudaMemcpyFromSymbol(host + 16, g_kt_max, 16 * 8) == cudaSuccess;
    return ok ? GVA_OK : GVA_ERR_CUDA;
}
#endif

int gva_get_device_status(int *code_out) {
    int v = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, g_status, sizeof(int));
    const int zero = 0;
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
    if (code_out) *code_out = v;
    if (e != cudaSuccess) return GVA_ERR_CUDA;
    return v == 0 ? GVA_OK : GVA_ERR_DEVICE_CHECK;
}

}  // extern "C"
