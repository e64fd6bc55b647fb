// Host side of the C ABI: argument validation, plane and workspace layout,
// act-order resolution, the M-based dispatcher and the entry points.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <new>
#include <vector>

#include "pq_internal.cuh"

namespace {
thread_local char g_last_error[512] = "";
}

namespace pq {

int32_t fail(int32_t code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return code;
}

int32_t cuda_fail(cudaError_t e, const char* where) {
    return fail(PQ_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

int npad(int N) { return (N + kStrip - 1) / kStrip * kStrip; }

int w2_bp(int K) { return (K / kGroup + 7) / 8 * 8; }

Planes plane_layout(const pq_desc& d) {
    Planes l = {};
    const size_t Np = (size_t)npad(d.N), K = (size_t)d.K, G = K / kGroup;
    size_t off = 0;
    if (d.fmt == PQ_FMT_W4_AFFINE) {
        const size_t GA = K / kAffineGroup;
        l.codes_off = off;
        off = align_up(off + Np * (K / 2), kAlign);
        l.scales_off = off;
        off = align_up(off + GA * Np * 2, kAlign);
        l.biases_off = off;
        off = align_up(off + GA * Np * 2, kAlign);
        l.zeros_off = l.perm_off = off;
        l.total = off;
        return l;
    }
    l.codes_off = off;
    off = align_up(off + Np * (d.fmt == PQ_FMT_W4_GPTQ ? K / 2 : K / 4), kAlign);
    l.scales_off = off;
    // W4: [G][Npad]; W2: [Npad][Bp] (each row's block scales padded to whole 16-byte chunks)
    off = align_up(off + (d.fmt == PQ_FMT_W4_GPTQ ? G * Np * 2 : Np * (size_t)w2_bp(d.K) * 2), kAlign);
    l.zeros_off = off;
    if (d.fmt == PQ_FMT_W4_GPTQ && d.zp == PQ_ZP_EXPLICIT_U8) off = align_up(off + G * Np, kAlign);
    l.perm_off = off;
    if (d.fmt == PQ_FMT_W4_GPTQ && d.has_gidx) off = align_up(off + K * 4, kAlign);
    l.total = off;
    return l;
}

Workspace workspace_layout(const pq_desc& d) {
    Workspace w = {};
    const size_t M = (size_t)d.max_m, K = (size_t)d.K;
    size_t off = 0;
    w.status_off = off;
    w.flags_off = 256;
    off = align_up(kWsFixedBytes, kAlign);
    w.xg_off = off;
    if (d.fmt == PQ_FMT_W4_GPTQ && d.has_gidx) off = align_up(off + M * K * 2, kAlign);
    w.sk_off = off;
    w.sk_bytes = (size_t)split_k_slices(d) * npad(d.N) * 16 * 4;
    off = align_up(off + w.sk_bytes, kAlign);
    w.gp_off = off;
    w.gp_rows = gemm_partial_rows(d.max_m);
    w.gp_bytes = w.gp_rows ? (size_t)2 * kGemmMaxCtas * w.gp_rows * kGemmTileCols * 4 : 0;
    off = align_up(off + w.gp_bytes, kAlign);
    w.q_off = w.xs_off = w.sq_off = w.qa_off = off;
    if (d.fmt == PQ_FMT_W2_PQ2) {
        w.q_off = off;
        off = align_up(off + M * K, kAlign);
        w.xs_off = off;
        off = align_up(off + M * (K / (size_t)d.act_group) * 4, kAlign);
        w.sq_off = off;
        off = align_up(off + M * (K / kGroup) * 4, kAlign);
        w.qa_off = off;
        off = align_up(off + M * K * 2, kAlign);
    } else if (d.fmt == PQ_FMT_W4_AFFINE && d.max_m > kActDecodeMaxM) {
        // the GEMM's sums of x over every 64-group
        w.xs_off = off;
        off = align_up(off + M * (K / kAffineGroup) * 4, kAlign);
    }
    w.total = off;
    return w;
}

ActLayout act_layout(const pq_desc& d, int M) {
    ActLayout l = {};
    const size_t m = (size_t)M, K = (size_t)d.K;
    size_t off = 0;
    l.q8_off = off;
    if (!act_codes_bf16(M)) off = align_up(off + m * K, kAlign);
    l.xs_off = off;
    off = align_up(off + m * (K / (size_t)d.act_group) * 4, kAlign);
    l.sq_off = off;
    off = align_up(off + m * (K / kGroup) * 4, kAlign);
    l.qa_off = off;
    if (act_codes_bf16(M)) off = align_up(off + m * K * 2, kAlign);
    l.total = off;
    return l;
}

static ActPlanes act_planes(const pq_desc& d, int M, void* base) {
    const ActLayout l = act_layout(d, M);
    uint8_t* b = static_cast<uint8_t*>(base);
    ActPlanes a;
    a.q8 = reinterpret_cast<int8_t*>(b + l.q8_off);
    a.qa = reinterpret_cast<uint16_t*>(b + l.qa_off);
    a.sq = reinterpret_cast<int32_t*>(b + l.sq_off);
    a.xs = reinterpret_cast<float*>(b + l.xs_off);
    return a;
}

static int32_t validate_desc(const pq_desc* d) {
    if (!d) return fail(PQ_ERR_INVALID_ARG, "descriptor is NULL");
    if (d->fmt != PQ_FMT_W4_GPTQ && d->fmt != PQ_FMT_W2_PQ2 && d->fmt != PQ_FMT_W4_AFFINE)
        return fail(PQ_ERR_INVALID_ARG, "fmt %d is not PQ_FMT_W4_GPTQ, PQ_FMT_W2_PQ2 or PQ_FMT_W4_AFFINE", d->fmt);
    if (d->N < 1) return fail(PQ_ERR_SHAPE, "N = %d must be >= 1", d->N);
    if (d->K < kGroup || d->K % kGroup)
        return fail(PQ_ERR_SHAPE, "K = %d must be a positive multiple of 128", d->K);
    if (d->fmt == PQ_FMT_W4_AFFINE) {
        if (d->group != kAffineGroup)
            return fail(PQ_ERR_UNSUPPORTED, "group = %d; the affine 4-bit format takes 64", d->group);
    } else if (d->group != kGroup) {
        return fail(PQ_ERR_UNSUPPORTED, "group = %d; only 128 is supported", d->group);
    }
    if (d->act_dtype != PQ_F16 && d->act_dtype != PQ_BF16)
        return fail(PQ_ERR_INVALID_ARG, "act_dtype %d is not PQ_F16 or PQ_BF16", d->act_dtype);
    if (d->out_dtype != PQ_F16 && d->out_dtype != PQ_BF16)
        return fail(PQ_ERR_INVALID_ARG, "out_dtype %d is not PQ_F16 or PQ_BF16", d->out_dtype);
    if (d->max_m < 1 || d->max_m > (1 << 20))
        return fail(PQ_ERR_SHAPE, "max_m = %d must lie in 1..2^20", d->max_m);
    if ((int64_t)d->N * d->K > (int64_t)1 << 36)
        return fail(PQ_ERR_SHAPE, "N*K = %lld exceeds 2^36", (long long)d->N * d->K);
    if (d->fmt == PQ_FMT_W4_AFFINE) {
        if (d->zp != PQ_ZP_SYMMETRIC_8)
            return fail(PQ_ERR_ZP_CONVENTION, "the affine 4-bit format has biases, not zero points; zp must be PQ_ZP_SYMMETRIC_8");
        if (d->has_gidx) return fail(PQ_ERR_UNSUPPORTED, "the affine 4-bit format has no act order");
    } else if (d->fmt == PQ_FMT_W4_GPTQ) {
        if (d->zp != PQ_ZP_SYMMETRIC_8 && d->zp != PQ_ZP_EXPLICIT_U8)
            return fail(PQ_ERR_INVALID_ARG, "zp %d is not a PQ_ZP_* convention", d->zp);
        if (d->has_gidx != 0 && d->has_gidx != 1)
            return fail(PQ_ERR_INVALID_ARG, "has_gidx must be 0 or 1");
    } else {
        if (d->zp != PQ_ZP_SYMMETRIC_8)
            return fail(PQ_ERR_ZP_CONVENTION, "ternary PQ2 has no zero points; zp must be PQ_ZP_SYMMETRIC_8");
        if (d->has_gidx) return fail(PQ_ERR_UNSUPPORTED, "ternary PQ2 has no act order");
        if (d->act_group != kGroup && d->act_group != d->K)
            return fail(PQ_ERR_UNSUPPORTED, "act_group = %d must be 128 or K (%d)", d->act_group, d->K);
        // the activation quantiser stages one row (K * 2 bytes) in shared memory
        if (d->K > 65536) return fail(PQ_ERR_UNSUPPORTED, "ternary PQ2 needs K <= 65536, got K = %d", d->K);
    }
    return PQ_OK;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

static int32_t begin_handle(const pq_desc* d, void* d_prepared, size_t prepared_bytes,
                            void* d_ws, size_t ws_bytes, pq_prepared** out,
                            pq_prepared** made) {
    if (!out) return fail(PQ_ERR_INVALID_ARG, "out handle pointer is NULL");
    *out = nullptr;
    if (!d_prepared) return fail(PQ_ERR_INVALID_ARG, "prepared buffer is NULL");
    if (!d_ws) return fail(PQ_ERR_INVALID_ARG, "workspace buffer is NULL");
    if (((uintptr_t)d_prepared & (kAlign - 1)) || ((uintptr_t)d_ws & (kAlign - 1)))
        return fail(PQ_ERR_ALIGN, "prepared and workspace buffers must be 256-byte aligned");
    Planes pl = plane_layout(*d);
    Workspace wl = workspace_layout(*d);
    if (prepared_bytes < pl.total)
        return fail(PQ_ERR_BUFFER_TOO_SMALL, "prepared buffer has %zu bytes, needs %zu", prepared_bytes, pl.total);
    if (ws_bytes < wl.total)
        return fail(PQ_ERR_BUFFER_TOO_SMALL, "workspace has %zu bytes, needs %zu", ws_bytes, wl.total);
    pq_prepared* p = new (std::nothrow) pq_prepared();
    if (!p) return fail(PQ_ERR_INVALID_ARG, "host allocation of the handle failed");
    p->d = *d;
    p->Npad = npad(d->N);
    p->G = d->K / kGroup;
    uint8_t* base = static_cast<uint8_t*>(d_prepared);
    p->base = base;
    p->codes = base + pl.codes_off;
    p->scales = reinterpret_cast<uint16_t*>(base + pl.scales_off);
    p->zeros = (d->fmt == PQ_FMT_W4_GPTQ && d->zp == PQ_ZP_EXPLICIT_U8) ? base + pl.zeros_off : nullptr;
    p->perm = (d->fmt == PQ_FMT_W4_GPTQ && d->has_gidx) ? reinterpret_cast<int32_t*>(base + pl.perm_off) : nullptr;
    p->biases = d->fmt == PQ_FMT_W4_AFFINE ? reinterpret_cast<uint16_t*>(base + pl.biases_off) : nullptr;
    p->ws = static_cast<uint8_t*>(d_ws);
    p->ws_bytes = ws_bytes;
    p->wl = wl;
    p->status = reinterpret_cast<uint32_t*>(p->ws + wl.status_off);
    p->gemm_state = nullptr;
    cudaError_t e = cudaGetDevice(&p->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
    if (e != cudaSuccess) { delete p; return cuda_fail(e, "device query"); }
    *made = p;
    return PQ_OK;
}

static int32_t finish_handle(pq_prepared* p, cudaStream_t s, pq_prepared** out) {
    // the status word and the GEMM's shared-tile flags start at zero; every
    // launch leaves the flags zero
    cudaError_t e = cudaMemsetAsync(p->ws, 0, kWsFixedBytes, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) { pq::gemm_free(p); delete p; return cuda_fail(e, "prepare"); }
    if (gemm_supported(p->d)) {
        int32_t rc = gemm_init(p);
        if (rc != PQ_OK) { delete p; return rc; }
    }
    *out = p;
    return PQ_OK;
}

// Dispatcher: M-based variant choice (pure function of desc, M, SM count).
static int32_t choose_variant(const pq_desc& d, int M) {
    if (d.fmt == PQ_FMT_W4_GPTQ || d.fmt == PQ_FMT_W4_AFFINE) {
        if (M <= 16) return PQ_VARIANT_W4_GEMV;
        return gemm_supported(d) ? PQ_VARIANT_W4_GEMM : PQ_VARIANT_W4_GEMV;
    }
    // one token: the fused CUDA-core kernel; two: the quantise pre-pass and
    // the CUDA-core kernel; 3..16: the cluster split-K decode (one launch,
    // quantiser in the cluster).  Measured on GB300 over the 7B projection
    // shapes (per call, CUDA graphs of 8 layers): at M = 2 the pre-pass
    // path 6.4 / 10.0 / 10.8 us (4096 x 4096 / 11008 x 4096 / 4096 x 11008)
    // against 6.4 / 11.0 / 11.9 for the cluster decode; at M = 4 9.3 / 13.5 /
    // 17.1 for the int8 split-K path against 6.5 / 11.2 / 12.3; at M = 16
    // 9.0 / 15.0 / 17.3 for the bf16 split-K path against 8.5 / 13.9 / 16.0.
    // Longer rows than the cluster holds take the split-K paths.
    if (M == 1 && w2_gemv_fits(d, M, true)) return PQ_VARIANT_W2_GEMV_FUSED;
    if (M == 2 && w2_gemv_fits(d, M, false)) return PQ_VARIANT_W2_GEMV;
    if (M <= 16 && w2_cl_fits(d, M)) return PQ_VARIANT_W2_GEMV_CL;
    if (M <= 8 && split_k_slices(d) > 0) return PQ_VARIANT_W2_GEMV_TC;
    if (M <= 16 && split_k_slices(d) > 0) return PQ_VARIANT_W2_GEMV_BF;
    if (M <= 16 && w2_gemv_fits(d, M, false)) return PQ_VARIANT_W2_GEMV;
    return gemm_supported(d) ? PQ_VARIANT_W2_GEMM : PQ_VARIANT_W2_GEMV;
}

static bool variant_runs(const pq_desc& d, int M, int v) {
    switch (v) {
        case PQ_VARIANT_W4_GEMV:
            return d.fmt == PQ_FMT_W4_GPTQ || (d.fmt == PQ_FMT_W4_AFFINE && w4_affine_runs(d, M));
        case PQ_VARIANT_W4_GEMM:
            // affine layers need the sums of x, which the workspace holds when max_m > 16
            return (d.fmt == PQ_FMT_W4_GPTQ || (d.fmt == PQ_FMT_W4_AFFINE && d.max_m > kActDecodeMaxM)) &&
                   gemm_supported(d);
        case PQ_VARIANT_W2_GEMV_FUSED: return d.fmt == PQ_FMT_W2_PQ2 && w2_gemv_fits(d, M, true);
        case PQ_VARIANT_W2_GEMV: return d.fmt == PQ_FMT_W2_PQ2 && w2_gemv_fits(d, M, false);
        case PQ_VARIANT_W2_GEMM: return d.fmt == PQ_FMT_W2_PQ2 && gemm_supported(d);
        case PQ_VARIANT_W2_GEMV_TC: return d.fmt == PQ_FMT_W2_PQ2 && M <= 16 && split_k_slices(d) > 0;
        case PQ_VARIANT_W2_GEMV_BF: return d.fmt == PQ_FMT_W2_PQ2 && M <= 16 && split_k_slices(d) > 0;
        case PQ_VARIANT_W2_GEMV_CL: return w2_cl_fits(d, M);
        default: return false;
    }
}

// The kernels that run on quantised activations held by the caller, the
// same choice as pq_linear makes: for M <= 2 the buffer holds int8
// plane-order codes (the CUDA-core GEMV without its fused quantiser; the
// int8 split-K decode for rows it cannot hold), for M = 3..16 bf16 codes in
// tensor-core order (the cluster decode without its quantiser; the bf16
// split-K decode for rows too long for the cluster), above that the same
// bf16 codes for the GEMM.  -1: none runs for (d, M).
static int act_variant(const pq_desc& d, int M) {
    if (M > kActDecodeMaxM) return gemm_supported(d) ? PQ_VARIANT_W2_GEMM : -1;
    if (act_codes_bf16(M)) {
        if (w2_cl_fits(d, M)) return PQ_VARIANT_W2_GEMV_CL;
        return split_k_slices(d) > 0 ? PQ_VARIANT_W2_GEMV_BF : (gemm_supported(d) ? PQ_VARIANT_W2_GEMM : -1);
    }
    if (w2_gemv_fits(d, M, false)) return PQ_VARIANT_W2_GEMV;
    if (split_k_slices(d) > 0) return PQ_VARIANT_W2_GEMV_TC;
    return -1;
}

}  // namespace pq

using namespace pq;

extern "C" {

const char* pq_last_error(void) { return g_last_error; }

size_t pq_prepared_bytes(const pq_desc* d) {
    if (validate_desc(d) != PQ_OK) return 0;
    return plane_layout(*d).total;
}

size_t pq_workspace_bytes(const pq_desc* d) {
    if (validate_desc(d) != PQ_OK) return 0;
    return workspace_layout(*d).total;
}

int32_t pq_prepare_w4(const pq_desc* d, const uint32_t* d_qweight, const uint16_t* d_scales,
                      const uint8_t* d_zeros, const int32_t* h_g_idx, void* d_prepared,
                      size_t prepared_bytes, void* d_workspace, size_t workspace_bytes,
                      void* stream, pq_prepared** out) {
    int32_t rc = validate_desc(d);
    if (rc != PQ_OK) return rc;
    if (d->fmt != PQ_FMT_W4_GPTQ) return fail(PQ_ERR_INVALID_ARG, "pq_prepare_w4 needs fmt = PQ_FMT_W4_GPTQ");
    if (!d_qweight || !d_scales) return fail(PQ_ERR_INVALID_ARG, "qweight and scales must be non-NULL");
    if (!aligned16(d_qweight) || !aligned16(d_scales) || (d_zeros && !aligned16(d_zeros)))
        return fail(PQ_ERR_ALIGN, "qweight, scales and zeros must be 16-byte aligned");
    if (d->zp == PQ_ZP_SYMMETRIC_8 && d_zeros)
        return fail(PQ_ERR_ZP_CONVENTION, "zero points supplied but the convention is PQ_ZP_SYMMETRIC_8 (z = 8)");
    if (d->zp == PQ_ZP_EXPLICIT_U8 && !d_zeros)
        return fail(PQ_ERR_ZP_CONVENTION, "convention PQ_ZP_EXPLICIT_U8 needs unpacked uint8 zero points [K/128][N]");
    if (d->has_gidx && !h_g_idx) return fail(PQ_ERR_GIDX, "has_gidx = 1 but g_idx is NULL");
    if (!d->has_gidx && h_g_idx) return fail(PQ_ERR_GIDX, "g_idx supplied but has_gidx = 0");

    std::vector<int32_t> perm;
    if (d->has_gidx) {
        // Act order: every group 0..G-1 must own exactly 128 rows, so that the
        // stable sort by group yields contiguous 128-row runs.
        const int K = d->K, G = K / kGroup;
        std::vector<int32_t> count(G, 0);
        for (int k = 0; k < K; ++k) {
            int32_t g = h_g_idx[k];
            if (g < 0 || g >= G)
                return fail(PQ_ERR_GIDX, "g_idx[%d] = %d lies outside [0, %d)", k, g, G);
            ++count[g];
        }
        for (int g = 0; g < G; ++g)
            if (count[g] != kGroup)
                return fail(PQ_ERR_GIDX, "g_idx group %d has %d rows; every sorted group must be one "
                            "contiguous run of 128 rows", g, count[g]);
        // stable counting sort: rows in ascending k within each group
        std::vector<int32_t> next(G);
        for (int g = 0; g < G; ++g) next[g] = g * kGroup;
        perm.assign(K, 0);
        for (int k = 0; k < K; ++k) perm[next[h_g_idx[k]]++] = k;
    }

    pq_prepared* p = nullptr;
    rc = begin_handle(d, d_prepared, prepared_bytes, d_workspace, workspace_bytes, out, &p);
    if (rc != PQ_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (d->has_gidx)
        e = cudaMemcpyAsync(p->perm, perm.data(), perm.size() * 4, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = launch_prepare_w4(p, d_qweight, d_scales, d_zeros, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);   // perm host buffer lives until here
    if (e != cudaSuccess) { delete p; return cuda_fail(e, "pq_prepare_w4"); }
    return finish_handle(p, s, out);
}

int32_t pq_prepare_w2(const pq_desc* d, const uint8_t* d_raw, size_t row_stride_bytes,
                      void* d_prepared, size_t prepared_bytes, void* d_workspace,
                      size_t workspace_bytes, void* stream, pq_prepared** out) {
    int32_t rc = validate_desc(d);
    if (rc != PQ_OK) return rc;
    if (d->fmt != PQ_FMT_W2_PQ2) return fail(PQ_ERR_INVALID_ARG, "pq_prepare_w2 needs fmt = PQ_FMT_W2_PQ2");
    if (!d_raw) return fail(PQ_ERR_INVALID_ARG, "raw PQ2 rows must be non-NULL");
    const size_t width = (size_t)(d->K / kGroup) * 34;
    if (row_stride_bytes < width)
        return fail(PQ_ERR_SHAPE, "row stride %zu is below the %zu bytes of one row", row_stride_bytes, width);
    pq_prepared* p = nullptr;
    rc = begin_handle(d, d_prepared, prepared_bytes, d_workspace, workspace_bytes, out, &p);
    if (rc != PQ_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_prepare_w2(p, d_raw, row_stride_bytes, s);
    if (e != cudaSuccess) { delete p; return cuda_fail(e, "pq_prepare_w2"); }
    return finish_handle(p, s, out);
}

int32_t pq_prepare_affine4(const pq_desc* d, const uint32_t* d_wq, const uint16_t* d_scales,
                           const uint16_t* d_biases, void* d_prepared, size_t prepared_bytes, void* d_workspace,
                           size_t workspace_bytes, void* stream, pq_prepared** out) {
    int32_t rc = validate_desc(d);
    if (rc != PQ_OK) return rc;
    if (d->fmt != PQ_FMT_W4_AFFINE) return fail(PQ_ERR_INVALID_ARG, "pq_prepare_affine4 needs fmt = PQ_FMT_W4_AFFINE");
    if (!d_wq || !d_scales || !d_biases) return fail(PQ_ERR_INVALID_ARG, "codes, scales and biases must be non-NULL");
    pq_prepared* p = nullptr;
    rc = begin_handle(d, d_prepared, prepared_bytes, d_workspace, workspace_bytes, out, &p);
    if (rc != PQ_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_prepare_affine4(p, d_wq, d_scales, d_biases, s);
    if (e != cudaSuccess) { delete p; return cuda_fail(e, "pq_prepare_affine4"); }
    return finish_handle(p, s, out);
}

int32_t pq_plan(const pq_desc* d, int32_t M, int32_t num_sms, pq_plan_info* out) {
    int32_t rc = validate_desc(d);
    if (rc != PQ_OK) return rc;
    if (!out) return fail(PQ_ERR_INVALID_ARG, "plan output is NULL");
    if (M < 1 || M > d->max_m) return fail(PQ_ERR_SHAPE, "M = %d must lie in 1..max_m (%d)", M, d->max_m);
    if (num_sms < 1) return fail(PQ_ERR_INVALID_ARG, "num_sms = %d must be >= 1", num_sms);
    pq_prepared tmp = {};
    tmp.d = *d;
    tmp.Npad = npad(d->N);
    tmp.G = d->K / kGroup;
    tmp.num_sms = num_sms;
    tmp.wl = workspace_layout(*d);
    memset(out, 0, sizeof *out);
    out->variant = choose_variant(*d, M);
    if (!variant_runs(*d, M, out->variant))
        return fail(PQ_ERR_UNSUPPORTED, "no kernel runs fmt %d at M = %d", d->fmt, M);
    switch (out->variant) {
        case PQ_VARIANT_W4_GEMV: plan_w4_gemv(&tmp, M, out); break;
        case PQ_VARIANT_W2_GEMV_FUSED: plan_w2_gemv(&tmp, M, true, out); break;
        case PQ_VARIANT_W2_GEMV: plan_w2_gemv(&tmp, M, false, out); break;
        case PQ_VARIANT_W2_GEMV_TC: plan_w2_tc(&tmp, M, out); break;
        case PQ_VARIANT_W2_GEMV_BF: plan_w2_bf(&tmp, M, out); break;
        case PQ_VARIANT_W2_GEMV_CL: plan_w2_cl(&tmp, M, out); break;
        default: plan_gemm(&tmp, M, out); break;
    }
    return PQ_OK;
}

int32_t pq_linear_variant(const void* d_x, const pq_prepared* p, void* d_y, int32_t M,
                          int32_t variant, void* stream) {
    if (!p) return fail(PQ_ERR_INVALID_ARG, "handle is NULL");
    if (!d_x || !d_y) return fail(PQ_ERR_INVALID_ARG, "x and y must be non-NULL");
    if (!aligned16(d_x) || !aligned16(d_y)) return fail(PQ_ERR_ALIGN, "x and y must be 16-byte aligned");
    if (M < 1 || M > p->d.max_m) return fail(PQ_ERR_SHAPE, "M = %d must lie in 1..max_m (%d)", M, p->d.max_m);
    const pq_desc& d = p->d;
    int v = variant == PQ_VARIANT_AUTO ? choose_variant(d, M) : variant;
    if (!variant_runs(d, M, v))
        return fail(PQ_ERR_UNSUPPORTED, "variant %d cannot run fmt %d at M = %d", v, d.fmt, M);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    switch (v) {
        case PQ_VARIANT_W4_GEMV:
            e = launch_w4_gemv(p, d_x, d_y, M, s);   // resolves act order itself
            break;
        case PQ_VARIANT_W4_GEMM:
            if (d.has_gidx) e = launch_gather(p, d_x, M, s);
            if (e == cudaSuccess)
                e = launch_w4_gemm(p, d.has_gidx ? p->ws + p->wl.xg_off : d_x, d_y, M, s);
            break;
        case PQ_VARIANT_W2_GEMV_FUSED:
            e = launch_w2_gemv(p, d_x, d_y, M, true, ws_act(p), s);
            break;
        case PQ_VARIANT_W2_GEMV:
            e = launch_w2_quantize(p, d_x, M, false, ws_act(p), s);
            if (e == cudaSuccess) e = launch_w2_gemv(p, d_x, d_y, M, false, ws_act(p), s);
            break;
        case PQ_VARIANT_W2_GEMM:
            e = launch_w2_quantize(p, d_x, M, true, ws_act(p), s);
            if (e == cudaSuccess) e = launch_w2_gemm(p, d_y, M, ws_act(p), s);
            break;
        case PQ_VARIANT_W2_GEMV_TC:
            e = launch_w2_quantize(p, d_x, M, false, ws_act(p), s);
            if (e == cudaSuccess) e = launch_w2_tc(p, d_y, M, ws_act(p), s);
            break;
        case PQ_VARIANT_W2_GEMV_BF:
            e = launch_w2_quantize(p, d_x, M, true, ws_act(p), s);
            if (e == cudaSuccess) e = launch_w2_bf(p, d_y, M, ws_act(p), s);
            break;
        case PQ_VARIANT_W2_GEMV_CL:
            e = launch_w2_cl(p, d_x, d_y, M, s);
            break;
    }
    if (e != cudaSuccess) return cuda_fail(e, "pq_linear launch");
    return PQ_OK;
}

int32_t pq_linear(const void* d_x, const pq_prepared* p, void* d_y, int32_t M, void* stream) {
    return pq_linear_variant(d_x, p, d_y, M, PQ_VARIANT_AUTO, stream);
}

size_t pq_act_bytes(const pq_desc* d, int32_t M) {
    if (validate_desc(d) != PQ_OK) return 0;
    if (d->fmt != PQ_FMT_W2_PQ2) {
        fail(PQ_ERR_INVALID_ARG, "quantised activations exist for ternary PQ2 layers only");
        return 0;
    }
    if (M < 1 || M > d->max_m) {
        fail(PQ_ERR_SHAPE, "M = %d must lie in 1..max_m (%d)", M, d->max_m);
        return 0;
    }
    return act_layout(*d, M).total;
}

// Checks of a quantised-activation buffer (producers and readers alike).
static int32_t check_act(const pq_prepared* p, const void* d_act, size_t act_bytes, int32_t M) {
    if (!p) return fail(PQ_ERR_INVALID_ARG, "handle is NULL");
    if (p->d.fmt != PQ_FMT_W2_PQ2) return fail(PQ_ERR_INVALID_ARG, "handle is not ternary PQ2");
    if (M < 1 || M > p->d.max_m) return fail(PQ_ERR_SHAPE, "M = %d must lie in 1..max_m (%d)", M, p->d.max_m);
    if (!d_act) return fail(PQ_ERR_INVALID_ARG, "activation buffer is NULL");
    if ((uintptr_t)d_act & (kAlign - 1)) return fail(PQ_ERR_ALIGN, "activation buffer must be 256-byte aligned");
    const size_t need = act_layout(p->d, M).total;
    if (act_bytes < need)
        return fail(PQ_ERR_BUFFER_TOO_SMALL, "activation buffer has %zu bytes, needs %zu for M = %d", act_bytes,
                    need, M);
    return PQ_OK;
}

int32_t pq_quantize_act(const void* d_x, const pq_prepared* p, void* d_act, size_t act_bytes, int32_t M,
                        void* stream) {
    int32_t rc = check_act(p, d_act, act_bytes, M);
    if (rc != PQ_OK) return rc;
    if (!d_x) return fail(PQ_ERR_INVALID_ARG, "x is NULL");
    if (!aligned16(d_x)) return fail(PQ_ERR_ALIGN, "x must be 16-byte aligned");
    cudaError_t e = launch_w2_quantize(p, d_x, M, act_codes_bf16(M), act_planes(p->d, M, d_act),
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PQ_OK : cuda_fail(e, "pq_quantize_act");
}

int32_t pq_norm_quantize(const void* d_h, const void* d_r, const pq_norm* norm, const pq_prepared* p,
                         void* d_r_out, void* d_norm_out, void* d_act, size_t act_bytes, int32_t M,
                         void* stream) {
    int32_t rc = check_act(p, d_act, act_bytes, M);
    if (rc != PQ_OK) return rc;
    if (!d_h || !norm || !norm->gamma) return fail(PQ_ERR_INVALID_ARG, "h, norm and norm->gamma must be non-NULL");
    if (!aligned16(d_h) || (d_r && !aligned16(d_r)) || (d_r_out && !aligned16(d_r_out)) ||
        (d_norm_out && !aligned16(d_norm_out)) || !aligned16(norm->gamma))
        return fail(PQ_ERR_ALIGN, "h, r, r_out, norm_out and gamma must be 16-byte aligned");
    if (!(norm->eps > 0.0f) || !(norm->eps < 3.0e38f))
        return fail(PQ_ERR_INVALID_ARG, "eps must be positive and finite");
    if (norm->unit_offset != 0 && norm->unit_offset != 1)
        return fail(PQ_ERR_INVALID_ARG, "unit_offset must be 0 or 1");
    const int B = norm->had_block;
    if (B != 0 && (B < 2 || B > 1024 || (B & (B - 1)) || p->d.K % B))
        return fail(PQ_ERR_INVALID_ARG, "had_block = %d must be 0 or a power of two in 2..1024 dividing K = %d", B,
                    p->d.K);
    NormArgs n;
    n.h = d_h;
    n.r = d_r;
    n.r_out = d_r_out;
    n.norm_out = d_norm_out;
    n.gamma = norm->gamma;
    n.signs = norm->signs;
    n.eps = norm->eps;
    n.unit_offset = norm->unit_offset;
    n.had_block = B;
    cudaError_t e = launch_w2_norm_quantize(p, n, M, act_codes_bf16(M), act_planes(p->d, M, d_act),
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PQ_OK : cuda_fail(e, "pq_norm_quantize");
}

int32_t pq_linear_act(const void* d_act, size_t act_bytes, const pq_prepared* p, void* d_y, int32_t M,
                      void* stream) {
    int32_t rc = check_act(p, d_act, act_bytes, M);
    if (rc != PQ_OK) return rc;
    if (!d_y) return fail(PQ_ERR_INVALID_ARG, "y is NULL");
    if (!aligned16(d_y)) return fail(PQ_ERR_ALIGN, "y must be 16-byte aligned");
    const int v = act_variant(p->d, M);
    if (v < 0) return fail(PQ_ERR_UNSUPPORTED, "no kernel runs quantised activations for K = %d at M = %d", p->d.K, M);
    const ActPlanes a = act_planes(p->d, M, const_cast<void*>(d_act));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (v == PQ_VARIANT_W2_GEMV) e = launch_w2_gemv(p, nullptr, d_y, M, false, a, s);
    else if (v == PQ_VARIANT_W2_GEMV_TC) e = launch_w2_tc(p, d_y, M, a, s);
    else if (v == PQ_VARIANT_W2_GEMV_BF) e = launch_w2_bf(p, d_y, M, a, s);
    else if (v == PQ_VARIANT_W2_GEMV_CL) e = launch_w2_cl_act(p, d_y, M, a, s);
    else e = launch_w2_gemm(p, d_y, M, a, s);
    return e == cudaSuccess ? PQ_OK : cuda_fail(e, "pq_linear_act");
}

int32_t pq_device_status(const pq_prepared* p, void* stream) {
    if (!p) return fail(PQ_ERR_INVALID_ARG, "handle is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, p->status, 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(p->status, 0, 4, s);
    // A GEMM that gave up a bounded wait may have left shared-tile flags
    // raised (a contributor counted its part, the owner never consumed it):
    // clear them, so the next launch on this workspace starts from zero.
    if (e == cudaSuccess && word != 0) e = cudaMemsetAsync(p->ws + 256, 0, kWsFixedBytes - 256, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "pq_device_status");
    if (word != 0) return fail((int32_t)word, "device status word held %d", (int32_t)word);
    return PQ_OK;
}

void pq_destroy(pq_prepared* p) {
    if (!p) return;
    gemm_free(p);
    delete p;
}

int32_t pq_debug_unpack(const pq_prepared* p, float* d_w, void* stream) {
    if (!p || !d_w) return fail(PQ_ERR_INVALID_ARG, "handle and output must be non-NULL");
    cudaError_t e = launch_debug_unpack(p, d_w, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PQ_OK : cuda_fail(e, "pq_debug_unpack");
}

int32_t pq_debug_w2a8_quantize(const void* d_x, const pq_prepared* p, int8_t* d_q, float* d_xs,
                               int32_t M, void* stream) {
    if (!p || !d_x || !d_q || !d_xs) return fail(PQ_ERR_INVALID_ARG, "NULL argument");
    if (p->d.fmt != PQ_FMT_W2_PQ2) return fail(PQ_ERR_INVALID_ARG, "handle is not ternary PQ2");
    if (M < 1 || M > p->d.max_m) return fail(PQ_ERR_SHAPE, "M = %d must lie in 1..max_m", M);
    if (!aligned16(d_x)) return fail(PQ_ERR_ALIGN, "x must be 16-byte aligned");
    cudaError_t e = launch_w2_debug_quantize(p, d_x, d_q, d_xs, M, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PQ_OK : cuda_fail(e, "pq_debug_w2a8_quantize");
}

int32_t pq_debug_w2a8_group_sums(const void* d_x, const pq_prepared* p, int32_t* d_S, int32_t M,
                                 void* stream) {
    if (!p || !d_x || !d_S) return fail(PQ_ERR_INVALID_ARG, "NULL argument");
    if (p->d.fmt != PQ_FMT_W2_PQ2) return fail(PQ_ERR_INVALID_ARG, "handle is not ternary PQ2");
    if (M < 1 || M > p->d.max_m) return fail(PQ_ERR_SHAPE, "M = %d must lie in 1..max_m", M);
    if (!aligned16(d_x)) return fail(PQ_ERR_ALIGN, "x must be 16-byte aligned");
    cudaError_t e = launch_w2_debug_sums(p, d_x, d_S, M, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PQ_OK : cuda_fail(e, "pq_debug_w2a8_group_sums");
}

int32_t pq_debug_act_unpack(const void* d_act, size_t act_bytes, const pq_prepared* p, int32_t M, int8_t* d_q,
                            float* d_xs, int32_t* d_sq, void* stream) {
    int32_t rc = check_act(p, d_act, act_bytes, M);
    if (rc != PQ_OK) return rc;
    if (!d_q || !d_xs || !d_sq) return fail(PQ_ERR_INVALID_ARG, "NULL output");
    cudaError_t e = launch_debug_act_unpack(p, act_planes(p->d, M, const_cast<void*>(d_act)), M,
                                            act_codes_bf16(M), d_q, d_xs, d_sq, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PQ_OK : cuda_fail(e, "pq_debug_act_unpack");
}

int32_t pq_debug_expire_wait(const pq_prepared* p, int32_t spin_limit, void* stream) {
    if (!p) return fail(PQ_ERR_INVALID_ARG, "handle is NULL");
    if (spin_limit < 1 || spin_limit > (1 << 24))
        return fail(PQ_ERR_INVALID_ARG, "spin_limit = %d must lie in 1..2^24", spin_limit);
    cudaError_t e = launch_expire_wait(p, spin_limit, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PQ_OK : cuda_fail(e, "pq_debug_expire_wait");
}

}  // extern "C"
