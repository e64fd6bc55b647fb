// Internal declarations shared by the translation units of libpq.
// Host handle layout, device helpers and the kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include <atomic>

#include "../../include/pq.h"

namespace pq {

constexpr int kGroup = 128;          // weights per scale group along K
constexpr int kAffineGroup = 64;     // inputs per scale and bias of the affine 4-bit format
constexpr int kStrip = 16;           // output rows per GEMV strip (mma M)
constexpr size_t kAlign = 256;       // plane / workspace section alignment

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Kernel-native planes inside the caller's prepared allocation.
//   W4: codes [Npad][K/2] bytes; row n, 32-bit word j holds rows k'=8j..8j+7
//       of the (sorted) K order with k'=8j+2i in nibble i and k'=8j+2i+1 in
//       nibble i+4, so one mask of 0x000F000F yields two consecutive k.
//       scales [G][Npad] fp16, zeros [G][Npad] u8 (explicit zero points),
//       perm [K] int32 (act order: prepared row k' is original row perm[k']).
//   W2: codes [Npad][K/4] bytes, the PQ2 code bytes of each block in their
//       original order; scales [Npad][Bp] fp16, Bp = K/128 rounded up to 8
//       (zero padded) so every row's block scales start on a 16-byte boundary.
//   W4 affine: codes as W4, K-permuted inside every 128 inputs (prepared k'
//       = 32t + 8w + r of a block holds input 16t + 8w + r for w < 2 and
//       64 + 16t + 8(w - 2) + r for w >= 2, so the lane of the decode kernel
//       that owns k' 32t..32t+31 finds its first 16 inputs in the block's
//       first 64-group and the other 16 in its second); scales and biases
//       [K/64][Npad] in the activation dtype.
struct Planes {
    size_t codes_off, scales_off, zeros_off, perm_off, biases_off, total;
};

// Scratch inside the caller's workspace.  The first kWsFixedBytes are laid
// out the same for every descriptor, so handles that share one workspace
// agree on them: the device status word, then the state that lasts from one
// launch to the next (the GEMM's shared-tile flags, zero between launches).
// The rest is scratch written and read within one call, laid out per
// descriptor.
struct Workspace {
    size_t status_off;      // uint32 device status word (offset 0)
    size_t flags_off;       // GEMM shared-tile flags [kGemmMaxCtas] u32 (fixed offset 256)
    size_t xg_off;          // W4 act order: gathered x [max_m][K] (16-bit)
    size_t q_off;           // W2: int8 q [max_m][K] in plane order
    size_t xs_off;          // W2: fp32 scales [max_m][K/act_group]; affine (max_m > 16):
                            //   the GEMM's fp32 sums of x over each 64-group [max_m][K/64]
    size_t sq_off;          // W2: int32 sum of q per block [max_m][K/128]
    size_t qa_off;          // W2 GEMM: q as bf16 [max_m][K]
    size_t sk_off;          // split-K decode: partial sums [slices][Npad][16] fp32
    size_t sk_bytes;        //   (0 when the descriptor has no split-K path)
    size_t gp_off;          // prefill GEMM: partial tiles [2 * kGemmMaxCtas][gp_rows][128] fp32
    size_t gp_bytes;        //   (0 bytes when max_m <= 16: the GEMM then splits no tile)
    int gp_rows;
    size_t total;
};

// W4 decode for M > 1 splits K into slices of this many 128-row groups.
constexpr int kSliceGroups = 4;
inline int w4_slices(int K) { return (K / kGroup + kSliceGroups - 1) / kSliceGroups; }
// The one-token W4 kernel keeps the activation row in shared memory beside
// its weight ring, which bounds K; longer rows take the split-K kernel.
constexpr int kW4OneTokenMaxK = 81408;
// ... the same for affine 4-bit layers (a larger ring item and the row's
// 64-group sums beside the row)
constexpr int kW4AffineOneTokenMaxK = 76416;
// ... and holds the rows of up to this many tokens (more: split-K).
constexpr int kW4RowTokens = 4;
// Ternary decode for M > 1 (int8 tensor cores) splits K into slices of this
// many 128-weight blocks.
constexpr int kW2SliceBlocks = 8;
inline int w2_slices(int K) { return (K / kGroup + kW2SliceBlocks - 1) / kW2SliceBlocks; }
// K slices whose partial sums the workspace holds (0: no split-K path).
inline int split_k_slices(const pq_desc& d) {
    if (d.fmt == PQ_FMT_W4_AFFINE) return (d.max_m > 1 || d.K > kW4AffineOneTokenMaxK) ? w4_slices(d.K) : 0;
    if (d.fmt == PQ_FMT_W4_GPTQ) return (d.max_m > 1 || d.K > kW4OneTokenMaxK) ? w4_slices(d.K) : 0;
    return d.max_m > 1 ? w2_slices(d.K) : 0;
}

// The prefill GEMM gives every CTA an equal share of the 128-row groups of
// its last tiles; a CTA that holds part of a tile writes it to one of its two
// partial-tile slots (and raises its flag when the tile's owner adds the
// parts).  The workspace holds slots and flags for this many CTAs (the grid
// never exceeds it).
constexpr int kGemmMaxCtas = 160;
constexpr int kGemmFlagBytes = 768;      // kGemmMaxCtas u32 flags, 256-byte aligned
constexpr size_t kWsFixedBytes = 256 + kGemmFlagBytes;
constexpr int kGemmTileRows = 192;       // tokens per GEMM tile
constexpr int kGemmTileCols = 128;       // output features per GEMM tile
inline int gemm_partial_rows(int max_m) {
    if (max_m <= 16) return 0;
    return max_m >= kGemmTileRows ? kGemmTileRows : (max_m + 15) / 16 * 16;
}

// Quantised activations of a ternary layer: what the quantiser (or the fused
// norm producer) writes and the ternary kernels read.  The handle's workspace
// holds one set; callers of pq_quantize_act / pq_norm_quantize hold others in
// a buffer of their own (act_layout).
struct ActPlanes {
    int8_t* q8;      // int8 q [M][K] in plane order (CUDA-core and int8 decodes)
    uint16_t* qa;    // q as bf16 [M][K] in tensor-core operand order (cluster and bf16 decodes, GEMM)
    int32_t* sq;     // int32 sum of q per 128-block [M][K/128]
    float* xs;       // fp32 scales [M][K/act_group]
};
// Caller-held activation buffer for M tokens: int8 plane-order codes when
// M <= 2 (the CUDA-core decode), bf16 codes in tensor-core order otherwise
// (the cluster decode at M = 3..16, its split-K fallback, and the GEMM);
// scales and block sums in both cases.  Sections start on 256-byte
// boundaries.
struct ActLayout {
    size_t q8_off, xs_off, sq_off, qa_off, total;
};
constexpr int kActDecodeMaxM = 16;   // decode kernels up to here, the GEMM above
constexpr int kActInt8MaxM = 2;      // int8 codes up to here, bf16 codes above
inline bool act_codes_bf16(int M) { return M > kActInt8MaxM; }

Planes plane_layout(const pq_desc& d);
Workspace workspace_layout(const pq_desc& d);
ActLayout act_layout(const pq_desc& d, int M);
int npad(int N);
int w2_bp(int K);   // W2 scale-plane row length in blocks (a multiple of 8)

}  // namespace pq

struct pq_prepared {
    pq_desc d;
    int Npad, G;
    int device, num_sms;
    uint8_t* base;
    uint8_t* codes;
    uint16_t* scales;
    uint8_t* zeros;
    int32_t* perm;
    uint16_t* biases;       // affine 4-bit: [K/64][Npad] biases (scales in `scales`)
    uint8_t* ws;
    size_t ws_bytes;
    pq::Workspace wl;
    uint32_t* status;
    void* gemm_state;       // tensor maps for the tcgen05 GEMM (owned)
};

namespace pq {

// ---- error reporting (api.cu) ----
int32_t fail(int32_t code, const char* fmt, ...);
int32_t cuda_fail(cudaError_t e, const char* where);

// ---- kernel attributes, per device ----
// cudaFuncSetAttribute applies to the current device only.  Each kernel
// keeps, per device, the largest dynamic shared memory it has been allowed
// (one record per kernel, shared by every launcher of that kernel, so one
// launcher can never lower the size another relies on) and the attribute is
// only ever raised.  Devices beyond kMaxDevices are configured on every
// launch (raised to the size that launch needs).
constexpr int kMaxDevices = 64;
struct SmemAttr {
    std::atomic<size_t> bytes[kMaxDevices];
};

template <auto Kernel>
SmemAttr& smem_record() {
    static SmemAttr rec;
    return rec;
}

template <auto Kernel>
cudaError_t ensure_smem(size_t bytes) {
    SmemAttr& rec = smem_record<Kernel>();
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool tracked = dev >= 0 && dev < kMaxDevices;
    size_t cur = tracked ? rec.bytes[dev].load() : 0;
    if (cur >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess && tracked)
        while (cur < bytes && !rec.bytes[dev].compare_exchange_weak(cur, bytes)) {
        }
    return e;
}

// the same for the shared-memory carveout preference (set once per device)
template <auto Kernel>
cudaError_t ensure_max_carveout() {
    static std::atomic<int> done[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices && done[dev].load()) return cudaSuccess;
    e = cudaFuncSetAttribute(Kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess && dev >= 0 && dev < kMaxDevices) done[dev].store(1);
    return e;
}

// ---- launch helper: PDL attribute so a kernel may start while its
//      predecessor on the stream drains; kernels order their reads of
//      predecessor outputs after griddepcontrol.wait. ----
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                   cudaStream_t stream, bool pdl, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same with the cooperative attribute as well: every CTA of the grid is
// resident at once (for kernels whose CTAs wait on one another's flags).
template <typename... KArgs, typename... Args>
cudaError_t launch_cooperative(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t stream, bool pdl, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same with a thread-block cluster of `cluster` CTAs along x (the grid's
// x a multiple of it): the CTAs of a cluster run at the same time and share
// their shared memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                           int cluster, bool pdl, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---- launchers (one per translation unit) ----
cudaError_t launch_prepare_w4(const pq_prepared* p, const uint32_t* qweight,
                              const uint16_t* scales, const uint8_t* zeros,
                              cudaStream_t s);
cudaError_t launch_prepare_w2(const pq_prepared* p, const uint8_t* raw,
                              size_t row_stride, cudaStream_t s);
cudaError_t launch_prepare_affine4(const pq_prepared* p, const uint32_t* wq, const uint16_t* scales,
                                   const uint16_t* biases, cudaStream_t s);
// the whole-row decode kernel runs an affine 4-bit layer at M tokens
bool w4_affine_runs(const pq_desc& d, int M);
cudaError_t launch_debug_unpack(const pq_prepared* p, float* w, cudaStream_t s);
cudaError_t launch_expire_wait(const pq_prepared* p, int spin_limit, cudaStream_t s);

void plan_w4_gemv(const pq_prepared* p, int M, pq_plan_info* info);
// x in the caller's order; act order is resolved inside (the whole-row
// kernel gathers through the permutation, split-K after a gather launch)
cudaError_t launch_w4_gemv(const pq_prepared* p, const void* x, void* y, int M,
                           cudaStream_t s);
cudaError_t launch_gather(const pq_prepared* p, const void* x, int M, cudaStream_t s);
// split-K decode, second pass: y = sum of the slices' partials (x rs[m])
cudaError_t launch_sk_reduce(const pq_prepared* p, void* y, int M, int nslices, const float* rs, cudaStream_t s);

void plan_w2_gemv(const pq_prepared* p, int M, bool fused, pq_plan_info* info);
bool w2_gemv_fits(const pq_desc& d, int M, bool fused);
ActPlanes ws_act(const pq_prepared* p);       // the handle's own workspace set
cudaError_t launch_w2_quantize(const pq_prepared* p, const void* x, int M,
                               bool bf16_codes, const ActPlanes& a, cudaStream_t s);
// fused producer: residual add, RMSNorm, optional random-sign Hadamard, then
// the same quantiser (one CTA per token row)
struct NormArgs {
    const void* h;          // [M][K] act dtype
    const void* r;          // [M][K] act dtype or NULL
    void* r_out;            // [M][K] act dtype or NULL (may equal h or r)
    void* norm_out;         // [M][K] act dtype or NULL
    const void* gamma;      // [K] act dtype
    const int8_t* signs;    // [K] or NULL
    float eps;
    int unit_offset;
    int had_block;          // 0 or a power of two 2..1024
};
cudaError_t launch_w2_norm_quantize(const pq_prepared* p, const NormArgs& n, int M,
                                    bool bf16_codes, const ActPlanes& a, cudaStream_t s);
cudaError_t launch_w2_gemv(const pq_prepared* p, const void* x, void* y, int M,
                           bool fused, const ActPlanes& a, cudaStream_t s);
bool w2_tc_runs(const pq_prepared* p, int M);
void plan_w2_tc(const pq_prepared* p, int M, pq_plan_info* info);
cudaError_t launch_w2_tc(const pq_prepared* p, void* y, int M, const ActPlanes& a, cudaStream_t s);
void plan_w2_bf(const pq_prepared* p, int M, pq_plan_info* info);
// the same decode on bf16 mma.sync; reads the bf16 codes (a.qa)
cudaError_t launch_w2_bf(const pq_prepared* p, void* y, int M, const ActPlanes& a, cudaStream_t s);
// the cluster split-K decode (quantiser in the cluster, one launch)
bool w2_cl_fits(const pq_desc& d, int M);
void plan_w2_cl(const pq_prepared* p, int M, pq_plan_info* info);
cudaError_t launch_w2_cl(const pq_prepared* p, const void* x, void* y, int M, cudaStream_t s);
// ... the same on quantised activations (bf16 codes, a.qa and a.xs)
cudaError_t launch_w2_cl_act(const pq_prepared* p, void* y, int M, const ActPlanes& a, cudaStream_t s);
cudaError_t launch_w2_debug_quantize(const pq_prepared* p, const void* x, int8_t* q,
                                     float* xs, int M, cudaStream_t s);
cudaError_t launch_w2_debug_sums(const pq_prepared* p, const void* x, int32_t* S,
                                 int M, cudaStream_t s);
cudaError_t launch_debug_act_unpack(const pq_prepared* p, const ActPlanes& a, int M, bool bf16_codes,
                                    int8_t* q, float* xs, int32_t* sq, cudaStream_t s);

bool gemm_supported(const pq_desc& d);
void plan_gemm(const pq_prepared* p, int M, pq_plan_info* info);
int32_t gemm_init(pq_prepared* p);        // builds tensor maps (host)
void gemm_free(pq_prepared* p);
cudaError_t launch_w4_gemm(const pq_prepared* p, const void* x, void* y, int M,
                           cudaStream_t s);
cudaError_t launch_w2_gemm(const pq_prepared* p, void* y, int M, const ActPlanes& a,
                           cudaStream_t s);

}  // namespace pq

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
namespace pqd {

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ldg_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;  // (a & b) | c
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Programmatic dependent launch: wait for the predecessor grid's memory,
// and let the successor grid be scheduled.
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float to_float(uint16_t v, bool bf16) {
    return bf16 ? __bfloat162float(__ushort_as_bfloat16(v))
                : __half2float(__ushort_as_half(v));
}

__device__ __forceinline__ uint16_t from_float(float v, bool bf16) {
    return bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(v))
                : __half_as_ushort(__float2half_rn(v));
}

// Sums of x over the 64-input groups of the affine 4-bit format: eight lanes
// of a warp (lanes 8j..8j+7) hold one 16-byte chunk (eight inputs) each; a
// lane adds its chunk in order, then the eight partial sums are added as a
// fixed tree (xor 1, 2, 4), so every lane ends with the same group total and
// every kernel that forms the sums this way gets the same bits.
__device__ __forceinline__ float chunk_sum8(uint4 u, bool bf16) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        s += to_float((uint16_t)(w[i] & 0xFFFFu), bf16);
        s += to_float((uint16_t)(w[i] >> 16), bf16);
    }
    return s;
}
__device__ __forceinline__ float team8_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    return v;
}

}  // namespace pqd
