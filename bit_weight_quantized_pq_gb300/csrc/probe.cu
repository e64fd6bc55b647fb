// Copy-only read probe: the yardstick for the decode GEMVs ("Kernel
// experiments: recorded evidence", Test 24, bw_probe: a plain streaming read
// of the same bytes with no decode work, timed the same way as the kernels it
// judges).  Every 16-byte chunk of the buffer is loaded once with a 16-byte
// non-allocating load; the words are XOR-folded into one checksum per CTA,
// which one thread folds into sink word (CTA index mod 64), so no load is
// dead code and no word takes more than a few atomics per launch.
#include "pq_internal.cuh"

namespace {

using namespace pq;
using namespace pqd;

constexpr int kProbeThreads = 256;
constexpr int kProbeUnroll = 4;   // independent 16-byte loads in flight per thread
constexpr int kProbeSinkWords = 64;

__global__ void __launch_bounds__(kProbeThreads)
read_probe_kernel(const uint4* __restrict__ src, size_t n16, uint32_t* __restrict__ sink, int dependent) {
    pdl_trigger();
    if (dependent) pdl_wait();
    const size_t stride = (size_t)gridDim.x * kProbeThreads;
    size_t i = (size_t)blockIdx.x * kProbeThreads + threadIdx.x;
    uint32_t acc = 0;
    // consecutive threads read consecutive chunks (512 contiguous bytes per
    // warp and load); each thread keeps kProbeUnroll loads in flight
    for (; i + (kProbeUnroll - 1) * stride < n16; i += kProbeUnroll * stride) {
        uint4 v[kProbeUnroll];
#pragma unroll
        for (int u = 0; u < kProbeUnroll; ++u) v[u] = ldg_stream(src + i + u * stride);
#pragma unroll
        for (int u = 0; u < kProbeUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
    for (; i < n16; i += stride) {
        const uint4 v = ldg_stream(src + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    __shared__ uint32_t part[kProbeThreads / 32];
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t a = 0;
#pragma unroll
        for (int w = 0; w < kProbeThreads / 32; ++w) a ^= part[w];
        atomicXor(sink + (blockIdx.x & (kProbeSinkWords - 1)), a);
    }
}

}  // namespace

extern "C" int32_t pq_probe_read(const void* d_src, size_t bytes, uint32_t* d_sink, int32_t ctas_per_sm,
                                 int32_t dependent, void* stream) {
    using namespace pq;
    if (!d_src || !d_sink) return fail(PQ_ERR_INVALID_ARG, "source and sink must be non-NULL");
    if (((uintptr_t)d_src & 15) || (bytes & 15))
        return fail(PQ_ERR_ALIGN, "the probe reads 16-byte chunks: source address and size must be multiples of 16");
    if (((uintptr_t)d_sink & 3)) return fail(PQ_ERR_ALIGN, "sink must be 4-byte aligned");
    if (bytes == 0) return fail(PQ_ERR_SHAPE, "nothing to read");
    if (ctas_per_sm < 0 || ctas_per_sm > 8) return fail(PQ_ERR_INVALID_ARG, "ctas_per_sm = %d must lie in 0..8", ctas_per_sm);
    if (dependent != 0 && dependent != 1) return fail(PQ_ERR_INVALID_ARG, "dependent must be 0 or 1");
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "pq_probe_read device query");
    const size_t n16 = bytes / 16;
    const size_t per_cta = (size_t)kProbeThreads * kProbeUnroll;
    size_t grid = (size_t)sms * (ctas_per_sm ? ctas_per_sm : 8);
    const size_t need = (n16 + per_cta - 1) / per_cta;
    if (grid > need) grid = need;
    e = launch(read_probe_kernel, dim3((unsigned)grid), dim3(kProbeThreads), 0, static_cast<cudaStream_t>(stream), true,
               static_cast<const uint4*>(d_src), n16, d_sink, (int)dependent);
    return e == cudaSuccess ? PQ_OK : cuda_fail(e, "pq_probe_read launch");
}
