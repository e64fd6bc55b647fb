// Load-time repacking into kernel-native planes, the dequantising debug
// export, and the bounded-wait expiry check.
//
// W4 ("mate: Marlin-class W4A16 GEMM ... #6", prepare_w4a16_from_gptq_frame):
// GPTQ qweight [K/8][N] (N-contiguous words) becomes a K-contiguous code plane
// per output row, rows of K permuted by the act-order sort.  W2 ("Kernel
// experiments: recorded evidence", Test 1 prepare_pq2 / Test 4 shared
// prepared layout): the 34-byte blocks split into a code plane and a scale
// plane; payload stays 34 bytes per 128 weights.
#include "pq_internal.cuh"

namespace {

using namespace pq;

// One thread per (row n, 32-bit word j of the prepared row): word j holds the
// prepared rows k' = 8j..8j+7, k' = 8j+2i in nibble i and 8j+2i+1 in nibble
// i+4.  Prepared row k' reads original row perm[k'] (or k').
__global__ void repack_w4_codes(const uint32_t* __restrict__ qweight, const int32_t* __restrict__ perm,
                                uint32_t* __restrict__ codes, int N, int Npad, int K) {
    const int words_per_row = K / 8;
    const long long total = (long long)Npad * words_per_row;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int n = (int)(idx % Npad);            // n fastest: coalesced qweight reads
        const int j = (int)(idx / Npad);
        uint32_t word = 0;
        if (n < N) {
#pragma unroll
            for (int o = 0; o < 8; ++o) {
                const int kp = 8 * j + o;
                const int k = perm ? perm[kp] : kp;
                const uint32_t code = (qweight[(size_t)(k >> 3) * N + n] >> (4 * (k & 7))) & 0xFu;
                const int nib = (o >> 1) + ((o & 1) << 2);
                word |= code << (4 * nib);
            }
        }
        codes[(size_t)n * words_per_row + j] = word;
    }
}

// [G][N] -> [G][Npad] copy with zero padding (scales fp16 or zero points u8).
template <typename T>
__global__ void pad_columns(const T* __restrict__ src, T* __restrict__ dst, int G, int N, int Npad) {
    const long long total = (long long)G * Npad;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int n = (int)(idx % Npad);
        const int g = (int)(idx / Npad);
        dst[idx] = n < N ? src[(size_t)g * N + n] : T(0);
    }
}

// One thread per (row n, block b < Bp): 32 code bytes to the code plane, the
// little-endian fp16 scale to the [Npad][Bp] scale plane (padding blocks 0).
__global__ void repack_w2(const uint8_t* __restrict__ raw, size_t stride, uint8_t* __restrict__ codes,
                          uint16_t* __restrict__ scales, int N, int Npad, int K, int Bp) {
    const int B = K / kGroup;
    const long long total = (long long)Npad * Bp;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int b = (int)(idx % Bp);
        const int n = (int)(idx / Bp);
        if (b >= B) {
            scales[(size_t)n * Bp + b] = 0;
            continue;
        }
        uint8_t* dst = codes + (size_t)n * (K / 4) + (size_t)b * 32;
        uint16_t sc = 0;
        if (n < N) {
            const uint8_t* blk = raw + (size_t)n * stride + (size_t)b * 34;
            sc = (uint16_t)blk[0] | ((uint16_t)blk[1] << 8);
#pragma unroll
            for (int i = 0; i < 32; ++i) dst[i] = blk[2 + i];
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) dst[i] = 0;
        }
        scales[(size_t)n * Bp + b] = sc;
    }
}

// Affine 4-bit ("qwen CUDA: --prompt-precision int8 ... #1176": codes with a
// scale and a bias per 64 inputs).  Input k of prepared position k' inside a
// 128-input block: k' = 32t + 8w + r holds 16t + 8w + r (w < 2) or
// 64 + 16t + 8(w - 2) + r (w >= 2).
__device__ __forceinline__ int affine_src(int kp) {
    const int blk = kp & ~127, r = kp & 127;
    const int t = r >> 5, w = (r >> 3) & 3, o = r & 7;
    return blk + (w < 2 ? 16 * t + 8 * w + o : 64 + 16 * t + 8 * (w - 2) + o);
}

// One thread per (row n, 32-bit word j of the prepared row), nibble order as
// repack_w4_codes; the source words are output-row major [N][K/8].
__global__ void repack_affine4_codes(const uint32_t* __restrict__ wq, uint32_t* __restrict__ codes, int N,
                                     int Npad, int K) {
    const int words_per_row = K / 8;
    const long long total = (long long)Npad * words_per_row;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int j = (int)(idx % words_per_row);     // j fastest: coalesced reads of a row
        const int n = (int)(idx / words_per_row);
        uint32_t word = 0;
        if (n < N) {
#pragma unroll
            for (int o = 0; o < 8; ++o) {
                const int k = affine_src(8 * j + o);
                const uint32_t code = (wq[(size_t)n * words_per_row + (k >> 3)] >> (4 * (k & 7))) & 0xFu;
                const int nib = (o >> 1) + ((o & 1) << 2);
                word |= code << (4 * nib);
            }
        }
        codes[(size_t)n * words_per_row + j] = word;
    }
}

// [N][G] -> [G][Npad] (16-bit scales or biases), zero padding past N.
__global__ void transpose_groups(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst, int G, int N,
                                 int Npad) {
    const long long total = (long long)G * Npad;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int n = (int)(idx % Npad);
        const int g = (int)(idx / Npad);
        dst[idx] = n < N ? src[(size_t)n * G + g] : (uint16_t)0;
    }
}

__device__ __forceinline__ float f16_bits(uint16_t v) { return __half2float(__ushort_as_half(v)); }

// Dequantised fp32 W[K][N] from the affine planes: RN(s * q + b), the
// product exact in fp32.
__global__ void unpack_affine4(const pq_prepared prep, float* __restrict__ w) {
    const int K = prep.d.K, N = prep.d.N, Np = prep.Npad;
    const bool bf16 = prep.d.act_dtype == PQ_BF16;
    const long long total = (long long)K * N;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int n = (int)(idx % N);
        const int kp = (int)(idx / N);
        const uint32_t word = reinterpret_cast<const uint32_t*>(prep.codes)[(size_t)n * (K / 8) + kp / 8];
        const int o = kp & 7;
        const int nib = (o >> 1) + ((o & 1) << 2);
        const int code = (word >> (4 * nib)) & 0xF;
        const int k = affine_src(kp);
        const int g = k / kAffineGroup;
        const float s = pqd::to_float(prep.scales[(size_t)g * Np + n], bf16);
        const float b = pqd::to_float(prep.biases[(size_t)g * Np + n], bf16);
        w[(size_t)k * N + n] = __fadd_rn(__fmul_rn(s, (float)code), b);
    }
}

// Dequantised fp32 W[K][N] in original row order from the W4 planes.
__global__ void unpack_w4(const pq_prepared prep, float* __restrict__ w) {
    const int K = prep.d.K, N = prep.d.N, Np = prep.Npad;
    const long long total = (long long)K * N;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int n = (int)(idx % N);
        const int kp = (int)(idx / N);
        const uint32_t word = reinterpret_cast<const uint32_t*>(prep.codes)[(size_t)n * (K / 8) + kp / 8];
        const int o = kp & 7;
        const int nib = (o >> 1) + ((o & 1) << 2);
        const int code = (word >> (4 * nib)) & 0xF;
        const int g = kp / kGroup;
        const int z = prep.zeros ? prep.zeros[(size_t)g * Np + n] : 8;
        const float s = f16_bits(prep.scales[(size_t)g * Np + n]);
        const int k = prep.perm ? prep.perm[kp] : kp;
        w[(size_t)k * N + n] = (float)(code - z) * s;
    }
}

__global__ void unpack_w2(const pq_prepared prep, float* __restrict__ w, int Bp) {
    const int K = prep.d.K, N = prep.d.N;
    const long long total = (long long)K * N;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int n = (int)(idx % N);
        const int k = (int)(idx / N);
        const uint8_t byte = prep.codes[(size_t)n * (K / 4) + k / 4];
        const int code = (byte >> (2 * (k & 3))) & 3;
        const float s = f16_bits(prep.scales[(size_t)n * Bp + k / kGroup]);
        w[(size_t)k * N + n] = (float)(code - 1) * s;
    }
}

// A wait that nothing satisfies: poll an mbarrier with a bound, then record
// PQ_ERR_DEVICE_TIMEOUT and return.  This is the same bounded-wait pattern the
// tcgen05 GEMM pipeline uses, exercised on purpose.
__global__ void expire_wait(uint32_t* status, int spin_limit) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        const uint32_t a = (uint32_t)__cvta_generic_to_shared(&bar);
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(a));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        uint32_t done = 0;
        for (int i = 0; i < spin_limit && !done; ++i) {
            asm volatile("{\n\t.reg .pred p;\n\t"
                         "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\t"
                         "selp.u32 %0, 1, 0, p;\n\t}"
                         : "=r"(done) : "r"(a) : "memory");
        }
        if (!done) atomicCAS(status, 0u, (uint32_t)(int32_t)PQ_ERR_DEVICE_TIMEOUT);
    }
}

int grid_for(long long total, int block) {
    long long g = (total + block - 1) / block;
    if (g > 65535LL * 16) g = 65535LL * 16;
    return (int)(g < 1 ? 1 : g);
}

}  // namespace

namespace pq {

cudaError_t launch_prepare_w4(const pq_prepared* p, const uint32_t* qweight, const uint16_t* scales,
                              const uint8_t* zeros, cudaStream_t s) {
    const pq_desc& d = p->d;
    const long long words = (long long)p->Npad * (d.K / 8);
    repack_w4_codes<<<grid_for(words, 256), 256, 0, s>>>(qweight, p->perm,
                                                          reinterpret_cast<uint32_t*>(p->codes),
                                                          d.N, p->Npad, d.K);
    const long long gn = (long long)p->G * p->Npad;
    pad_columns<uint16_t><<<grid_for(gn, 256), 256, 0, s>>>(scales, p->scales, p->G, d.N, p->Npad);
    if (zeros) pad_columns<uint8_t><<<grid_for(gn, 256), 256, 0, s>>>(zeros, p->zeros, p->G, d.N, p->Npad);
    return cudaGetLastError();
}

cudaError_t launch_prepare_w2(const pq_prepared* p, const uint8_t* raw, size_t row_stride, cudaStream_t s) {
    const int Bp = w2_bp(p->d.K);
    const long long total = (long long)p->Npad * Bp;
    repack_w2<<<grid_for(total, 256), 256, 0, s>>>(raw, row_stride, p->codes, p->scales, p->d.N,
                                                   p->Npad, p->d.K, Bp);
    return cudaGetLastError();
}

cudaError_t launch_prepare_affine4(const pq_prepared* p, const uint32_t* wq, const uint16_t* scales,
                                   const uint16_t* biases, cudaStream_t s) {
    const long long words = (long long)p->Npad * (p->d.K / 8);
    repack_affine4_codes<<<grid_for(words, 256), 256, 0, s>>>(wq, reinterpret_cast<uint32_t*>(p->codes), p->d.N,
                                                             p->Npad, p->d.K);
    const int G = p->d.K / kAffineGroup;
    const long long planes = (long long)G * p->Npad;
    transpose_groups<<<grid_for(planes, 256), 256, 0, s>>>(scales, p->scales, G, p->d.N, p->Npad);
    transpose_groups<<<grid_for(planes, 256), 256, 0, s>>>(biases, p->biases, G, p->d.N, p->Npad);
    return cudaGetLastError();
}

cudaError_t launch_debug_unpack(const pq_prepared* p, float* w, cudaStream_t s) {
    const long long total = (long long)p->d.K * p->d.N;
    if (p->d.fmt == PQ_FMT_W4_AFFINE)
        unpack_affine4<<<grid_for(total, 256), 256, 0, s>>>(*p, w);
    else if (p->d.fmt == PQ_FMT_W4_GPTQ)
        unpack_w4<<<grid_for(total, 256), 256, 0, s>>>(*p, w);
    else
        unpack_w2<<<grid_for(total, 256), 256, 0, s>>>(*p, w, w2_bp(p->d.K));
    return cudaGetLastError();
}

cudaError_t launch_expire_wait(const pq_prepared* p, int spin_limit, cudaStream_t s) {
    expire_wait<<<1, 32, 0, s>>>(p->status, spin_limit);
    return cudaGetLastError();
}

}  // namespace pq
