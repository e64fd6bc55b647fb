// Ternary W2A8 decode path ("Kernel experiments: recorded evidence"):
//   * activation quantiser (Test 6 group quantiser; Test 21 plane order and
//     per-group integer sum): per activation group, scale = max|a| / 127 in
//     fp32, q = clamp(rint_even(a / scale), -127, 127), int8 stored so that
//     plane s of a 32-bit code word meets one int32 of activations;
//   * GEMV: per 128-weight block the exact int32 sum
//     S = sum (code - 1) * q = sum code * q - sum q, formed with dp4a on the
//     four 2-bit planes of each code word (Test 6 DP4A dot, Test 21 minus-one
//     correction), then y += S * ws (* xs) in fp32.
// GB300 design: persistent CTAs of 16 warps; every lane streams the 32 code
// bytes of its own block (and lanes 0..3 the block scales of the step) with
// cp.async into a per-warp ring, issued before the dependency wait and before
// quantisation, and forms the block's exact int32 sum alone.  The quantiser
// runs inside every CTA for M = 1 (no second launch, no scratch) or as a
// pre-pass into the workspace.
#include "gemv_common.cuh"

namespace {

using namespace pq;
using namespace pqd;
using namespace pqg;

constexpr int kThreads = 256;     // quantise pre-pass CTA
constexpr int kWarps = 8;         // split-K and cluster decode CTAs: 8 warps
// The one- and two-token GEMV: 16 warps a CTA, persistent over rows, with a
// ring of 4 row steps a warp, so that two CTAs fit an SM at every 7B shape
// (measured on GB300 over the merged one-token decode pass: 6.66 us per
// ternary call against 6.76 with 8 warps and 6 steps; 5 steps leave room
// for one CTA per SM at K = 11008 and lose 10%).
constexpr int kGemvWarps = 16;
static_assert(kGemvWarps % 4 == 0, "the quantiser reads the warps' maxima four at a time");
constexpr int kDepth = 4;         // cp.async ring depth (row steps) per warp
constexpr int kItemB = 1024 + 64; // one warp step: 32 blocks of 32 code bytes + 32 block scales
// Shared-memory stride of one block's 128 plane-ordered activation codes: the
// 16 extra bytes put the lanes of a warp (one block each) on different banks.
constexpr int kQStride = 144;

__device__ __forceinline__ float warp_sum_f(float v) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float group_scale(float amax) {
    return __fdiv_rn(amax, 127.0f);              // correctly rounded fp32 quotient
}

__device__ __forceinline__ int quant_one(float a, float scale) {
    const float div = scale > 0.f ? scale : 1.0f;
    float r = rintf(__fdiv_rn(a, div));          // nearest, ties to even
    r = fminf(127.f, fmaxf(-127.f, r));
    return (int)r;
}

// Divisor of one activation group: the scale s and rn = RN(1/s).  Scales
// below 2^-100 (and s = 0) take the plain correctly rounded division.
struct QDiv {
    float s, rn;
    bool plain;
};

__device__ __forceinline__ QDiv make_qdiv(float scale) {
    QDiv q;
    q.plain = !(scale >= 0x1p-100f);
    q.s = scale;
    q.rn = q.plain ? 1.0f : __frcp_rn(scale);
    return q;
}


// q = clamp(rint(RN(a / s)), -127, 127) without a division per element.
// With rn = RN(1/s), y = RN(a * rn) lies within one ulp of a / s, so the
// residual a - s*y is exact in one FMA, and RN(y + rn * (a - s*y)) is the
// correctly rounded quotient (Markstein's theorem on the final correction
// step of Newton-Raphson division).  |a| <= 127 s bounds the quotient, and
// s >= 2^-100 keeps every intermediate normal or the quotient far below 1/2.
// Adding 1.5 * 2^23 then rounds the quotient to an integer, ties to even, in
// the low mantissa bits: the result's bit pattern is 0x4B400000 + q, whose
// low byte is q as int8.  Two activations at a time on the packed fp32 pipe
// (each lane an IEEE operation, so the same bits as the scalar sequence).
// The clamp is never reached here: s = RN(amax / 127) >= (amax / 127)(1 -
// 2^-24) for the group's own maximum, so |a / s| < 127.00001 and the rounded
// quotient stays within +-127 (finite activations).
constexpr uint32_t kQMagic = 0x4B400000u;    // bit pattern of 1.5 * 2^23

__device__ __forceinline__ void quant_pair(float a0, float a1, const QDiv& d, uint32_t& t0, uint32_t& t1) {
    asm("{\n\t.reg .b64 ra, rn, rs, ry, re, rm;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rn, {%4, %4};\n\t"
        "mov.b64 rs, {%5, %5};\n\t"
        "mov.b64 rm, {%6, %6};\n\t"
        "mul.rn.f32x2 ry, ra, rn;\n\t"
        "fma.rn.f32x2 re, rs, ry, ra;\n\t"
        "fma.rn.f32x2 ry, re, rn, ry;\n\t"
        "add.rn.f32x2 ry, ry, rm;\n\t"
        "mov.b64 {%0, %1}, ry;\n\t}"
        : "=r"(t0), "=r"(t1)
        : "f"(a0), "f"(a1), "f"(d.rn), "f"(-d.s), "f"(12582912.0f));
}

// Largest |value| of the eight 16-bit activations of a 16-byte chunk, as
// the bit pattern of a non-negative value (fp16 and bf16 patterns of
// non-negative finite values order like the values).
__device__ __forceinline__ uint32_t chunk_absmax_bits(const uint4& u) {
    constexpr uint32_t kAbs = 0x7FFF7FFFu;
    const uint32_t v = __vmaxu2(__vmaxu2(u.x & kAbs, u.y & kAbs), __vmaxu2(u.z & kAbs, u.w & kAbs));
    return max(v & 0xFFFFu, v >> 16);
}

template <bool BF16IN>
__device__ __forceinline__ float bits16_to_float(uint32_t b) {
    return BF16IN ? __uint_as_float(b << 16) : __half2float(__ushort_as_half((uint16_t)b));
}

// Divisors of bf16 activation groups from a table.  A bf16 maximum
// a >= 2^-93 is 2^e (1 + j/128), j its 7 mantissa bits, and scaling by a
// power of two commutes with correct rounding while results stay normal, so
// s = RN(a / 127) = 2^e RN((1 + j/128) / 127) and RN(1/s) = 2^-e RN(1/s0)
// for s0 = RN((1 + j/128) / 127) exactly (here s >= 2^-100 and 1/s <= 2^100
// are normal).  A kernel that quantises fills the 128 pairs (s0, RN(1/s0))
// with the same correctly rounded division and reciprocal before it waits
// for its input; a group's divisor is then two shared-memory loads and two
// integer adds on the exponent fields instead of both operations on the
// critical path.  Smaller maxima (and fp16 inputs) take make_qdiv.
constexpr int kQTab = 128;
__device__ __forceinline__ void qtab_fill(float* tab) {    // every thread; the caller synchronises
    for (int j = threadIdx.x; j < kQTab; j += blockDim.x) {
        const float s0 = group_scale(1.0f + (float)j * (1.0f / 128.0f));
        tab[j] = s0;
        tab[kQTab + j] = __frcp_rn(s0);
    }
}
template <bool BF16IN>
__device__ __forceinline__ QDiv qdiv_of(uint32_t amax_bits, const float* tab) {
    const float a = bits16_to_float<BF16IN>(amax_bits);
    if (!BF16IN || tab == nullptr || !(a >= 0x1p-93f)) return make_qdiv(group_scale(a));
    const uint32_t j = amax_bits & 0x7Fu;
    const uint32_t de = (((amax_bits >> 7) & 0xFFu) - 127u) << 23;   // 2^e on the exponent field (mod 2^32)
    QDiv q;
    q.s = __uint_as_float(__float_as_uint(tab[j]) + de);
    q.rn = __uint_as_float(__float_as_uint(tab[kQTab + j]) - de);
    q.plain = false;
    return q;
}

template <bool BF16IN>
__device__ __forceinline__ void unpack8(const uint4& u, float (&a)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (BF16IN) {
            a[2 * j] = __uint_as_float(w[j] << 16);
            a[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        } else {
            a[2 * j] = __half2float(__ushort_as_half((uint16_t)(w[j] & 0xFFFF)));
            a[2 * j + 1] = __half2float(__ushort_as_half((uint16_t)(w[j] >> 16)));
        }
    }
}

// Quantise one activation row xr[0..K), already in shared memory, with
// activation group AG (128 or K).  All threads of the CTA call it
// (blockDim.x a multiple of 32, at most 512).  Thread u of a stride step
// takes the 16 consecutive elements 16u..16u+15, so a 128-block is 8
// consecutive lanes; the loops stay rolled (the code runs once per launch).
//   PLANE: int8 codes in plane order (block b, in-block index i stored at
//          b*qstride + (i%4)*32 + i/4);
//   else:  codes as bf16 (exact integers) in the tensor-core operand order
//          described below.
// sq receives the int32 sum of q of every 128-block and xs the fp32 scale of
// every activation group.  `red` is 33 floats
// of shared scratch; `rowi` alternates its halves between consecutive rows.
template <bool PLANE, bool BF16IN>
__device__ void quantize_row(const uint16_t* xr, int K, int AG, int8_t* q8, uint16_t* qbf, int32_t* sq,
                             float* xs, float* red, int rowi, const float* qtab, int qstride = kGroup) {
    const int tid = threadIdx.x, T = blockDim.x, lane = tid & 31;
    const int U = K / 16;                         // 16-element units
    const int UR = (U + 31) / 32 * 32;            // whole warps in every step
    QDiv row{};
    if (AG != kGroup) {                           // one group per row: row amax first
        uint32_t mb = 0;
#pragma unroll 1
        for (int u = tid; u < U; u += T) {
            mb = max(mb, chunk_absmax_bits(*reinterpret_cast<const uint4*>(xr + 16 * u)));
            mb = max(mb, chunk_absmax_bits(*reinterpret_cast<const uint4*>(xr + 16 * u + 8)));
        }
        const uint32_t wm = __reduce_max_sync(0xffffffffu, mb);
        uint32_t* r = reinterpret_cast<uint32_t*>(red) + 16 * (rowi & 1);
        if (lane == 0) r[tid >> 5] = wm;
        __syncthreads();
        uint32_t am = r[0];
        for (int w = 1; w < (T >> 5); ++w) am = max(am, r[w]);
        row = qdiv_of<BF16IN>(am, qtab);
        if (tid == 0) xs[0] = row.s;
    }
#pragma unroll 1
    for (int u = tid; u < UR; u += T) {
        const bool ok = u < U;
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        const uint4 ulo = ok ? *reinterpret_cast<const uint4*>(xr + 16 * u) : z;
        const uint4 uhi = ok ? *reinterpret_cast<const uint4*>(xr + 16 * u + 8) : z;
        float a[16];
        {
            float lo[8], hi[8];
            unpack8<BF16IN>(ulo, lo);
            unpack8<BF16IN>(uhi, hi);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                a[j] = lo[j];
                a[8 + j] = hi[j];
            }
        }
        QDiv dv = row;
        if (AG == kGroup) {
            uint32_t mb = max(chunk_absmax_bits(ulo), chunk_absmax_bits(uhi));
#pragma unroll
            for (int o = 4; o > 0; o >>= 1) mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, o));
            dv = qdiv_of<BF16IN>(mb, qtab);
            if (ok && (lane & 7) == 0) xs[u / 8] = dv.s;
        }
        // t[j] = 0x4B400000 + q[j]
        uint32_t t[16];
        if (dv.plain) {
#pragma unroll
            for (int j = 0; j < 16; ++j) t[j] = kQMagic + (uint32_t)quant_one(a[j], dv.s);
        } else {
#pragma unroll
            for (int j = 0; j < 16; j += 2) quant_pair(a[j], a[j + 1], dv, t[j], t[j + 1]);
        }
        // the block's sum of q (the decode kernels subtract it): the offset
        // words added with wrap-around, minus 16 offsets
        uint32_t su = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) su += t[j];
        int s = (int)(su - 16u * kQMagic);
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (ok && (lane & 7) == 0) sq[u / 8] = s;
        if (PLANE) {
            if (ok) {
                // plane p, in-block bytes 4*(u%8) .. +3 hold elements i0+p, i0+4+p, i0+8+p, i0+12+p
                // (the low bytes of their offset words)
                int8_t* dst = q8 + (size_t)(u / 8) * qstride + 4 * (u % 8);
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const uint32_t lo = __byte_perm(t[p], t[4 + p], 0x0040);
                    const uint32_t hi = __byte_perm(t[8 + p], t[12 + p], 0x0040);
                    *reinterpret_cast<uint32_t*>(dst + p * 32) = __byte_perm(lo, hi, 0x5410);
                }
            }
        } else if (ok) {
            // Tensor-core operand order: inside every 16-element block position
            // p holds element pi(p), pi = 0,8,1,9,2,10,3,11,4,12,5,13,6,14,7,15,
            // the order in which the GEMM's converter unpacks a 32-bit code word.
            // q = t - 1.5 * 2^23 exactly, then two codes to bf16 (exact) at once.
            uint32_t w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(t[j]) - 12582912.0f,
                                                               __uint_as_float(t[8 + j]) - 12582912.0f);
                w[j] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            uint4* dst = reinterpret_cast<uint4*>(qbf + 16 * (size_t)u);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
    }
}

// The same quantiser on 8-element units for the one-token GEMV, whose CTA
// has twice the threads of a 16-element-unit pass over a 4096-wide row:
// thread v of a step takes elements 8v..8v+7 (a 128-block is 16 consecutive
// lanes), the same roundings in the same order, so the same codes, scales
// and block sums.  Int8 codes in plane order only: half-unit vv of block b
// puts elements 8vv + p and 8vv + 4 + p into bytes 2vv, 2vv + 1 of plane p.
template <bool BF16IN>
__device__ void quantize_row_planes8(const uint16_t* xr, int K, int AG, int8_t* q8, int32_t* sq, float* xs,
                                     float* red, int rowi, int qstride, const float* qtab) {
    const int tid = threadIdx.x, T = blockDim.x, lane = tid & 31;
    const int H = K / 8;                          // 8-element units
    const int HR = (H + 31) / 32 * 32;            // whole warps in every step
    QDiv row{};
    if (AG != kGroup) {                           // one group per row: row amax first
        uint32_t mb = 0;
#pragma unroll 1
        for (int v = tid; v < H; v += T) mb = max(mb, chunk_absmax_bits(*reinterpret_cast<const uint4*>(xr + 8 * v)));
        const uint32_t wm = __reduce_max_sync(0xffffffffu, mb);
        uint32_t* r = reinterpret_cast<uint32_t*>(red) + 16 * (rowi & 1);   // 16-byte aligned
        if (lane == 0) r[tid >> 5] = wm;
        __syncthreads();
        // the warps' maxima four at a time (T / 32 is a multiple of 4)
        uint32_t am = 0;
#pragma unroll 4
        for (int w = 0; w < (T >> 5); w += 4) {
            const uint4 v = *reinterpret_cast<const uint4*>(r + w);
            am = max(am, max(max(v.x, v.y), max(v.z, v.w)));
        }
        row = qdiv_of<BF16IN>(am, qtab);
        if (tid == 0) xs[0] = row.s;
    }
#pragma unroll 1
    for (int v = tid; v < HR; v += T) {
        const bool ok = v < H;
        const uint4 u = ok ? *reinterpret_cast<const uint4*>(xr + 8 * v) : make_uint4(0u, 0u, 0u, 0u);
        float a[8];
        unpack8<BF16IN>(u, a);
        QDiv dv = row;
        if (AG == kGroup) {
            uint32_t mb = chunk_absmax_bits(u);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, o));
            dv = qdiv_of<BF16IN>(mb, qtab);
            if (ok && (lane & 15) == 0) xs[v / 16] = dv.s;
        }
        uint32_t t[8];
        if (dv.plain) {
#pragma unroll
            for (int j = 0; j < 8; ++j) t[j] = kQMagic + (uint32_t)quant_one(a[j], dv.s);
        } else {
#pragma unroll
            for (int j = 0; j < 8; j += 2) quant_pair(a[j], a[j + 1], dv, t[j], t[j + 1]);
        }
        uint32_t su = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) su += t[j];
        int s = (int)(su - 8u * kQMagic);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (ok && (lane & 15) == 0) sq[v / 16] = s;
        if (ok) {
            uint16_t* dst = reinterpret_cast<uint16_t*>(q8 + (size_t)(v / 16) * qstride + 2 * (v % 16));
#pragma unroll
            for (int p = 0; p < 4; ++p) dst[16 * p] = (uint16_t)__byte_perm(t[p], t[4 + p], 0x0040);
        }
    }
}

// Four unsigned bytes of a times four signed bytes of b, plus c.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Sum of code * q over one 16-byte chunk (64 weights = half a block):
// code words cw[0..3] (bytes 16h..16h+15 of the block), q planes of the
// block at qb (128 bytes, plane order).  Plane s of word w holds the codes of
// in-block weights 16(4h+w)+4i+s, i = 0..3, which is exactly int32 word
// (4h+w) of plane s.  Plane s is taken in place (word & 3 << 2s in every
// byte): unsigned bytes code * 4^s <= 192 against the signed activation
// bytes, so plane s's sum is 4^s times its dot and comes back exactly by an
// arithmetic shift.
__device__ __forceinline__ int chunk_dot(const uint4& c, const int8_t* qb, int h) {
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
    int acc[4] = {0, 0, 0, 0};          // one chain per plane: four dependent dp4a each
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const uint4 qv = *reinterpret_cast<const uint4*>(qb + s * 32 + 16 * h);
        const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
        for (int w = 0; w < 4; ++w) acc[s] = dp4a_us(cw[w] & (0x03030303u << (2 * s)), qw[w], acc[s]);
    }
    return (acc[0] + (acc[1] >> 2)) + ((acc[2] >> 4) + (acc[3] >> 6));
}

// The same sum over a whole block with the block's activation codes held in
// registers (q[8s + 4h + w] is plane s's word 4h + w), one accumulator per
// plane over both halves, so the planes' scalings come off once a block.
__device__ __forceinline__ int block_dot_reg(const uint4& c0, const uint4& c1, const uint32_t (&q)[32]) {
    const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    int acc[4] = {0, 0, 0, 0};
#pragma unroll
    for (int s = 0; s < 4; ++s)
#pragma unroll
        for (int w = 0; w < 8; ++w) acc[s] = dp4a_us(cw[w] & (0x03030303u << (2 * s)), q[8 * s + w], acc[s]);
    return (acc[0] + (acc[1] >> 2)) + ((acc[2] >> 4) + (acc[3] >> 6));
}

// dynamic shared memory of the GEMV:
//   ring [kGemvWarps][kDepth][kItemB] | q [MT][K/128][kQStride] | sq [MT][K/128] |
//   xs [MT][K/AG] | red[33] | (fused) x rows [MT][K] 16-bit, 16-byte aligned
struct W2Smem {
    size_t q, sq, xs, red, x, total;
};
__host__ __device__ inline W2Smem w2_smem(int MT, int K, int AG, bool fused) {
    W2Smem l;
    l.q = (size_t)kGemvWarps * kDepth * kItemB;
    l.sq = l.q + (size_t)MT * (K / kGroup) * kQStride;
    l.xs = l.sq + (size_t)MT * (K / kGroup) * 4;
    l.red = (l.xs + (size_t)MT * (K / AG) * 4 + 15) / 16 * 16;   // 16-byte aligned (read as uint4)
    l.x = (l.red + 33 * 4 + 15) / 16 * 16;
    l.total = l.x + (fused ? (size_t)MT * K * 2 : 0);
    return l;
}
__host__ __device__ inline size_t w2_smem_bytes(int MT, int K, int AG, bool fused) {
    return w2_smem(MT, K, AG, fused).total;
}

// Persistent GEMV: warp gw of TW owns output rows gw, gw+TW, ...; a row is
// streamed in steps of 32 blocks (1 KB of codes), lane l copying the 32 code
// bytes of block 32*step + l (and lanes 0..3 the step's 32 block scales) with
// cp.async into a ring of kDepth steps, so every lane owns whole blocks and
// forms their exact int32 sums alone.  At one token two CTAs share an SM,
// so its instance is held to 64 registers a thread.
template <int MT, bool FUSED>
__global__ void __launch_bounds__(kGemvWarps * 32, MT == 1 ? 2 : 1)
w2_gemv_kernel(const uint16_t* __restrict__ x, int act_bf16, const uint8_t* __restrict__ codes,
               const uint16_t* __restrict__ wscales, const int8_t* __restrict__ q_ws,
               const int32_t* __restrict__ sq_ws, const float* __restrict__ xs_ws,
               uint16_t* __restrict__ y, int M, int N, int K, int Bp, int AG, int out_bf16, uint32_t* status) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ __align__(8) uint64_t xbar;
    __shared__ float qtab[FUSED ? 2 * kQTab : 1];
    const int B = K / kGroup, XG = K / AG;
    const W2Smem L = w2_smem(MT, K, AG, FUSED);
    int8_t* q_s = reinterpret_cast<int8_t*>(smem + L.q);
    int32_t* sq_s = reinterpret_cast<int32_t*>(smem + L.sq);
    float* xs_s = reinterpret_cast<float*>(smem + L.xs);
    float* red = reinterpret_cast<float*>(smem + L.red);
    uint16_t* x_s = reinterpret_cast<uint16_t*>(smem + L.x);

    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int steps = (B + 31) / 32;
    const int TW = gridDim.x * kGemvWarps, gw = blockIdx.x * kGemvWarps + warp;
    const int nrows = gw < N ? (N - 1 - gw) / TW + 1 : 0;
    const int total = nrows * steps;
    uint8_t* ring = smem + (size_t)warp * kDepth * kItemB;

    // steps are issued strictly in order and tracked by counters
    int is_i = 0, is_row = gw, is_it = 0, is_slot = 0;
    // one-token rows of one step (K <= 4096): the issue reduced to pointer
    // steps (lane l always copies block l); warps with two rows or more also
    // take the loop below with the activation codes in registers
    const bool one_step = MT == 1 && steps == 1;
    const uint8_t* o_src = codes + (size_t)gw * (K / 4) + 32 * lane;
    const uint16_t* o_ssrc = wscales + (size_t)gw * Bp + 8 * lane;
    const size_t o_cstep = (size_t)TW * (K / 4), o_sstep = (size_t)TW * Bp;
    const uint32_t ring_u32 = smem_u32(ring);
    const bool o_code = lane < B, o_scale = lane < 4 && 8 * lane < Bp;
    auto issue_next = [&]() {
        if (one_step) {
            if (is_i < total) {
                const uint32_t slot = ring_u32 + (uint32_t)(is_slot * kItemB);
                if (o_code) {
                    cp_async16(slot + 32 * lane, o_src);
                    cp_async16(slot + 32 * lane + 16, o_src + 16);
                }
                if (o_scale) cp_async16(slot + 1024 + 16 * lane, o_ssrc);
                o_src += o_cstep;
                o_ssrc += o_sstep;
            }
            ++is_i;
            if (++is_slot == kDepth) is_slot = 0;
            cp_commit();
            return;
        }
        if (is_i < total) {
            const int b = lane + 32 * is_it;
            uint8_t* slot = ring + (size_t)is_slot * kItemB;
            if (b < B) {
                const uint8_t* src = codes + (size_t)is_row * (K / 4) + 32 * (size_t)b;
                cp_async16(smem_u32(slot + 32 * lane), src);
                cp_async16(smem_u32(slot + 32 * lane + 16), src + 16);
            }
            if (lane < 4 && 32 * is_it + 8 * lane < Bp)
                cp_async16(smem_u32(slot + 1024 + 16 * lane), wscales + (size_t)is_row * Bp + 32 * is_it + 8 * lane);
            if (++is_it == steps) {
                is_it = 0;
                is_row += TW;
            }
        }
        ++is_i;
        if (++is_slot == kDepth) is_slot = 0;
        cp_commit();     // one (possibly empty) group per step keeps the wait count uniform
    };

    // Weights do not depend on the predecessor, but only kPreSteps of the
    // ring's steps go out before the dependency wait and the rest after the
    // activation input is requested: with every SM's whole ring in flight
    // the input reached the CTAs later (measured on GB300 over the merged
    // one-token pass: 6.29 us per call with all four steps issued early,
    // 6.14 with two, 6.17 with three, 6.29 with one).
    constexpr int kPreSteps = 2;
    for (int d = 0; d < kPreSteps; ++d) issue_next();
    if (FUSED && threadIdx.x == 0) rows_init(smem_u32(&xbar));
    if (FUSED && act_bf16) qtab_fill(qtab);
    if (FUSED) __syncthreads();
    pdl_wait();
    if (FUSED) {
        // the activation rows by bulk copy on their own barrier, then the
        // quantiser reads them from shared memory
        if (threadIdx.x == 0) rows_load(smem_u32(x_s), x, (uint32_t)(M * K * 2), smem_u32(&xbar));
        for (int d = kPreSteps; d < kDepth; ++d) issue_next();
        if (!rows_wait(smem_u32(&xbar), status)) {
            rows_drain(smem_u32(&xbar));
            cp_wait<0>();
            return;
        }
        for (int m = 0; m < M; ++m)
            if (act_bf16)
                quantize_row_planes8<true>(x_s + (size_t)m * K, K, AG, q_s + (size_t)m * B * kQStride, sq_s + m * B,
                                           xs_s + m * XG, red, m, kQStride, qtab);
            else
                quantize_row_planes8<false>(x_s + (size_t)m * K, K, AG, q_s + (size_t)m * B * kQStride, sq_s + m * B,
                                            xs_s + m * XG, red, m, kQStride, nullptr);
    } else {
        for (int d = kPreSteps; d < kDepth; ++d) issue_next();
        const int qv = M * K / 16;
        for (int i = threadIdx.x; i < qv; i += blockDim.x)
            *reinterpret_cast<uint4*>(q_s + (size_t)(i >> 3) * kQStride + 16 * (i & 7)) = ldg_v4(q_ws + 16 * (size_t)i);
        for (int i = threadIdx.x; i < M * B; i += blockDim.x) sq_s[i] = sq_ws[i];
        for (int i = threadIdx.x; i < M * XG; i += blockDim.x) xs_s[i] = xs_ws[i];
    }
    __syncthreads();

    if (one_step && total >= 2) {
        // one token, rows of one step (K <= 4096): lane l always takes block
        // l, so its 128 activation codes, their sum and scale stay in
        // registers and the loop reads only the weights from shared memory
        // (the same sums in the same order as the general loop below;
        // measured on GB300 over the merged one-token pass: 6.44 -> 6.30 us
        // per call).  Warps with a single row keep the general loop: there
        // the register copy cost more than it saved (4096 x 4096 alone,
        // 3.88 against 4.07 us per call).
        const bool valid = lane < B;
        uint32_t qr[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint4 v = valid ? *reinterpret_cast<const uint4*>(q_s + (size_t)lane * kQStride + 16 * j)
                                  : make_uint4(0u, 0u, 0u, 0u);
            qr[4 * j] = v.x; qr[4 * j + 1] = v.y; qr[4 * j + 2] = v.z; qr[4 * j + 3] = v.w;
        }
        const int sqb = valid ? sq_s[lane] : 0;
        const float xsb = (AG == kGroup && valid) ? xs_s[lane] : 1.f;
        const float xrow = xs_s[0];
        int rs1 = 0, n1 = gw;
        for (int i = 0; i < total; ++i) {
            cp_wait<kDepth - 1>();
            __syncwarp();
            const uint8_t* slot = ring + (size_t)rs1 * kItemB;
            if (++rs1 == kDepth) rs1 = 0;
            const uint4 cw0 = *reinterpret_cast<const uint4*>(slot + 32 * lane);
            const uint4 cw1 = *reinterpret_cast<const uint4*>(slot + 32 * lane + 16);
            const float ws = valid ? __half2float(__ushort_as_half(
                                         reinterpret_cast<const uint16_t*>(slot + 1024)[lane])) : 0.f;
            __syncwarp();
            issue_next();
            float term = 0.f;
            if (valid) {
                const int S = block_dot_reg(cw0, cw1, qr) - sqb;
                term = (float)S * ws;
                if (AG == kGroup) term *= xsb;
            }
            float v = warp_sum_f(0.f + term);
            if (AG != kGroup) v *= xrow;
            if (lane == 0) y[n1] = from_float(v, out_bf16 != 0);
            n1 += TW;
        }
        cp_wait<0>();
        return;
    }

    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.f;
    int rs = 0, it = 0, n = gw;
    for (int i = 0; i < total; ++i) {
        cp_wait<kDepth - 1>();
        __syncwarp();
        const uint8_t* slot = ring + (size_t)rs * kItemB;
        if (++rs == kDepth) rs = 0;
        const uint4 cw0 = *reinterpret_cast<const uint4*>(slot + 32 * lane);
        const uint4 cw1 = *reinterpret_cast<const uint4*>(slot + 32 * lane + 16);
        const int b = lane + 32 * it;
        const bool valid = b < B;
        const float ws = valid ? __half2float(__ushort_as_half(
                                     reinterpret_cast<const uint16_t*>(slot + 1024)[lane])) : 0.f;
        __syncwarp();                             // slot fully read before it is refilled
        issue_next();
        if (valid) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m < M) {
                    const int8_t* qb = q_s + ((size_t)m * B + b) * kQStride;
                    const int dot = chunk_dot(cw0, qb, 0) + chunk_dot(cw1, qb, 1);
                    const int S = dot - sq_s[m * B + b];      // exact block sum of (code-1)*q
                    float term = (float)S * ws;
                    if (AG == kGroup) term *= xs_s[m * XG + b];
                    acc[m] += term;
                }
            }
        }
        if (++it == steps) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m < M) {
                    float v = warp_sum_f(acc[m]);
                    if (AG != kGroup) v *= xs_s[m * XG];
                    if (lane == 0) y[(size_t)m * N + n] = from_float(v, out_bf16 != 0);
                }
                acc[m] = 0.f;
            }
            it = 0;
            n += TW;
        }
    }
    cp_wait<0>();
}

// Split-K ternary decode for M = 2..16 on the int8 tensor cores
// (mma.sync m16n8k32, s8 x s8 -> exact s32).  The K order inside a block is
// the plane order the quantiser writes: k32 step s of a block takes plane s,
// and its k-slots 4t..4t+3 / 16+4t..16+4t+3 are plane words t / 4+t, i.e.
// in-block weights 16w+4i+s.  So the A fragment of lane (g, t) is
// (code word w >> 2s) & 0x03030303 of rows g and g+8 for w = t, 4+t -- the
// codes 0..2 as int8 -- and the B fragment is the same plane words of the
// activation codes; the block sum of (code - 1) * q is the s32 result minus
// the block's sum of q, exact as in the CUDA-core kernel.
// Work tile = (block of 8 strips, K slice of kW2SliceBlocks blocks): the 8
// warps of a CTA take the 8 strips of a block on the CTA's one slice, the
// CTA stages the slice's activation codes of all tokens once, each warp
// writes fp32 partial sums of its strip, and a second launch adds the
// slices in fixed order (deterministic).
namespace w2sk {
constexpr int SB = kW2SliceBlocks;         // blocks per slice
// a row's block scales of a slice are copied as 16-byte chunks (8 scales):
// the slice must start on an 8-block boundary of the scale plane
static_assert(SB % 8 == 0, "ternary split-K slices must be a multiple of 8 blocks");
constexpr int D = 2;                       // slices in flight per warp
constexpr int CODE_B = SB * 512;           // [block][16 rows][32 code bytes]
constexpr int SC_B = 16 * SB * 2;          // [16 rows][SB] fp16 block scales
constexpr int ITEM_B = CODE_B + SC_B;
constexpr int RING = kWarps * D * ITEM_B;
constexpr int QROW_B = SB * kGroup + 16;   // one token's codes of the slice + 16 B
constexpr int Q_B = 16 * QROW_B;
constexpr int SQ_B = 16 * SB * 4;          // [16 tokens][SB] int32 block sums of q
constexpr int XS_B = 16 * SB * 4;          // [16 tokens][SB] activation scales
constexpr size_t SMEM = (size_t)RING + Q_B + SQ_B + XS_B;
}  // namespace w2sk

__device__ __forceinline__ void imma16832(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int NT, bool AG128>
__global__ void __launch_bounds__(kWarps * 32)
w2_tc_kernel(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ wscales,
             const int8_t* __restrict__ q_ws, const int32_t* __restrict__ sq_ws, const float* __restrict__ xs_ws,
             float* __restrict__ part, int M, int Npad, int K, int Bp, int nslices, int cps) {
    using namespace w2sk;
    extern __shared__ __align__(16) uint8_t smem[];

    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int B = K / kGroup;
    const int slice = (int)blockIdx.x % nslices, c = (int)blockIdx.x / nslices;
    const int bb = slice * SB, nb = B - bb < SB ? B - bb : SB;
    const int nstrips = Npad / kStrip;
    const int nblk = (nstrips + kWarps - 1) / kWarps;
    int total = c < nblk ? (nblk - 1 - c) / cps + 1 : 0;
    if (total > 0 && kWarps * (c + (total - 1) * cps) + warp >= nstrips) --total;
    uint8_t* ring = smem + (size_t)warp * D * ITEM_B;
    uint8_t* q_s = smem + RING;
    int32_t* sq_s = reinterpret_cast<int32_t*>(smem + RING + Q_B);
    float* xs_s = reinterpret_cast<float*>(smem + RING + Q_B + SQ_B);

    // copy lane: row r = lane / 2, 16-byte half h = lane % 2 of each block;
    // rows 4..7 (mod 8) store their halves swapped, so the four word loads of
    // a fragment never share a bank
    const int cr = lane >> 1, ch = lane & 1;
    const int cdst = cr * 32 + ((ch ^ ((cr >> 2) & 1)) << 4);
    int is_i = 0, is_slot = 0;
    auto issue_next = [&]() {
        if (is_i < total) {
            const int n0 = (kWarps * (c + is_i * cps) + warp) * kStrip;
            uint8_t* slot = ring + (size_t)is_slot * ITEM_B;
            const uint8_t* src = codes + (size_t)(n0 + cr) * (K / 4) + (size_t)bb * 32 + 16 * ch;
            for (int j = 0; j < nb; ++j) cp_async16(smem_u32(slot + j * 512 + cdst), src + 32 * j);
            // block scales: 16 rows x SB fp16, one 16-byte chunk per row
            if (lane < 16)
                cp_async16(smem_u32(slot + CODE_B + 16 * lane), wscales + (size_t)(n0 + lane) * Bp + bb);
        }
        ++is_i;
        if (++is_slot == D) is_slot = 0;
        cp_commit();
    };

    for (int d = 0; d < D; ++d) issue_next();          // weights before the dependency wait
    pdl_wait();
    // the slice's activation codes, block sums and scales of all 16 tokens
    // (tokens >= M and blocks past K are zero-filled)
    for (int i = threadIdx.x; i < 16 * SB * 8; i += blockDim.x) {
        const int m = i / (SB * 8), j = (i / 8) % SB, cc = i % 8;
        const bool ok = m < M && j < nb;
        cp_async16_zfill(smem_u32(q_s + m * QROW_B + j * kGroup + 16 * cc),
                         ok ? q_ws + (size_t)m * K + (size_t)(bb + j) * kGroup + 16 * cc : q_ws, ok);
    }
    for (int i = threadIdx.x; i < 16 * SB; i += blockDim.x) {
        const int m = i / SB, j = i % SB;
        const bool ok = m < M && j < nb;
        sq_s[i] = ok ? sq_ws[(size_t)m * B + bb + j] : 0;
        xs_s[i] = ok ? (AG128 ? xs_ws[(size_t)m * B + bb + j] : xs_ws[m]) : 0.f;
    }
    cp_commit();
    cp_wait<0>();
    __syncthreads();

    // per-lane shared-memory offsets of the fragments
    const int wrow = (((0 ^ ((g >> 2) & 1)) << 4) | (4 * t)) + g * 32;    // row g, word t (half 0)
    const int wrow4 = ((((1 ^ ((g >> 2) & 1)) << 4) | (4 * t))) + g * 32; // row g, word 4+t (half 1)
    int rs = 0;
    for (int i = 0; i < total; ++i) {
        const int strip = kWarps * (c + i * cps) + warp, n0 = strip * kStrip;
        cp_wait<D - 1>();
        __syncwarp();
        const uint8_t* slot = ring + (size_t)rs * ITEM_B;
        if (++rs == D) rs = 0;
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        for (int j = 0; j < nb; ++j) {
            const uint8_t* cb = slot + j * 512;
            const uint32_t c0 = *reinterpret_cast<const uint32_t*>(cb + wrow);        // row g, word t
            const uint32_t c1 = *reinterpret_cast<const uint32_t*>(cb + 256 + wrow);  // row g+8, word t
            const uint32_t c2 = *reinterpret_cast<const uint32_t*>(cb + wrow4);       // row g, word 4+t
            const uint32_t c3 = *reinterpret_cast<const uint32_t*>(cb + 256 + wrow4); // row g+8, word 4+t
            const uint16_t* scr = reinterpret_cast<const uint16_t*>(slot + CODE_B);
            const float wsa = __half2float(__ushort_as_half(scr[g * SB + j]));
            const float wsb = __half2float(__ushort_as_half(scr[(g + 8) * SB + j]));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint8_t* qb = q_s + (nt * 8 + g) * QROW_B + j * kGroup + 4 * t;
                int d[4] = {0, 0, 0, 0};
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint32_t b0 = *reinterpret_cast<const uint32_t*>(qb + 32 * s);
                    const uint32_t b1 = *reinterpret_cast<const uint32_t*>(qb + 32 * s + 16);
                    imma16832(d, (c0 >> (2 * s)) & 0x03030303u, (c1 >> (2 * s)) & 0x03030303u,
                              (c2 >> (2 * s)) & 0x03030303u, (c3 >> (2 * s)) & 0x03030303u, b0, b1);
                }
                // d: rows g / g+8 x tokens nt*8 + 2t, +1; subtract the block sums of q
                const int m0 = nt * 8 + 2 * t;
                const int s0 = d[0] - sq_s[m0 * SB + j], s1 = d[1] - sq_s[(m0 + 1) * SB + j];
                const int s2 = d[2] - sq_s[m0 * SB + j], s3 = d[3] - sq_s[(m0 + 1) * SB + j];
                if (AG128) {
                    const float x0 = xs_s[m0 * SB + j], x1 = xs_s[(m0 + 1) * SB + j];
                    acc[nt][0] = fmaf((float)s0 * wsa, x0, acc[nt][0]);
                    acc[nt][1] = fmaf((float)s1 * wsa, x1, acc[nt][1]);
                    acc[nt][2] = fmaf((float)s2 * wsb, x0, acc[nt][2]);
                    acc[nt][3] = fmaf((float)s3 * wsb, x1, acc[nt][3]);
                } else {
                    acc[nt][0] = fmaf((float)s0, wsa, acc[nt][0]);
                    acc[nt][1] = fmaf((float)s1, wsa, acc[nt][1]);
                    acc[nt][2] = fmaf((float)s2, wsb, acc[nt][2]);
                    acc[nt][3] = fmaf((float)s3, wsb, acc[nt][3]);
                }
            }
        }
        __syncwarp();                                    // slot read: refill it
        issue_next();
        float* ps = part + ((size_t)slice * Npad + n0) * 16;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            *reinterpret_cast<float2*>(ps + g * 16 + nt * 8 + 2 * t) = make_float2(acc[nt][0], acc[nt][1]);
            *reinterpret_cast<float2*>(ps + (g + 8) * 16 + nt * 8 + 2 * t) = make_float2(acc[nt][2], acc[nt][3]);
        }
    }
    cp_wait<0>();
}

// Pre-pass: one CTA per activation row into the workspace; the row is
// staged in dynamic shared memory (K * 2 bytes).
template <bool PLANE>
__global__ void __launch_bounds__(kThreads)
w2_quantize_kernel(const uint16_t* __restrict__ x, int act_bf16, int K, int AG, int8_t* q8,
                   uint16_t* qbf, int32_t* sq, float* xs, uint32_t* status) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ float red[33];
    __shared__ __align__(8) uint64_t xbar;
    __shared__ float qtab[2 * kQTab];
    uint16_t* x_s = reinterpret_cast<uint16_t*>(smem);
    pdl_trigger();
    if (threadIdx.x == 0) rows_init(smem_u32(&xbar));
    if (act_bf16) qtab_fill(qtab);
    __syncthreads();
    pdl_wait();
    const int m = blockIdx.x;
    if (threadIdx.x == 0) rows_load(smem_u32(x_s), x + (size_t)m * K, (uint32_t)K * 2, smem_u32(&xbar));
    if (!rows_wait(smem_u32(&xbar), status)) {
        rows_drain(smem_u32(&xbar));
        return;
    }
    int8_t* qm = PLANE ? q8 + (size_t)m * K : nullptr;
    uint16_t* qbm = PLANE ? nullptr : qbf + (size_t)m * K;
    if (act_bf16)
        quantize_row<PLANE, true>(x_s, K, AG, qm, qbm, sq + (size_t)m * (K / kGroup), xs + (size_t)m * (K / AG), red, 0,
                                  qtab);
    else
        quantize_row<PLANE, false>(x_s, K, AG, qm, qbm, sq + (size_t)m * (K / kGroup), xs + (size_t)m * (K / AG), red, 0,
                                   nullptr);
}

// Fused activation producer ("Kernel experiments: recorded evidence",
// section E, Test 18 and Diagram 5): residual add, RMSNorm, the optional
// random-sign Hadamard transform and the group quantiser in one pass over a
// token row, so the normalised row never goes back to memory.  One CTA of
// kThreads threads per row; every step is fp32 with the two roundings to
// the activation dtype the page makes.  The floating point decides int8
// codes, so every operation is an explicitly rounded fp32 operation
// (__fadd_rn / __fmul_rn; nothing is contracted into an FMA, and the one
// FMA form used, RN(+-1 * v + o), rounds exactly a sum or difference) in a
// fixed order:
//   * sum of squares over 2048 lanes, lane i taking elements i, i + 2048, ...
//     in turn (the page's 2048-wide accumulator; thread t owns lanes
//     8t..8t+7), then the lanes added by halving (i += i + h, h = 1024..1);
//   * inv = RN(1 / RN(sqrt(RN(RN(sum / K) + eps))));
//   * n = RN_act(RN(u * inv) * w), w = gamma (+ 1 when unit_offset);
//   * transform: sign flip, butterflies (a, b) -> (a + b, a - b) at strides
//     1, 2, ..., B/2 inside each block of B, times RN(1/sqrt(B)), RN_act;
//   * then quantize_row, the same code as the quantise pre-pass.
// The residual output is written in the second pass, which reads h and r
// again element by element before writing, so r_out may be h or r itself.
constexpr int kNormLanes = 2048;
static_assert(kNormLanes == 8 * kThreads, "one 16-byte chunk of lanes per thread");

template <bool BF16IN>
__device__ __forceinline__ void load8(const uint16_t* src, float (&v)[8]) {
    unpack8<BF16IN>(*reinterpret_cast<const uint4*>(src), v);
}

template <bool BF16IN>
__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        w[j] = (uint32_t)from_float(v[2 * j], BF16IN) | ((uint32_t)from_float(v[2 * j + 1], BF16IN) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <bool BF16IN>
__device__ __forceinline__ void residual8(const uint16_t* h, const uint16_t* r, size_t k, float (&u)[8]) {
    load8<BF16IN>(h + k, u);
    if (r) {
        float b[8];
        load8<BF16IN>(r + k, b);
#pragma unroll
        for (int j = 0; j < 8; ++j) u[j] = __fadd_rn(u[j], b[j]);
    }
}

template <bool PLANE, bool BF16IN>
__global__ void __launch_bounds__(kThreads)
w2_norm_quant_kernel(const uint16_t* h, const uint16_t* r, uint16_t* r_out,
                     uint16_t* __restrict__ norm_out, const uint16_t* __restrict__ gamma,
                     const int8_t* __restrict__ signs, float eps, int unit_offset, int had_block, float had_scale,
                     int K, int AG, int8_t* q8, uint16_t* qbf, int32_t* sq, float* xs) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ float lanes[kNormLanes];
    __shared__ float red[33];
    __shared__ float qtab[2 * kQTab];
    uint16_t* row = reinterpret_cast<uint16_t*>(smem);        // [K] the row handed to the quantiser
    float* fbuf = lanes;                                        // transform chunk, after the sum
    pdl_trigger();
    if (BF16IN) qtab_fill(qtab);                                // ordered before use by the barriers below
    pdl_wait();
    const int tid = threadIdx.x;
    const size_t m = blockIdx.x;
    const uint16_t* hm = h + m * K;
    const uint16_t* rm = r ? r + m * K : nullptr;

    // pass 1: lane sums of u^2
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
    for (int k = 8 * tid; k < K; k += kNormLanes) {
        float u[8];
        residual8<BF16IN>(hm, rm, k, u);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], __fmul_rn(u[j], u[j]));
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) lanes[8 * tid + j] = acc[j];
    __syncthreads();
#pragma unroll 1
    for (int hh = kNormLanes / 2; hh >= 32; hh >>= 1) {
        for (int i = tid; i < hh; i += kThreads) lanes[i] = __fadd_rn(lanes[i], lanes[i + hh]);
        __syncthreads();
    }
    if (tid < 32) {                  // halving steps 16 .. 1 inside the first warp
        float x = lanes[tid];
#pragma unroll
        for (int hh = 16; hh >= 1; hh >>= 1) x = __fadd_rn(x, __shfl_down_sync(0xffffffffu, x, hh));
        if (tid == 0) lanes[0] = x;
    }
    __syncthreads();
    const float var = __fdiv_rn(lanes[0], (float)K);
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(var, eps)));
    __syncthreads();                                            // lanes[0] read: fbuf may reuse it

    // pass 2: residual out, normalised row and its transform.  Thread t holds
    // elements c0 + 8t .. c0 + 8t + 7 of each 2048-element chunk, so the
    // butterflies of strides 1, 2, 4 stay in its registers, strides 8 .. 128
    // pair lanes of one warp (shuffles) and strides 256, 512 pair warps
    // (shared memory).  Every stage forms each output with one rounded add or
    // subtract of the same two inputs as the plain stage-by-stage transform.
    int lb = 0;
    while ((1 << lb) < had_block) ++lb;
    const int lane = tid & 31;
#pragma unroll 1
    for (int c0 = 0; c0 < K; c0 += kNormLanes) {
        const int k = c0 + 8 * tid;
        const bool valid = k < K;
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (valid) {
            float u[8], w[8];
            residual8<BF16IN>(hm, rm, k, u);
            load8<BF16IN>(gamma + k, w);
            if (r_out) *reinterpret_cast<uint4*>(r_out + m * K + k) = pack8<BF16IN>(u);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float wj = unit_offset ? __fadd_rn(w[j], 1.0f) : w[j];
                v[j] = __fmul_rn(__fmul_rn(u[j], inv), wj);
            }
            const uint4 nb = pack8<BF16IN>(v);
            if (norm_out) *reinterpret_cast<uint4*>(norm_out + m * K + k) = nb;
            if (lb == 0) *reinterpret_cast<uint4*>(row + k) = nb;
            unpack8<BF16IN>(nb, v);                              // the rounded row enters the transform
            if (signs) {
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = signs[k + j] < 0 ? -v[j] : v[j];
            }
        }
        if (lb == 0) continue;                                   // uniform across the CTA
#pragma unroll
        for (int l = 0; l < 3; ++l) {
            if (l < lb) {
                const int hs = 1 << l;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (!(j & hs)) {
                        const float a = v[j], b = v[j + hs];
                        v[j] = __fadd_rn(a, b);
                        v[j + hs] = __fsub_rn(a, b);
                    }
            }
        }
        // cross-thread stages: the lower partner keeps a + b, the upper one
        // o - v = a - b, both as RN(sgn * v + o) with sgn = +-1 (the product
        // is exact, so the one rounding is that of the sum or difference)
#pragma unroll 1
        for (int l = 3; l < lb && l < 8; ++l) {
            const int mk = 1 << (l - 3);
            const float sgn = (lane & mk) ? -1.0f : 1.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = __fmaf_rn(sgn, v[j], __shfl_xor_sync(0xffffffffu, v[j], mk));
        }
#pragma unroll 1
        for (int l = 8; l < lb; ++l) {
            const int tm = 1 << (l - 3);                         // partner thread: tid ^ tm
            const float sgn = (tid & tm) ? -1.0f : 1.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) fbuf[8 * tid + j] = v[j];
            __syncthreads();
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = __fmaf_rn(sgn, v[j], fbuf[8 * (tid ^ tm) + j]);
            __syncthreads();
        }
        if (valid) {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = __fmul_rn(v[j], had_scale);
            *reinterpret_cast<uint4*>(row + k) = pack8<BF16IN>(v);
        }
    }
    __syncthreads();

    quantize_row<PLANE, BF16IN>(row, K, AG, PLANE ? q8 + m * K : nullptr, PLANE ? nullptr : qbf + m * K,
                                sq + m * (K / kGroup), xs + m * (K / AG), red, 0, BF16IN ? qtab : nullptr);
}

// Test export: plane-order workspace codes back to natural order.
__global__ void unplane_kernel(const int8_t* __restrict__ qp, int8_t* __restrict__ q, int total) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const int blk = i / kGroup, j = i % kGroup;
        q[i] = qp[(size_t)blk * kGroup + (j % 4) * 32 + j / 4];
    }
}

// Test export: exact block sums S[m][n][b] with the GEMV's chunk_dot and
// minus-one correction.  One warp per output row.
// Test export: bf16 tensor-core-order codes back to natural-order int8 (the
// inverse of the order pi in quantize_row: element e of a 16-element block
// sits at position 2e for e < 8 and 2(e - 8) + 1 otherwise).
__global__ void unorder_bf16_kernel(const uint16_t* __restrict__ qa, int8_t* __restrict__ q, int total) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const int e = i % 16, pos = e < 8 ? 2 * e : 2 * (e - 8) + 1;
        q[i] = (int8_t)__float2int_rn(__bfloat162float(__ushort_as_bfloat16(qa[i - e + pos])));
    }
}

__global__ void w2_sums_kernel(const uint8_t* __restrict__ codes, const int8_t* __restrict__ q_ws,
                               const int32_t* __restrict__ sq_ws, int32_t* __restrict__ S, int M, int N,
                               int K) {
    const int n = blockIdx.x, lane = threadIdx.x;
    const int C = K / 64, B = K / kGroup;
    for (int m = 0; m < M; ++m) {
        for (int base = 0; base < C; base += 32) {
            const int c = base + lane;
            const bool valid = c < C;
            int dot = 0;
            if (valid)
                dot = chunk_dot(ldg_v4(codes + (size_t)n * (K / 4) + 16 * (size_t)c),
                                q_ws + (size_t)m * K + (size_t)(c >> 1) * kGroup, c & 1);
            const int pair = dot + __shfl_xor_sync(0xffffffffu, dot, 1);
            if (valid && !(lane & 1))
                S[((size_t)m * N + n) * B + (c >> 1)] = pair - sq_ws[(size_t)m * B + (c >> 1)];
        }
    }
}

// Two CTAs per SM for every M: after the activations arrive the time is
// bound by instruction issue, so more warps per SM win over leaving room
// for the next launch's early weight copies (measured on GB300).
constexpr int kCtasPerSmM1 = 2;

// The grid is two CTAs per SM, so the SMs must hold two and not three: with
// room for a third, the block scheduler fills some SMs with three and leaves
// others idle (measured on GB300: the 4-bit-shaped ternary decode pass over
// 32 layers ran on 122-141 of the 152 SMs; 1.044 -> 0.936 ms once the
// request was padded).  A CTA that asks for at least 76 KB of dynamic shared
// memory leaves no room for a third (3 x (76 KB + the 1 KB the runtime
// reserves) > 228 KB).
constexpr size_t kW2TwoPerSmSmem = 76 * 1024;
inline size_t w2_launch_smem(size_t smem) { return smem < kW2TwoPerSmSmem ? kW2TwoPerSmSmem : smem; }

int w2_grid(const pq_prepared* p, int M) {
    const int need = (p->d.N + kGemvWarps - 1) / kGemvWarps;   // at least one row per warp
    const int cap = p->num_sms * (M <= 1 ? kCtasPerSmM1 : 2);
    return need < cap ? need : cap;
}

template <int MT, bool FUSED>
cudaError_t launch_gemv_t(const pq_prepared* p, const void* x, void* y, int M, const ActPlanes& a,
                          cudaStream_t s) {
    const pq_desc& d = p->d;
    const size_t smem = w2_launch_smem(w2_smem_bytes(MT, d.K, d.act_group, FUSED));
    cudaError_t e = ensure_smem<w2_gemv_kernel<MT, FUSED>>(smem);
    if (e == cudaSuccess) e = ensure_max_carveout<w2_gemv_kernel<MT, FUSED>>();
    if (e != cudaSuccess) return e;
    return launch(w2_gemv_kernel<MT, FUSED>, dim3(w2_grid(p, M)), dim3(kGemvWarps * 32), smem, s, true,
                  static_cast<const uint16_t*>(x), d.act_dtype == PQ_BF16 ? 1 : 0,
                  static_cast<const uint8_t*>(p->codes), static_cast<const uint16_t*>(p->scales),
                  static_cast<const int8_t*>(a.q8), static_cast<const int32_t*>(a.sq),
                  static_cast<const float*>(a.xs), static_cast<uint16_t*>(y), M, d.N,
                  d.K, w2_bp(d.K), d.act_group, d.out_dtype == PQ_BF16 ? 1 : 0, p->status);
}

// The pre-pass stages one activation row (K * 2 bytes) in shared memory.
template <bool PLANE>
cudaError_t quantize_smem_attr(int K) {
    const size_t smem = (size_t)K * 2;
    return smem > 48 * 1024 ? ensure_smem<w2_quantize_kernel<PLANE>>(smem) : cudaSuccess;
}

int mt_for(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16; }

// CTAs per K slice of the tensor-core decode: about two per SM in total, at
// most one per block of 8 strips.
int tc_cps(const pq_prepared* p) {
    const int ns = w2_slices(p->d.K);
    const int nblk = (p->Npad / kStrip + kWarps - 1) / kWarps;
    int cps = 2 * p->num_sms / ns;
    if (cps < 1) cps = 1;
    return cps < nblk ? cps : nblk;
}

// The same split-K decode on bf16 mma.sync (m16n8k16) with exact integer
// operands, for GB300 where the legacy int8 tensor path is slow.  A k16 step
// is one 32-bit code word u of a block (weights 16u .. 16u + 15, field f at
// bits 2f); its k-slots 2p, 2p + 1 take fields p and p + 8, so one shift and
// one LOP3 place a pair of codes in the two bf16 halves (128 + c) and one
// packed subtract of 129 gives the exact pair (c - 1).  The activations are
// the quantiser's bf16 codes in tensor-core order (position 2p of every 16
// holds element p, 2p + 1 element p + 8): the same k-slot order, so the B
// fragment is two 32-bit words.  A block's 8 MMAs accumulate its sum of
// (c - 1) * q in fp32 from zero: at most 128 * 2 * 127 in magnitude, exact,
// so the result equals the int8 kernel's bit for bit.
namespace w2bf {
constexpr int SB = kW2SliceBlocks;          // blocks per slice (the int8 kernel's slices)
constexpr int D = 2;                        // slices in flight per warp
constexpr int CODE_B = SB * 512;            // [block][16 rows][32 code bytes]
constexpr int SC_B = 16 * SB * 2;           // [16 rows][SB] fp16 block scales
constexpr int ITEM_B = CODE_B + SC_B;
constexpr int RING = kWarps * D * ITEM_B;
constexpr int QROW_B = SB * kGroup * 2 + 16;   // one token's bf16 codes of the slice + 16 B
constexpr int Q_B = 16 * QROW_B;
constexpr int XS_B = 16 * SB * 4;           // [16 tokens][SB] activation scales
constexpr size_t SMEM = (size_t)RING + Q_B + XS_B;
}  // namespace w2bf

__device__ __forceinline__ uint32_t tern_pair(uint32_t w, int p) {
    // fields p and p + 8 of a code word -> bf16 pair (c_p - 1, c_{p+8} - 1)
    const uint32_t t = lop3_and_or(w >> (2 * p), 0x00030003u, 0x43004300u);    // 128 + c in each half
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(t), "r"(0x43014301u));       // - 129
    return d;
}

template <int NT, bool AG128>
__global__ void __launch_bounds__(kWarps * 32)
w2_bf_kernel(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ wscales,
             const uint16_t* __restrict__ qa_ws, const float* __restrict__ xs_ws, float* __restrict__ part, int M,
             int Npad, int K, int Bp, int nslices, int cps) {
    using namespace w2bf;
    extern __shared__ __align__(16) uint8_t smem[];

    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int B = K / kGroup;
    const int slice = (int)blockIdx.x % nslices, c = (int)blockIdx.x / nslices;
    const int bb = slice * SB, nb = B - bb < SB ? B - bb : SB;
    const int nstrips = Npad / kStrip;
    const int nblk = (nstrips + kWarps - 1) / kWarps;
    int total = c < nblk ? (nblk - 1 - c) / cps + 1 : 0;
    if (total > 0 && kWarps * (c + (total - 1) * cps) + warp >= nstrips) --total;
    uint8_t* ring = smem + (size_t)warp * D * ITEM_B;
    uint8_t* q_s = smem + RING;
    float* xs_s = reinterpret_cast<float*>(smem + RING + Q_B);

    // copy lane: row r = lane / 2, 16-byte half h = lane % 2 of each block;
    // rows 4..7 (mod 8) store their halves swapped (the word loads of rows g
    // of a warp then fall on different banks)
    const int cr = lane >> 1, ch = lane & 1;
    const int cdst = cr * 32 + ((ch ^ ((cr >> 2) & 1)) << 4);
    int is_i = 0, is_slot = 0;
    auto issue_next = [&]() {
        if (is_i < total) {
            const int n0 = (kWarps * (c + is_i * cps) + warp) * kStrip;
            uint8_t* slot = ring + (size_t)is_slot * ITEM_B;
            const uint8_t* src = codes + (size_t)(n0 + cr) * (K / 4) + (size_t)bb * 32 + 16 * ch;
            for (int j = 0; j < nb; ++j) cp_async16(smem_u32(slot + j * 512 + cdst), src + 32 * j);
            if (lane < 16)
                cp_async16(smem_u32(slot + CODE_B + 16 * lane), wscales + (size_t)(n0 + lane) * Bp + bb);
        }
        ++is_i;
        if (++is_slot == D) is_slot = 0;
        cp_commit();
    };

    for (int d = 0; d < D; ++d) issue_next();          // weights before the dependency wait
    pdl_wait();
    // the slice's bf16 activation codes and scales of all 16 tokens (tokens
    // >= M and blocks past K zero-filled): 16 chunks of 16 bytes per block
    for (int i = threadIdx.x; i < 16 * SB * 16; i += blockDim.x) {
        const int m = i / (SB * 16), j = (i / 16) % SB, cc = i % 16;
        const bool ok = m < M && j < nb;
        cp_async16_zfill(smem_u32(q_s + m * QROW_B + j * (kGroup * 2) + 16 * cc),
                         ok ? qa_ws + (size_t)m * K + (size_t)(bb + j) * kGroup + 8 * cc : qa_ws, ok);
    }
    for (int i = threadIdx.x; i < 16 * SB; i += blockDim.x) {
        const int m = i / SB, j = i % SB;
        const bool ok = m < M && j < nb;
        xs_s[i] = ok ? (AG128 ? xs_ws[(size_t)m * B + bb + j] : xs_ws[m]) : 0.f;
    }
    cp_commit();
    cp_wait<0>();
    __syncthreads();

    // shared-memory offsets of rows g and g + 8 inside a block (two 16-byte halves each)
    const int rg0 = g * 32 + ((0 ^ ((g >> 2) & 1)) << 4), rg1 = g * 32 + ((1 ^ ((g >> 2) & 1)) << 4);
    int rs = 0;
    for (int i = 0; i < total; ++i) {
        const int strip = kWarps * (c + i * cps) + warp, n0 = strip * kStrip;
        cp_wait<D - 1>();
        __syncwarp();
        const uint8_t* slot = ring + (size_t)rs * ITEM_B;
        if (++rs == D) rs = 0;
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        for (int j = 0; j < nb; ++j) {
            const uint8_t* cb = slot + j * 512;
            const uint4 wa0 = *reinterpret_cast<const uint4*>(cb + rg0);          // row g, words 0..3
            const uint4 wa1 = *reinterpret_cast<const uint4*>(cb + rg1);          // row g, words 4..7
            const uint4 wb0 = *reinterpret_cast<const uint4*>(cb + 256 + rg0);    // row g + 8
            const uint4 wb1 = *reinterpret_cast<const uint4*>(cb + 256 + rg1);
            const uint32_t wa[8] = {wa0.x, wa0.y, wa0.z, wa0.w, wa1.x, wa1.y, wa1.z, wa1.w};
            const uint32_t wb[8] = {wb0.x, wb0.y, wb0.z, wb0.w, wb1.x, wb1.y, wb1.z, wb1.w};
            const uint16_t* scr = reinterpret_cast<const uint16_t*>(slot + CODE_B);
            const float wsa = __half2float(__ushort_as_half(scr[g * SB + j]));
            const float wsb = __half2float(__ushort_as_half(scr[(g + 8) * SB + j]));
            float d[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t a0 = tern_pair(wa[u], t), a1 = tern_pair(wb[u], t);
                const uint32_t a2 = tern_pair(wa[u], t + 4), a3 = tern_pair(wb[u], t + 4);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint8_t* qb = q_s + (nt * 8 + g) * QROW_B + (j * kGroup + 16 * u + 2 * t) * 2;
                    const uint32_t b0 = *reinterpret_cast<const uint32_t*>(qb);
                    const uint32_t b1 = *reinterpret_cast<const uint32_t*>(qb + 16);
                    asm volatile(
                        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
                        "{%8,%9}, {%0,%1,%2,%3};"
                        : "+f"(d[nt][0]), "+f"(d[nt][1]), "+f"(d[nt][2]), "+f"(d[nt][3])
                        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
                }
            }
            // d: rows g / g+8 x tokens nt*8 + 2t, +1: the exact block sums
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (AG128) {
                    const int m0 = nt * 8 + 2 * t;
                    const float x0 = xs_s[m0 * SB + j], x1 = xs_s[(m0 + 1) * SB + j];
                    acc[nt][0] = fmaf(d[nt][0] * wsa, x0, acc[nt][0]);
                    acc[nt][1] = fmaf(d[nt][1] * wsa, x1, acc[nt][1]);
                    acc[nt][2] = fmaf(d[nt][2] * wsb, x0, acc[nt][2]);
                    acc[nt][3] = fmaf(d[nt][3] * wsb, x1, acc[nt][3]);
                } else {
                    acc[nt][0] = fmaf(d[nt][0], wsa, acc[nt][0]);
                    acc[nt][1] = fmaf(d[nt][1], wsa, acc[nt][1]);
                    acc[nt][2] = fmaf(d[nt][2], wsb, acc[nt][2]);
                    acc[nt][3] = fmaf(d[nt][3], wsb, acc[nt][3]);
                }
            }
        }
        __syncwarp();                                    // slot read: refill it
        issue_next();
        float* ps = part + ((size_t)slice * Npad + n0) * 16;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            *reinterpret_cast<float2*>(ps + g * 16 + nt * 8 + 2 * t) = make_float2(acc[nt][0], acc[nt][1]);
            *reinterpret_cast<float2*>(ps + (g + 8) * 16 + nt * 8 + 2 * t) = make_float2(acc[nt][2], acc[nt][3]);
        }
    }
    cp_wait<0>();
}

template <int NT, bool AG128>
cudaError_t launch_bf_t(const pq_prepared* p, void* y, int M, const ActPlanes& a, cudaStream_t s) {
    const pq_desc& d = p->d;
    cudaError_t e = ensure_smem<w2_bf_kernel<NT, AG128>>(w2bf::SMEM);
    if (e != cudaSuccess) return e;
    const int ns = w2_slices(d.K), cps = tc_cps(p);
    e = launch(w2_bf_kernel<NT, AG128>, dim3(ns * cps), dim3(kWarps * 32), w2bf::SMEM, s, true,
                           static_cast<const uint8_t*>(p->codes), static_cast<const uint16_t*>(p->scales),
                           static_cast<const uint16_t*>(a.qa), static_cast<const float*>(a.xs),
                           reinterpret_cast<float*>(p->ws + p->wl.sk_off), M, p->Npad, d.K, w2_bp(d.K), ns, cps);
    if (e != cudaSuccess) return e;
    return pq::launch_sk_reduce(p, y, M, ns, AG128 ? nullptr : static_cast<const float*>(a.xs), s);
}

template <int NT, bool AG128>
cudaError_t launch_tc_t(const pq_prepared* p, void* y, int M, const ActPlanes& a, cudaStream_t s) {
    const pq_desc& d = p->d;
    cudaError_t e = ensure_smem<w2_tc_kernel<NT, AG128>>(w2sk::SMEM);
    if (e != cudaSuccess) return e;
    const int ns = w2_slices(d.K), cps = tc_cps(p);
    e = launch(w2_tc_kernel<NT, AG128>, dim3(ns * cps), dim3(kWarps * 32), w2sk::SMEM, s, true,
                           static_cast<const uint8_t*>(p->codes), static_cast<const uint16_t*>(p->scales),
                           static_cast<const int8_t*>(a.q8), static_cast<const int32_t*>(a.sq),
                           static_cast<const float*>(a.xs),
                           reinterpret_cast<float*>(p->ws + p->wl.sk_off), M, p->Npad, d.K, w2_bp(d.K), ns, cps);
    if (e != cudaSuccess) return e;
    // per-row activation scales multiply the slice sum (per-block ones are in the partials)
    return pq::launch_sk_reduce(p, y, M, ns, AG128 ? nullptr : static_cast<const float*>(a.xs), s);
}

// Cluster split-K ternary decode, M = 1..16, one launch from the caller's
// activations to y.  A cluster of CL CTAs covers one group of 8R strips
// (16 output rows each) over the whole K: CTA r of the cluster takes K slice
// r (SB blocks of 128, SB a multiple of 4) and the strips' weights of that
// slice, warp w the strips 8i + w of the group.
//   1. Each CTA streams its weight items (16 rows x up to 4 blocks of codes
//      and block scales) into per-warp rings before the dependency wait,
//      then stages its slice of every token row.
//   2. Per-row activation scales (act_group = K): each CTA finds every
//      token's largest |x| over its slice; after a cluster barrier it reads
//      the other CTAs' maxima from their shared memory, so every CTA holds
//      the row maxima and quantises its own slice exactly as the pre-pass
//      quantises the row (the same helpers, the same group scale).  Per-block
//      scales (act_group = 128) need nothing from the other CTAs.
//   3. The codes go to shared memory as fp16 in tensor-core order (position
//      2p of every 16 holds element p, 2p + 1 element p + 8), element e
//      multiplied by 4^-(e mod 4) (exact).  For the A operand a lane with
//      k-slot pair t takes code fields t, t + 8 of a code word with one LOP3
//      into two fp16 halves 1024 + 4^t c (the field lands in mantissa bits
//      2t, 2t + 1 below bit 10: exact for every code 0..3), and fields
//      t + 4, t + 12 after a shift by 8.  So every product is
//      1024 * 4^-t * q + c * q, an integer; a block's sum stays below 2^23
//      in magnitude and the fp32 sum is exact; the block sum of (c - 1) q is
//      that sum minus W = sum_e (1024 * 4^-(e mod 4) + 1) q_e, formed by the
//      quantiser.  The B fragments of both 8-token tiles come from one
//      ldmatrix.x4.
//   4. Each warp scales a block's exact sum by the row's block scale (and
//      the token's block scale for act_group = 128) into fp32 accumulators,
//      block by block in K order, and stores the strip's slice sums in its
//      CTA's shared memory; after a second cluster barrier every strip is
//      summed over the slices in the order 0, 1, ..., CL - 1 from the CTAs'
//      shared memory (deterministic), times the token's row scale, into y.
//      A third barrier keeps every CTA's shared memory until all have read.
// ACT: the input is a quantised-activation buffer (bf16 codes in tensor-core
// order and the fp32 scales, as the pre-pass writes them) instead of x;
// step 2 is skipped and the codes are converted in place, so the result
// equals that of the same kernel quantising x itself, bit for bit.
// Every CTA of a cluster passes every cluster barrier: there is no early exit.
namespace w2cl {
constexpr int kMaxCL = 8;                   // CTAs per cluster (portable size)
constexpr int CB = 4;                       // blocks per ring item
constexpr int D = 3;                        // items in flight per warp
constexpr int CODE_B = CB * 512;            // [block][16 rows][32 code bytes]
constexpr int ITEM_B = CODE_B + 16 * 8;     // + [16 rows][4] fp16 block scales
constexpr int RING = kWarps * D * ITEM_B;
constexpr int kMaxR = 6;                    // strips per warp
constexpr int kMaxSB = 24;                  // blocks per slice (K <= 24576)
__host__ __device__ constexpr int xrow_b(int SB) { return SB * kGroup * 2 + 16; }
// strips of a group each CTA adds up (strip s of the group goes to CTA s % CL)
__host__ __device__ constexpr int owned(int R, int CL) { return (kWarps * R + CL - 1) / CL; }
struct Lay {
    int xq, wsum, xsb, part, small, total;
};
__host__ __device__ inline Lay lay(int SB, int R, int CL) {
    Lay l;
    l.xq = RING;                                        // [16][SB*128] x, then codes (16-bit)
    l.wsum = l.xq + 16 * xrow_b(SB);                    // [16][SB] fp32 W
    l.xsb = l.wsum + 16 * SB * 4;                       // [16][SB] fp32 per-block activation scales
    l.part = l.xsb + 16 * SB * 4;                       // [owned][CL][16 rows][16 tokens] fp32 slice sums
    l.small = l.part + owned(R, CL) * CL * 1024;        // amax[kMaxCL][16] u32 | rs, rn, plain [16] | mbarrier
    l.total = l.small + kMaxCL * 16 * 4 + 3 * 16 * 4 + 16;
    return l;
}
}  // namespace w2cl

__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" :: "r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(a));
}
__device__ __forceinline__ void ldsm_x2(uint32_t a, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(a));
}
// fp16 pair (lo, hi) = (q0 * sc, q1 * sc) from t = 0x4B400000 + q words
// (the quantiser's form); exact for |q| <= 127 and sc a power of two.
__device__ __forceinline__ uint32_t scaled_codes_f16x2(uint32_t t0, uint32_t t1, float sc) {
    uint32_t r;
    asm("{\n\t.reg .b64 a, s, c, v;\n\t.reg .f32 lo, hi;\n\t"
        "mov.b64 a, {%1, %2};\n\t"
        "mov.b64 s, {%3, %3};\n\t"
        "mov.b64 c, {%4, %4};\n\t"
        "fma.rn.f32x2 v, a, s, c;\n\t"
        "mov.b64 {lo, hi}, v;\n\t"
        "cvt.rn.f16x2.f32 %0, hi, lo;\n\t}"
        : "=r"(r)
        : "r"(t0), "r"(t1), "f"(sc), "f"(-12582912.0f * sc));
    return r;
}
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int NT, bool AG128, bool BF16IN, bool ACT>
__global__ void __launch_bounds__(kWarps * 32, 2)
w2_cl_kernel(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ wscales,
             const uint16_t* __restrict__ x, const float* __restrict__ xs_act, uint16_t* __restrict__ y,
             uint32_t* __restrict__ status, int M, int N, int Npad, int K, int Bp, int SB, int R, int out_bf16) {
    using namespace w2cl;
    extern __shared__ __align__(16) uint8_t smem[];
    pdl_trigger();
    int ncl;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(ncl));
    const Lay L = lay(SB, R, ncl);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int B = K / kGroup;
    const int rank = (int)cluster_ctarank();
    const int grp = (int)blockIdx.x / ncl;
    const int bb0 = rank * SB, nbs = B - bb0 < SB ? (B - bb0 > 0 ? B - bb0 : 0) : SB;   // blocks of this slice
    const int nch = (nbs + CB - 1) / CB;                                                  // ring items per strip
    const int nstrips = Npad / kStrip;
    uint8_t* ring = smem + (size_t)warp * D * ITEM_B;
    uint8_t* xq = smem + L.xq;
    float* wsum = reinterpret_cast<float*>(smem + L.wsum);
    float* xsb = reinterpret_cast<float*>(smem + L.xsb);
    float* part = reinterpret_cast<float*>(smem + L.part);
    uint32_t* amax = reinterpret_cast<uint32_t*>(smem + L.small);          // [kMaxCL][16]: CTA q's maxima
    float* rs_s = reinterpret_cast<float*>(smem + L.small + kMaxCL * 64);
    float* rn_s = reinterpret_cast<float*>(smem + L.small + kMaxCL * 64 + 64);
    uint32_t* pl_s = reinterpret_cast<uint32_t*>(smem + L.small + kMaxCL * 64 + 128);
    uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + L.small + kMaxCL * 64 + 192);
    if (threadIdx.x == 0) rows_init(smem_u32(xbar));
    __syncthreads();

    // this warp's items: strip i (0..R-1) of the group, chunk c of the slice
    const int nitems = R * nch;
    auto strip_of = [&](int i) { return grp * kWarps * R + kWarps * i + warp; };
    const int cr = lane >> 1, chh = lane & 1;
    const int cdst = cr * 32 + ((chh ^ ((cr >> 2) & 1)) << 4);
    int is_i = 0, is_slot = 0;
    auto issue_next = [&]() {
        if (is_i < nitems) {
            const int i = is_i / nch, c = is_i % nch;
            const int st = strip_of(i);
            if (st < nstrips) {
                const int n0 = st * kStrip, bb = bb0 + c * CB;
                const int nb = B - bb < CB ? B - bb : CB;
                uint8_t* slot = ring + (size_t)is_slot * ITEM_B;
                const uint8_t* src = codes + (size_t)(n0 + cr) * (K / 4) + (size_t)bb * 32 + 16 * chh;
                for (int j = 0; j < nb; ++j) cp_async16(smem_u32(slot + j * 512 + cdst), src + 32 * j);
                if (lane < 16) cp_async8(smem_u32(slot + CODE_B + 8 * lane), wscales + (size_t)(n0 + lane) * Bp + bb);
            }
        }
        ++is_i;
        if (++is_slot == D) is_slot = 0;
        cp_commit();
    };
    for (int d = 0; d < D; ++d) issue_next();          // weights before the dependency wait
    // barrier 0: no CTA stores into another's shared memory before all have
    // started (arrive now, wait before the first such store)
    cluster_arrive_relaxed();
    pdl_wait();

    // ---- stage this slice of the M token rows: one bulk copy per row on an
    //      mbarrier (not a cp.async group, so waiting for it does not wait
    //      for the weight items issued before).  Rows >= M and blocks past K
    //      are never read as codes (the quantiser writes zeros there).
    const int XR = xrow_b(SB);
    if (threadIdx.x == 0) {
        const uint32_t bytes = (uint32_t)nbs * kGroup * 2;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                     :: "r"(smem_u32(xbar)), "r"(bytes * (uint32_t)M) : "memory");
        for (int m = 0; m < M; ++m)
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                :: "r"(smem_u32(xq + m * XR)), "l"(x + (size_t)m * K + (size_t)bb0 * kGroup), "r"(bytes),
                   "r"(smem_u32(xbar)) : "memory");
    }
    // on a timeout the status word is set; the CTA still passes every
    // cluster barrier (its outputs are then not meaningful)
    if (!rows_wait(smem_u32(xbar), status)) rows_drain(smem_u32(xbar));

    // ---- row maxima over the slice, stored into every CTA of the cluster
    //      (slot `rank`), then over the cluster (act_group = K)
    cluster_wait();                                     // barrier 0
    if (!AG128 && !ACT) {
        for (int m = warp; m < M; m += kWarps) {
            uint32_t mb = 0;
            for (int cc = lane; cc < nbs * 16; cc += 32)
                mb = max(mb, chunk_absmax_bits(*reinterpret_cast<const uint4*>(xq + m * XR + 16 * cc)));
            mb = __reduce_max_sync(0xffffffffu, mb);
            if (lane < ncl) dsmem_st_u32(dsmem_map(smem_u32(amax + rank * 16 + m), (uint32_t)lane), mb);
        }
        cluster_arrive();                               // barrier 1: every CTA's maxima stored
        cluster_wait();
    }
    if (!AG128 && ACT && threadIdx.x < M) rs_s[threadIdx.x] = xs_act[threadIdx.x];
    if (!AG128 && !ACT && threadIdx.x < M) {
        const int m = threadIdx.x;
        uint32_t mb = 0;
#pragma unroll
        for (int q = 0; q < kMaxCL; ++q)             // unrolled: the loads go out together
            if (q < ncl) mb = max(mb, amax[q * 16 + m]);
        const QDiv dv = make_qdiv(group_scale(bits16_to_float<BF16IN>(mb)));
        rs_s[m] = dv.s;
        rn_s[m] = dv.rn;
        pl_s[m] = dv.plain ? 1u : 0u;
    }
    __syncthreads();

    // ---- quantise the slice in place: 16-element unit u of token m per thread
    //      (a 128-block is 8 consecutive threads); codes to fp16 x 4^-(e mod 4)
    {
        const int upr = SB * 8;                          // units per token row of the slice
        for (int i = threadIdx.x; i < 16 * upr; i += blockDim.x) {
            const int m = i / upr, u = i % upr;
            // ok is the same for the 8 threads of a block (one token, one block)
            const bool ok = m < M && u < nbs * 8;
            uint8_t* ux = xq + m * XR + 32 * u;
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            const uint4 ulo = ok ? *reinterpret_cast<const uint4*>(ux) : z;       // rows >= M were never staged
            const uint4 uhi = ok ? *reinterpret_cast<const uint4*>(ux + 16) : z;
            uint32_t tq[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) tq[j] = kQMagic;                        // q = 0
            int w = 0;
            if (ACT) {
                // the codes as the pre-pass wrote them: word p holds elements
                // p and p + 8 as bf16 (exact integers)
                if (ok) {
                    const uint32_t wi[8] = {ulo.x, ulo.y, ulo.z, ulo.w, uhi.x, uhi.y, uhi.z, uhi.w};
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        tq[j] = kQMagic + (uint32_t)(int)__uint_as_float(wi[j] << 16);
                        tq[8 + j] = kQMagic + (uint32_t)(int)__uint_as_float(wi[j] & 0xFFFF0000u);
                    }
                }
                if (AG128 && (u & 7) == 0) xsb[m * SB + u / 8] = ok ? xs_act[(size_t)m * B + bb0 + u / 8] : 0.f;
            }
            QDiv dv;
            if (ACT) {
                dv.s = 0.f;
                dv.rn = 0.f;
                dv.plain = false;
            } else if (AG128) {
                uint32_t mb = max(chunk_absmax_bits(ulo), chunk_absmax_bits(uhi));
#pragma unroll
                for (int o = 4; o > 0; o >>= 1) mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, o));
                dv = make_qdiv(group_scale(bits16_to_float<BF16IN>(mb)));
                if ((u & 7) == 0) xsb[m * SB + u / 8] = ok ? dv.s : 0.f;
            } else {
                dv.s = rs_s[m];
                dv.rn = rn_s[m];
                dv.plain = pl_s[m] != 0;
            }
            if (ok && !ACT) {
                float a[16];
                {
                    float lo[8], hi[8];
                    unpack8<BF16IN>(ulo, lo);
                    unpack8<BF16IN>(uhi, hi);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        a[j] = lo[j];
                        a[8 + j] = hi[j];
                    }
                }
                if (dv.plain) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) tq[j] = kQMagic + (uint32_t)quant_one(a[j], dv.s);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; j += 2) quant_pair(a[j], a[j + 1], dv, tq[j], tq[j + 1]);
                }
            }
            // W over the unit: weights 1025, 257, 65, 17 for e mod 4 = 0..3
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int q = (int)(tq[j] - kQMagic);
                w += q * (j % 4 == 0 ? 1025 : j % 4 == 1 ? 257 : j % 4 == 2 ? 65 : 17);
            }
#pragma unroll
            for (int o = 4; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
            if ((u & 7) == 0) wsum[m * SB + u / 8] = (float)w;
            // word j: elements j and j + 8 times 4^-(j mod 4), exact, as fp16:
            // (magic + q) * sc - magic * sc in one packed FMA
            uint32_t wd[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float sc = j % 4 == 0 ? 1.f : j % 4 == 1 ? 0.25f : j % 4 == 2 ? 0.0625f : 0.015625f;
                wd[j] = scaled_codes_f16x2(tq[j], tq[8 + j], sc);
            }
            *reinterpret_cast<uint4*>(ux) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
            *reinterpret_cast<uint4*>(ux + 16) = make_uint4(wd[4], wd[5], wd[6], wd[7]);
        }
    }
    __syncthreads();

    const uint32_t msk = 0x00030003u << (2 * t);
    // ---- the strips: exact block sums on fp16 mma.sync, scaled into fp32
    const int rg0 = g * 32 + ((0 ^ ((g >> 2) & 1)) << 4), rg1 = g * 32 + ((1 ^ ((g >> 2) & 1)) << 4);
    // ldmatrix row of this lane: token (lane & 7) + 8 (lane >> 4), 16-byte half (lane >> 3) & 1
    const uint32_t bl = smem_u32(xq) + (uint32_t)(((lane & 7) + 8 * (lane >> 4)) * XR + ((lane >> 3) & 1) * 16);
    int rsl = 0;
    float acc[NT][4];
    for (int it = 0; it < nitems; ++it) {
        const int i = it / nch, c = it % nch;
        const int st = strip_of(i);
        cp_wait<D - 1>();
        __syncwarp();
        const uint8_t* slot = ring + (size_t)rsl * ITEM_B;
        if (++rsl == D) rsl = 0;
        if (c == 0) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        }
        if (st < nstrips) {
            const int jb = c * CB, nb = nbs - jb < CB ? nbs - jb : CB;
            const uint16_t* scr = reinterpret_cast<const uint16_t*>(slot + CODE_B);
            for (int jj = 0; jj < nb; ++jj) {
                const int j = jb + jj;                  // block of the slice
                const uint8_t* cb = slot + jj * 512;
                const uint4 wa0 = *reinterpret_cast<const uint4*>(cb + rg0);
                const uint4 wa1 = *reinterpret_cast<const uint4*>(cb + rg1);
                const uint4 wb0 = *reinterpret_cast<const uint4*>(cb + 256 + rg0);
                const uint4 wb1 = *reinterpret_cast<const uint4*>(cb + 256 + rg1);
                const uint32_t wa[8] = {wa0.x, wa0.y, wa0.z, wa0.w, wa1.x, wa1.y, wa1.z, wa1.w};
                const uint32_t wb[8] = {wb0.x, wb0.y, wb0.z, wb0.w, wb1.x, wb1.y, wb1.z, wb1.w};
                float d[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
                const uint32_t bj = bl + (uint32_t)(j * kGroup * 2);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const uint32_t a0 = lop3_and_or(wa[u], msk, 0x64006400u);
                    const uint32_t a1 = lop3_and_or(wb[u], msk, 0x64006400u);
                    const uint32_t a2 = lop3_and_or(wa[u] >> 8, msk, 0x64006400u);
                    const uint32_t a3 = lop3_and_or(wb[u] >> 8, msk, 0x64006400u);
                    if (NT == 2) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(bj + 32 * u, b0, b1, b2, b3);
                        mma_f16(d[0], a0, a1, a2, a3, b0, b1);
                        mma_f16(d[NT - 1], a0, a1, a2, a3, b2, b3);
                    } else {
                        uint32_t b0, b1;
                        ldsm_x2(bj + 32 * u, b0, b1);
                        mma_f16(d[0], a0, a1, a2, a3, b0, b1);
                    }
                }
                const float wsa = __half2float(__ushort_as_half(scr[g * 4 + jj]));
                const float wsb = __half2float(__ushort_as_half(scr[(g + 8) * 4 + jj]));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int m0 = nt * 8 + 2 * t;
                    const float W0 = wsum[m0 * SB + j], W1 = wsum[(m0 + 1) * SB + j];
                    const float s0 = d[nt][0] - W0, s1 = d[nt][1] - W1;
                    const float s2 = d[nt][2] - W0, s3 = d[nt][3] - W1;
                    if (AG128) {
                        const float x0 = xsb[m0 * SB + j], x1 = xsb[(m0 + 1) * SB + j];
                        acc[nt][0] = fmaf(s0 * wsa, x0, acc[nt][0]);
                        acc[nt][1] = fmaf(s1 * wsa, x1, acc[nt][1]);
                        acc[nt][2] = fmaf(s2 * wsb, x0, acc[nt][2]);
                        acc[nt][3] = fmaf(s3 * wsb, x1, acc[nt][3]);
                    } else {
                        acc[nt][0] = fmaf(s0, wsa, acc[nt][0]);
                        acc[nt][1] = fmaf(s1, wsa, acc[nt][1]);
                        acc[nt][2] = fmaf(s2, wsb, acc[nt][2]);
                        acc[nt][3] = fmaf(s3, wsb, acc[nt][3]);
                    }
                }
            }
        }
        __syncwarp();                                   // slot read: refill it
        issue_next();
        if (c == nch - 1) {
            // this slice's sums of strip i (rows g, g + 8 x tokens nt*8 + 2t, + 1)
            // into slot `rank` of the owning CTA's shared memory
            const int sg = kWarps * i + warp;
            const uint32_t ps = dsmem_map(smem_u32(part + ((size_t)(sg / ncl) * ncl + rank) * 256),
                                          (uint32_t)(sg % ncl));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                dsmem_st_f2(ps + 4u * (g * 16 + nt * 8 + 2 * t), acc[nt][0], acc[nt][1]);
                dsmem_st_f2(ps + 4u * ((g + 8) * 16 + nt * 8 + 2 * t), acc[nt][2], acc[nt][3]);
            }
        }
    }
    cp_wait<0>();
    cluster_arrive();                                   // barrier 2: every slice sum stored
    cluster_wait();

    // ---- the strips this CTA owns (s % CL == rank), one warp each, from its
    //      own shared memory; lane: row r = lane / 2, tokens 8h .. 8h + 7.
    //      No CTA touches another's shared memory after barrier 2.
    {
        const int r = lane >> 1, h = lane & 1;
        const int nsg = kWarps * R;                     // strips of the group
        for (int o = warp; o < owned(R, ncl); o += kWarps) {
            const int sg = o * ncl + rank;
            const int st = grp * nsg + sg;
            if (sg >= nsg || st >= nstrips) continue;
            const float* src = part + (size_t)o * ncl * 256 + r * 16 + 8 * h;
            float a8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int q = 0; q < kMaxCL; ++q) {          // unrolled: the loads go out together, the adds in slice order
                if (q < ncl) {
                    const float4 v0 = *reinterpret_cast<const float4*>(src + q * 256);
                    const float4 v1 = *reinterpret_cast<const float4*>(src + q * 256 + 4);
                    a8[0] += v0.x; a8[1] += v0.y; a8[2] += v0.z; a8[3] += v0.w;
                    a8[4] += v1.x; a8[5] += v1.y; a8[6] += v1.z; a8[7] += v1.w;
                }
            }
            const int n = st * kStrip + r;
            if (n < N) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int m = 8 * h + j;
                    if (m < M) y[(size_t)m * N + n] = from_float(AG128 ? a8[j] : a8[j] * rs_s[m], out_bf16 != 0);
                }
            }
        }
    }
}

}  // namespace

namespace pq {

bool w2_gemv_fits(const pq_desc& d, int M, bool fused) {
    if (M > 16 || (fused && M > 4)) return false;
    return w2_smem_bytes(mt_for(M), d.K, d.act_group, fused) <= 224 * 1024;
}

void plan_w2_gemv(const pq_prepared* p, int M, bool fused, pq_plan_info* info) {
    info->variant = fused ? PQ_VARIANT_W2_GEMV_FUSED : PQ_VARIANT_W2_GEMV;
    info->grid = w2_grid(p, M);
    info->block = kGemvWarps * 32;
    info->smem_bytes = (int)w2_launch_smem(w2_smem_bytes(mt_for(M), p->d.K, p->d.act_group, fused));
    info->launches = fused ? 1 : 2;
    info->m_tile = mt_for(M);
    info->k_split = 1;
}

bool w2_tc_runs(const pq_prepared* p, int M) {
    return p->d.fmt == PQ_FMT_W2_PQ2 && M >= 1 && M <= 16 && p->wl.sk_bytes > 0;
}

void plan_w2_tc(const pq_prepared* p, int M, pq_plan_info* info) {
    info->variant = PQ_VARIANT_W2_GEMV_TC;
    info->grid = w2_slices(p->d.K) * tc_cps(p);
    info->block = kWarps * 32;
    info->smem_bytes = (int)w2sk::SMEM;
    info->launches = 3;                       // quantise, GEMV, slice sum
    info->m_tile = M <= 8 ? 8 : 16;
    info->k_split = w2_slices(p->d.K);
}

void plan_w2_bf(const pq_prepared* p, int M, pq_plan_info* info) {
    plan_w2_tc(p, M, info);
    info->variant = PQ_VARIANT_W2_GEMV_BF;
    info->smem_bytes = (int)w2bf::SMEM;
}

// Shape of the cluster decode: K slices of SB blocks (a multiple of 4, so
// the block scales of a ring item are one aligned 8-byte copy), at most
// eight of them (CL CTAs per cluster), and R strips per warp, chosen so
// that the clusters fit on the GPU at once (about two CTAs per SM) where
// four strips per warp suffice.
struct ClShape {
    int CL, SB, R, groups;
    size_t smem;
};
static bool cl_shape(const pq_desc& d, int Npad, int num_sms, ClShape* out) {
    const int B = d.K / kGroup;
    if (B < 1) return false;
    int SB = (B + w2cl::kMaxCL - 1) / w2cl::kMaxCL;
    SB = (SB + 3) / 4 * 4;
    if (SB > w2cl::kMaxSB) return false;
    ClShape c;
    c.SB = SB;
    c.CL = (B + SB - 1) / SB;
    const int nstrips = Npad / kStrip;
    // the fewest strips per warp whose clusters are all resident at once
    // (228 KB of shared memory per SM, 1 KB of it reserved per CTA)
    for (c.R = 1;; ++c.R) {
        const int per_sm = (int)((228 * 1024) / ((size_t)w2cl::lay(SB, c.R, c.CL).total + 1024));
        int rc = (per_sm < 2 ? per_sm : 2) * (num_sms > 0 ? num_sms : 1) / c.CL;
        c.groups = (nstrips + kWarps * c.R - 1) / (kWarps * c.R);
        if (c.groups <= (rc < 1 ? 1 : rc) || c.R == w2cl::kMaxR) break;
    }
    c.smem = (size_t)w2cl::lay(SB, c.R, c.CL).total;
    *out = c;
    return true;
}

bool w2_cl_fits(const pq_desc& d, int M) {
    ClShape c;
    return d.fmt == PQ_FMT_W2_PQ2 && M >= 1 && M <= 16 && cl_shape(d, (int)npad(d.N), 152, &c);
}

void plan_w2_cl(const pq_prepared* p, int M, pq_plan_info* info) {
    ClShape c = {};
    cl_shape(p->d, p->Npad, p->num_sms, &c);
    info->variant = PQ_VARIANT_W2_GEMV_CL;
    info->grid = c.groups * c.CL;
    info->block = kWarps * 32;
    info->smem_bytes = (int)c.smem;
    info->launches = 1;
    info->m_tile = M <= 8 ? 8 : 16;
    info->k_split = c.CL;
}

template <int NT, bool AG128, bool BF16IN, bool ACT>
static cudaError_t launch_cl_t(const pq_prepared* p, const void* x, const float* xs_act, void* y, int M,
                               const ClShape& c, cudaStream_t s) {
    const pq_desc& d = p->d;
    cudaError_t e = ensure_smem<w2_cl_kernel<NT, AG128, BF16IN, ACT>>(c.smem);
    if (e != cudaSuccess) return e;
    return launch_cluster(w2_cl_kernel<NT, AG128, BF16IN, ACT>, dim3((unsigned)(c.groups * c.CL)),
                          dim3(kWarps * 32), c.smem, s, c.CL, true, static_cast<const uint8_t*>(p->codes),
                          static_cast<const uint16_t*>(p->scales), static_cast<const uint16_t*>(x), xs_act,
                          static_cast<uint16_t*>(y), p->status, M, d.N, p->Npad, d.K, w2_bp(d.K), c.SB, c.R,
                          d.out_dtype == PQ_BF16 ? 1 : 0);
}

template <bool ACT>
static cudaError_t launch_cl(const pq_prepared* p, const void* x, const float* xs_act, void* y, int M,
                             cudaStream_t s) {
    ClShape c;
    if (!cl_shape(p->d, p->Npad, p->num_sms, &c)) return cudaErrorInvalidValue;
    const bool ag = p->d.act_group == kGroup, bf = ACT || p->d.act_dtype == PQ_BF16;
    if (M <= 8) {
        if (ag) return bf ? launch_cl_t<1, true, true, ACT>(p, x, xs_act, y, M, c, s)
                          : launch_cl_t<1, true, false, ACT>(p, x, xs_act, y, M, c, s);
        return bf ? launch_cl_t<1, false, true, ACT>(p, x, xs_act, y, M, c, s)
                  : launch_cl_t<1, false, false, ACT>(p, x, xs_act, y, M, c, s);
    }
    if (ag) return bf ? launch_cl_t<2, true, true, ACT>(p, x, xs_act, y, M, c, s)
                      : launch_cl_t<2, true, false, ACT>(p, x, xs_act, y, M, c, s);
    return bf ? launch_cl_t<2, false, true, ACT>(p, x, xs_act, y, M, c, s)
              : launch_cl_t<2, false, false, ACT>(p, x, xs_act, y, M, c, s);
}

cudaError_t launch_w2_cl(const pq_prepared* p, const void* x, void* y, int M, cudaStream_t s) {
    return launch_cl<false>(p, x, nullptr, y, M, s);
}

cudaError_t launch_w2_cl_act(const pq_prepared* p, void* y, int M, const ActPlanes& a, cudaStream_t s) {
    return launch_cl<true>(p, a.qa, a.xs, y, M, s);
}

ActPlanes ws_act(const pq_prepared* p) {
    ActPlanes a;
    a.q8 = reinterpret_cast<int8_t*>(p->ws + p->wl.q_off);
    a.qa = reinterpret_cast<uint16_t*>(p->ws + p->wl.qa_off);
    a.sq = reinterpret_cast<int32_t*>(p->ws + p->wl.sq_off);
    a.xs = reinterpret_cast<float*>(p->ws + p->wl.xs_off);
    return a;
}

// After the quantiser (plane order).
cudaError_t launch_w2_tc(const pq_prepared* p, void* y, int M, const ActPlanes& a, cudaStream_t s) {
    const bool ag128 = p->d.act_group == kGroup;
    if (M <= 8) return ag128 ? launch_tc_t<1, true>(p, y, M, a, s) : launch_tc_t<1, false>(p, y, M, a, s);
    return ag128 ? launch_tc_t<2, true>(p, y, M, a, s) : launch_tc_t<2, false>(p, y, M, a, s);
}

// After the quantiser (bf16 codes in tensor-core order).
cudaError_t launch_w2_bf(const pq_prepared* p, void* y, int M, const ActPlanes& a, cudaStream_t s) {
    const bool ag128 = p->d.act_group == kGroup;
    if (M <= 8) return ag128 ? launch_bf_t<1, true>(p, y, M, a, s) : launch_bf_t<1, false>(p, y, M, a, s);
    return ag128 ? launch_bf_t<2, true>(p, y, M, a, s) : launch_bf_t<2, false>(p, y, M, a, s);
}

cudaError_t launch_w2_quantize(const pq_prepared* p, const void* x, int M, bool bf16_codes, const ActPlanes& a,
                               cudaStream_t s) {
    const pq_desc& d = p->d;
    const uint16_t* xx = static_cast<const uint16_t*>(x);
    const int abf = d.act_dtype == PQ_BF16 ? 1 : 0;
    const size_t smem = (size_t)d.K * 2;
    cudaError_t e = bf16_codes ? quantize_smem_attr<false>(d.K) : quantize_smem_attr<true>(d.K);
    if (e != cudaSuccess) return e;
    if (bf16_codes)
        return launch(w2_quantize_kernel<false>, dim3(M), dim3(kThreads), smem, s, true, xx, abf, d.K,
                      d.act_group, a.q8, a.qa, a.sq, a.xs, p->status);
    return launch(w2_quantize_kernel<true>, dim3(M), dim3(kThreads), smem, s, true, xx, abf, d.K, d.act_group,
                  a.q8, a.qa, a.sq, a.xs, p->status);
}

template <bool PLANE, bool BF16IN>
cudaError_t launch_norm_t(const pq_prepared* p, const NormArgs& n, int M, const ActPlanes& a, cudaStream_t s) {
    const pq_desc& d = p->d;
    const size_t smem = (size_t)d.K * 2;
    if (smem > 48 * 1024) {
        cudaError_t e = ensure_smem<w2_norm_quant_kernel<PLANE, BF16IN>>(smem);
        if (e != cudaSuccess) return e;
    }
    const float had_scale = n.had_block ? (float)(1.0 / sqrt((double)n.had_block)) : 1.0f;
    return launch(w2_norm_quant_kernel<PLANE, BF16IN>, dim3(M), dim3(kThreads), smem, s, true,
                  static_cast<const uint16_t*>(n.h), static_cast<const uint16_t*>(n.r),
                  static_cast<uint16_t*>(n.r_out), static_cast<uint16_t*>(n.norm_out),
                  static_cast<const uint16_t*>(n.gamma), n.signs, n.eps, n.unit_offset, n.had_block, had_scale,
                  d.K, d.act_group, a.q8, a.qa, a.sq, a.xs);
}

cudaError_t launch_w2_norm_quantize(const pq_prepared* p, const NormArgs& n, int M, bool bf16_codes,
                                    const ActPlanes& a, cudaStream_t s) {
    const bool bf16 = p->d.act_dtype == PQ_BF16;
    if (bf16_codes) return bf16 ? launch_norm_t<false, true>(p, n, M, a, s) : launch_norm_t<false, false>(p, n, M, a, s);
    return bf16 ? launch_norm_t<true, true>(p, n, M, a, s) : launch_norm_t<true, false>(p, n, M, a, s);
}

cudaError_t launch_w2_gemv(const pq_prepared* p, const void* x, void* y, int M, bool fused, const ActPlanes& a,
                           cudaStream_t s) {
    switch (mt_for(M)) {
        case 1: return fused ? launch_gemv_t<1, true>(p, x, y, M, a, s) : launch_gemv_t<1, false>(p, x, y, M, a, s);
        case 2: return fused ? launch_gemv_t<2, true>(p, x, y, M, a, s) : launch_gemv_t<2, false>(p, x, y, M, a, s);
        case 4: return fused ? launch_gemv_t<4, true>(p, x, y, M, a, s) : launch_gemv_t<4, false>(p, x, y, M, a, s);
        case 8: return launch_gemv_t<8, false>(p, x, y, M, a, s);
        default: return launch_gemv_t<16, false>(p, x, y, M, a, s);
    }
}

cudaError_t launch_w2_debug_quantize(const pq_prepared* p, const void* x, int8_t* q, float* xs, int M,
                                     cudaStream_t s) {
    cudaError_t e = launch_w2_quantize(p, x, M, false, ws_act(p), s);
    if (e != cudaSuccess) return e;
    const int total = M * p->d.K;
    unplane_kernel<<<(total + 255) / 256, 256, 0, s>>>(reinterpret_cast<const int8_t*>(p->ws + p->wl.q_off), q,
                                                        total);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return cudaMemcpyAsync(xs, p->ws + p->wl.xs_off, (size_t)M * (p->d.K / p->d.act_group) * 4,
                           cudaMemcpyDeviceToDevice, s);
}

cudaError_t launch_debug_act_unpack(const pq_prepared* p, const ActPlanes& a, int M, bool bf16_codes, int8_t* q,
                                   float* xs, int32_t* sq, cudaStream_t s) {
    const int total = M * p->d.K;
    const int blocks = (total + 255) / 256;
    if (bf16_codes)
        unorder_bf16_kernel<<<blocks, 256, 0, s>>>(a.qa, q, total);
    else
        unplane_kernel<<<blocks, 256, 0, s>>>(a.q8, q, total);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(xs, a.xs, (size_t)M * (p->d.K / p->d.act_group) * 4, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(sq, a.sq, (size_t)M * (p->d.K / kGroup) * 4, cudaMemcpyDeviceToDevice, s);
    return e;
}

cudaError_t launch_w2_debug_sums(const pq_prepared* p, const void* x, int32_t* S, int M, cudaStream_t s) {
    cudaError_t e = launch_w2_quantize(p, x, M, false, ws_act(p), s);
    if (e != cudaSuccess) return e;
    w2_sums_kernel<<<p->d.N, 32, 0, s>>>(p->codes, reinterpret_cast<const int8_t*>(p->ws + p->wl.q_off),
                                         reinterpret_cast<const int32_t*>(p->ws + p->wl.sq_off), S, M,
                                         p->d.N, p->d.K);
    return cudaGetLastError();
}

}  // namespace pq

// ---------------------------------------------------------------------------
// Allocation-free ternary decode (pq_linear_w2a8_static).
//
// For callers that cannot allocate device memory at all: code running inside
// a host framework that owns every device buffer and forbids new allocations
// once it is serving, or that cannot afford the device-wide synchronisation an
// allocation may cause.  The quantised activations, their per-block sums and
// their scales live in the file-scope array below instead of the handle's
// workspace.  It is part of this library's device image: every GPU that loads
// the library holds these bytes until the process exits.
// ---------------------------------------------------------------------------
#include <mutex>

namespace {

constexpr size_t kStaticScratchBytes = 128 * 1024;
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
uint8_t* g_static_addr[kMaxDevices] = {};

struct StaticLayout {
    size_t q, sq, xs, total;
};

StaticLayout static_layout(const pq_desc& d, int M) {
    StaticLayout l;
    l.q = 0;
    l.sq = align_up((size_t)M * d.K, kAlign);
    l.xs = align_up(l.sq + (size_t)M * (d.K / kGroup) * 4, kAlign);
    l.total = align_up(l.xs + (size_t)M * (d.K / d.act_group) * 4, kAlign);
    return l;
}

// Device address of the array for the current device.  The name of a
// __device__ variable in host code is only a host-side stand-in, so the
// address is asked from the runtime once per device, with that device
// current, and kept for the life of the process's primary context on that
// device (a cudaDeviceReset ends that context and the library with it: load
// the library again before calling it after one).
cudaError_t static_scratch_address(uint8_t** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_addr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess) return e;
        g_static_addr[dev] = static_cast<uint8_t*>(ptr);
    }
    *out = g_static_addr[dev];
    return cudaSuccess;
}

template <int MT>
cudaError_t launch_static_gemv(const pq_prepared* p, const void* x, void* y, int M, const uint8_t* scratch,
                               const StaticLayout& l, cudaStream_t s) {
    const pq_desc& d = p->d;
    const size_t smem = w2_launch_smem(w2_smem_bytes(MT, d.K, d.act_group, false));
    cudaError_t e = ensure_smem<w2_gemv_kernel<MT, false>>(smem);
    if (e == cudaSuccess) e = ensure_max_carveout<w2_gemv_kernel<MT, false>>();
    if (e != cudaSuccess) return e;
    return launch(w2_gemv_kernel<MT, false>, dim3(w2_grid(p, M)), dim3(kGemvWarps * 32), smem, s, true,
                  static_cast<const uint16_t*>(x), d.act_dtype == PQ_BF16 ? 1 : 0,
                  static_cast<const uint8_t*>(p->codes), static_cast<const uint16_t*>(p->scales),
                  reinterpret_cast<const int8_t*>(scratch + l.q), reinterpret_cast<const int32_t*>(scratch + l.sq),
                  reinterpret_cast<const float*>(scratch + l.xs), static_cast<uint16_t*>(y), M, d.N, d.K,
                  w2_bp(d.K), d.act_group, d.out_dtype == PQ_BF16 ? 1 : 0, p->status);
}

}  // namespace

extern "C" int32_t pq_linear_w2a8_static(const void* d_x, const pq_prepared* p, void* d_y, int32_t M,
                                         void* stream) {
    using namespace pq;
    if (!p) return fail(PQ_ERR_INVALID_ARG, "handle is NULL");
    if (!d_x || !d_y) return fail(PQ_ERR_INVALID_ARG, "x and y must be non-NULL");
    if (((uintptr_t)d_x & 15) || ((uintptr_t)d_y & 15)) return fail(PQ_ERR_ALIGN, "x and y must be 16-byte aligned");
    if (p->d.fmt != PQ_FMT_W2_PQ2) return fail(PQ_ERR_INVALID_ARG, "pq_linear_w2a8_static needs a ternary PQ2 handle");
    if (M < 1 || M > 16) return fail(PQ_ERR_SHAPE, "pq_linear_w2a8_static runs M = 1..16, got M = %d", M);
    if (M > p->d.max_m) return fail(PQ_ERR_SHAPE, "M = %d must lie in 1..max_m (%d)", M, p->d.max_m);
    if (!w2_gemv_fits(p->d, M, false))
        return fail(PQ_ERR_UNSUPPORTED, "M = %d, K = %d does not fit the decode GEMV's shared memory", M, p->d.K);
    const StaticLayout l = static_layout(p->d, M);
    if (l.total > kStaticScratchBytes)
        return fail(PQ_ERR_BUFFER_TOO_SMALL,
                    "M = %d, K = %d needs %zu bytes of static scratch; the library reserves %zu "
                    "(M*K must stay below about 120000)", M, p->d.K, l.total, kStaticScratchBytes);
    uint8_t* scratch = nullptr;
    cudaError_t e = static_scratch_address(&scratch);
    if (e != cudaSuccess) return cuda_fail(e, "static scratch address");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // every byte the GEMV reads (q, the block sums and the scales of all M rows)
    // is rewritten by the pre-pass first, so nothing needs clearing
    const pq_desc& d = p->d;
    e = quantize_smem_attr<true>(d.K);
    if (e != cudaSuccess) return cuda_fail(e, "pq_linear_w2a8_static configure");
    e = launch(w2_quantize_kernel<true>, dim3(M), dim3(kThreads), (size_t)d.K * 2, s, true,
               static_cast<const uint16_t*>(d_x), d.act_dtype == PQ_BF16 ? 1 : 0, d.K, d.act_group,
               reinterpret_cast<int8_t*>(scratch + l.q), static_cast<uint16_t*>(nullptr),
               reinterpret_cast<int32_t*>(scratch + l.sq), reinterpret_cast<float*>(scratch + l.xs), p->status);
    if (e == cudaSuccess) {
        switch (mt_for(M)) {
            case 1: e = launch_static_gemv<1>(p, d_x, d_y, M, scratch, l, s); break;
            case 2: e = launch_static_gemv<2>(p, d_x, d_y, M, scratch, l, s); break;
            case 4: e = launch_static_gemv<4>(p, d_x, d_y, M, scratch, l, s); break;
            case 8: e = launch_static_gemv<8>(p, d_x, d_y, M, scratch, l, s); break;
            default: e = launch_static_gemv<16>(p, d_x, d_y, M, scratch, l, s); break;
        }
    }
    return e == cudaSuccess ? PQ_OK : cuda_fail(e, "pq_linear_w2a8_static launch");
}
