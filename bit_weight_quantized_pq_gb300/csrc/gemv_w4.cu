// W4A16 decode GEMV, M = 1..16: y[m][n] = sum_g s[g][n] * sum_{k in g} (q[n][k] - z[g][n]) * x[m][k].
//
// The decode shape of "mate: Marlin-class W4A16 GEMM for mp_31 ... #6" (the
// GEMV "that reads each weight once"): every packed code byte is streamed from
// HBM exactly once.  GB300 design:
//   * M = 1..4: persistent CTAs of 8 warps loop over 16-row strips; the
//     warps of a CTA split K into contiguous runs of 128-row groups and
//     reduce each strip through shared memory in a fixed order
//     (deterministic); the activation rows sit once in shared memory
//     (under act order permuted there by the kernel, no gather launch);
//   * M = 5..16 (and rows too long for shared memory): split K across CTAs
//     (slices of four groups), the CTA's
//     activation slice for all tokens in shared memory, fp32 partial sums
//     per slice, added in a fixed order inside a thread-block cluster
//     (8 slices or fewer, K <= 4096, M <= 8) or by a second,
//     programmatically dependent launch;
//   * every lane streams its own 16-byte code chunks (and the scale slices of
//     the same groups) with cp.async into a per-warp ring, so the next items
//     are in flight without holding registers;
//   * codes become exact fp16/bf16 values (q - z) with one LOP3 per two
//     weights (nibble OR exponent bits: 1024+q / 128+q) and one packed
//     subtract, consumed directly as the A fragment of mma.m16n8k16 (weights
//     are the 16-row operand, tokens the 8 columns);
//   * each 128-row group accumulates into a fresh fp32 fragment which is then
//     scaled by s[g][n] once, in fp32;
//   * weight copies for the first D groups are issued before
//     griddepcontrol.wait, so under programmatic dependent launch the weight
//     stream overlaps the previous kernel; activations are copied only after.
#include "gemv_common.cuh"

namespace {

using namespace pq;
using namespace pqd;
using namespace pqg;

constexpr int kWarps = 8;

template <bool BF16>
__device__ __forceinline__ uint32_t dq_pair(uint32_t v, uint32_t zc) {
    // two 4-bit codes (bits 0..3 and 16..19 of v) -> exact (q - z) pair
    constexpr uint32_t kMagic = BF16 ? 0x43004300u : 0x64006400u;  // 128 / 1024 per half
    const uint32_t t = lop3_and_or(v, 0x000F000Fu, kMagic);
    uint32_t d;
    if (BF16)
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(t), "r"(zc));
    else
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(t), "r"(zc));
    return d;
}

template <bool BF16>
__device__ __forceinline__ uint32_t zero_pair(int z) {
    // (magic + z) in both halves: 128 + z (bf16) and 1024 + z (fp16) for
    // z < 16 have the mantissa field z, so the bit pattern is magic | z
    return ((BF16 ? 0x4300u : 0x6400u) | (uint32_t)z) * 0x00010001u;
}

template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    if (BF16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Lane (g = lane/4, t = lane%4) of a warp covering one 16-row strip:
//   k16 step j (0..7) of a group maps mma k-slots {2t,2t+1} to group rows
//   32t+4j+{0,1} and slots {2t+8,2t+9} to 32t+4j+{2,3}, so one lane's A
//   operands are the 32 consecutive rows 32t..32t+31 of output rows n0+g and
//   n0+g+8 (one 16-byte code chunk each), and its B operands are
//   x[token][32t..32t+31] (64 consecutive bytes).

// Whole-row kernel for M = 1..MT tokens (MT = 1 or 4).  The same lane
// mapping and exact unpack, with the per-item bookkeeping amortised over
// items of four 128-row groups (4 KB of codes per warp, double buffered) and
// the activation rows of all tokens in shared memory.  MMA column g is token
// g: with MT = 1 every lane feeds the one row into all eight columns (the
// seven extra columns repeat column 0 and are ignored), so no operand needs
// masking; with MT > 1 lane (g, t) feeds token g (zeros for g >= M) and holds
// tokens 2t, 2t + 1 of its two rows.
namespace m1 {
constexpr int IG = 4;                                   // groups per item
constexpr int D = 2;                                    // items per warp ring
constexpr int CODE_B = IG * 1024, SC_B = IG * 32, ZP_B = IG * 16;
constexpr int ITEM_B = CODE_B + SC_B + ZP_B;
constexpr int RING = kWarps * D * ITEM_B;
// affine 4-bit layers: two scales and two biases (one per 64-group) per row
// and 128-group instead of one scale and one zero point
constexpr int SC_BA = IG * 64, BI_BA = IG * 64;
constexpr int ITEM_BA = CODE_B + SC_BA + BI_BA;
constexpr int RING_A = kWarps * D * ITEM_BA;
// activation row stride in elements: rows of several tokens start 16 bytes
// apart in the bank map, so the eight token rows of a fragment load spread
inline int xstride(int K, int MT) { return MT == 1 ? K : K + 8; }
// under act order the rows arrive in the caller's order in a second buffer
// and are permuted inside shared memory
// (affine layers add the sum of x over every 64-group of every token, fp32)
inline size_t smem(int K, int MT, bool gather = false, bool affine = false) {
    return (size_t)(affine ? RING_A : RING) + (size_t)MT * xstride(K, MT) * 2 + (gather ? (size_t)MT * K * 2 : 0) +
           (affine ? (size_t)MT * (K / kAffineGroup) * 4 : 0);
}
// static shared memory of the kernel: the strips' fixed-order reduction buffer
inline size_t smem_static(int MT) { return sizeof(float) * 2 * kWarps * MT * 16; }
}  // namespace m1
// the activation rows must fit beside the ring, with the static buffer, in
// the 227 KB a CTA may hold (one token: K <= 81408); longer rows take the
// split-K kernel below
inline bool m1_fits(int K, int MT, bool gather = false, bool affine = false) {
    return m1::smem(K, MT, gather, affine) + m1::smem_static(MT) <= 227 * 1024;
}
static_assert(m1::RING + 2 * (size_t)kW4OneTokenMaxK + sizeof(float) * 2 * kWarps * 16 <= 227 * 1024,
              "one-token row bound");
static_assert(m1::RING_A + 2 * (size_t)kW4AffineOneTokenMaxK + 4 * (size_t)(kW4AffineOneTokenMaxK / kAffineGroup) +
                      sizeof(float) * 2 * kWarps * 16 <=
                  227 * 1024,
              "one-token affine row bound");

// Act order: the kernel resolves the permutation itself (activation k' of
// the prepared order is x[perm[k']]), so no gather launch precedes it.  The
// rows arrive in the caller's order by coalesced copies into a second
// shared-memory buffer and are permuted there (scattered global loads would
// cost one L1 request per element).  The permutation is a prepared plane,
// independent of the predecessor: the first kPermAhead chunks of each thread
// are loaded before the dependency wait.
constexpr int kPermAhead = 4;

// Permute 8 prepared-order activations k' = 8c..8c+7 (indices in pa, pb) of
// each token from the caller-order rows xraw into the operand rows xrow.
template <int MT>
__device__ __forceinline__ void gather_chunk(const uint16_t* xraw, uint16_t* xrow, int XS, int K, int M, int c,
                                             const int4& pa, const int4& pb) {
    const int idx[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if (m < M) {
            uint16_t v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = xraw[(size_t)m * K + idx[j]];
            uint4 u;
            u.x = (uint32_t)v[0] | ((uint32_t)v[1] << 16);
            u.y = (uint32_t)v[2] | ((uint32_t)v[3] << 16);
            u.z = (uint32_t)v[4] | ((uint32_t)v[5] << 16);
            u.w = (uint32_t)v[6] | ((uint32_t)v[7] << 16);
            *reinterpret_cast<uint4*>(xrow + (size_t)m * XS + 8 * c) = u;
        }
    }
}

// AFF (affine 4-bit, "qwen CUDA: --prompt-precision int8 ... #1176"):
// w = s * q + b per 64-group.  The prepared K order puts words 0, 1 of a
// lane's 16-byte chunk in the 128-group's first 64-group and words 2, 3 in
// its second, so each 64-group gets its own MMA accumulators and scale; the
// bias adds b * (sum of x over the 64-group), the sums formed once per CTA.
template <int MT, bool BF16, bool ASYM, bool GATHER, bool AFF>
__global__ void __launch_bounds__(kWarps * 32)
gemv_w4_m1_kernel(const uint16_t* __restrict__ x, const uint8_t* __restrict__ codes,
                  const uint16_t* __restrict__ scales, const uint8_t* __restrict__ zeros,
                  const uint16_t* __restrict__ biases, const int32_t* __restrict__ perm, uint16_t* __restrict__ y,
                  int M, int N, int Npad, int K, int out_bf16) {
    using namespace m1;
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ float red[2][kWarps][MT * 16];           // [strip parity][warp][token][row]

    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int G = K / kGroup;
    const int gb = (G * warp) / kWarps, ge = (G * (warp + 1)) / kWarps;
    const int ips = (ge - gb + IG - 1) / IG;               // items per strip
    const int nstrips = Npad / kStrip;
    const int my_strips = nstrips > (int)blockIdx.x ? (nstrips - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int total = my_strips * ips;
    constexpr int ITEM = AFF ? ITEM_BA : ITEM_B;
    constexpr int RINGB = AFF ? RING_A : RING;
    constexpr int SCB = AFF ? SC_BA : SC_B;
    uint8_t* ring = smem + (size_t)warp * D * ITEM;
    const uint16_t* xrow = reinterpret_cast<const uint16_t*>(smem + RINGB);

    int is_i = 0, is_strip = (int)blockIdx.x, is_grp = gb, is_slot = 0;
    auto issue_next = [&]() {
        if (is_i < total) {
            const int n0 = is_strip * kStrip;
            const int ng = ge - is_grp < IG ? ge - is_grp : IG;
            uint8_t* slot = ring + (size_t)is_slot * ITEM;
            const uint8_t* ra = codes + (size_t)(n0 + g) * (K / 2) + (size_t)is_grp * 64 + 16 * t;
#pragma unroll
            for (int q = 0; q < IG; ++q) {
                if (q < ng) {
                    cp_async16(smem_u32(slot + q * 1024 + lane * 16), ra + 64 * q);
                    cp_async16(smem_u32(slot + q * 1024 + 512 + lane * 16), ra + 64 * q + (size_t)8 * (K / 2));
                }
            }
            if (AFF) {
                // lane l < 4 ng: 64-group 2 is_grp + l / 2, 8-row half l % 2, at
                // item offset 64 (l / 4) + 32 ((l / 2) % 2) + 16 (l % 2); biases
                // likewise from lane 16
                if (lane < 4 * ng)
                    cp_async16(smem_u32(slot + CODE_B + 16 * lane),
                               scales + (size_t)(2 * is_grp + (lane >> 1)) * Npad + n0 + 8 * (lane & 1));
                else if (lane >= 16 && lane < 16 + 4 * ng)
                    cp_async16(smem_u32(slot + CODE_B + SC_BA + 16 * (lane - 16)),
                               biases + (size_t)(2 * is_grp + ((lane - 16) >> 1)) * Npad + n0 + 8 * (lane & 1));
            } else if (lane < 2 * ng)
                cp_async16(smem_u32(slot + CODE_B + 16 * lane),
                           scales + (size_t)(is_grp + (lane >> 1)) * Npad + n0 + 8 * (lane & 1));
            if (ASYM && lane >= 8 && lane < 8 + ng)
                cp_async16(smem_u32(slot + CODE_B + SC_B + 16 * (lane - 8)), zeros + (size_t)(is_grp + lane - 8) * Npad + n0);
            is_grp += IG;
            if (is_grp >= ge) {
                is_grp = gb;
                is_strip += gridDim.x;
            }
        }
        ++is_i;
        if (++is_slot == D) is_slot = 0;
        cp_commit();
    };

    for (int d = 0; d < D; ++d) issue_next();          // weights before the dependency wait
    const int XS = MT == 1 ? K : K + 8, KC = K / 8;
    int4 pa[kPermAhead], pb[kPermAhead];
    if (GATHER) {
#pragma unroll
        for (int j = 0; j < kPermAhead; ++j) {
            const int c = threadIdx.x + j * (int)blockDim.x;
            if (c < KC) {
                pa[j] = __ldg(reinterpret_cast<const int4*>(perm + 8 * (size_t)c));
                pb[j] = __ldg(reinterpret_cast<const int4*>(perm + 8 * (size_t)c + 4));
            }
        }
    }
    pdl_wait();
    // The rows by cp.async, waited together with the two prefetched items: on
    // GB300 this measured faster than a bulk copy on its own mbarrier here
    // (the ternary GEMV, with six items in flight, takes the bulk copy).
    uint16_t* xraw = reinterpret_cast<uint16_t*>(smem + RINGB + (size_t)MT * XS * 2);  // act order only
    // affine: sums of x over each 64-group of each token (0 for tokens >= M)
    const int GA = K / kAffineGroup;
    float* xsum = reinterpret_cast<float*>(smem + RINGB + (size_t)MT * XS * 2);
    uint16_t* xdst = GATHER ? xraw : const_cast<uint16_t*>(xrow);
    const int XD = GATHER ? K : XS;
    for (int i = threadIdx.x; i < M * KC; i += blockDim.x) {
        const int m = i / KC, c = i - m * KC;
        cp_async16(smem_u32(xdst + (size_t)m * XD + 8 * c), x + (size_t)m * K + 8 * (size_t)c);
    }
    cp_commit();
    cp_wait<0>();
    __syncthreads();
    if (GATHER) {
#pragma unroll
        for (int j = 0; j < kPermAhead; ++j) {
            const int c = threadIdx.x + j * (int)blockDim.x;
            if (c < KC) gather_chunk<MT>(xraw, const_cast<uint16_t*>(xrow), XS, K, M, c, pa[j], pb[j]);
        }
        for (int c = threadIdx.x + kPermAhead * (int)blockDim.x; c < KC; c += blockDim.x)
            gather_chunk<MT>(xraw, const_cast<uint16_t*>(xrow), XS, K, M, c,
                             __ldg(reinterpret_cast<const int4*>(perm + 8 * (size_t)c)),
                             __ldg(reinterpret_cast<const int4*>(perm + 8 * (size_t)c + 4)));
        __syncthreads();
    }
    if (AFF) {
        // eight lanes a sum, one 16-byte chunk each: a warp reads 512
        // consecutive bytes of a row (no two lanes of a phase on one bank)
        const int tasks = MT * GA * 8;                   // a multiple of 16
        for (int i0 = warp * 32; i0 < tasks; i0 += kWarps * 32) {
            const int i = i0 + lane, sidx = i >> 3, c = i & 7;
            const int m = sidx / GA, ga = sidx - m * GA;
            float v = 0.f;
            if (i < tasks && m < M)
                v = chunk_sum8(*reinterpret_cast<const uint4*>(xrow + (size_t)m * XS + (size_t)ga * kAffineGroup + 8 * c),
                               BF16);
            v = team8_sum(v);
            if (i < tasks && c == 0) xsum[sidx] = v;
        }
        __syncthreads();
    }

    int rs = 0;
    const bool xlane = MT == 1 || g < M;                 // this lane's token column is live
    const uint16_t* xtok = xrow + (MT == 1 ? 0 : (size_t)g * XS);
    for (int j = 0; j < my_strips; ++j) {
      // rows g and g+8 x tokens 2t and 2t+1 (MT = 1: column 2t, token 0)
      float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
      // a warp with an empty K-range (K < 1024) still joins the reduction
      for (int cg = gb; cg < ge; cg += IG) {
        cp_wait<D - 1>();
        __syncwarp();
        const uint8_t* slot = ring + (size_t)rs * ITEM;
        if (++rs == D) rs = 0;
        const int ng = ge - cg < IG ? ge - cg : IG;
        uint4 ca[IG], cb[IG];
        float sa[IG], sb[IG];
        int za[IG], zb[IG];
        // affine: raw 16-bit scales and biases of rows g / g + 8, first and
        // second 64-group: {s_A(g) | s_A(g+8) << 16, s_B(g) | s_B(g+8) << 16}
        uint32_t sp[IG][2], bp[IG][2];
#pragma unroll
        for (int q = 0; q < IG; ++q) {
            if (q < ng) {
                ca[q] = *reinterpret_cast<const uint4*>(slot + q * 1024 + lane * 16);
                cb[q] = *reinterpret_cast<const uint4*>(slot + q * 1024 + 512 + lane * 16);
                if (AFF) {
                    const uint16_t* sc = reinterpret_cast<const uint16_t*>(slot + CODE_B + 64 * q);
                    const uint16_t* bi = reinterpret_cast<const uint16_t*>(slot + CODE_B + SC_BA + 64 * q);
                    sp[q][0] = (uint32_t)sc[g] | ((uint32_t)sc[g + 8] << 16);
                    sp[q][1] = (uint32_t)sc[16 + g] | ((uint32_t)sc[16 + g + 8] << 16);
                    bp[q][0] = (uint32_t)bi[g] | ((uint32_t)bi[g + 8] << 16);
                    bp[q][1] = (uint32_t)bi[16 + g] | ((uint32_t)bi[16 + g + 8] << 16);
                } else {
                    const uint16_t* sc = reinterpret_cast<const uint16_t*>(slot + CODE_B + 32 * q);
                    sa[q] = __half2float(__ushort_as_half(sc[g]));
                    sb[q] = __half2float(__ushort_as_half(sc[g + 8]));
                    za[q] = ASYM ? (int)slot[CODE_B + SCB + 16 * q + g] : 8;
                    zb[q] = ASYM ? (int)slot[CODE_B + SCB + 16 * q + g + 8] : 8;
                }
            }
        }
        __syncwarp();                                    // slot read: refill it
        issue_next();
#pragma unroll
        for (int q = 0; q < IG; ++q) {
            if (q < ng) {
                uint32_t xh[16];
                const uint16_t* xs = xtok + (size_t)(cg + q) * kGroup;
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    // word v of the lane's chunk: inputs 32t + 8v of the group,
                    // or for affine layers 16t + 8v (v < 2) / 64 + 16t + 8(v - 2)
                    const int off = AFF ? (v < 2 ? 16 * t + 8 * v : 64 + 16 * t + 8 * (v - 2)) : 32 * t + 8 * v;
                    const uint4 u = xlane ? *reinterpret_cast<const uint4*>(xs + off) : make_uint4(0u, 0u, 0u, 0u);
                    xh[4 * v] = u.x; xh[4 * v + 1] = u.y; xh[4 * v + 2] = u.z; xh[4 * v + 3] = u.w;
                }
                const uint32_t zca = zero_pair<BF16>(AFF ? 0 : za[q]), zcb = zero_pair<BF16>(AFF ? 0 : zb[q]);
                // d0, d1: words 0, 1 (the first 64-group for affine layers);
                // e0, e1: words 2, 3 (the second)
                float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
                float e0[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
                const uint32_t wa[4] = {ca[q].x, ca[q].y, ca[q].z, ca[q].w};
                const uint32_t wb[4] = {cb[q].x, cb[q].y, cb[q].z, cb[q].w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    float (&f0)[4] = (AFF && w >= 2) ? e0 : d0;
                    float (&f1)[4] = (AFF && w >= 2) ? e1 : d1;
                    mma16816<BF16>(f0, dq_pair<BF16>(wa[w], zca), dq_pair<BF16>(wb[w], zcb),
                                   dq_pair<BF16>(wa[w] >> 4, zca), dq_pair<BF16>(wb[w] >> 4, zcb),
                                   xh[4 * w], xh[4 * w + 1]);
                    mma16816<BF16>(f1, dq_pair<BF16>(wa[w] >> 8, zca), dq_pair<BF16>(wb[w] >> 8, zcb),
                                   dq_pair<BF16>(wa[w] >> 12, zca), dq_pair<BF16>(wb[w] >> 12, zcb),
                                   xh[4 * w + 2], xh[4 * w + 3]);
                }
                if (AFF) {
                    const float sAa = to_float((uint16_t)(sp[q][0] & 0xFFFF), BF16), sAb = to_float((uint16_t)(sp[q][0] >> 16), BF16);
                    const float sBa = to_float((uint16_t)(sp[q][1] & 0xFFFF), BF16), sBb = to_float((uint16_t)(sp[q][1] >> 16), BF16);
                    acc0 = fmaf(sBa, e0[0] + e1[0], fmaf(sAa, d0[0] + d1[0], acc0));
                    acc1 = fmaf(sBb, e0[2] + e1[2], fmaf(sAb, d0[2] + d1[2], acc1));
                    if (MT > 1) {
                        acc2 = fmaf(sBa, e0[1] + e1[1], fmaf(sAa, d0[1] + d1[1], acc2));
                        acc3 = fmaf(sBb, e0[3] + e1[3], fmaf(sAb, d0[3] + d1[3], acc3));
                    }
                    // bias: b * (sum of x over the 64-group), tokens 2t / 2t + 1
                    // (token 0 when MT = 1; lanes past the tokens skip it)
                    const float bAa = to_float((uint16_t)(bp[q][0] & 0xFFFF), BF16), bAb = to_float((uint16_t)(bp[q][0] >> 16), BF16);
                    const float bBa = to_float((uint16_t)(bp[q][1] & 0xFFFF), BF16), bBb = to_float((uint16_t)(bp[q][1] >> 16), BF16);
                    const int ga = 2 * (cg + q);
                    if (MT == 1) {
                        const float xA = xsum[ga], xB = xsum[ga + 1];
                        acc0 = fmaf(bBa, xB, fmaf(bAa, xA, acc0));
                        acc1 = fmaf(bBb, xB, fmaf(bAb, xA, acc1));
                    } else if (2 * t < MT) {
                        const float* x0 = xsum + (size_t)(2 * t) * GA + ga;
                        const float* x1 = x0 + GA;
                        acc0 = fmaf(bBa, x0[1], fmaf(bAa, x0[0], acc0));
                        acc1 = fmaf(bBb, x0[1], fmaf(bAb, x0[0], acc1));
                        acc2 = fmaf(bBa, x1[1], fmaf(bAa, x1[0], acc2));
                        acc3 = fmaf(bBb, x1[1], fmaf(bAb, x1[0], acc3));
                    }
                } else {
                    acc0 = fmaf(sa[q], d0[0] + d1[0], acc0);
                    acc1 = fmaf(sb[q], d0[2] + d1[2], acc1);
                    if (MT > 1) {
                        acc2 = fmaf(sa[q], d0[1] + d1[1], acc2);
                        acc3 = fmaf(sb[q], d0[3] + d1[3], acc3);
                    }
                }
            }
        }
      }
      // strip done: fixed-order reduction over the K-split warps
      if (MT == 1) {
          if (t == 0) {
              red[j & 1][warp][g] = acc0;
              red[j & 1][warp][g + 8] = acc1;
          }
      } else {
          if (2 * t < MT) {
              red[j & 1][warp][(2 * t) * 16 + g] = acc0;
              red[j & 1][warp][(2 * t) * 16 + g + 8] = acc1;
              red[j & 1][warp][(2 * t + 1) * 16 + g] = acc2;
              red[j & 1][warp][(2 * t + 1) * 16 + g + 8] = acc3;
          }
      }
      __syncthreads();
      if (warp == (j % kWarps)) {
          const int n0 = ((int)blockIdx.x + j * (int)gridDim.x) * kStrip;
          for (int o = lane; o < MT * 16; o += 32) {
              const int tok = o >> 4, r = o & 15;
              float s = red[j & 1][0][o];
#pragma unroll
              for (int w = 1; w < kWarps; ++w) s += red[j & 1][w][o];
              if (tok < M && n0 + r < N) y[(size_t)tok * N + n0 + r] = from_float(s, out_bf16 != 0);
          }
      }
    }
    cp_wait<0>();
}

template <int MT, bool BF16, bool ASYM, bool GATHER, bool AFF = false>
cudaError_t launch_m1_t(const pq_prepared* p, const void* x, void* y, int M, cudaStream_t s) {
    const pq_desc& d = p->d;
    const size_t smem = m1::smem(d.K, MT, GATHER, AFF);
    // residency for this shared-memory size, per device: (smem << 8) | CTAs per SM
    static std::atomic<uint64_t> occ[kMaxDevices];
    cudaError_t e = ensure_smem<gemv_w4_m1_kernel<MT, BF16, ASYM, GATHER, AFF>>(smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    const int dev = p->device;
    const uint64_t rec = dev >= 0 && dev < kMaxDevices ? occ[dev].load(std::memory_order_relaxed) : 0;
    if ((rec >> 8) == smem) {
        per_sm = (int)(rec & 0xFF);
    } else {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_w4_m1_kernel<MT, BF16, ASYM, GATHER, AFF>,
                                                          kWarps * 32, smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kMaxDevices) occ[dev].store(((uint64_t)smem << 8) | (uint64_t)(per_sm & 0xFF));
    }
    const int nstrips = p->Npad / kStrip;
    const int cap = p->num_sms * (per_sm < 1 ? 1 : per_sm);
    return launch(gemv_w4_m1_kernel<MT, BF16, ASYM, GATHER, AFF>, dim3(nstrips < cap ? nstrips : cap),
                  dim3(kWarps * 32), smem, s, true, static_cast<const uint16_t*>(x),
                  static_cast<const uint8_t*>(p->codes), static_cast<const uint16_t*>(p->scales),
                  static_cast<const uint8_t*>(p->zeros), static_cast<const uint16_t*>(AFF ? p->biases : nullptr),
                  static_cast<const int32_t*>(GATHER ? p->perm : nullptr), static_cast<uint16_t*>(y), M, d.N,
                  p->Npad, d.K, d.out_dtype == PQ_BF16 ? 1 : 0);
}

// x in the caller's order: the kernel gathers through the act-order
// permutation when the layer has one (unless x was gathered already)
template <int MT>
cudaError_t launch_m1_mt(const pq_prepared* p, const void* x, void* y, int M, bool gathered, cudaStream_t s) {
    const bool bf16 = p->d.act_dtype == PQ_BF16;
    const bool asym = p->zeros != nullptr;
    if (p->d.fmt == PQ_FMT_W4_AFFINE)
        return bf16 ? launch_m1_t<MT, true, false, false, true>(p, x, y, M, s)
                    : launch_m1_t<MT, false, false, false, true>(p, x, y, M, s);
    if (p->d.has_gidx && !gathered) {
        if (bf16) return asym ? launch_m1_t<MT, true, true, true>(p, x, y, M, s) : launch_m1_t<MT, true, false, true>(p, x, y, M, s);
        return asym ? launch_m1_t<MT, false, true, true>(p, x, y, M, s) : launch_m1_t<MT, false, false, true>(p, x, y, M, s);
    }
    if (bf16) return asym ? launch_m1_t<MT, true, true, false>(p, x, y, M, s) : launch_m1_t<MT, true, false, false>(p, x, y, M, s);
    return asym ? launch_m1_t<MT, false, true, false>(p, x, y, M, s) : launch_m1_t<MT, false, false, false>(p, x, y, M, s);
}

// Token-column width of the whole-row kernel for M tokens, 0 if it does not
// apply: then split-K.  Up to 4 tokens whenever their rows fit in shared
// memory (measured on GB300 over the 7B shapes: 7.2 / 8.5 us per call at
// M = 2 / 4 against 8.9 / 9.1 split-K, even where the rows leave one CTA per
// SM; at M = 8 an 8-token variant measured 9.4 against 8.5 split-K).
int m1_tile_affine(int M, int K) {
    if (M <= 1) return m1_fits(K, 1, false, true) ? 1 : 0;
    return M <= kW4RowTokens && m1_fits(K, 4, false, true) ? 4 : 0;
}

int m1_tile(int M, int K) {
    if (M <= 1) return m1_fits(K, 1) ? 1 : 0;
    return M <= kW4RowTokens && m1_fits(K, 4) ? 4 : 0;
}

// CTAs of the whole-row kernel per SM (dynamic + static shared memory + the
// 1 KB the runtime reserves per CTA, against the SM's 228 KB)
inline int m1_per_sm(int K, int MT, bool gather) {
    const size_t per_cta = m1::smem(K, MT, gather) + sizeof(float) * 2 * kWarps * MT * 16 + 1024;
    return (int)((size_t)228 * 1024 / per_cta);
}

// Act order on the whole-row kernel: permuted in its shared memory when the
// second copy of the rows fits there without costing residency, else after a
// gather launch (measured on GB300, 5120-wide rows: one token 7.4 us against
// 8.0 with the gather launch; four tokens of a 27648-row layer 28.4 us at
// one CTA per SM against 26.2 at two).
bool m1_gathers(const pq_prepared* p, int M) {
    const int mt = m1_tile(M, p->d.K);
    return p->d.has_gidx && mt > 0 && m1_fits(p->d.K, mt, true) &&
           m1_per_sm(p->d.K, mt, true) >= m1_per_sm(p->d.K, mt, false);
}

cudaError_t launch_m1(const pq_prepared* p, const void* x, void* y, int M, bool gathered, cudaStream_t s) {
    const int mt = p->d.fmt == PQ_FMT_W4_AFFINE ? m1_tile_affine(M, p->d.K) : m1_tile(M, p->d.K);
    switch (mt) {
        case 1: return launch_m1_mt<1>(p, x, y, M, gathered, s);
        case 4: return launch_m1_mt<4>(p, x, y, M, gathered, s);
        default: return cudaErrorInvalidValue;
    }
}

// Split-K decode for M = 2..16 tokens (and single rows too long for the
// kernel above).  Work tile = (block of 8 strips, K slice of kSliceGroups
// groups); the 8 warps of a CTA take the 8 strips of a block, all on the
// CTA's one slice, so the CTA copies its activation slice [16][512] into
// shared memory once and every strip it visits reuses it -- the activations
// are read from L2 once per CTA instead of once per strip and group.  Each
// warp writes its strip's fp32 partial sums for the slice to the workspace;
// a second, programmatically dependent launch adds the slices in the fixed
// order 0, 1, ... and writes y (deterministic).  Nothing waits on another CTA.
// CLU (at most 8 slices, at most kCluBlocks strip blocks per CTA, M <= 8): the
// ns CTAs of one strip block run as a thread-block cluster instead; each
// warp stores its strip's slice sums into the shared memory of the CTA that
// owns the strip (strip i of the CTA's sequence: CTA i % ns), and after one
// cluster barrier the owner adds them in slice order and writes y: one
// launch, the same sums in the same order, so the same bits.
namespace sk {
constexpr int SG = kSliceGroups;                      // groups per slice
constexpr int D = 2;                                  // slices in flight per warp
constexpr int CODE_B = SG * 1024, SC_B = SG * 32, ZP_B = SG * 16;
constexpr int ITEM_B = CODE_B + SC_B + ZP_B;
constexpr int RING = kWarps * D * ITEM_B;
// affine 4-bit layers: two scales and two biases per row and group
constexpr int SC_BA = SG * 64, BI_BA = SG * 64;
constexpr int ITEM_BA = CODE_B + SC_BA + BI_BA;
constexpr int RING_A = kWarps * D * ITEM_BA;
// one token's activation slice (SG groups of 16 chunks of 16 bytes) + 16
// bytes, so consecutive tokens start one bank group apart
constexpr int XROW_B = SG * kGroup * 2 + 16;
constexpr size_t SMEM = (size_t)RING + 16 * XROW_B;
// affine: + the sums of x over the slice's 64-groups, [16 tokens][2 SG] fp32
constexpr int XSUM_N = 16 * 2 * SG;
constexpr size_t SMEM_A = (size_t)RING_A + 16 * XROW_B + XSUM_N * 4;
// cluster mode: the strips a CTA owns, [owned][ns][16 rows][16 tokens] fp32,
// after the other regions (owned = ceil(8 tmax / ns), tmax the CTA's strip blocks)
constexpr int kCluBlocks = 3;       // 4-bit: two CTAs per SM with 24 KB of sums
constexpr int kCluBlocksA = 2;      // affine: its larger ring leaves room for 16 KB
inline size_t clu_part_bytes(int tmax, int ns) { return (size_t)((kWarps * tmax + ns - 1) / ns) * ns * 1024; }
static_assert((XSUM_N * 8) % (kWarps * 32) == 0, "whole warps form the slice sums");
}  // namespace sk

// Position of 16-byte chunk c (0..15) inside a group's 256 activation bytes:
// chunks 8..15 swap pairs, so the four lanes t of a B-fragment load (chunks
// 4t+v) land on four different bank groups.
__device__ __forceinline__ int xchunk(int c) { return c ^ (((c >> 3) & 1) << 1); }

// Affine 4-bit layers: inputs 8cc..8cc+7 of a 128-input block (chunk cc) are
// prepared chunk 4t + w, with cc = 2t + w (w < 2) or 8 + 2t + (w - 2)
// (w >= 2), so the activation slice is stored in the prepared order and the
// operand loads are those of the other layers.
__device__ __forceinline__ int aff_chunk(int cc) {
    return cc < 8 ? 4 * (cc >> 1) + (cc & 1) : 4 * ((cc - 8) >> 1) + 2 + (cc & 1);
}

// AFF: affine 4-bit layers (w = s * q + b per 64-group): words 0, 1 of a
// lane's chunk accumulate apart from words 2, 3 (the two 64-groups of the
// group), each scaled by its own s, and b * (sum of x over the 64-group) is
// added from the slice's sums, formed once per CTA.
template <int NT, bool BF16, bool ASYM, bool AFF, bool CLU = false>
__global__ void __launch_bounds__(kWarps * 32)
gemv_w4_sk_kernel(const uint16_t* __restrict__ x, const uint8_t* __restrict__ codes,
                  const uint16_t* __restrict__ scales, const uint8_t* __restrict__ zeros,
                  const uint16_t* __restrict__ biases, float* __restrict__ part, int M, int Npad, int K, int nslices,
                  int cps, uint16_t* __restrict__ y, int N, int out_bf16) {
    using namespace sk;
    extern __shared__ __align__(16) uint8_t smem[];
    constexpr int ITEM = AFF ? ITEM_BA : ITEM_B;
    constexpr int RINGB = AFF ? RING_A : RING;
    float* own = reinterpret_cast<float*>(smem + (AFF ? SMEM_A : SMEM));   // cluster mode: owned strips' sums

    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int G = K / kGroup;
    const int slice = (int)blockIdx.x % nslices, c = (int)blockIdx.x / nslices;
    const int gb = slice * SG, ng = G - gb < SG ? G - gb : SG;
    const int nstrips = Npad / kStrip;
    const int nblk = (nstrips + kWarps - 1) / kWarps;
    // this warp's strips: 8b + warp for blocks b = c, c + cps, ... (< nstrips)
    int total = c < nblk ? (nblk - 1 - c) / cps + 1 : 0;
    if (total > 0 && kWarps * (c + (total - 1) * cps) + warp >= nstrips) --total;
    uint8_t* ring = smem + (size_t)warp * D * ITEM;
    uint8_t* xsl = smem + RINGB;
    float* xsum = reinterpret_cast<float*>(smem + RINGB + 16 * XROW_B);   // affine: [16][2 SG]

    int is_i = 0, is_slot = 0;
    auto issue_next = [&]() {
        if (is_i < total) {
            const int n0 = (kWarps * (c + is_i * cps) + warp) * kStrip;
            uint8_t* slot = ring + (size_t)is_slot * ITEM;
            const uint8_t* ra = codes + (size_t)(n0 + g) * (K / 2) + (size_t)gb * 64 + 16 * t;
#pragma unroll
            for (int q = 0; q < SG; ++q) {
                if (q < ng) {
                    cp_async16(smem_u32(slot + q * 1024 + lane * 16), ra + 64 * q);
                    cp_async16(smem_u32(slot + q * 1024 + 512 + lane * 16), ra + 64 * q + (size_t)8 * (K / 2));
                }
            }
            if (AFF) {
                // as in the whole-row kernel: lane l < 4 ng the scales of
                // 64-group 2 gb + l / 2, rows 8 (l % 2) .. + 7; lanes 16.. the biases
                if (lane < 4 * ng)
                    cp_async16(smem_u32(slot + CODE_B + 16 * lane),
                               scales + (size_t)(2 * gb + (lane >> 1)) * Npad + n0 + 8 * (lane & 1));
                else if (lane >= 16 && lane < 16 + 4 * ng)
                    cp_async16(smem_u32(slot + CODE_B + SC_BA + 16 * (lane - 16)),
                               biases + (size_t)(2 * gb + ((lane - 16) >> 1)) * Npad + n0 + 8 * (lane & 1));
            } else if (lane < 2 * ng) {
                cp_async16(smem_u32(slot + CODE_B + 16 * lane),
                           scales + (size_t)(gb + (lane >> 1)) * Npad + n0 + 8 * (lane & 1));
            }
            if (ASYM && lane >= 8 && lane < 8 + ng)
                cp_async16(smem_u32(slot + CODE_B + SC_B + 16 * (lane - 8)), zeros + (size_t)(gb + lane - 8) * Npad + n0);
        }
        ++is_i;
        if (++is_slot == D) is_slot = 0;
        cp_commit();
    };

    for (int d = 0; d < D; ++d) issue_next();          // weights before the dependency wait
    // cluster mode, barrier 0: no CTA stores into another's shared memory
    // before every CTA of the cluster has started (wait before the first store)
    if (CLU) cluster_arrive_relaxed();
    pdl_wait();
    // the activation slice of all 16 token rows (rows >= M and groups past K
    // are zero-filled)
    for (int i = threadIdx.x; i < 16 * SG * 16; i += blockDim.x) {
        const int m = i / (SG * 16), q = (i / 16) % SG, cc = i % 16;
        const bool ok = m < M && q < ng;
        cp_async16_zfill(smem_u32(xsl + m * XROW_B + q * 256 + xchunk(AFF ? aff_chunk(cc) : cc) * 16),
                         ok ? x + (size_t)m * K + (size_t)(gb + q) * kGroup + 8 * cc : x, ok);
    }
    cp_commit();
    cp_wait<0>();
    __syncthreads();
    if (AFF) {
        // sum of x over 64-group h of group q for every token: eight lanes a
        // sum, the chunks in their natural order (as the whole-row kernel)
        for (int i = threadIdx.x; i < XSUM_N * 8; i += blockDim.x) {
            const int sidx = i >> 3, cl = i & 7;
            const int m = sidx / (2 * SG), qh = sidx - m * (2 * SG);
            const uint4 u = *reinterpret_cast<const uint4*>(xsl + m * XROW_B + (qh >> 1) * 256 +
                                                            xchunk(aff_chunk(8 * (qh & 1) + cl)) * 16);
            const float v = team8_sum(chunk_sum8(u, BF16));
            if (cl == 0) xsum[sidx] = v;
        }
        __syncthreads();
    }

    int rs = 0;
    for (int i = 0; i < total; ++i) {
        const int strip = kWarps * (c + i * cps) + warp;
        const int n0 = strip * kStrip;
        cp_wait<D - 1>();
        __syncwarp();
        const uint8_t* slot = ring + (size_t)rs * ITEM;
        if (++rs == D) rs = 0;
        uint4 ca[SG], cb[SG];
        float sa[SG], sb[SG];
        int za[SG], zb[SG];
        // affine: raw 16-bit scales / biases of rows g, g + 8: [q][0] the
        // first 64-group, [q][1] the second
        uint32_t sp[SG][2], bp[SG][2];
#pragma unroll
        for (int q = 0; q < SG; ++q) {
            if (q < ng) {
                ca[q] = *reinterpret_cast<const uint4*>(slot + q * 1024 + lane * 16);
                cb[q] = *reinterpret_cast<const uint4*>(slot + q * 1024 + 512 + lane * 16);
                if (AFF) {
                    const uint16_t* sc = reinterpret_cast<const uint16_t*>(slot + CODE_B + 64 * q);
                    const uint16_t* bi = reinterpret_cast<const uint16_t*>(slot + CODE_B + SC_BA + 64 * q);
                    sp[q][0] = (uint32_t)sc[g] | ((uint32_t)sc[g + 8] << 16);
                    sp[q][1] = (uint32_t)sc[16 + g] | ((uint32_t)sc[16 + g + 8] << 16);
                    bp[q][0] = (uint32_t)bi[g] | ((uint32_t)bi[g + 8] << 16);
                    bp[q][1] = (uint32_t)bi[16 + g] | ((uint32_t)bi[16 + g + 8] << 16);
                } else {
                    const uint16_t* sc = reinterpret_cast<const uint16_t*>(slot + CODE_B + 32 * q);
                    sa[q] = __half2float(__ushort_as_half(sc[g]));
                    sb[q] = __half2float(__ushort_as_half(sc[g + 8]));
                    za[q] = ASYM ? (int)slot[CODE_B + SC_B + 16 * q + g] : 8;
                    zb[q] = ASYM ? (int)slot[CODE_B + SC_B + 16 * q + g + 8] : 8;
                }
            }
        }
        __syncwarp();                                    // slot read: refill it
        issue_next();
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
        for (int q = 0; q < SG; ++q) {
            if (q < ng) {
                const uint32_t zca = zero_pair<BF16>(AFF ? 0 : za[q]), zcb = zero_pair<BF16>(AFF ? 0 : zb[q]);
                const uint32_t wa[4] = {ca[q].x, ca[q].y, ca[q].z, ca[q].w};
                const uint32_t wb[4] = {cb[q].x, cb[q].y, cb[q].z, cb[q].w};
                uint32_t a[4][2][4];                     // A fragments of the 8 k16 steps
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    a[w][0][0] = dq_pair<BF16>(wa[w], zca);
                    a[w][0][1] = dq_pair<BF16>(wb[w], zcb);
                    a[w][0][2] = dq_pair<BF16>(wa[w] >> 4, zca);
                    a[w][0][3] = dq_pair<BF16>(wb[w] >> 4, zcb);
                    a[w][1][0] = dq_pair<BF16>(wa[w] >> 8, zca);
                    a[w][1][1] = dq_pair<BF16>(wb[w] >> 8, zcb);
                    a[w][1][2] = dq_pair<BF16>(wa[w] >> 12, zca);
                    a[w][1][3] = dq_pair<BF16>(wb[w] >> 12, zcb);
                }
                // affine: the rows' scales and biases (A: first 64-group, B: second)
                float sAg = 0.f, sAh = 0.f, sBg = 0.f, sBh = 0.f, bAg = 0.f, bAh = 0.f, bBg = 0.f, bBh = 0.f;
                if (AFF) {
                    sAg = to_float((uint16_t)(sp[q][0] & 0xFFFFu), BF16);
                    sAh = to_float((uint16_t)(sp[q][0] >> 16), BF16);
                    sBg = to_float((uint16_t)(sp[q][1] & 0xFFFFu), BF16);
                    sBh = to_float((uint16_t)(sp[q][1] >> 16), BF16);
                    bAg = to_float((uint16_t)(bp[q][0] & 0xFFFFu), BF16);
                    bAh = to_float((uint16_t)(bp[q][0] >> 16), BF16);
                    bBg = to_float((uint16_t)(bp[q][1] & 0xFFFFu), BF16);
                    bBh = to_float((uint16_t)(bp[q][1] >> 16), BF16);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    // B fragments: token nt*8 + g, chunks 4t..4t+3 of group q
                    const uint8_t* xr = xsl + (nt * 8 + g) * XROW_B + q * 256;
                    uint32_t xh[16];
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const uint4 u = *reinterpret_cast<const uint4*>(xr + (4 * t + (v ^ (t & 2))) * 16);
                        xh[4 * v] = u.x; xh[4 * v + 1] = u.y; xh[4 * v + 2] = u.z; xh[4 * v + 3] = u.w;
                    }
                    // d0, d1: words 0, 1 (the first 64-group for affine layers);
                    // e0, e1: words 2, 3 (the second)
                    float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
                    float e0[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        float (&f0)[4] = (AFF && w >= 2) ? e0 : d0;
                        float (&f1)[4] = (AFF && w >= 2) ? e1 : d1;
                        mma16816<BF16>(f0, a[w][0][0], a[w][0][1], a[w][0][2], a[w][0][3], xh[4 * w], xh[4 * w + 1]);
                        mma16816<BF16>(f1, a[w][1][0], a[w][1][1], a[w][1][2], a[w][1][3], xh[4 * w + 2],
                                       xh[4 * w + 3]);
                    }
                    if (AFF) {
                        // tokens nt*8 + 2t, + 1: their 64-group sums of group q
                        const float2 x0 = *reinterpret_cast<const float2*>(xsum + (nt * 8 + 2 * t) * (2 * SG) + 2 * q);
                        const float2 x1 = *reinterpret_cast<const float2*>(xsum + (nt * 8 + 2 * t + 1) * (2 * SG) + 2 * q);
                        acc[nt][0] = fmaf(sBg, e0[0] + e1[0], fmaf(sAg, d0[0] + d1[0], acc[nt][0]));
                        acc[nt][1] = fmaf(sBg, e0[1] + e1[1], fmaf(sAg, d0[1] + d1[1], acc[nt][1]));
                        acc[nt][2] = fmaf(sBh, e0[2] + e1[2], fmaf(sAh, d0[2] + d1[2], acc[nt][2]));
                        acc[nt][3] = fmaf(sBh, e0[3] + e1[3], fmaf(sAh, d0[3] + d1[3], acc[nt][3]));
                        acc[nt][0] = fmaf(bBg, x0.y, fmaf(bAg, x0.x, acc[nt][0]));
                        acc[nt][1] = fmaf(bBg, x1.y, fmaf(bAg, x1.x, acc[nt][1]));
                        acc[nt][2] = fmaf(bBh, x0.y, fmaf(bAh, x0.x, acc[nt][2]));
                        acc[nt][3] = fmaf(bBh, x1.y, fmaf(bAh, x1.x, acc[nt][3]));
                    } else {
                        acc[nt][0] = fmaf(sa[q], d0[0] + d1[0], acc[nt][0]);
                        acc[nt][1] = fmaf(sa[q], d0[1] + d1[1], acc[nt][1]);
                        acc[nt][2] = fmaf(sb[q], d0[2] + d1[2], acc[nt][2]);
                        acc[nt][3] = fmaf(sb[q], d0[3] + d1[3], acc[nt][3]);
                    }
                }
            }
        }
        // partials of this slice: rows n0+g, n0+g+8; tokens nt*8 + 2t, +1
        if (CLU) {
            if (i == 0) cluster_wait();                 // barrier 0 (the loop's trip count is the same in every CTA)
            const int sidx = kWarps * i + warp;         // the CTA's strip sequence
            const uint32_t ps = dsmem_map(smem_u32(own + ((size_t)(sidx / nslices) * nslices + slice) * 256),
                                          (uint32_t)(sidx % nslices));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                dsmem_st_f2(ps + 4u * (g * 16 + nt * 8 + 2 * t), acc[nt][0], acc[nt][1]);
                dsmem_st_f2(ps + 4u * ((g + 8) * 16 + nt * 8 + 2 * t), acc[nt][2], acc[nt][3]);
            }
        } else {
            float* ps = part + ((size_t)slice * Npad + n0) * 16;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                *reinterpret_cast<float2*>(ps + g * 16 + nt * 8 + 2 * t) = make_float2(acc[nt][0], acc[nt][1]);
                *reinterpret_cast<float2*>(ps + (g + 8) * 16 + nt * 8 + 2 * t) = make_float2(acc[nt][2], acc[nt][3]);
            }
        }
        (void)strip;
    }
    cp_wait<0>();
    if (CLU) {
        // a warp with no strip still passes barrier 0 before barrier 1
        if (total == 0) cluster_wait();
        cluster_arrive();                               // barrier 1: every slice sum stored
        cluster_wait();
        // the strips this CTA owns, one warp each: sum the slices 0, 1, ...
        // in order from this CTA's own shared memory; lane: row r = lane / 2,
        // tokens 8h .. 8h + 7
        const int r = lane >> 1, h = lane & 1;
        const int tmax = nblk > c ? (nblk - 1 - c) / cps + 1 : 0;        // the CTA's strip blocks
        const int nown = (kWarps * tmax + nslices - 1) / nslices;
        for (int o = warp; o < nown; o += kWarps) {
            const int sidx = o * nslices + slice;
            if (sidx >= kWarps * tmax) continue;
            const int st = kWarps * (c + (sidx / kWarps) * cps) + sidx % kWarps;
            if (st >= nstrips) continue;
            const float* src = own + (size_t)o * nslices * 256 + r * 16 + 8 * h;
            float a8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int q = 0; q < 8; ++q) {               // at most 8 slices in a cluster: unrolled, the
                if (q < nslices) {                      // loads go out together, the adds in slice order
                    const float4 v0 = *reinterpret_cast<const float4*>(src + q * 256);
                    const float4 v1 = *reinterpret_cast<const float4*>(src + q * 256 + 4);
                    a8[0] += v0.x; a8[1] += v0.y; a8[2] += v0.z; a8[3] += v0.w;
                    a8[4] += v1.x; a8[5] += v1.y; a8[6] += v1.z; a8[7] += v1.w;
                }
            }
            const int n = st * kStrip + r;
            if (n < N) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (8 * h + j < M) y[(size_t)(8 * h + j) * N + n] = from_float(a8[j], out_bf16 != 0);
            }
        }
    }
}

// Second pass of the split-K decode: y[m][n] = sum over the slices s, in the
// order 0, 1, ..., of part[s][n][m] (times rs[m] when a per-token scale is
// given).  One thread per (row, four tokens); the partials come from L2.
__global__ void __launch_bounds__(256)
sk_reduce_kernel(const float* __restrict__ part, const float* __restrict__ rs, uint16_t* __restrict__ y, int M,
                 int N, int Npad, int nslices, int out_bf16) {
    pdl_trigger();
    pdl_wait();
    const int qm = (M + 3) / 4;
    const long long total = (long long)N * qm;
    for (long long i = blockIdx.x * 256ll + threadIdx.x; i < total; i += (long long)gridDim.x * 256) {
        const int n = (int)(i / qm), m0 = 4 * (int)(i % qm);
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        for (int s0 = 0; s0 < nslices; s0 += 8) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (s0 + u < nslices)
                    v[u] = __ldcg(reinterpret_cast<const float4*>(part + ((size_t)(s0 + u) * Npad + n) * 16 + m0));
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (s0 + u < nslices) {
                    a0 += v[u].x; a1 += v[u].y; a2 += v[u].z; a3 += v[u].w;
                }
        }
        const float a[4] = {a0, a1, a2, a3};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (m0 + j < M) y[(size_t)(m0 + j) * N + n] = from_float(rs ? a[j] * rs[m0 + j] : a[j], out_bf16 != 0);
    }
}

// CTAs per slice: about two per SM in total, at most one per strip block.
int sk_cps(const pq_prepared* p) {
    const int ns = w4_slices(p->d.K);
    const int nblk = (p->Npad / kStrip + kWarps - 1) / kWarps;
    int cps = 2 * p->num_sms / ns;
    if (cps < 1) cps = 1;
    return cps < nblk ? cps : nblk;
}

// Cluster mode: CTAs per slice such that every cluster is resident at once.
// Clusters must fit inside one GPC, so fewer of them fit than CTAs would:
// about 85% of two CTAs per SM (measured: 36 clusters of eight 94 KB CTAs
// on 152 SMs); a second wave would cost a whole pass.
int sk_cps_cluster(const pq_prepared* p) {
    const int ns = w4_slices(p->d.K);
    const int nblk = (p->Npad / kStrip + kWarps - 1) / kWarps;
    int cps = (2 * p->num_sms * 27 / 32) / ns;
    if (cps < 1) cps = 1;
    return cps < nblk ? cps : nblk;
}
// The strip blocks the busiest CTA of the cluster grid walks, and whether the
// slices run as clusters (at most 8 of them, and few enough strip blocks that
// the slice sums fit beside the ring at two CTAs per SM).
int sk_tmax(const pq_prepared* p) {
    const int nblk = (p->Npad / kStrip + kWarps - 1) / kWarps, cps = sk_cps_cluster(p);
    return (nblk + cps - 1) / cps;
}
// Only for one 8-token tile (M <= 8): measured over the 7B per-projection
// pass (32 layers x 7 projections in stream order, the cluster kernels
// between two-launch ones) the cluster path took 7.89 against 8.23 us per
// call at M = 8 but 8.89 against 8.69 at M = 16, although chains of one
// shape favoured it at both.
bool sk_cluster(const pq_prepared* p, int M) {
    const bool aff = p->d.fmt == PQ_FMT_W4_AFFINE;
    return M <= 8 && w4_slices(p->d.K) <= 8 && sk_tmax(p) <= (aff ? sk::kCluBlocksA : sk::kCluBlocks);
}

template <int NT, bool BF16, bool ASYM, bool AFF, bool CLU>
cudaError_t launch_sk_t(const pq_prepared* p, const void* x, void* y, int M, cudaStream_t s) {
    const pq_desc& d = p->d;
    const int ns = w4_slices(d.K), cps = CLU ? sk_cps_cluster(p) : sk_cps(p);
    const size_t smem = (AFF ? sk::SMEM_A : sk::SMEM) + (CLU ? sk::clu_part_bytes(sk_tmax(p), ns) : 0);
    cudaError_t e = ensure_smem<gemv_w4_sk_kernel<NT, BF16, ASYM, AFF, CLU>>(smem);
    if (e != cudaSuccess) return e;
    auto kern = gemv_w4_sk_kernel<NT, BF16, ASYM, AFF, CLU>;
    const uint16_t* xx = static_cast<const uint16_t*>(x);
    const uint8_t* cd = static_cast<const uint8_t*>(p->codes);
    const uint16_t* sc = static_cast<const uint16_t*>(p->scales);
    const uint8_t* zp = static_cast<const uint8_t*>(p->zeros);
    const uint16_t* bi = static_cast<const uint16_t*>(AFF ? p->biases : nullptr);
    float* part = reinterpret_cast<float*>(p->ws + p->wl.sk_off);
    uint16_t* yy = static_cast<uint16_t*>(y);
    const int ob = d.out_dtype == PQ_BF16 ? 1 : 0;
    if (CLU)
        return launch_cluster(kern, dim3(ns * cps), dim3(kWarps * 32), smem, s, ns, true, xx, cd, sc, zp, bi, part, M,
                              p->Npad, d.K, ns, cps, yy, d.N, ob);
    e = launch(kern, dim3(ns * cps), dim3(kWarps * 32), smem, s, true, xx, cd, sc, zp, bi, part, M, p->Npad, d.K, ns,
               cps, yy, d.N, ob);
    if (e != cudaSuccess) return e;
    return pq::launch_sk_reduce(p, y, M, ns, nullptr, s);
}

template <int NT, bool BF16, bool ASYM, bool AFF>
cudaError_t launch_sk_c(const pq_prepared* p, const void* x, void* y, int M, cudaStream_t s) {
    return sk_cluster(p, M) ? launch_sk_t<NT, BF16, ASYM, AFF, true>(p, x, y, M, s)
                            : launch_sk_t<NT, BF16, ASYM, AFF, false>(p, x, y, M, s);
}

template <int NT>
cudaError_t launch_sk(const pq_prepared* p, const void* x, void* y, int M, cudaStream_t s) {
    const bool bf16 = p->d.act_dtype == PQ_BF16;
    const bool asym = p->zeros != nullptr;
    if (p->d.fmt == PQ_FMT_W4_AFFINE)
        return bf16 ? launch_sk_c<NT, true, false, true>(p, x, y, M, s)
                    : launch_sk_c<NT, false, false, true>(p, x, y, M, s);
    if (bf16) return asym ? launch_sk_c<NT, true, true, false>(p, x, y, M, s) : launch_sk_c<NT, true, false, false>(p, x, y, M, s);
    return asym ? launch_sk_c<NT, false, true, false>(p, x, y, M, s) : launch_sk_c<NT, false, false, false>(p, x, y, M, s);
}

// Act order: x'[m][k'] = x[m][perm[k']] into the workspace (one pass, before
// the GEMV / GEMM reads it).
__global__ void gather_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm,
                              uint16_t* __restrict__ xg, int M, int K) {
    pdl_trigger();
    pdl_wait();
    const long long total = (long long)M * K;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int m = (int)(i / K), kp = (int)(i % K);
        xg[i] = x[(size_t)m * K + perm[kp]];
    }
}

// Persistent grid: as many CTAs as are resident at once (every CTA starts in
// the first wave), at most one per strip.  `per_sm` is the residency.
int grid_for(const pq_prepared* p, int per_sm) {
    const int nstrips = p->Npad / kStrip;
    const int cap = p->num_sms * (per_sm < 1 ? 1 : per_sm);
    return nstrips < cap ? nstrips : cap;
}

// residency estimate for the host-only planner (shared memory bound)
int est_per_sm(size_t smem) {
    const size_t sm_bytes = 228 * 1024, per_cta = smem + 8 * 1024 + 1024;   // + static + reserved
    int n = (int)(sm_bytes / per_cta);
    return n < 1 ? 1 : (n > 3 ? 3 : n);
}

}  // namespace

namespace pq {

bool w4_affine_runs(const pq_desc& d, int M) {
    // the whole-row kernel where the rows fit, else split-K (16-token tiles)
    return d.fmt == PQ_FMT_W4_AFFINE && M >= 1 && (m1_tile_affine(M, d.K) > 0 || split_k_slices(d) > 0);
}

void plan_w4_gemv(const pq_prepared* p, int M, pq_plan_info* info) {
    info->variant = PQ_VARIANT_W4_GEMV;
    const bool aff = p->d.fmt == PQ_FMT_W4_AFFINE;
    const int mt = aff ? m1_tile_affine(M, p->d.K) : m1_tile(M, p->d.K);
    const bool one = mt > 0;
    info->block = kWarps * 32;
    // the whole-row kernel permutes act-order activations itself where both
    // copies of the rows fit; otherwise a gather launch comes first
    const bool self_gather = m1_gathers(p, M);
    info->launches = (p->d.has_gidx && !self_gather ? 1 : 0) + (one ? 1 : 2);   // (gather) GEMV (slice sum)
    if (one) {
        const size_t smem = m1::smem(p->d.K, mt, self_gather, aff);
        info->grid = grid_for(p, est_per_sm(smem));
        info->smem_bytes = (int)smem;
        info->m_tile = mt;
        info->k_split = kWarps;
    } else {
        const bool clu = sk_cluster(p, M);
        info->grid = w4_slices(p->d.K) * (clu ? sk_cps_cluster(p) : sk_cps(p));
        info->smem_bytes = (int)((aff ? sk::SMEM_A : sk::SMEM) +
                                 (clu ? sk::clu_part_bytes(sk_tmax(p), w4_slices(p->d.K)) : 0));
        if (clu) info->launches -= 1;                    // the slices are added inside the cluster
        info->m_tile = M <= 8 ? 8 : 16;
        info->k_split = w4_slices(p->d.K);
    }
}

// x in the caller's order (under act order the whole-row kernel gathers
// through the permutation; split-K reads a gathered copy in the workspace)
cudaError_t launch_w4_gemv(const pq_prepared* p, const void* x, void* y, int M, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    const bool aff = p->d.fmt == PQ_FMT_W4_AFFINE;
    auto tile = [&](int m) { return aff ? m1_tile_affine(m, p->d.K) : m1_tile(m, p->d.K); };
    if (M <= 16 && tile(M) && (!p->d.has_gidx || m1_gathers(p, M))) return launch_m1(p, x, y, M, false, s);
    const bool gathered = p->d.has_gidx;
    if (gathered) {
        e = launch_gather(p, x, M, s);
        x = p->ws + p->wl.xg_off;
    }
    for (int m0 = 0; m0 < M && e == cudaSuccess; m0 += 16) {
        // M > 16 (forced variant only): 16-token column tiles, stream ordered
        const int mm = M - m0 < 16 ? M - m0 : 16;
        const void* xs = static_cast<const uint16_t*>(x) + (size_t)m0 * p->d.K;
        void* ys = static_cast<uint16_t*>(y) + (size_t)m0 * p->d.N;
        if (tile(mm)) e = launch_m1(p, xs, ys, mm, gathered, s);
        else if (p->wl.sk_bytes == 0) e = cudaErrorInvalidValue;   // workspace sized for M = 1
        else if (mm <= 8) e = launch_sk<1>(p, xs, ys, mm, s);
        else e = launch_sk<2>(p, xs, ys, mm, s);
    }
    return e;
}

cudaError_t launch_sk_reduce(const pq_prepared* p, void* y, int M, int nslices, const float* rs, cudaStream_t s) {
    const long long total = (long long)p->d.N * ((M + 3) / 4);
    long long blocks = (total + 255) / 256;
    const long long cap = 4ll * p->num_sms;
    if (blocks > cap) blocks = cap;
    return launch(sk_reduce_kernel, dim3((unsigned)blocks), dim3(256), 0, s, true,
                  reinterpret_cast<const float*>(p->ws + p->wl.sk_off), rs, static_cast<uint16_t*>(y), M, p->d.N,
                  p->Npad, nslices, p->d.out_dtype == PQ_BF16 ? 1 : 0);
}

cudaError_t launch_gather(const pq_prepared* p, const void* x, int M, cudaStream_t s) {
    const long long total = (long long)M * p->d.K;
    long long blocks = (total + 255) / 256;
    if (blocks > 4 * 1024) blocks = 4 * 1024;
    return launch(gather_kernel, dim3((unsigned)blocks), dim3(256), 0, s, true,
                  static_cast<const uint16_t*>(x), static_cast<const int32_t*>(p->perm),
                  reinterpret_cast<uint16_t*>(p->ws + p->wl.xg_off), M, p->d.K);
}

}  // namespace pq
