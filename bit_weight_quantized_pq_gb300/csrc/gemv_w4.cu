// W4A16 decode GEMV, M = 1..16: y[m][n] = sum_g s[g][n] * sum_{k in g} (q[n][k] - z[g][n]) * x[m][k].
//
// The decode shape of "mate: Marlin-class W4A16 GEMM for mp_31 ... #6" (the
// GEMV "that reads each weight once"): every packed code byte is streamed from
// HBM exactly once.  GB300 design:
//   * persistent CTAs of 8 warps loop over 16-row strips; the warps of a CTA
//     split K into contiguous runs of 128-row groups and reduce each strip
//     through shared memory in a fixed order (deterministic);
//   * every lane streams its own 16-byte code chunks (and the activation and
//     scale slices of the same group) with cp.async into a per-warp ring of D
//     groups, so D groups per lane are in flight without holding registers,
//     across strip boundaries;
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

// Token tiles: MR = 1 (one token), 8 (tokens 1..8) or 16 (9..16).
template <int MR>
struct Cfg {
    static constexpr int NT = MR <= 8 ? 1 : 2;                // n8 tiles
    static constexpr int D = MR == 1 ? 6 : (MR == 8 ? 6 : 4); // ring depth (groups)
    static constexpr int CODE_B = 2 * 32 * 16;                // [row half][lane][16 B]
    // M = 1: the activation row sits once in shared memory for the whole CTA;
    // else each item carries its activation slices [nt][v][lane][16 B]
    static constexpr int X_B = MR == 1 ? 0 : NT * 4 * 32 * 16;
    static constexpr int SC_B = 32, ZP_B = 16;
    static constexpr int ITEM_B = CODE_B + X_B + SC_B + ZP_B;
    static constexpr int RING = kWarps * D * ITEM_B;
    static size_t smem(int K) { return (size_t)RING + (MR == 1 ? (size_t)K * 2 : 0); }
};

// Lane (g = lane/4, t = lane%4) of a warp covering one 16-row strip:
//   k16 step j (0..7) of a group maps mma k-slots {2t,2t+1} to group rows
//   32t+4j+{0,1} and slots {2t+8,2t+9} to 32t+4j+{2,3}, so one lane's A
//   operands are the 32 consecutive rows 32t..32t+31 of output rows n0+g and
//   n0+g+8 (one 16-byte code chunk each), and its B operands are
//   x[token][32t..32t+31] (64 consecutive bytes).
template <int MR, bool BF16, bool ASYM>
__global__ void __launch_bounds__(kWarps * 32)
gemv_w4_kernel(const uint16_t* __restrict__ x, const uint8_t* __restrict__ codes,
               const uint16_t* __restrict__ scales, const uint8_t* __restrict__ zeros,
               uint16_t* __restrict__ y, int M, int N, int Npad, int K, int out_bf16) {
    using C = Cfg<MR>;
    constexpr int NT = C::NT, D = C::D;
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ float red[2][kWarps][NT][4][32];

    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int G = K / kGroup;
    const int gb = (G * warp) / kWarps, ge = (G * (warp + 1)) / kWarps;
    const int gpw = ge - gb;
    const int nstrips = Npad / kStrip;
    const int my_strips = nstrips > (int)blockIdx.x ? (nstrips - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int total = my_strips * gpw;
    uint8_t* ring = smem + (size_t)warp * D * C::ITEM_B;
    const uint16_t* xrow = reinterpret_cast<const uint16_t*>(smem + C::RING);   // M = 1 only

    // activation slices of group grp for this lane (M > 1)
    auto copy_x = [&](uint8_t* slot, int grp) {
        uint8_t* xs = slot + C::CODE_B;
        const uint16_t* xg = x + (size_t)grp * kGroup + 32 * t;
        if (MR != 1) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int m = nt * 8 + g;
                const bool ok = m < M;
                const uint16_t* src = ok ? xg + (size_t)m * K : x;
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    cp_async16_zfill(smem_u32(xs + ((nt * 4 + v) * 32 + lane) * 16), src + (ok ? 8 * v : 0), ok);
            }
        }
    };

    // Items are issued strictly in order: item i is strip i / gpw of this CTA,
    // group gb + i % gpw, ring slot i % D, tracked by counters (no division).
    int is_i = 0, is_strip = (int)blockIdx.x, is_grp = gb, is_slot = 0;
    auto issue_next = [&](bool with_x) {
        if (is_i < total) {
            const int n0 = is_strip * kStrip;
            uint8_t* slot = ring + (size_t)is_slot * C::ITEM_B;
            const uint8_t* ra = codes + (size_t)(n0 + g) * (K / 2) + (size_t)is_grp * 64 + 16 * t;
            cp_async16(smem_u32(slot + lane * 16), ra);
            cp_async16(smem_u32(slot + 512 + lane * 16), ra + (size_t)8 * (K / 2));
            uint8_t* sc = slot + C::CODE_B + C::X_B;
            if (lane < 2) cp_async16(smem_u32(sc + 16 * lane), scales + (size_t)is_grp * Npad + n0 + 8 * lane);
            if (ASYM && lane == 2) cp_async16(smem_u32(sc + C::SC_B), zeros + (size_t)is_grp * Npad + n0);
            if (with_x) copy_x(slot, is_grp);
            if (++is_grp == ge) {
                is_grp = gb;
                is_strip += gridDim.x;
            }
        }
        ++is_i;
        if (++is_slot == D) is_slot = 0;
        cp_commit();   // one group per item (possibly empty) keeps the wait count uniform
    };

    // weights of the first D items before the dependency wait; their
    // activation slices after it
    for (int d = 0; d < D; ++d) issue_next(false);
    pdl_wait();
    if (MR == 1) {
        // the whole activation row, once, by all threads of the CTA
        for (int i = threadIdx.x; i < K / 8; i += blockDim.x)
            cp_async16(smem_u32(xrow + 8 * i), x + 8 * (size_t)i);
    } else {
        for (int d = 0, grp = gb; d < D && d < total; ++d) {
            copy_x(ring + (size_t)d * C::ITEM_B, grp);
            if (++grp == ge) grp = gb;
        }
    }
    cp_commit();
    cp_wait<0>();          // the first D items, weights and activations
    if (MR == 1) __syncthreads(); else __syncwarp();
    int rg = gb;           // group of the next item to consume

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

    int rs = 0;            // ring slot of the next item to consume
    for (int j = 0; j < my_strips; ++j) {
        const int n0 = ((int)blockIdx.x + j * (int)gridDim.x) * kStrip;
        for (int gi = 0; gi < gpw; ++gi) {
            (void)gi;
            cp_wait<D - 1>();
            __syncwarp();
            const uint8_t* slot = ring + (size_t)rs * C::ITEM_B;
            if (++rs == D) rs = 0;
            const uint4 ca = *reinterpret_cast<const uint4*>(slot + lane * 16);
            const uint4 cb = *reinterpret_cast<const uint4*>(slot + 512 + lane * 16);
            uint32_t xh[NT][16];
            if (MR == 1) {
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    uint4 u = make_uint4(0, 0, 0, 0);
                    if (g == 0) u = *reinterpret_cast<const uint4*>(xrow + (size_t)rg * kGroup + 32 * t + 8 * v);
                    xh[0][4 * v] = u.x; xh[0][4 * v + 1] = u.y; xh[0][4 * v + 2] = u.z; xh[0][4 * v + 3] = u.w;
                }
            } else {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const uint4 u = *reinterpret_cast<const uint4*>(slot + C::CODE_B + ((nt * 4 + v) * 32 + lane) * 16);
                        xh[nt][4 * v] = u.x; xh[nt][4 * v + 1] = u.y; xh[nt][4 * v + 2] = u.z; xh[nt][4 * v + 3] = u.w;
                    }
            }
            const uint16_t* sc = reinterpret_cast<const uint16_t*>(slot + C::CODE_B + C::X_B);
            const float sa = __half2float(__ushort_as_half(sc[g]));
            const float sb = __half2float(__ushort_as_half(sc[g + 8]));
            int za = 8, zb = 8;
            if (ASYM) {
                const uint8_t* zp = slot + C::CODE_B + C::X_B + C::SC_B;
                za = zp[g];
                zb = zp[g + 8];
            }
            __syncwarp();                      // every lane has read the slot
            issue_next(true);                  // refill it D items ahead
            if (++rg == ge) rg = gb;

            const uint32_t zca = zero_pair<BF16>(za), zcb = zero_pair<BF16>(zb);
            // four independent accumulator chains (two MMAs each) instead of
            // one chain of eight dependent MMAs
            float d[4][NT][4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) d[c][nt][0] = d[c][nt][1] = d[c][nt][2] = d[c][nt][3] = 0.f;
            const uint32_t wa[4] = {ca.x, ca.y, ca.z, ca.w};
            const uint32_t wb[4] = {cb.x, cb.y, cb.z, cb.w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int sh = 8 * h;
                    const uint32_t a0 = dq_pair<BF16>(wa[w] >> sh, zca);
                    const uint32_t a1 = dq_pair<BF16>(wb[w] >> sh, zcb);
                    const uint32_t a2 = dq_pair<BF16>(wa[w] >> (sh + 4), zca);
                    const uint32_t a3 = dq_pair<BF16>(wb[w] >> (sh + 4), zcb);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma16816<BF16>(d[(w & 1) * 2 + h][nt], a0, a1, a2, a3, xh[nt][4 * w + 2 * h],
                                       xh[nt][4 * w + 2 * h + 1]);
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float s4[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) s4[q] = (d[0][nt][q] + d[1][nt][q]) + (d[2][nt][q] + d[3][nt][q]);
                acc[nt][0] = fmaf(sa, s4[0], acc[nt][0]);
                acc[nt][1] = fmaf(sa, s4[1], acc[nt][1]);
                acc[nt][2] = fmaf(sb, s4[2], acc[nt][2]);
                acc[nt][3] = fmaf(sb, s4[3], acc[nt][3]);
            }
        }
        // strip done: fixed-order reduction over the K-split warps
        float (*rb)[NT][4][32] = red[j & 1];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                rb[warp][nt][q][lane] = acc[nt][q];
                acc[nt][q] = 0.f;
            }
        __syncthreads();
        if (warp == (j % kWarps)) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float s = rb[0][nt][q][lane];
#pragma unroll
                    for (int w = 1; w < kWarps; ++w) s += rb[w][nt][q][lane];
                    const int n = n0 + g + ((q & 2) ? 8 : 0);
                    const int m = nt * 8 + 2 * t + (q & 1);
                    if (m < M && n < N) y[(size_t)m * N + n] = from_float(s, out_bf16 != 0);
                }
        }
    }
    cp_wait<0>();
}

// M = 1 specialisation.  The same lane mapping and exact unpack, with the
// per-item bookkeeping amortised over items of four 128-row groups (4 KB of
// codes per warp, double buffered), and every lane feeding the one activation
// row into all eight MMA columns (the seven extra columns repeat column 0 and
// are ignored), so no operand needs masking.
namespace m1 {
constexpr int IG = 4;                                   // groups per item
constexpr int D = 2;                                    // items per warp ring
constexpr int CODE_B = IG * 1024, SC_B = IG * 32, ZP_B = IG * 16;
constexpr int ITEM_B = CODE_B + SC_B + ZP_B;
constexpr int RING = kWarps * D * ITEM_B;
inline size_t smem(int K) { return (size_t)RING + (size_t)K * 2; }
}  // namespace m1
// the activation row must fit beside the ring (K <= 81920); longer rows take
// the 8-token tile with one live column
inline bool m1_fits(int K) { return m1::smem(K) <= 227 * 1024; }

template <bool BF16, bool ASYM>
__global__ void __launch_bounds__(kWarps * 32)
gemv_w4_m1_kernel(const uint16_t* __restrict__ x, const uint8_t* __restrict__ codes,
                  const uint16_t* __restrict__ scales, const uint8_t* __restrict__ zeros,
                  uint16_t* __restrict__ y, int N, int Npad, int K, int out_bf16) {
    using namespace m1;
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ float red[2][kWarps][2][32];

    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int G = K / kGroup;
    const int gb = (G * warp) / kWarps, ge = (G * (warp + 1)) / kWarps;
    const int ips = (ge - gb + IG - 1) / IG;               // items per strip
    const int nstrips = Npad / kStrip;
    const int my_strips = nstrips > (int)blockIdx.x ? (nstrips - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int total = my_strips * ips;
    uint8_t* ring = smem + (size_t)warp * D * ITEM_B;
    const uint16_t* xrow = reinterpret_cast<const uint16_t*>(smem + RING);

    int is_i = 0, is_strip = (int)blockIdx.x, is_grp = gb, is_slot = 0;
    auto issue_next = [&]() {
        if (is_i < total) {
            const int n0 = is_strip * kStrip;
            const int ng = ge - is_grp < IG ? ge - is_grp : IG;
            uint8_t* slot = ring + (size_t)is_slot * ITEM_B;
            const uint8_t* ra = codes + (size_t)(n0 + g) * (K / 2) + (size_t)is_grp * 64 + 16 * t;
#pragma unroll
            for (int q = 0; q < IG; ++q) {
                if (q < ng) {
                    cp_async16(smem_u32(slot + q * 1024 + lane * 16), ra + 64 * q);
                    cp_async16(smem_u32(slot + q * 1024 + 512 + lane * 16), ra + 64 * q + (size_t)8 * (K / 2));
                }
            }
            if (lane < 2 * ng)
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
    pdl_wait();
    // The row by cp.async, waited together with the two prefetched items: on
    // GB300 this measured faster than a bulk copy on its own mbarrier here
    // (the ternary GEMV, with six items in flight, takes the bulk copy).
    for (int i = threadIdx.x; i < K / 8; i += blockDim.x)
        cp_async16(smem_u32(xrow + 8 * i), x + 8 * (size_t)i);
    cp_commit();
    cp_wait<0>();
    __syncthreads();

    int rs = 0;
    for (int j = 0; j < my_strips; ++j) {
      float acc0 = 0.f, acc1 = 0.f;                      // rows g and g+8 (column 2t)
      // a warp with an empty K-range (K < 1024) still joins the reduction
      for (int cg = gb; cg < ge; cg += IG) {
        cp_wait<D - 1>();
        __syncwarp();
        const uint8_t* slot = ring + (size_t)rs * ITEM_B;
        if (++rs == D) rs = 0;
        const int ng = ge - cg < IG ? ge - cg : IG;
        uint4 ca[IG], cb[IG];
        float sa[IG], sb[IG];
        int za[IG], zb[IG];
#pragma unroll
        for (int q = 0; q < IG; ++q) {
            if (q < ng) {
                ca[q] = *reinterpret_cast<const uint4*>(slot + q * 1024 + lane * 16);
                cb[q] = *reinterpret_cast<const uint4*>(slot + q * 1024 + 512 + lane * 16);
                const uint16_t* sc = reinterpret_cast<const uint16_t*>(slot + CODE_B + 32 * q);
                sa[q] = __half2float(__ushort_as_half(sc[g]));
                sb[q] = __half2float(__ushort_as_half(sc[g + 8]));
                za[q] = ASYM ? (int)slot[CODE_B + SC_B + 16 * q + g] : 8;
                zb[q] = ASYM ? (int)slot[CODE_B + SC_B + 16 * q + g + 8] : 8;
            }
        }
        __syncwarp();                                    // slot read: refill it
        issue_next();
#pragma unroll
        for (int q = 0; q < IG; ++q) {
            if (q < ng) {
                uint32_t xh[16];
                const uint16_t* xs = xrow + (size_t)(cg + q) * kGroup + 32 * t;
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const uint4 u = *reinterpret_cast<const uint4*>(xs + 8 * v);
                    xh[4 * v] = u.x; xh[4 * v + 1] = u.y; xh[4 * v + 2] = u.z; xh[4 * v + 3] = u.w;
                }
                const uint32_t zca = zero_pair<BF16>(za[q]), zcb = zero_pair<BF16>(zb[q]);
                float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
                const uint32_t wa[4] = {ca[q].x, ca[q].y, ca[q].z, ca[q].w};
                const uint32_t wb[4] = {cb[q].x, cb[q].y, cb[q].z, cb[q].w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    mma16816<BF16>(d0, dq_pair<BF16>(wa[w], zca), dq_pair<BF16>(wb[w], zcb),
                                   dq_pair<BF16>(wa[w] >> 4, zca), dq_pair<BF16>(wb[w] >> 4, zcb),
                                   xh[4 * w], xh[4 * w + 1]);
                    mma16816<BF16>(d1, dq_pair<BF16>(wa[w] >> 8, zca), dq_pair<BF16>(wb[w] >> 8, zcb),
                                   dq_pair<BF16>(wa[w] >> 12, zca), dq_pair<BF16>(wb[w] >> 12, zcb),
                                   xh[4 * w + 2], xh[4 * w + 3]);
                }
                acc0 = fmaf(sa[q], d0[0] + d1[0], acc0);
                acc1 = fmaf(sb[q], d0[2] + d1[2], acc1);
            }
        }
      }
      // strip done: fixed-order reduction over the K-split warps
      if (t == 0) {
          red[j & 1][warp][0][g] = acc0;
          red[j & 1][warp][1][g] = acc1;
      }
      __syncthreads();
      if (warp == (j % kWarps) && lane < 16) {
          const int r = lane & 7, hf = lane >> 3;
          float s = red[j & 1][0][hf][r];
#pragma unroll
          for (int w = 1; w < kWarps; ++w) s += red[j & 1][w][hf][r];
          const int n = ((int)blockIdx.x + j * (int)gridDim.x) * kStrip + r + 8 * hf;
          if (n < N) y[n] = from_float(s, out_bf16 != 0);
      }
    }
    cp_wait<0>();
}

template <bool BF16, bool ASYM>
cudaError_t launch_m1_t(const pq_prepared* p, const void* x, void* y, cudaStream_t s) {
    const pq_desc& d = p->d;
    const size_t smem = m1::smem(d.K);
    static thread_local size_t configured = 0;
    static thread_local int per_sm = 1;
    if (configured != smem) {
        cudaError_t e = cudaFuncSetAttribute(gemv_w4_m1_kernel<BF16, ASYM>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_w4_m1_kernel<BF16, ASYM>,
                                                              kWarps * 32, smem);
        if (e != cudaSuccess) return e;
        configured = smem;
    }
    const int nstrips = p->Npad / kStrip;
    const int cap = p->num_sms * (per_sm < 1 ? 1 : per_sm);
    return launch(gemv_w4_m1_kernel<BF16, ASYM>, dim3(nstrips < cap ? nstrips : cap), dim3(kWarps * 32), smem, s,
                  true, static_cast<const uint16_t*>(x), static_cast<const uint8_t*>(p->codes),
                  static_cast<const uint16_t*>(p->scales), static_cast<const uint8_t*>(p->zeros),
                  static_cast<uint16_t*>(y), d.N, p->Npad, d.K, d.out_dtype == PQ_BF16 ? 1 : 0);
}

cudaError_t launch_m1(const pq_prepared* p, const void* x, void* y, cudaStream_t s) {
    const bool bf16 = p->d.act_dtype == PQ_BF16;
    const bool asym = p->zeros != nullptr;
    if (bf16) return asym ? launch_m1_t<true, true>(p, x, y, s) : launch_m1_t<true, false>(p, x, y, s);
    return asym ? launch_m1_t<false, true>(p, x, y, s) : launch_m1_t<false, false>(p, x, y, s);
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

template <int MR, bool BF16, bool ASYM>
cudaError_t launch_t(const pq_prepared* p, const void* x, void* y, int M, cudaStream_t s) {
    const pq_desc& d = p->d;
    const size_t smem = Cfg<MR>::smem(d.K);
    static thread_local size_t configured = 0;
    static thread_local int per_sm = 1;
    if (configured != smem) {
        cudaError_t e = cudaFuncSetAttribute(gemv_w4_kernel<MR, BF16, ASYM>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_w4_kernel<MR, BF16, ASYM>, kWarps * 32,
                                                              smem);
        if (e != cudaSuccess) return e;
        configured = smem;
    }
    return launch(gemv_w4_kernel<MR, BF16, ASYM>, dim3(grid_for(p, per_sm)), dim3(kWarps * 32), smem, s, true,
                  static_cast<const uint16_t*>(x), static_cast<const uint8_t*>(p->codes),
                  static_cast<const uint16_t*>(p->scales), static_cast<const uint8_t*>(p->zeros),
                  static_cast<uint16_t*>(y), M, d.N, p->Npad, d.K, d.out_dtype == PQ_BF16 ? 1 : 0);
}

template <int MR>
cudaError_t launch_mr(const pq_prepared* p, const void* x, void* y, int M, cudaStream_t s) {
    const bool bf16 = p->d.act_dtype == PQ_BF16;
    const bool asym = p->zeros != nullptr;
    if (bf16) return asym ? launch_t<MR, true, true>(p, x, y, M, s) : launch_t<MR, true, false>(p, x, y, M, s);
    return asym ? launch_t<MR, false, true>(p, x, y, M, s) : launch_t<MR, false, false>(p, x, y, M, s);
}

}  // namespace

namespace pq {

void plan_w4_gemv(const pq_prepared* p, int M, pq_plan_info* info) {
    info->variant = PQ_VARIANT_W4_GEMV;
    const bool one = M <= 1 && m1_fits(p->d.K);
    const size_t smem = one ? m1::smem(p->d.K) : M <= 8 ? Cfg<8>::smem(p->d.K) : Cfg<16>::smem(p->d.K);
    info->grid = grid_for(p, est_per_sm(smem));
    info->block = kWarps * 32;
    info->smem_bytes = (int)smem;
    info->launches = p->d.has_gidx ? 2 : 1;
    info->m_tile = one ? 1 : M <= 8 ? 8 : 16;
    info->k_split = kWarps;
}

cudaError_t launch_w4_gemv(const pq_prepared* p, const void* x, void* y, int M, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    for (int m0 = 0; m0 < M && e == cudaSuccess; m0 += 16) {
        // M > 16 (forced variant only): 16-token column tiles
        const int mm = M - m0 < 16 ? M - m0 : 16;
        const void* xs = static_cast<const uint16_t*>(x) + (size_t)m0 * p->d.K;
        void* ys = static_cast<uint16_t*>(y) + (size_t)m0 * p->d.N;
        if (mm == 1 && m1_fits(p->d.K)) e = launch_m1(p, xs, ys, s);
        else if (mm <= 8) e = launch_mr<8>(p, xs, ys, mm, s);
        else e = launch_mr<16>(p, xs, ys, mm, s);
    }
    return e;
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
