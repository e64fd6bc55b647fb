// W4A16 decode GEMV, M = 1..16: y[m][n] = sum_g s[g][n] * sum_{k in g} (q[n][k] - z[g][n]) * x[m][k].
//
// The decode shape of "mate: Marlin-class W4A16 GEMM for mp_31 ... #6" (the
// GEMV "that reads each weight once"): every packed code byte is streamed from
// HBM exactly once with 16-byte loads.  GB300 design:
//   * a warp owns a strip of 16 output rows and a contiguous run of 128-row
//     groups; the warps of a CTA split K and reduce through shared memory in a
//     fixed order (deterministic);
//   * codes are turned into exact fp16/bf16 values (q - z) with one LOP3 per
//     two weights (nibble OR exponent bits: 1024+q / 128+q) and one packed
//     subtract, and consumed directly as the A fragment of
//     mma.m16n8k16 (weights are the 16-row operand, tokens the 8 columns);
//   * each 128-row group accumulates into a fresh fp32 fragment that is then
//     scaled by s[g][n] and added to the running sum, so the scale is applied
//     exactly once per group in fp32;
//   * weight loads for the first groups are issued before griddepcontrol.wait,
//     so under programmatic dependent launch the weight stream overlaps the
//     previous kernel's tail; activations are read only after the wait.
#include "pq_internal.cuh"

namespace {

using namespace pq;
using namespace pqd;

constexpr int kMaxWarps = 16;

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
    // (magic + z) in both halves; magic + z <= 1039 / 143 is exact
    const uint32_t h = BF16 ? (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(128.0f + z))
                            : (uint32_t)__half_as_ushort(__float2half_rn(1024.0f + z));
    return h | (h << 16);
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

struct GroupRegs {
    uint4 ca, cb;      // codes of rows g and g+8: 32 consecutive k each
    uint16_t sa, sb;   // scales of rows g, g+8
    uint8_t za, zb;    // zero points of rows g, g+8
};

template <bool ASYM>
__device__ __forceinline__ void load_group(GroupRegs& r, const uint8_t* rowA, const uint8_t* rowB,
                                           const uint16_t* sc, const uint8_t* zp, int grp, int Npad) {
    r.ca = ldg_stream(rowA + (size_t)grp * 64);
    r.cb = ldg_stream(rowB + (size_t)grp * 64);
    r.sa = __ldg(sc + (size_t)grp * Npad);
    r.sb = __ldg(sc + (size_t)grp * Npad + 8);
    if (ASYM) {
        r.za = __ldg(zp + (size_t)grp * Npad);
        r.zb = __ldg(zp + (size_t)grp * Npad + 8);
    } else {
        r.za = r.zb = 8;
    }
}

// Lane (g = lane/4, t = lane%4) of a warp covering one 16-row strip:
//   k16 step j (0..7) of a group maps mma k-slots {2t,2t+1} to group rows
//   32t+4j+{0,1} and slots {2t+8,2t+9} to 32t+4j+{2,3}, so one lane's A
//   operands are the 32 consecutive rows 32t..32t+31 of rows n0+g and
//   n0+g+8, and its B operands are x[token g][32t..32t+31] (consecutive).
template <int NT, bool BF16>
__device__ __forceinline__ void group_mma(float (&acc)[NT][4], const GroupRegs& r,
                                          const uint32_t (&xh)[NT][16]) {
    const uint32_t zca = zero_pair<BF16>(r.za), zcb = zero_pair<BF16>(r.zb);
    float d[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
    const uint32_t wa[4] = {r.ca.x, r.ca.y, r.ca.z, r.ca.w};
    const uint32_t wb[4] = {r.cb.x, r.cb.y, r.cb.z, r.cb.w};
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
                mma16816<BF16>(d[nt], a0, a1, a2, a3, xh[nt][4 * w + 2 * h], xh[nt][4 * w + 2 * h + 1]);
        }
    }
    const float sa = __half2float(__ushort_as_half(r.sa));
    const float sb = __half2float(__ushort_as_half(r.sb));
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        acc[nt][0] = fmaf(sa, d[nt][0], acc[nt][0]);
        acc[nt][1] = fmaf(sa, d[nt][1], acc[nt][1]);
        acc[nt][2] = fmaf(sb, d[nt][2], acc[nt][2]);
        acc[nt][3] = fmaf(sb, d[nt][3], acc[nt][3]);
    }
}

template <int NT>
__device__ __forceinline__ void load_x(uint32_t (&xh)[NT][16], const uint16_t* __restrict__ x, int M,
                                       int K, int grp, int g, int t) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int m = nt * 8 + g;
        if (m < M) {
            const uint16_t* src = x + (size_t)m * K + (size_t)grp * kGroup + 32 * t;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 u = ldg_v4(src + 8 * v);
                xh[nt][4 * v + 0] = u.x;
                xh[nt][4 * v + 1] = u.y;
                xh[nt][4 * v + 2] = u.z;
                xh[nt][4 * v + 3] = u.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) xh[nt][i] = 0u;
        }
    }
}

template <int NT, bool BF16, bool ASYM>
__global__ void __launch_bounds__(kMaxWarps * 32)
gemv_w4_kernel(const uint16_t* __restrict__ x, const uint8_t* __restrict__ codes,
               const uint16_t* __restrict__ scales, const uint8_t* __restrict__ zeros,
               uint16_t* __restrict__ y, int M, int N, int Npad, int K, int out_bf16) {
    __shared__ float red[kMaxWarps][NT][4][32];
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = blockDim.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int n0 = blockIdx.x * kStrip;
    const int G = K / kGroup;
    const int gb = (G * warp) / W, ge = (G * (warp + 1)) / W;

    const uint8_t* rowA = codes + (size_t)(n0 + g) * (K / 2) + 16 * t;
    const uint8_t* rowB = rowA + (size_t)8 * (K / 2);
    const uint16_t* sc = scales + n0 + g;
    const uint8_t* zp = ASYM ? zeros + n0 + g : nullptr;

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

    // two-group pipeline stages, double buffered in registers
    GroupRegs cur0, cur1, nxt0, nxt1;
    if (gb < ge) load_group<ASYM>(cur0, rowA, rowB, sc, zp, gb, Npad);
    if (gb + 1 < ge) load_group<ASYM>(cur1, rowA, rowB, sc, zp, gb + 1, Npad);
    pdl_wait();   // x may be the previous kernel's output
    uint32_t xh[NT][16];
    for (int grp = gb; grp < ge; grp += 2) {
        if (grp + 2 < ge) load_group<ASYM>(nxt0, rowA, rowB, sc, zp, grp + 2, Npad);
        if (grp + 3 < ge) load_group<ASYM>(nxt1, rowA, rowB, sc, zp, grp + 3, Npad);
        load_x<NT>(xh, x, M, K, grp, g, t);
        group_mma<NT, BF16>(acc, cur0, xh);
        if (grp + 1 < ge) {
            load_x<NT>(xh, x, M, K, grp + 1, g, t);
            group_mma<NT, BF16>(acc, cur1, xh);
        }
        cur0 = nxt0;
        cur1 = nxt1;
    }

#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) red[warp][nt][i][lane] = acc[nt][i];
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float s = 0.f;
                for (int w = 0; w < W; ++w) s += red[w][nt][i][lane];   // fixed order
                const int n = n0 + g + ((i & 2) ? 8 : 0);
                const int m = nt * 8 + 2 * t + (i & 1);
                if (m < M && n < N) y[(size_t)m * N + n] = from_float(s, out_bf16 != 0);
            }
        }
    }
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

template <int NT, bool BF16, bool ASYM>
cudaError_t launch_t(const pq_prepared* p, const void* x, void* y, int M, int warps, cudaStream_t s) {
    const pq_desc& d = p->d;
    return launch(gemv_w4_kernel<NT, BF16, ASYM>, dim3(p->Npad / kStrip), dim3(warps * 32), 0, s, true,
                  static_cast<const uint16_t*>(x), static_cast<const uint8_t*>(p->codes),
                  static_cast<const uint16_t*>(p->scales), static_cast<const uint8_t*>(p->zeros),
                  static_cast<uint16_t*>(y), M, d.N, p->Npad, d.K, d.out_dtype == PQ_BF16 ? 1 : 0);
}

int warps_for(int G) {
    // at least two groups per warp, at most 16 warps
    int w = G / 2;
    if (w > kMaxWarps) w = kMaxWarps;
    if (w < 1) w = 1;
    return w;
}

}  // namespace

namespace pq {

void plan_w4_gemv(const pq_prepared* p, int M, pq_plan_info* info) {
    info->variant = PQ_VARIANT_W4_GEMV;
    info->grid = p->Npad / kStrip;
    info->block = warps_for(p->G) * 32;
    info->smem_bytes = 0;
    info->launches = p->d.has_gidx ? 2 : 1;
    info->m_tile = M <= 8 ? 8 : 16;
    info->k_split = warps_for(p->G);
}

cudaError_t launch_w4_gemv(const pq_prepared* p, const void* x, void* y, int M, cudaStream_t s) {
    const bool bf16 = p->d.act_dtype == PQ_BF16;
    const bool asym = p->zeros != nullptr;
    const int warps = warps_for(p->G);
    cudaError_t e = cudaSuccess;
    for (int m0 = 0; m0 < M && e == cudaSuccess; m0 += 16) {
        // M > 16 (only when no GEMM variant exists): 16-token column tiles
        const int mm = M - m0 < 16 ? M - m0 : 16;
        const void* xs = static_cast<const uint16_t*>(x) + (size_t)m0 * p->d.K;
        void* ys = static_cast<uint16_t*>(y) + (size_t)m0 * p->d.N;
        if (mm <= 8) {
            if (bf16) e = asym ? launch_t<1, true, true>(p, xs, ys, mm, warps, s) : launch_t<1, true, false>(p, xs, ys, mm, warps, s);
            else      e = asym ? launch_t<1, false, true>(p, xs, ys, mm, warps, s) : launch_t<1, false, false>(p, xs, ys, mm, warps, s);
        } else {
            if (bf16) e = asym ? launch_t<2, true, true>(p, xs, ys, mm, warps, s) : launch_t<2, true, false>(p, xs, ys, mm, warps, s);
            else      e = asym ? launch_t<2, false, true>(p, xs, ys, mm, warps, s) : launch_t<2, false, false>(p, xs, ys, mm, warps, s);
        }
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
