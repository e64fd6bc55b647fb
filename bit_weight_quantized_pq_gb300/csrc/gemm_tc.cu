// Prefill GEMM (M >= 17) on the 5th-generation tensor cores.
//
// Computes the same layer as the decode GEMV -- W4A16: y = sum_g s[g][n] *
// sum_{k in g} x[m][k] (q[n][k] - z[g][n]) ("mate: Marlin-class W4A16 GEMM ...
// #6", the 128-row-tile prefill kernel that unpacks int4 before the MMA);
// affine 4-bit: y = sum_h s[h][n] sum_{k in h} x[m][k] q[n][k] + b[h][n] X[m][h]
// over the 64-input groups h, X the sums of x over them ("qwen CUDA:
// --prompt-precision int8 ... #1176": the group's dot on the tensor cores,
// then s times it plus b times the group's sum of x, in fp32);
// ternary W2A8: y = sum_b ws[n][b] xs[m][b] sum_{k in b} q[m][k] (code - 1)
// ("Kernel experiments: recorded evidence", Test 7 int8 tensor-core MMQ and
// Test 21: an exact integer dot per 128-group, then the scales in fp32).
//
// Every MMA operand is exact (|q - z| <= 15, |q| <= 15, |code - 1| <= 2 and
// the quantised activations |q| <= 127 are exact in bf16, and every
// 128-term block dot of the ternary path, at most 2 * 127 * 128 < 2^24 in
// magnitude, is exact in the fp32 accumulator); every scale is applied once
// per group in fp32 by the epilogue.
// Registers: the block is launched with 512 x 128; warps 0-7 give theirs down
// to 64 and warps 8-15 take 192 (setmaxnreg), which adds up to exactly the
// launch allocation.  The host refuses to launch if the compiled kernel does
// not use exactly 128 registers per thread, or spills.
// Every mbarrier wait is bounded (about one second of wall time); on expiry the
// kernel records PQ_ERR_DEVICE_TIMEOUT in the status word, stops every role,
// waits for its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <new>

#include "pq_internal.cuh"

namespace {

using namespace pq;
using namespace pqd;

constexpr int BN = kGemmTileCols;  // weight rows per tile (128, the MMA M)
constexpr int BK = 64;             // inputs per half stage (one 128-byte swizzle atom of bf16)
constexpr int kThreads = 512;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait: false if the CTA is aborting or ~1 s passed (then it aborts
// the CTA and records the timeout).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             uint32_t* status) {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        if (mbar_try(bar, parity)) return true;
        if ((i & 255) == 255) {
            if (*abort_flag) return false;
            const uint64_t now = globaltimer();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > 1000000000ull) {
                *abort_flag = 1;
                atomicCAS(status, 0u, (uint32_t)(int32_t)PQ_ERR_DEVICE_TIMEOUT);
                return false;
            }
        }
    }
}

// Bounded wait for a peer CTA's flag to reach 8 (its 8 epilogue warps wrote
// their rows); every lane polls with acquire semantics, so its later loads
// of the part see the peer's stores.
__device__ __forceinline__ bool wait_flag(const uint32_t* flag, volatile int* abort_flag, uint32_t* status) {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        uint32_t v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v >= 8u) return true;
        if ((i & 63) == 63) {
            if (*abort_flag) return false;
            const uint64_t now = globaltimer();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > 1000000000ull) {
                *abort_flag = 1;
                atomicCAS(status, 0u, (uint32_t)(int32_t)PQ_ERR_DEVICE_TIMEOUT);
                return false;
            }
        }
    }
}

// a short bounded poll used only while draining on exit
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try(bar, parity) && globaltimer() - t0 < 200000000ull) {
    }
}

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar) : "memory");
}

// K-major SWIZZLE_128B operand descriptor: rows of 128 bytes, 8-row atoms of
// 1024 bytes (stride byte offset), tile base 1024-byte aligned.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)1 << 16;                 // leading byte offset (unused for this layout)
    d |= (uint64_t)(1024 >> 4) << 32;       // stride byte offset
    d |= (uint64_t)1 << 46;                 // descriptor version for this architecture
    d |= (uint64_t)2 << 61;                 // SWIZZLE_128B
    return d;
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 columns of this warp's 32 TMEM lanes; the registers are valid only
// after the matching wait (which names them, so no use moves above it)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait16(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :: "memory");
}
// and for 32 columns
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
                   "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait32(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
                   "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :: "memory");
}
// CW columns (16 or 32) by one load
template <int CW>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, uint32_t (&r)[CW]) {
    if constexpr (CW == 32) tmem_ld32(taddr, r);
    else tmem_ld16(taddr, r);
}
template <int CW>
__device__ __forceinline__ void tmem_waitn(uint32_t (&r)[CW]) {
    if constexpr (CW == 32) tmem_wait32(r);
    else tmem_wait16(r);
}

// a0 += t0 * s0, a1 += t1 * s1 in one packed fp32 FMA (each lane an IEEE
// fma, so the same bits as two fmaf)
__device__ __forceinline__ void ffma2(float& a0, float& a1, float t0, float t1, float s0, float s1) {
    asm("{\n\t.reg .b64 ra, rt, rs;\n\tmov.b64 ra, {%0, %1};\n\tmov.b64 rt, {%2, %3};\n\t"
        "mov.b64 rs, {%4, %5};\n\tfma.rn.f32x2 ra, rt, rs, ra;\n\tmov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a0), "+f"(a1) : "f"(t0), "f"(t1), "f"(s0), "f"(s1));
}

// Two codes (bits of `mask` in each 16-bit half of v) -> magic + code, and
// with SUB the exact (code - z) pair.
template <bool BF16, bool SUB = true>
__device__ __forceinline__ uint32_t dq_pair(uint32_t v, uint32_t mask, uint32_t zc) {
    constexpr uint32_t kMagic = BF16 ? 0x43004300u : 0x64006400u;   // 128 / 1024 per half
    const uint32_t t = lop3_and_or(v, mask, kMagic);
    if (!SUB) return t;
    uint32_t d;
    if (BF16)
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(t), "r"(zc));
    else
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(t), "r"(zc));
    return d;
}


// Work of one CTA.  Tile t covers tokens (t % mblocks) * bm and output
// features (t / mblocks) * BN; its work is G = K / 128 groups.  CTA c first
// takes the whole tiles c, c + P, ..., c + (ndp - 1) P, then the contiguous
// range [B0 + c Wsk / P, B0 + (c + 1) Wsk / P) of the remaining tiles'
// groups, counted tile after tile (B0 = ndp P G, Wsk = T G - B0).  So every
// CTA gets the same number of groups, and a tile may be shared by a few
// consecutive CTAs c_lo < ... < c_hi.  The tile is the last segment of c_lo
// (whose range holds the tile's first group: the owner) and the first
// segment of every later one.  The parts are added in CTA order (fixed, so
// the result does not depend on timing) in one of two ways:
//   * own = 1 (a tile is shared by two CTAs at most, the long ranges of
//     large M): the later CTAs finish their parts early, write them to their
//     fp32 slot 0 and count them done on their flag; the owner, at the end
//     of its range, waits for the flags, adds the parts to its own and
//     writes y.  Nothing waits on the owner, and the grid is launched
//     cooperatively (all CTAs resident), so every wait ends.
//   * own = 0 (many CTAs per tile, small M): every part goes to a slot
//     (slot 1 for the owner's) and gemm_wt_fixup_kernel, a second launch,
//     adds them; spread over many CTAs this is faster than one owner
//     reading many parts.
// Without partial slots (Wsk = 0) the schedule is the plain one: tiles c,
// c + P, ... to the end.
// All counts stay below 2^31 (the host shares tiles out only then), and
// c Wsk / P is evaluated as c per + (c rem) / P with Wsk = per P + rem, so the
// kernels need no 64-bit division.
struct Sched {
    int bm;                    // tokens per tile
    int P, G, T, ndp;
    int B0, Wsk, per, rem;
    int mblocks;               // token tiles; t / mblocks = (t * mb_mul) >> mb_shift for t < 2^31
    uint32_t mb_mul;
    int mb_shift;
    int own;                   // 1: owners add the parts; 0: the fixup kernel does
};

// Tile t -> first token and first output feature.  The division by the
// run-time tile count uses a precomputed multiplier (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994):
// with l = ceil(log2 d) and m = ceil(2^(31+l) / d), floor(t m / 2^(31+l)) =
// floor(t / d) for every t < 2^31; it needs fewer registers than a divide.
__host__ __device__ __forceinline__ void tile_origin(const Sched& sc, int t, int& m0, int& n0) {
    const int nb = (int)(((unsigned long long)(uint32_t)t * sc.mb_mul) >> sc.mb_shift);
    m0 = (t - nb * sc.mblocks) * sc.bm;
    n0 = nb * BN;
}

// kind: 0 whole tile; 1 part of a tile another CTA owns (to this CTA's
// slot 0); 2 part of a tile this CTA owns (adds the later CTAs' parts and
// writes y, or with own = 0 goes to slot 1)
struct Seg {
    int tile, g0, g1, kind;
};

__host__ __device__ __forceinline__ int sk_start(const Sched& sc, int c) {
    return sc.B0 + c * sc.per + (c * sc.rem) / sc.P;
}

// This CTA's shared group range [u0, u1) and its first tile, computed once
// (the host keeps T G below 2^31 when it shares tiles out).
struct Range {
    int u0, u1, t0;
    int steps;                 // k-steps of all this CTA's segments (two per group)
};

// The idx-th segment of CTA c's work; false past the end.
// (r points at shared memory and is read when needed: the epilogue keeps
// no copy of it in registers.)
__device__ __forceinline__ bool seg_at(const Sched& sc, const volatile Range* rp, int c, int idx, Seg& out) {
    if (idx < sc.ndp) {
        out.tile = c + idx * sc.P;
        out.g0 = 0;
        out.g1 = sc.G;
        out.kind = 0;
        return out.tile < sc.T;
    }
    const int j = idx - sc.ndp;
    const int u0 = rp->u0, u1 = rp->u1;
    const int t = rp->t0 + j, tu = t * sc.G;
    if (u0 >= u1 || tu >= u1) return false;
    out.tile = t;
    out.g0 = (u0 > tu ? u0 : tu) - tu;
    out.g1 = (u1 < tu + sc.G ? u1 : tu + sc.G) - tu;
    out.kind = (out.g0 == 0 && out.g1 == sc.G) ? 0 : (out.g0 > 0 ? 1 : 2);
    return true;
}

struct GemmArgs {
    uint16_t* y;
    float* part;               // partial slots [2 P][BN / 4][part_rows] float4 (or null)
    uint32_t* flags;           // [P] parts done: 8 contributor warps, then 8 owner warps
    int part_rows;
    const uint16_t* wscales;   // W4: [K/128][Npad] fp16; W2: [Npad][Bp] fp16; affine: [K/64][Npad] (act dtype)
    const uint16_t* wbiases;   // affine: [K/64][Npad] (act dtype)
    const float* xs;           // W2: activation scales [M][K/AG]; affine: sums of x [M][K/64]
    uint32_t* status;
    int M, N, Npad, K, Bp, out_bf16;
};

// ---------------------------------------------------------------------------
// Weight-stationary W4A16 GEMM: the converted weights are the MMA's A
// operand in tensor memory, the tokens its N dimension.
//
// The kernel above reads every converted weight stage from shared memory
// twice (two M = 128 MMAs of 128 tokens each) after writing it there, and
// the tensor core's operand reads alone take about all of an SM's
// shared-memory bandwidth at the dense bf16 rate.  Here the converter
// threads write the bf16 weights straight into tensor memory with
// tcgen05.st (lane = weight row, column c = inputs 2c, 2c + 1), and one
// MMA of M = 128 weight rows x N = 192 tokens x K = 16 reads them from
// there; shared memory carries only the TMA's activation and code tiles and
// the tensor core's activation reads, about 40% less traffic per flop.
// The accumulator is weight rows x tokens, so every epilogue thread holds
// one weight row: it reads its own group scale, with no staging.
//   warp 0      TMA producer: per 128-input group (one stage) two
//               activation tiles [192 tokens x 64 k] (SW128), two code
//               tiles [128 rows x 32 bytes] (+ zero points), 3 stages
//   warp 1      MMA issuer (one thread): per group eight MMAs (M = 128,
//               N = 192, K = 16, A from tensor memory) after three waits,
//               then three commits.  tcgen05.mma issue blocks while the
//               tensor pipe is busy, so the pipe idles whenever this thread
//               waits: a stage per group (not per 64 inputs) halves the
//               waits and commits a group costs (measured: 49% of the
//               thread's time issuing, 36% waiting with 64-input stages)
//   warps 4-7   converters: thread = weight row 32 (warp % 4) + lane;
//               128 codes a group -> exact bf16 (q - z) -> tcgen05.st
//               into one of 2 A stages (64 columns each)
//   warps 8-15  epilogue: weight row 32 (warp % 4) + lane, tokens 96 h ..
//               96 h + 95 (h = (warp - 8) / 4); two accumulator buffers of
//               192 columns
// Tensor memory: accumulators at columns 0 and 192, A stages at 384 + 64 s.
// Ternary layers with one activation scale per token row take the same
// kernel (W2): the converters write the exact bf16 (code - 1) in the
// quantiser's operand order, the epilogue applies the row's block scale per
// group and the token's activation scale once per tile.
// Bounded waits, the schedule (whole tiles, then shared ranges of groups)
// and the deterministic part sums are those of the kernel above.
namespace wt {
constexpr int TM = kGemmTileRows;       // tokens per tile (192, the MMA N)
constexpr int S2 = 3;                   // activation + code ring, one 128-input group a stage
constexpr int SA = 2;                   // A stages in tensor memory, one group each
constexpr int A_COL = 2 * TM;           // first A column
constexpr int A_STAGE = 64;             // columns of one A stage (128 inputs)
constexpr int X_BYTES = TM * BK * 2;    // 24 KB: one 64-input half of a stage's activations
constexpr int WC_BYTES = BN * BK / 2;   // 4 KB: one half's codes
constexpr int WZ_BYTES = BN;
constexpr int TH = TM / 2;              // tokens per epilogue thread
struct Smem {
    static constexpr int x = 0;
    static constexpr int c = x + S2 * 2 * X_BYTES;
    static constexpr int z = c + S2 * 2 * WC_BYTES;
    static constexpr int xw = z + S2 * WZ_BYTES;           // affine: sums of x, [8 epilogue warps][96] fp32
    static constexpr int bar = xw + 8 * TH * 4;
    static constexpr int nbar = 2 * S2 + 2 * SA + 5;
    static constexpr int misc = bar + nbar * 8;
    static constexpr int total = misc + 32;
};
constexpr int kSmem = Smem::total + 1024;
static_assert(A_COL + SA * A_STAGE <= 512, "tensor memory columns");
static_assert(TM % 32 == 0 && TM <= 256, "tokens per tile: the MMA's N and the part slots' rows");
static_assert(kSmem <= 227 * 1024, "shared memory of one CTA");
__host__ __device__ constexpr uint32_t idesc(uint32_t ab_fmt) {
    return (1u << 4) | (ab_fmt << 7) | (ab_fmt << 10) | ((uint32_t)(TM >> 3) << 17) | ((uint32_t)(BN >> 4) << 24);
}
}  // namespace wt

__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

// 16 columns of this warp's 32 lanes from registers
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
                    "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
                 : "memory");
}

// 32 columns of this warp's 32 lanes from registers
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                 :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
                    "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
                    "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
                    "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
                 : "memory");
}



// AFF: affine 4-bit layers (a scale and a bias per 64 inputs).  Each
// 64-input half of a group accumulates into its own buffer (half h -> buffer
// h), and the epilogue adds s * dot + b * X per half with the row's own s and
// b and the tokens' sums of x X (from the pre-pass), which every epilogue warp
// stages for its 96 tokens in shared memory of its own.  The prepared codes
// are in the decode order (a 16-byte chunk t of a 128-input block holds
// inputs 16t .. 16t + 15 of the first 64-group in its words 0-1 and of the
// second in words 2-3); the producer loads a block's 64 code bytes a row and
// the converter of half h takes words 2h, 2h + 1 of every chunk.
// AG128: ternary layers with one activation scale per token and 128-input
// block; the epilogue stages the scales of its tokens per group the same way
// as the affine sums of x and takes t * xs, then times the row's block scale.
template <bool W2, bool BF16, bool ASYM, bool AFF, bool AG128 = false>
__global__ void __launch_bounds__(kThreads, 1)
gemm_wt_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmC,
               const __grid_constant__ CUtensorMap tmZ, const GemmArgs args, const Sched sched) {
    using namespace wt;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(base);
    const uint32_t bar0 = sbase + wt::Smem::bar;
    auto full = [&](int s) { return bar0 + 8 * s; };
    auto empty = [&](int s) { return bar0 + 8 * (S2 + s); };
    auto afull = [&](int s) { return bar0 + 8 * (2 * S2 + s); };
    auto aempty = [&](int s) { return bar0 + 8 * (2 * S2 + SA + s); };
    auto accfull = [&](int b) { return bar0 + 8 * (2 * S2 + 2 * SA + b); };
    auto accempty = [&](int b) { return bar0 + 8 * (2 * S2 + 2 * SA + 2 + b); };
    const uint32_t mma_done = bar0 + 8 * (2 * S2 + 2 * SA + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + wt::Smem::misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + wt::Smem::misc + 4);
    Range* range_sm = reinterpret_cast<Range*>(base + wt::Smem::misc + 8);

    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int M = args.M, N = args.N;
    const int ntiles = sched.T;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S2; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1 + 4);   // MMA commit + 4 converter warps
        }
        for (int s = 0; s < SA; ++s) {
            mbar_init(afull(s), 4);
            mbar_init(aempty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accfull(b), 1);
            mbar_init(accempty(b), 8);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        Range r = {0, 0, 0, 0};
        if (sched.Wsk > 0) {
            r.u0 = sk_start(sched, blockIdx.x);
            r.u1 = sk_start(sched, blockIdx.x + 1);
            r.t0 = r.u0 / sched.G;
        }
        int whole = (sched.T - (int)blockIdx.x + sched.P - 1) / sched.P;
        if (whole > sched.ndp) whole = sched.ndp;
        r.steps = 2 * (whole * sched.G + (r.u1 - r.u0));
        *range_sm = r;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;"
                     :: "r"(smem_u32(tmem_slot)) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    const volatile Range* rng = range_sm;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        asm volatile("setmaxnreg.dec.sync.aligned.u32 64;");
        if (lane == 0) {
            pdl_wait();
            int it = 0;
            bool ok = true;
            Seg sg;
            for (int si = 0; ok && seg_at(sched, rng, blockIdx.x, si, sg); ++si) {
                int m0, n0;
                tile_origin(sched, sg.tile, m0, n0);
                for (int g = sg.g0; g < sg.g1; ++g, ++it) {
                    const int slot = it % S2;
                    if (!wait_bounded(empty(slot), ((it / S2) & 1) ^ 1, abort_flag, args.status)) { ok = false; break; }
                    // ternary code tiles are half as wide (2 bits a weight)
                    constexpr int CB = W2 ? WC_BYTES / 2 : WC_BYTES;
                    mbar_expect_tx(full(slot), 2 * X_BYTES + 2 * CB + (ASYM ? WZ_BYTES : 0));
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        tma_2d(sbase + wt::Smem::x + (2 * slot + hh) * X_BYTES, &tmX, (2 * g + hh) * BK, m0, full(slot));
                        if (!AFF)
                            tma_2d(sbase + wt::Smem::c + (2 * slot + hh) * WC_BYTES, &tmC,
                                   (2 * g + hh) * (W2 ? BK / 4 : BK / 2), n0, full(slot));
                    }
                    // affine: the block's 64 code bytes a row, [128 rows][64 bytes]
                    if (AFF) tma_2d(sbase + wt::Smem::c + 2 * slot * WC_BYTES, &tmC, g * (kGroup / 2), n0, full(slot));
                    if (ASYM) tma_2d(sbase + wt::Smem::z + slot * WZ_BYTES, &tmZ, n0, g, full(slot));
                }
            }
            const int first = it > S2 ? it - S2 : 0;
            for (int j = first; j < it; ++j) drain_wait(full(j % S2), (j / S2) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        asm volatile("setmaxnreg.dec.sync.aligned.u32 64;");
        if (lane == 0) {
            const uint32_t id = idesc(BF16 ? 1u : 0u);
            bool ok = true;
            const int ngroups = rng->steps / 2;
            for (int gc = 0; gc < ngroups; ++gc) {
                const int buf = gc & 1, slot = gc % S2, aslot = gc % SA;
                if (!wait_bounded(full(slot), (gc / S2) & 1, abort_flag, args.status) ||
                    !wait_bounded(afull(aslot), (gc / SA) & 1, abort_flag, args.status) ||
                    !wait_bounded(accempty(AFF ? 0 : buf), ((AFF ? gc : gc >> 1) & 1) ^ 1, abort_flag, args.status)) {
                    ok = false;
                    break;
                }
                fence_after();
                if constexpr (AFF) {
                    // half h into buffer h; buffer 0 was waited for above
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        if (hh == 1) {
                            if (!wait_bounded(accempty(1), (gc & 1) ^ 1, abort_flag, args.status)) { ok = false; break; }
                            fence_after();
                        }
                        const uint64_t db = sw128_desc(sbase + wt::Smem::x + (2 * slot + hh) * X_BYTES);
                        const uint32_t ta = tmem + A_COL + A_STAGE * aslot + 32 * hh;
#pragma unroll
                        for (int j = 0; j < BK / 16; ++j) mma_f16_ta(tmem + hh * TM, ta + 8 * j, db + 2 * j, id, j ? 1u : 0u);
                        mma_commit(accfull(hh));
                    }
                    if (!ok) break;
                    mma_commit(empty(slot));
                    mma_commit(aempty(aslot));
                } else {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const uint64_t db = sw128_desc(sbase + wt::Smem::x + (2 * slot + hh) * X_BYTES);
                        const uint32_t ta = tmem + A_COL + A_STAGE * aslot + 32 * hh;
#pragma unroll
                        for (int j = 0; j < BK / 16; ++j)
                            mma_f16_ta(tmem + buf * TM, ta + 8 * j, db + 2 * j, id, (hh || j) ? 1u : 0u);
                    }
                    mma_commit(empty(slot));
                    mma_commit(aempty(aslot));
                    mma_commit(accfull(buf));
                }
            }
            (void)ok;
            mma_commit(mma_done);
            drain_wait(mma_done, 0);
        }
    } else if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 64;");
    } else if (warp < 8) {
        // ------------------------------------------------ converters (warps 4-7)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 64;");
        const int q = warp & 3, r = 32 * q + lane;       // weight row of the tile
        const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16) + A_COL;
        const int ngroups = rng->steps / 2;
        for (int gc = 0; gc < ngroups; ++gc) {
            const int slot = gc % S2, aslot = gc % SA;
            if (!wait_bounded(full(slot), (gc / S2) & 1, abort_flag, args.status)) break;
            if (!wait_bounded(aempty(aslot), ((gc / SA) & 1) ^ 1, abort_flag, args.status)) break;
            fence_after();
            const uint32_t z = ASYM ? (uint32_t)base[wt::Smem::z + slot * WZ_BYTES + r] : 8u;
            const uint32_t zc = ((BF16 ? 0x4300u : 0x6400u) | z) * 0x00010001u;
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
                if (AFF) {
                    // words 2hh, 2hh + 1 of each 16-byte chunk t of row r's 64
                    // bytes: inputs 16t .. 16t + 15 of 64-group hh, exact q;
                    // two chunks (16 columns) at a time
                    const uint8_t* cs = base + wt::Smem::c + 2 * slot * WC_BYTES + r * 64;
                    const uint32_t zq = (BF16 ? 0x4300u : 0x6400u) * 0x00010001u;   // magic + 0: q exactly
#pragma unroll
                    for (int tp = 0; tp < 2; ++tp) {
                        uint32_t v[16];
#pragma unroll
                        for (int t2 = 0; t2 < 2; ++t2) {
                            const uint2 pr = *reinterpret_cast<const uint2*>(cs + 16 * (2 * tp + t2) + 8 * hh);
                            const uint32_t w[2] = {pr.x, pr.y};
#pragma unroll
                            for (int wi = 0; wi < 2; ++wi) {
                                v[8 * t2 + 4 * wi + 0] = dq_pair<BF16>(w[wi], 0x000F000Fu, zq);
                                v[8 * t2 + 4 * wi + 1] = dq_pair<BF16>(w[wi] >> 4, 0x000F000Fu, zq);
                                v[8 * t2 + 4 * wi + 2] = dq_pair<BF16>(w[wi] >> 8, 0x000F000Fu, zq);
                                v[8 * t2 + 4 * wi + 3] = dq_pair<BF16>(w[wi] >> 12, 0x000F000Fu, zq);
                            }
                        }
                        tmem_st16(trow + A_STAGE * aslot + 32 * hh + 16 * tp, v);
                    }
                    continue;
                }
                if (W2) {
                    // row r's 64 codes of half hh: 16 bytes, word j = inputs
                    // 16j .. 16j + 15 (code of input 16j + k at bits 2k);
                    // column 8j + c holds (code - 1) of inputs 16j + c and
                    // 16j + 8 + c, the order the quantiser gives the tokens;
                    // two words (16 columns) at a time
                    const uint4 w4 = *reinterpret_cast<const uint4*>(base + wt::Smem::c + (2 * slot + hh) * WC_BYTES +
                                                                     r * 16);
                    const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                    for (int jp = 0; jp < 2; ++jp) {
                        uint32_t v[16];
#pragma unroll
                        for (int j2 = 0; j2 < 2; ++j2)
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                v[8 * j2 + c] = dq_pair<true>(w[2 * jp + j2] >> (2 * c), 0x00030003u, 0x43014301u);
                        tmem_st16(trow + A_STAGE * aslot + 32 * hh + 16 * jp, v);
                    }
                    continue;
                }
                uint32_t v[32];
                {
                    // row r's 64 codes of half hh: 32 bytes, word j = inputs 8j .. 8j + 7
                    const uint8_t* cs = base + wt::Smem::c + (2 * slot + hh) * WC_BYTES + r * 32;
                    const uint4 w0 = *reinterpret_cast<const uint4*>(cs);
                    const uint4 w1 = *reinterpret_cast<const uint4*>(cs + 16);
                    const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        // column 4j + i: inputs 8j + 2i, 8j + 2i + 1 (nibbles i, i + 4)
                        v[4 * j + 0] = dq_pair<BF16>(w[j], 0x000F000Fu, zc);
                        v[4 * j + 1] = dq_pair<BF16>(w[j] >> 4, 0x000F000Fu, zc);
                        v[4 * j + 2] = dq_pair<BF16>(w[j] >> 8, 0x000F000Fu, zc);
                        v[4 * j + 3] = dq_pair<BF16>(w[j] >> 12, 0x000F000Fu, zc);
                    }
                }
                tmem_st32(trow + A_STAGE * aslot + 32 * hh, v);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(afull(aslot));
                mbar_arrive(empty(slot));
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 8-15)
        asm volatile("setmaxnreg.inc.sync.aligned.u32 192;");
        pdl_wait();                       // the output buffer follows the stream order
        const int q = warp & 3, h = (warp - 8) >> 2;
        const int r = 32 * q + lane;      // weight row of the tile
        // epilogue groups a 128-input group: affine layers promote each 64-input half
        constexpr int EPG = AFF ? 2 : 1;
        // per-token values staged a group (affine: sums of x; per-block
        // ternary: activation scales), [M][groups] in the workspace
        constexpr bool STAGE = AFF || AG128;
        const int GA = args.K / (AFF ? kAffineGroup : kGroup);
        float* xw = reinterpret_cast<float*>(base + wt::Smem::xw) + (warp - 8) * TH;   // affine
        int ec = 0;
        bool ok = true;
        float acc[TH];
        // this row's scale (and, affine, bias) of epilogue group e of tile
        // `tile`, 0 past the tiles or rows: W4 [G][Npad] fp16, ternary
        // [Npad][Bp] fp16, affine [K/64][Npad] in the activation dtype; and,
        // affine, the sums of x of this warp's tokens lane, lane + 32, lane + 64
        float s_next = 0.f, b_next = 0.f, x_next[3] = {0.f, 0.f, 0.f};
        auto prefetch = [&](int tile, int e) {
            s_next = b_next = 0.f;
            x_next[0] = x_next[1] = x_next[2] = 0.f;
            if (tile >= ntiles) return;
            int tm0, tn0;
            tile_origin(sched, tile, tm0, tn0);
            const int n = tn0 + r;
            if (n < args.Npad) {
                if (AFF) {
                    s_next = to_float(args.wscales[(size_t)e * args.Npad + n], BF16);
                    b_next = to_float(args.wbiases[(size_t)e * args.Npad + n], BF16);
                } else {
                    const uint16_t b = W2 ? args.wscales[(size_t)n * args.Bp + e] : args.wscales[(size_t)e * args.Npad + n];
                    s_next = __half2float(__ushort_as_half(b));
                }
            }
            if (STAGE) {
#pragma unroll
                for (int i = 0; i < 3; ++i) {
                    const int m = tm0 + TH * h + lane + 32 * i;
                    if (m < M) x_next[i] = args.xs[(size_t)m * GA + e];
                }
            }
        };
        Seg sg;
        bool have = seg_at(sched, rng, blockIdx.x, 0, sg);
        if (have) prefetch(sg.tile, EPG * sg.g0);
        for (int si = 0; ok && have; ++si) {
            const int tile = sg.tile, e1 = EPG * sg.g1;
#pragma unroll
            for (int j = 0; j < TH; ++j) acc[j] = 0.f;
            for (int e = EPG * sg.g0; e < e1; ++e, ++ec) {
                const float sc = s_next, bc = b_next;
                if (STAGE) {
                    // stage this group's per-token values for the warp's tokens
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 3; ++i) xw[lane + 32 * i] = x_next[i];
                    __syncwarp();
                }
                if (e + 1 < e1) {
                    prefetch(tile, e + 1);
                } else {
                    Seg nx;
                    if (seg_at(sched, rng, blockIdx.x, si + 1, nx)) prefetch(nx.tile, EPG * nx.g0);
                    else prefetch(ntiles, 0);
                }
                const int buf = ec & 1;
                if (!wait_bounded(accfull(buf), (ec >> 1) & 1, abort_flag, args.status)) { ok = false; break; }
                fence_after();
                const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + buf * TM + TH * h;
                // 32 columns a load (16 for the ternary instantiation, whose
                // extra registers would spill)
                constexpr int CW = W2 ? 16 : 32, NC = TH / CW;
                uint32_t rb0[CW], rb1[CW];
                tmem_ldn<CW>(taddr, rb0);
                tmem_waitn<CW>(rb0);
#pragma unroll
                for (int cc = 0; cc < NC; ++cc) {
                    uint32_t (&cur)[CW] = (cc & 1) ? rb1 : rb0;
                    uint32_t (&nxt)[CW] = (cc & 1) ? rb0 : rb1;
                    if (cc + 1 < NC) tmem_ldn<CW>(taddr + CW * (cc + 1), nxt);
#pragma unroll
                    for (int j = 0; j < CW; j += 4) {
                        if (AG128) {
                            // (t * xs[token]) * ws[row], as the scales' product order of the decode
                            const float4 xv = *reinterpret_cast<const float4*>(xw + CW * cc + j);
                            acc[CW * cc + j] = fmaf(__uint_as_float(cur[j]) * xv.x, sc, acc[CW * cc + j]);
                            acc[CW * cc + j + 1] = fmaf(__uint_as_float(cur[j + 1]) * xv.y, sc, acc[CW * cc + j + 1]);
                            acc[CW * cc + j + 2] = fmaf(__uint_as_float(cur[j + 2]) * xv.z, sc, acc[CW * cc + j + 2]);
                            acc[CW * cc + j + 3] = fmaf(__uint_as_float(cur[j + 3]) * xv.w, sc, acc[CW * cc + j + 3]);
                            continue;
                        }
                        ffma2(acc[CW * cc + j], acc[CW * cc + j + 1], __uint_as_float(cur[j]),
                              __uint_as_float(cur[j + 1]), sc, sc);
                        ffma2(acc[CW * cc + j + 2], acc[CW * cc + j + 3], __uint_as_float(cur[j + 2]),
                              __uint_as_float(cur[j + 3]), sc, sc);
                        if (AFF) {
                            // + b * (sum of x over the 64-group)
                            const float4 xv = *reinterpret_cast<const float4*>(xw + CW * cc + j);
                            ffma2(acc[CW * cc + j], acc[CW * cc + j + 1], xv.x, xv.y, bc, bc);
                            ffma2(acc[CW * cc + j + 2], acc[CW * cc + j + 3], xv.z, xv.w, bc, bc);
                        }
                    }
                    if (cc + 1 < NC) tmem_waitn<CW>(nxt);
                }
                fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(accempty(buf));
            }
            if (!ok) break;
            // segment done: this thread holds y[m0 + TH h + j][n0 + r], j < TH
            seg_at(sched, rng, blockIdx.x, si, sg);
            int m0, n0;
            tile_origin(sched, sg.tile, m0, n0);
            const int mt = m0 + TH * h;          // first token of this thread's columns
            const int n = n0 + r;
            if (W2 && !AG128) {
                // per-row activation scale of every token, before parts are added
#pragma unroll
                for (int j = 0; j < TH; ++j) acc[j] *= mt + j < M ? args.xs[mt + j] : 0.f;
            }
            // part slots: [token quad][BN rows] float4, a warp's store of one
            // quad 512 contiguous bytes
            const size_t qstride = BN;           // float4s between token quads
            const size_t slot_f4 = (size_t)(args.part_rows / 4) * BN;
            if (sg.kind == 1 || (sg.kind == 2 && !sched.own)) {
                float4* dst = reinterpret_cast<float4*>(args.part) + (size_t)(2 * blockIdx.x + sg.kind - 1) * slot_f4 +
                              (size_t)(TH * h / 4) * qstride + r;
#pragma unroll
                for (int jq = 0; jq < TH / 4; ++jq)
                    if (mt + 4 * jq < M)
                        __stcg(dst + jq * qstride,
                               make_float4(acc[4 * jq], acc[4 * jq + 1], acc[4 * jq + 2], acc[4 * jq + 3]));
                if (sched.own) {
                    __threadfence();
                    __syncwarp();
                    if (lane == 0) atomicAdd(args.flags + blockIdx.x, 1u);
                }
                have = seg_at(sched, rng, blockIdx.x, si + 1, sg);
                continue;
            }
            if (sg.kind == 2) {
                const int tu = sg.tile * sched.G;
                int c_hi = blockIdx.x;
                while (c_hi + 1 < sched.P && sk_start(sched, c_hi + 1) < tu + sched.G) ++c_hi;
                for (int c = blockIdx.x + 1; c <= c_hi; ++c) {
                    if (!wait_flag(args.flags + c, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    const float4* src = reinterpret_cast<const float4*>(args.part) + (size_t)(2 * c) * slot_f4 +
                                        (size_t)(TH * h / 4) * qstride + r;
#pragma unroll
                    for (int jq = 0; jq < TH / 4; ++jq) {
                        if (mt + 4 * jq < M) {
                            const float4 v = __ldcg(src + jq * qstride);
                            acc[4 * jq] += v.x;
                            acc[4 * jq + 1] += v.y;
                            acc[4 * jq + 2] += v.z;
                            acc[4 * jq + 3] += v.w;
                        }
                    }
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0)
                    for (int c = blockIdx.x + 1; c <= c_hi; ++c)
                        if (atomicAdd(args.flags + c, 1u) == 15u) atomicExch(args.flags + c, 0u);
            }
            if (n < N) {
#pragma unroll
                for (int j = 0; j < TH; ++j)
                    if (mt + j < M) args.y[(size_t)(mt + j) * N + n] = from_float(acc[j], args.out_bf16 != 0);
            }
            have = seg_at(sched, rng, blockIdx.x, si + 1, sg);
        }
    }

    fence_before();
    __syncthreads();
    if (warp == 0) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" :: "r"(tmem) : "memory");
    }
}

// Fixup of the shared tiles (own = 0).  Tile t is shared when some CTA c's
// range starts strictly inside it; the lowest such c handles it: its parts
// are those of CTAs c - 1 .. c_hi (c_hi the CTA holding the tile's last
// group), added in CTA order (fixed, so the result does not depend on timing)
// and rounded once.  The part of the owner c - 1 is its slot 1; every later
// CTA's part is its slot 0.  Parts are stored [token quad][BN rows] float4;
// one thread per (token quad, weight row) of a shared tile.
__global__ void __launch_bounds__(256)
gemm_wt_fixup_kernel(const float* __restrict__ part, uint16_t* __restrict__ y, const Sched sc, int M, int N,
                     int part_rows, int out_bf16) {
    pdl_trigger();
    pdl_wait();
    constexpr int kPer = (wt::TM / 4) * BN / 256;            // CTAs per boundary
    const int c = 1 + blockIdx.x / kPer;
    const int u = sk_start(sc, c);
    if (u % sc.G == 0) return;
    const int t = u / sc.G, tu = t * sc.G;
    if (c > 1 && sk_start(sc, c - 1) > tu) return;
    int c_hi = c;
    while (c_hi + 1 < sc.P && sk_start(sc, c_hi + 1) < tu + sc.G) ++c_hi;
    const int c_lo = c - 1;
    int m0, n0;
    tile_origin(sc, t, m0, n0);
    const int idx = (blockIdx.x % kPer) * 256 + threadIdx.x;
    const int tq = idx / BN, r = idx % BN;
    if (m0 + 4 * tq >= M) return;
    const size_t slot_f4 = (size_t)(part_rows / 4) * BN;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int cc = c_lo; cc <= c_hi; ++cc) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(part) + (size_t)(2 * cc + (cc == c_lo ? 1 : 0)) * slot_f4 +
                                (size_t)tq * BN + r);
        a.x += v.x;
        a.y += v.y;
        a.z += v.z;
        a.w += v.w;
    }
    const int n = n0 + r;
    if (n >= N) return;
    const float o[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (m0 + 4 * tq + j < M) y[(size_t)(m0 + 4 * tq + j) * N + n] = from_float(o[j], out_bf16 != 0);
}

// Affine layers: X[m][h] = sum of x[m][k] over 64-group h, fp32, for the
// GEMM's epilogue.  Eight lanes a group, one 16-byte chunk each (x is
// row-major, so lane i of the grid reads chunk i of the whole matrix).
template <bool BF16>
__global__ void __launch_bounds__(256)
affine_xsum_kernel(const uint16_t* __restrict__ x, float* __restrict__ xsum, long long chunks) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const long long stride = (long long)gridDim.x * blockDim.x;
    // whole warps take every step (chunks is a multiple of 16), so the
    // team sum's shuffles see all 32 lanes
    for (long long i0 = (long long)blockIdx.x * blockDim.x + (threadIdx.x & ~31); i0 < chunks; i0 += stride) {
        const long long i = i0 + lane;
        float v = 0.f;
        if (i < chunks) v = chunk_sum8(ldg_v4(x + 8 * i), BF16);
        v = team8_sum(v);
        if (i < chunks && (i & 7) == 0) xsum[i >> 3] = v;
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

// The schedule of a launch (see Sched).  Sharing the last one to two waves
// of tiles out by groups evens the CTAs' work, but the parts cost an extra
// write and read: about kOwnGroups groups of one CTA's time when owners add
// them, kFixupGroups with the fixup launch (~1.5 us per 128-row group of a
// 256 x 128 tile on GB300; measured).  So the shared schedule is taken only
// where the busiest CTA of the plain one does more than that much extra
// work.  *shared: some tile is shared.
constexpr int kOwnGroups = 5;
constexpr int kFixupGroups = 9;

Sched make_sched(const pq_prepared* p, int M, int bm, bool* shared) {
    const int mblocks = (M + bm - 1) / bm, nblocks = (p->d.N + BN - 1) / BN;
    Sched sc;
    sc.bm = bm;
    sc.T = mblocks * nblocks;
    sc.mblocks = mblocks;
    int l = 0;
    while ((1ll << l) < mblocks) ++l;
    sc.mb_shift = 31 + l;
    sc.mb_mul = (uint32_t)(((1ull << (31 + l)) + (unsigned long long)mblocks - 1) / (unsigned long long)mblocks);
    sc.G = p->d.K / kGroup;
    sc.per = sc.rem = 0;
    sc.B0 = sc.Wsk = 0;
    sc.own = 0;
    // plain: tiles c, c + P, ... (the busiest CTA does ceil(T / P) tiles)
    sc.P = sc.T < p->num_sms ? sc.T : p->num_sms;
    sc.ndp = (sc.T + sc.P - 1) / sc.P;
    *shared = false;
    const long long TG = (long long)sc.T * sc.G;
    if (p->wl.gp_bytes == 0 || M > p->d.max_m || TG >= (1ll << 30)) return sc;
    int P = p->num_sms < kGemmMaxCtas ? p->num_sms : kGemmMaxCtas;
    if (TG < P) P = (int)TG;
    const int ndp = sc.T >= P ? sc.T / P - 1 : 0;
    const long long B0 = (long long)ndp * P * sc.G, Wsk = TG - B0;
    const long long busiest = ndp * (long long)sc.G + (Wsk + P - 1) / P;     // groups of the busiest CTA
    const bool parts = (Wsk % ((long long)P * sc.G)) != 0;
    const bool own = Wsk / P >= sc.G;          // every tile shared by two CTAs at most
    if (parts && (long long)sc.ndp * sc.G <= busiest + (own ? kOwnGroups : kFixupGroups)) return sc;
    sc.P = P;
    sc.ndp = ndp;
    sc.B0 = (int)B0;
    sc.Wsk = (int)Wsk;
    sc.per = (int)(Wsk / P);
    sc.rem = (int)(Wsk % P);
    sc.own = own ? 1 : 0;
    *shared = parts;
    return sc;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool load_encode() {
    if (g_encode) return true;
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return false;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return true;
}

bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    return g_encode(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct GemmState {
    CUtensorMap codes, zeros;
};

template <bool W2, bool BF16, bool ASYM, bool AFF = false, bool AG128 = false>
cudaError_t launch_wt(const pq_prepared* p, const void* x, const float* xs, void* y, int M, cudaStream_t s) {
    const pq_desc& d = p->d;
    const GemmState* st = static_cast<const GemmState*>(p->gemm_state);
    CUtensorMap tmX;
    if (!encode_2d(&tmX, BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x, (uint64_t)d.K,
                   (uint64_t)M, (uint64_t)d.K * 2, BK, wt::TM, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    // the setmaxnreg split needs exactly 128 registers a thread at launch
    static std::atomic<int> regs_ok{0};
    if (!regs_ok.load(std::memory_order_relaxed)) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, gemm_wt_kernel<W2, BF16, ASYM, AFF, AG128>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != 128 || fa.localSizeBytes != 0) return cudaErrorInvalidDeviceFunction;
        regs_ok.store(1);
    }
    {
        cudaError_t e = ensure_smem<gemm_wt_kernel<W2, BF16, ASYM, AFF, AG128>>((size_t)wt::kSmem);
        if (e != cudaSuccess) return e;
    }
    GemmArgs args;
    args.y = static_cast<uint16_t*>(y);
    args.flags = reinterpret_cast<uint32_t*>(p->ws + p->wl.flags_off);
    args.part = reinterpret_cast<float*>(p->ws + p->wl.gp_off);
    args.part_rows = p->wl.gp_rows;
    args.wscales = p->scales;
    args.wbiases = AFF ? p->biases : nullptr;
    args.xs = xs;
    args.status = p->status;
    args.M = M;
    args.N = d.N;
    args.Npad = p->Npad;
    args.K = d.K;
    args.Bp = w2_bp(d.K);
    args.out_bf16 = d.out_dtype == PQ_BF16 ? 1 : 0;
    bool shared = false;
    const Sched sc = make_sched(p, M, wt::TM, &shared);
    if (shared && sc.own)
        return launch_cooperative(gemm_wt_kernel<W2, BF16, ASYM, AFF, AG128>, dim3(sc.P), dim3(kThreads), wt::kSmem, s, true, tmX,
                                  st->codes, st->zeros, args, sc);
    cudaError_t e = launch(gemm_wt_kernel<W2, BF16, ASYM, AFF, AG128>, dim3(sc.P), dim3(kThreads), wt::kSmem, s, true, tmX, st->codes,
                           st->zeros, args, sc);
    if (e != cudaSuccess || !shared) return e;
    constexpr int kPer = (wt::TM / 4) * BN / 256;
    return launch(gemm_wt_fixup_kernel, dim3((sc.P - 1) * kPer), dim3(256), 0, s, true,
                  reinterpret_cast<const float*>(args.part), args.y, sc, M, d.N, args.part_rows, args.out_bf16);
}

}  // namespace

namespace pq {

bool gemm_supported(const pq_desc&) { return true; }

void plan_gemm(const pq_prepared* p, int M, pq_plan_info* info) {
    info->variant = p->d.fmt == PQ_FMT_W2_PQ2 ? PQ_VARIANT_W2_GEMM : PQ_VARIANT_W4_GEMM;
    bool shared = false;
    const Sched sc = make_sched(p, M, wt::TM, &shared);
    info->grid = sc.P;
    info->block = kThreads;
    info->smem_bytes = wt::kSmem;
    // (gather) + (ternary quantise / affine sums pre-pass) + GEMM + (fixup of shared tiles)
    info->launches = 1 + (p->d.has_gidx ? 1 : 0) + (p->d.fmt != PQ_FMT_W4_GPTQ ? 1 : 0) +
                     (shared && !sc.own ? 1 : 0);
    info->m_tile = wt::TM;
    // CTAs sharing one output tile at most
    info->k_split = 1;
    if (sc.Wsk > 0) {
        const int per = sc.per > 0 ? sc.per : 1;           // groups per CTA, at least
        info->k_split = (sc.G + per - 1) / per + 1 < sc.P ? (sc.G + per - 1) / per + 1 : sc.P;
        if (!shared) info->k_split = 1;
    }
}

int32_t gemm_init(pq_prepared* p) {
    if (!load_encode()) return fail(PQ_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    GemmState* st = new (std::nothrow) GemmState();
    if (!st) return fail(PQ_ERR_INVALID_ARG, "host allocation failed");
    const pq_desc& d = p->d;
    bool ok;
    if (d.fmt == PQ_FMT_W4_AFFINE) {
        // a 128-input block's 64 code bytes per row
        ok = encode_2d(&st->codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, p->codes, (uint64_t)d.K / 2, (uint64_t)p->Npad,
                       (uint64_t)d.K / 2, kGroup / 2, BN, CU_TENSOR_MAP_SWIZZLE_NONE);
        st->zeros = st->codes;
    } else if (d.fmt == PQ_FMT_W4_GPTQ) {
        ok = encode_2d(&st->codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, p->codes, (uint64_t)d.K / 2, (uint64_t)p->Npad,
                       (uint64_t)d.K / 2, BK / 2, BN, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (ok && p->zeros)
            ok = encode_2d(&st->zeros, CU_TENSOR_MAP_DATA_TYPE_UINT8, p->zeros, (uint64_t)p->Npad, (uint64_t)p->G,
                           (uint64_t)p->Npad, BN, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
        else
            st->zeros = st->codes;
    } else {
        ok = encode_2d(&st->codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, p->codes, (uint64_t)d.K / 4, (uint64_t)p->Npad,
                       (uint64_t)d.K / 4, BK / 4, BN, CU_TENSOR_MAP_SWIZZLE_NONE);
        st->zeros = st->codes;
    }
    if (!ok) {
        delete st;
        return fail(PQ_ERR_CUDA, "tensor map encoding failed for the prepared planes");
    }
    p->gemm_state = st;
    return PQ_OK;
}

void gemm_free(pq_prepared* p) {
    delete static_cast<GemmState*>(p->gemm_state);
    p->gemm_state = nullptr;
}

cudaError_t launch_w4_gemm(const pq_prepared* p, const void* x, void* y, int M, cudaStream_t s) {
    const bool bf16 = p->d.act_dtype == PQ_BF16;
    if (p->d.fmt == PQ_FMT_W4_AFFINE) {
        // the sums of x over every 64-group, then the GEMM
        float* xsum = reinterpret_cast<float*>(p->ws + p->wl.xs_off);
        const long long chunks = (long long)M * p->d.K / 8;
        long long blocks = (chunks + 255) / 256;
        if (blocks > 4ll * p->num_sms) blocks = 4ll * p->num_sms;
        cudaError_t e = bf16 ? launch(affine_xsum_kernel<true>, dim3((unsigned)blocks), dim3(256), 0, s, true,
                                      static_cast<const uint16_t*>(x), xsum, chunks)
                             : launch(affine_xsum_kernel<false>, dim3((unsigned)blocks), dim3(256), 0, s, true,
                                      static_cast<const uint16_t*>(x), xsum, chunks);
        if (e != cudaSuccess) return e;
        return bf16 ? launch_wt<false, true, false, true>(p, x, xsum, y, M, s)
                    : launch_wt<false, false, false, true>(p, x, xsum, y, M, s);
    }
    if (p->zeros)
        return bf16 ? launch_wt<false, true, true>(p, x, nullptr, y, M, s)
                    : launch_wt<false, false, true>(p, x, nullptr, y, M, s);
    return bf16 ? launch_wt<false, true, false>(p, x, nullptr, y, M, s)
                : launch_wt<false, false, false>(p, x, nullptr, y, M, s);
}

// a.qa holds the bf16 codes and a.xs the activation scales written by the
// quantiser (the pre-pass or the fused norm producer)
cudaError_t launch_w2_gemm(const pq_prepared* p, void* y, int M, const ActPlanes& a, cudaStream_t s) {
    // per-block activation scales: the token-stationary kernel (a scale per
    // token and group); one scale per token row: the weight-stationary one
    if (p->d.act_group == kGroup) return launch_wt<true, true, false, false, true>(p, a.qa, a.xs, y, M, s);
    return launch_wt<true, true, false>(p, a.qa, a.xs, y, M, s);
}

}  // namespace pq
