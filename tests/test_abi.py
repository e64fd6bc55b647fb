"""Host-side checks of the C ABI (no GPU): the library builds and loads,
exports every function include/pq.h declares, its constants match the
header, sizes and layouts follow the prepared-plane definition, the
dispatcher's decisions, and the refusals that happen before any launch."""
from __future__ import annotations

import os
import re

import numpy as np
import pytest

import bit_weight_quantized_pq_gb300 as pq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pq.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    pq.build()
    pq.lib()


def header_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"PQ_API\s+[\w\s\*]+?\b(pq_\w+)\s*\(", text)))


def header_defines():
    text = open(HEADER).read()
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"#define\s+(PQ_\w+)\s+(-?\d+)", text)}


def test_exports_every_declared_function():
    names = header_functions()
    assert len(names) >= 14
    lib = pq.lib()
    for n in names:
        assert hasattr(lib, n), n
        assert n in pq._SIGNATURES, f"binding lacks {n}"


def test_constants_match_header():
    for name, val in header_defines().items():
        assert getattr(pq, name) == val, name


def test_struct_layout_matches_header():
    import ctypes
    text = open(HEADER).read()
    body = re.search(r"typedef struct pq_desc \{(.*?)\} pq_desc;", text, re.S).group(1)
    fields = re.findall(r"int32_t\s+(\w+);", body)
    assert [f for f, _ in pq.pq_desc._fields_] == fields
    assert ctypes.sizeof(pq.pq_desc) == 4 * len(fields)
    body = re.search(r"typedef struct pq_plan_info \{(.*?)\} pq_plan_info;", text, re.S).group(1)
    assert [f for f, _ in pq.pq_plan_info._fields_] == re.findall(r"int32_t\s+(\w+);", body)


def _al(v):
    return (v + 255) // 256 * 256


@pytest.mark.parametrize("N,K", [(4096, 4096), (27648, 5120), (100, 256)])
def test_w4_prepared_bytes(N, K):
    Np = (N + 15) // 16 * 16
    G = K // 128
    d = pq.make_desc(pq.PQ_FMT_W4_GPTQ, N, K)
    assert pq.pq_prepared_bytes(d) == _al(Np * K // 2) + _al(G * Np * 2)
    d = pq.make_desc(pq.PQ_FMT_W4_GPTQ, N, K, zp=pq.PQ_ZP_EXPLICIT_U8, has_gidx=1)
    assert pq.pq_prepared_bytes(d) == _al(Np * K // 2) + _al(G * Np * 2) + _al(G * Np) + _al(4 * K)


def test_w4_payload_matches_definition():
    # 4096 x 4096 symmetric: codes N*K/2 + scales N*K/128*2 bytes, nothing more
    d = pq.make_desc(pq.PQ_FMT_W4_GPTQ, 4096, 4096)
    assert pq.pq_prepared_bytes(d) == 8_650_752


@pytest.mark.parametrize("N,K", [(4096, 4096), (11008, 4096), (4096, 11008)])
def test_w2_payload_is_34_bytes_per_128(N, K):
    # code plane N*K/4 plus one fp16 scale per block; scale rows are padded to
    # whole 16-byte chunks (8 blocks), which adds nothing when K/128 % 8 == 0
    d = pq.make_desc(pq.PQ_FMT_W2_PQ2, N, K, act_group=K, max_m=1)
    B = K // 128
    Bp = (B + 7) // 8 * 8
    assert pq.pq_prepared_bytes(d) == _al(N * K // 4) + _al(N * Bp * 2)
    if B % 8 == 0:
        assert pq.pq_prepared_bytes(d) == N * K // 128 * 34


FIXED = 256 + 768                       # status word | GEMM shared-tile flags (same for every descriptor)


def test_workspace_sizes():
    # fixed region | gathered x | split-K partials (10 slices of 4 groups x
    # 5120 rows x 16 tokens, fp32)
    d = pq.make_desc(pq.PQ_FMT_W4_GPTQ, 5120, 5120, has_gidx=1, zp=pq.PQ_ZP_EXPLICIT_U8, max_m=16)
    assert pq.pq_workspace_bytes(d) == _al(FIXED) + _al(16 * 5120 * 2) + _al(10 * 5120 * 16 * 4)
    d = pq.make_desc(pq.PQ_FMT_W4_GPTQ, 5120, 5120, has_gidx=1, zp=pq.PQ_ZP_EXPLICIT_U8, max_m=1)
    assert pq.pq_workspace_bytes(d) == _al(FIXED) + _al(5120 * 2)
    # fixed region | split-K partials (4 slices of 8 blocks) | q | xs | sq | q as bf16
    d = pq.make_desc(pq.PQ_FMT_W2_PQ2, 4096, 4096, act_group=128, max_m=4)
    assert pq.pq_workspace_bytes(d) == (_al(FIXED) + _al(4 * 4096 * 16 * 4) + _al(4 * 4096) +
                                        _al(4 * 32 * 4) + _al(4 * 32 * 4) + _al(4 * 4096 * 2))
    # prefill: + two fp32 partial-tile slots for each of up to 160 CTAs
    # (rows: min(192, max_m rounded up to 16))
    d = pq.make_desc(pq.PQ_FMT_W4_GPTQ, 4096, 4096, max_m=2048)
    assert pq.pq_workspace_bytes(d) == _al(FIXED) + _al(8 * 4096 * 16 * 4) + 2 * 160 * 192 * 128 * 4
    d = pq.make_desc(pq.PQ_FMT_W4_GPTQ, 4096, 4096, max_m=100)
    assert pq.pq_workspace_bytes(d) == _al(FIXED) + _al(8 * 4096 * 16 * 4) + 2 * 160 * 112 * 128 * 4


@pytest.mark.parametrize("kw,code,msg", [
    (dict(fmt=7), pq.PQ_ERR_INVALID_ARG, "fmt 7"),
    (dict(K=200), pq.PQ_ERR_SHAPE, "multiple of 128"),
    (dict(N=0), pq.PQ_ERR_SHAPE, "N = 0"),
    (dict(group=64), pq.PQ_ERR_UNSUPPORTED, "only 128"),
    (dict(act_dtype=9), pq.PQ_ERR_INVALID_ARG, "act_dtype"),
    (dict(max_m=0), pq.PQ_ERR_SHAPE, "max_m"),
])
def test_descriptor_refusals(kw, code, msg):
    base = dict(fmt=pq.PQ_FMT_W4_GPTQ, N=64, K=256)
    base.update(kw)
    fmt, N, K = base.pop("fmt"), base.pop("N"), base.pop("K")
    d = pq.make_desc(fmt, N, K, **base)
    assert pq.pq_prepared_bytes(d) == 0
    assert msg in pq.pq_last_error()
    with pytest.raises(pq.PQError) as e:
        pq.pq_plan(d, 1, 152)
    assert e.value.status == code


@pytest.mark.parametrize("fmt,N,K,max_m,M,variant,m_tile,k_split", [
    # W4: up to 4 tokens whose rows fit in shared memory keep K split over
    # the CTA's warps; otherwise (up to 16 tokens) K is split across CTAs in
    # slices of 4 groups; beyond 16 the tensor-core GEMM
    (pq.PQ_FMT_W4_GPTQ, 4096, 4096, 16, 1, pq.PQ_VARIANT_W4_GEMV, 1, 8),
    (pq.PQ_FMT_W4_GPTQ, 4096, 4096, 16, 4, pq.PQ_VARIANT_W4_GEMV, 4, 8),
    (pq.PQ_FMT_W4_GPTQ, 11008, 4096, 16, 2, pq.PQ_VARIANT_W4_GEMV, 4, 8),
    (pq.PQ_FMT_W4_GPTQ, 4096, 11008, 16, 4, pq.PQ_VARIANT_W4_GEMV, 4, 8),
    (pq.PQ_FMT_W4_GPTQ, 4096, 11008, 16, 8, pq.PQ_VARIANT_W4_GEMV, 8, 22),
    (pq.PQ_FMT_W4_GPTQ, 11008, 4096, 16, 8, pq.PQ_VARIANT_W4_GEMV, 8, 8),
    (pq.PQ_FMT_W4_GPTQ, 27648, 5120, 16, 16, pq.PQ_VARIANT_W4_GEMV, 16, 10),
    (pq.PQ_FMT_W4_GPTQ, 64, 98304, 1, 1, pq.PQ_VARIANT_W4_GEMV, 8, 192),
    # GEMM: whole tiles (4-bit: 128 weight rows x 192 tokens; ternary: 256
    # tokens x 128 rows) for all but the last one to two waves, whose 128-row
    # groups are shared out evenly (a tile split over k_split CTAs at most)
    # where that evens the CTAs' work by more than the part sums cost
    (pq.PQ_FMT_W4_GPTQ, 14336, 4096, 2048, 2048, pq.PQ_VARIANT_W4_GEMM, 192, 2),
    (pq.PQ_FMT_W4_GPTQ, 4096, 4096, 2048, 2048, pq.PQ_VARIANT_W4_GEMM, 192, 2),
    (pq.PQ_FMT_W4_GPTQ, 4096, 4096, 2048, 256, pq.PQ_VARIANT_W4_GEMM, 192, 4),
    (pq.PQ_FMT_W4_GPTQ, 4096, 4096, 304, 304, pq.PQ_VARIANT_W4_GEMM, 192, 4),
    # W2: one token fused CUDA-core GEMV; two tokens quantise pre-pass +
    # CUDA-core GEMV; 3..16 the cluster split-K decode (k_split = CTAs per
    # cluster); rows too long for the cluster: the split-K decodes
    (pq.PQ_FMT_W2_PQ2, 4096, 4096, 1, 1, pq.PQ_VARIANT_W2_GEMV_FUSED, 1, 1),
    (pq.PQ_FMT_W2_PQ2, 4096, 4096, 16, 1, pq.PQ_VARIANT_W2_GEMV_FUSED, 1, 1),
    (pq.PQ_FMT_W2_PQ2, 4096, 4096, 16, 2, pq.PQ_VARIANT_W2_GEMV, 2, 1),
    (pq.PQ_FMT_W2_PQ2, 11008, 4096, 16, 4, pq.PQ_VARIANT_W2_GEMV_CL, 8, 8),
    (pq.PQ_FMT_W2_PQ2, 4096, 11008, 16, 16, pq.PQ_VARIANT_W2_GEMV_CL, 16, 8),
    (pq.PQ_FMT_W2_PQ2, 4096, 640, 16, 3, pq.PQ_VARIANT_W2_GEMV_CL, 8, 2),
    (pq.PQ_FMT_W2_PQ2, 64, 24704, 16, 4, pq.PQ_VARIANT_W2_GEMV_TC, 8, 25),
    (pq.PQ_FMT_W2_PQ2, 64, 24704, 16, 12, pq.PQ_VARIANT_W2_GEMV_BF, 16, 25),
    (pq.PQ_FMT_W2_PQ2, 11008, 4096, 2048, 2048, pq.PQ_VARIANT_W2_GEMM, 192, 2),
])
def test_dispatcher_choices(fmt, N, K, max_m, M, variant, m_tile, k_split):
    d = pq.make_desc(fmt, N, K, act_group=K, max_m=max_m)
    info = pq.pq_plan(d, M, 152)
    assert (info["variant"], info["m_tile"], info["k_split"]) == (variant, m_tile, k_split)
    assert info["grid"] >= 1 and info["block"] > 0 and info["smem_bytes"] > 0


def test_w2_cluster_decode_plan():
    # slices of a multiple of 4 blocks over at most 8 CTAs; strips per warp
    # chosen so that the clusters are resident at once; one launch
    for N, K, cl, grid in ((4096, 4096, 8, 256), (11008, 4096, 8, 232), (4096, 11008, 8, 256),
                           (22016, 4096, 8, 280), (200, 1280, 3, 6), (16, 128, 1, 1)):
        d = pq.make_desc(pq.PQ_FMT_W2_PQ2, N, K, act_group=K, max_m=16)
        info = pq.pq_plan(d, 16, 152)
        assert info["variant"] == pq.PQ_VARIANT_W2_GEMV_CL and info["launches"] == 1
        assert (info["k_split"], info["grid"]) == (cl, grid), (N, K, info)
        assert info["smem_bytes"] <= 227 * 1024


def test_w2_refusals():
    d = pq.make_desc(pq.PQ_FMT_W2_PQ2, 64, 256, act_group=64)
    assert pq.pq_prepared_bytes(d) == 0 and "act_group" in pq.pq_last_error()
    d = pq.make_desc(pq.PQ_FMT_W2_PQ2, 64, 256, zp=pq.PQ_ZP_EXPLICIT_U8)
    with pytest.raises(pq.PQError) as e:
        pq.pq_plan(d, 1, 152)
    assert e.value.status == pq.PQ_ERR_ZP_CONVENTION


# Fake, aligned, non-null device addresses: each refusal below is decided on
# the host before any CUDA call, so nothing is dereferenced.
FAKE = 1 << 20


def test_zero_point_convention_refused_both_ways():
    d = pq.make_desc(pq.PQ_FMT_W4_GPTQ, 64, 256, zp=pq.PQ_ZP_SYMMETRIC_8)
    with pytest.raises(pq.PQError) as e:
        pq.pq_prepare_w4(d, FAKE, FAKE, FAKE, None, FAKE, 1 << 20, FAKE, 1 << 20)
    assert e.value.status == pq.PQ_ERR_ZP_CONVENTION and "SYMMETRIC" in str(e.value)
    d = pq.make_desc(pq.PQ_FMT_W4_GPTQ, 64, 256, zp=pq.PQ_ZP_EXPLICIT_U8)
    with pytest.raises(pq.PQError) as e:
        pq.pq_prepare_w4(d, FAKE, FAKE, None, None, FAKE, 1 << 20, FAKE, 1 << 20)
    assert e.value.status == pq.PQ_ERR_ZP_CONVENTION and "EXPLICIT" in str(e.value)


def test_g_idx_refusals_name_the_invariant():
    K = 384
    d = pq.make_desc(pq.PQ_FMT_W4_GPTQ, 64, K, has_gidx=1)
    bad = np.repeat(np.array([0, 1, 2], dtype=np.int32), 128)
    bad[5] = 1                                   # group 0 has 127 rows, group 1 has 129
    with pytest.raises(pq.PQError) as e:
        pq.pq_prepare_w4(d, FAKE, FAKE, None, bad, FAKE, 1 << 20, FAKE, 1 << 20)
    assert e.value.status == pq.PQ_ERR_GIDX
    assert "group 0 has 127 rows" in str(e.value) and "contiguous run of 128" in str(e.value)
    bad = np.repeat(np.array([0, 1, 3], dtype=np.int32), 128)
    with pytest.raises(pq.PQError) as e:
        pq.pq_prepare_w4(d, FAKE, FAKE, None, bad, FAKE, 1 << 20, FAKE, 1 << 20)
    assert "outside [0, 3)" in str(e.value)
    with pytest.raises(pq.PQError) as e:
        pq.pq_prepare_w4(d, FAKE, FAKE, None, None, FAKE, 1 << 20, FAKE, 1 << 20)
    assert e.value.status == pq.PQ_ERR_GIDX


def test_alignment_and_buffer_refusals():
    d = pq.make_desc(pq.PQ_FMT_W4_GPTQ, 64, 256)
    with pytest.raises(pq.PQError) as e:
        pq.pq_prepare_w4(d, FAKE + 4, FAKE, None, None, FAKE, 1 << 20, FAKE, 1 << 20)
    assert e.value.status == pq.PQ_ERR_ALIGN
    with pytest.raises(pq.PQError) as e:
        pq.pq_prepare_w4(d, FAKE, FAKE, None, None, FAKE + 16, 1 << 20, FAKE, 1 << 20)
    assert e.value.status == pq.PQ_ERR_ALIGN
    with pytest.raises(pq.PQError) as e:
        pq.pq_prepare_w4(d, FAKE, FAKE, None, None, FAKE, 100, FAKE, 1 << 20)
    assert e.value.status == pq.PQ_ERR_BUFFER_TOO_SMALL
    with pytest.raises(pq.PQError) as e:
        pq.pq_prepare_w4(d, FAKE, FAKE, None, None, FAKE, 1 << 20, FAKE, 8)
    assert e.value.status == pq.PQ_ERR_BUFFER_TOO_SMALL


def test_linear_refusals_before_launch():
    with pytest.raises(pq.PQError) as e:
        pq.pq_linear(FAKE, None, FAKE, 1)
    assert e.value.status == pq.PQ_ERR_INVALID_ARG


def test_expire_wait_argument_refusal():
    with pytest.raises(pq.PQError):
        pq.pq_debug_expire_wait(None, 10)


def test_act_bytes_layout():
    # int8 plane-order codes (M <= 2: the CUDA-core decode) or bf16 codes
    # (M > 2: the cluster decode and the GEMM), fp32 scales and int32 block
    # sums, each section on a 256-byte boundary
    for K, AG, max_m in ((4096, 128, 2048), (11008, 11008, 64), (128, 128, 16)):
        d = pq.make_desc(pq.PQ_FMT_W2_PQ2, 256, K, act_group=AG, max_m=max_m)
        for M in (1, 2, 3, 8, 9, 16, 17, max_m):
            if M > max_m:
                continue
            codes = M * K if M <= 2 else 2 * M * K
            want = _al(codes) + _al(M * (K // AG) * 4) + _al(M * (K // 128) * 4)
            assert pq.pq_act_bytes(d, M) == want, (K, AG, M)


def test_act_bytes_refusals():
    d = pq.make_desc(pq.PQ_FMT_W4_GPTQ, 64, 256)
    assert pq.pq_act_bytes(d, 1) == 0
    assert "ternary" in pq.pq_last_error()
    d = pq.make_desc(pq.PQ_FMT_W2_PQ2, 64, 256, max_m=8)
    assert pq.pq_act_bytes(d, 9) == 0
    assert "max_m" in pq.pq_last_error()
    assert pq.pq_act_bytes(d, 0) == 0


def test_act_entry_points_refuse_without_a_handle():
    nrm = pq.pq_norm(FAKE, None, 1e-6, 0, 0)
    for call in (lambda: pq.pq_quantize_act(FAKE, None, FAKE, 1 << 20, 1),
                 lambda: pq.pq_norm_quantize(FAKE, None, nrm, None, None, None, FAKE, 1 << 20, 1),
                 lambda: pq.pq_linear_act(FAKE, 1 << 20, None, FAKE, 1),
                 lambda: pq.pq_debug_act_unpack(FAKE, 1 << 20, None, 1, FAKE, FAKE, FAKE)):
        with pytest.raises(pq.PQError) as e:
            call()
        assert e.value.status == pq.PQ_ERR_INVALID_ARG


def test_norm_struct_layout_matches_header():
    import ctypes
    text = open(HEADER).read()
    body = re.search(r"typedef struct pq_norm \{(.*?)\} pq_norm;", text, re.S).group(1)
    fields = re.findall(r"\b(\w+);", re.sub(r"/\*.*?\*/", "", body, flags=re.S))
    assert [f for f, _ in pq.pq_norm._fields_] == fields
    assert ctypes.sizeof(pq.pq_norm) == 8 + 8 + 4 + 4 + 4 + 4


@pytest.mark.parametrize("N,K,M,launches,smem", [
    # permuted in shared memory: weight ring (8 warps x 2 items of 4 groups of
    # codes, scales, zero points) + the operand row + the caller-order row
    (5120, 5120, 1, 1, 8 * 2 * (4 * 1024 + 4 * 32 + 4 * 16) + 2 * 5120 * 2),
    (27648, 5120, 1, 1, None),
    (5120, 5120, 4, 2, None),        # a second copy would cost residency: gather launch first
    (56, 16384, 1, 2, None),
    (40, 9216, 3, 1, None),          # one CTA per SM either way: permuted in shared memory
    (5120, 5120, 16, 3, None),       # split-K: gather, GEMV, slice sum
])
def test_act_order_decode_plan(N, K, M, launches, smem):
    d = pq.make_desc(pq.PQ_FMT_W4_GPTQ, N, K, zp=pq.PQ_ZP_EXPLICIT_U8, has_gidx=1, max_m=16)
    plan = pq.pq_plan(d, M, 152)
    assert plan["variant"] == pq.PQ_VARIANT_W4_GEMV
    assert plan["launches"] == launches
    d0 = pq.make_desc(pq.PQ_FMT_W4_GPTQ, N, K, zp=pq.PQ_ZP_EXPLICIT_U8, max_m=16)
    plain = pq.pq_plan(d0, M, 152)
    if M <= 4:
        # the self-permuting kernel holds the caller-order rows as well
        extra = plan["smem_bytes"] - plain["smem_bytes"]
        assert extra == (plain["m_tile"] * K * 2 if launches == 1 else 0)
    if smem is not None:
        assert plan["smem_bytes"] == smem


def test_affine4_planes_and_plan():
    # codes [Npad][K/2] + scales and biases [K/64][Npad] 16-bit
    SK_A = 8 * 2 * (4096 + 256 + 256) + 16 * (4 * 256 + 16) + 16 * 8 * 4   # affine split-K shared memory
    for N, K in ((4096, 4096), (100, 640)):
        Np = (N + 15) // 16 * 16
        slices = -(-K // 512)
        for max_m in (1, 4, 64):
            d = pq.make_desc(pq.PQ_FMT_W4_AFFINE, N, K, group=64, max_m=max_m)
            assert pq.pq_prepared_bytes(d) == _al(Np * K // 2) + 2 * _al(K // 64 * Np * 2)
            # status word and flags; split-K partials for M > 1; GEMM partial
            # tiles and the sums of x over every 64-group for max_m > 16
            ws = _al(FIXED)
            if max_m > 1:
                ws += _al(slices * Np * 16 * 4)
            if max_m > 16:
                ws += _al(2 * 160 * 64 * 128 * 4) + _al(max_m * (K // 64) * 4)
            assert pq.pq_workspace_bytes(d) == ws, (N, K, max_m)
        for M, mt in ((1, 1), (2, 4), (4, 4)):
            plan = pq.pq_plan(d, M, 152)
            assert plan["variant"] == pq.PQ_VARIANT_W4_GEMV and plan["launches"] == 1 and plan["m_tile"] == mt
        for M, mt in ((5, 8), (8, 8), (9, 16), (16, 16)):
            # one 8-token tile: the K slices of a strip block (8 or fewer) run
            # as a thread-block cluster and add their sums there (8 KB of
            # them), one launch; two tiles: a second launch adds them
            plan = pq.pq_plan(d, M, 152)
            clu = M <= 8
            assert plan["variant"] == pq.PQ_VARIANT_W4_GEMV and plan["launches"] == (1 if clu else 2)
            assert plan["m_tile"] == mt and plan["k_split"] == slices
            assert plan["smem_bytes"] == SK_A + (8 * 1024 if clu else 0)
        plan = pq.pq_plan(d, 64, 152)
        assert plan["variant"] == pq.PQ_VARIANT_W4_GEMM and plan["launches"] in (2, 3) and plan["m_tile"] == 192
    # one token past the whole-row bound (76416) takes split-K
    d = pq.make_desc(pq.PQ_FMT_W4_AFFINE, 64, 76416, group=64, max_m=1)
    assert pq.pq_plan(d, 1, 152)["launches"] == 1 and pq.pq_workspace_bytes(d) == _al(FIXED)
    d = pq.make_desc(pq.PQ_FMT_W4_AFFINE, 64, 76544, group=64, max_m=1)
    plan = pq.pq_plan(d, 1, 152)
    assert plan["launches"] == 2 and plan["smem_bytes"] == SK_A           # 150 slices: a second launch adds them


def test_affine4_refusals():
    d = pq.make_desc(pq.PQ_FMT_W4_AFFINE, 64, 256, group=64, max_m=8)
    with pytest.raises(pq.PQError) as e:
        pq.pq_plan(d, 9, 152)
    assert e.value.status == pq.PQ_ERR_SHAPE
    for kw, code in ((dict(group=128), pq.PQ_ERR_UNSUPPORTED), (dict(group=64, has_gidx=1), pq.PQ_ERR_UNSUPPORTED),
                     (dict(group=64, zp=pq.PQ_ZP_EXPLICIT_U8), pq.PQ_ERR_ZP_CONVENTION)):
        bad = pq.make_desc(pq.PQ_FMT_W4_AFFINE, 64, 256, max_m=1, **kw)
        assert pq.pq_prepared_bytes(bad) == 0
        with pytest.raises(pq.PQError) as e:
            pq.pq_prepare_affine4(bad, FAKE, FAKE, FAKE, FAKE, 1 << 20, FAKE, 1 << 20)
        assert e.value.status == code, kw
    # the 4-bit GPTQ frame keeps its group of 128
    with pytest.raises(pq.PQError) as e:
        pq.pq_prepare_w4(pq.make_desc(pq.PQ_FMT_W4_GPTQ, 64, 256, group=64), FAKE, FAKE, None, None, FAKE,
                         1 << 20, FAKE, 1 << 20)
    assert e.value.status == pq.PQ_ERR_UNSUPPORTED


def test_probe_refusals_before_launch():
    for args, code in (((FAKE + 8, 64, FAKE, 0, 0), pq.PQ_ERR_ALIGN), ((FAKE, 60, FAKE, 0, 0), pq.PQ_ERR_ALIGN),
                       ((FAKE, 0, FAKE, 0, 0), pq.PQ_ERR_SHAPE), ((FAKE, 64, FAKE, 9, 0), pq.PQ_ERR_INVALID_ARG),
                       ((FAKE, 64, FAKE, 0, 2), pq.PQ_ERR_INVALID_ARG), ((None, 64, FAKE, 0, 0), pq.PQ_ERR_INVALID_ARG)):
        with pytest.raises(pq.PQError) as e:
            pq.pq_probe_read(*args)
        assert e.value.status == code, args
