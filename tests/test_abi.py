"""The C-ABI library loads, exports every symbol include/lora_gemm.h declares,
and its host-only entry points behave as documented (no GPU needed)."""
import os
import re
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lora_gemm.h")


@pytest.fixture(scope="module")
def L():
    from rank_adapter_gemm_gb300 import build
    build.build()
    import rank_adapter_gemm_gb300 as lib
    return lib


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lora_[a-z0-9_]+)\s*\(", text)))


def test_header_declarations_are_exported(L):
    from rank_adapter_gemm_gb300 import _lib
    declared = _declared()
    assert set(declared) == set(_lib.EXPORTED)
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.library_path()], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (lora_[a-z0-9_]+)$", out, flags=re.M))
    for name in declared:
        assert name in exported, name
    lib = _lib.load()
    for name in declared:
        assert hasattr(lib, name)


def test_abi_version_and_status_strings(L):
    assert L.lora_abi_version() == L.LORA_ABI_VERSION
    from rank_adapter_gemm_gb300 import _lib
    for code, name in _lib.STATUS.items():
        assert L.lora_status_string(code).startswith(name)
    assert L.lora_status_string(999) == "LORA_ERR_UNKNOWN"


def test_scale_rule_matches_oracle(L):
    for alpha, r, rs, a_s in [(16, 64, False, 1.0), (32, 16, True, 1.0), (0, 16, False, 0.5), (32, 16, False, 0.7),
                              (8, 8, True, 2.0), (16, 0, False, 1.0)]:
        assert L.lora_scale(alpha, r, rs, a_s) == oracle.scale(alpha, r, rs, a_s)


def test_pack_slot_table_layout_and_checks(L):
    S, n, r_max = 3, 2, 32
    buf = np.zeros(L.lora_slot_table_bytes(S, n), np.uint8)
    ranks = np.array([16, 0, 32], np.int32)
    scales = np.array([2.0, 1.0, 0.5], np.float32)
    A = np.array([0x1000, 0x1010, 0, 0, 0x2000, 0x2010], np.uint64)
    B = np.array([0x3000, 0x3010, 0, 0, 0x4000, 0x4010], np.uint64)
    L.lora_pack_slot_table(buf, S, n, r_max, ranks, scales, A, B)
    w = buf.view(np.int32)
    assert list(w[:4]) == [0x41526F4C, S, n, r_max]
    assert list(w[4:7]) == [16, 0, 32]
    assert list(buf[32:44].view(np.float32)) == [2.0, 1.0, 0.5]
    ptrs = buf[48:].view(np.uint64)
    assert list(ptrs[:6]) == list(A) and list(ptrs[6:12]) == list(B)
    bad = [
        (dict(ranks=np.array([12, 0, 32], np.int32)), 3),          # not a multiple of 8
        (dict(ranks=np.array([16, 0, 40], np.int32)), 3),          # above r_max
        (dict(A=np.array([0, 0x1010, 0, 0, 0x2000, 0x2010], np.uint64)), 5),   # null on a used slot
        (dict(B=np.array([0x3008, 0x3010, 0, 0, 0x4000, 0x4010], np.uint64)), 2),  # misaligned
    ]
    for kw, status in bad:
        args = dict(ranks=ranks, scales=scales, A=A, B=B)
        args.update(kw)
        with pytest.raises(L.LoraError) as e:
            L.lora_pack_slot_table(buf, S, n, r_max, args["ranks"], args["scales"], args["A"], args["B"])
        assert e.value.status == status


def test_workspace_bytes(L):
    sh = L.make_shape(32, 64, 4096, [4096, 1024, 1024])
    nbytes = L.lora_workspace_bytes(256, sh)
    xa = 3 * 256 * 64 * 4
    hl = 3 * 256 * 64 * 2  # prefill xa as bf16 hi and lo, rank padded to 64
    # control block, the shrink output xa, the fused kernel's accumulator (same
    # size as xa), the prefill path's hi/lo parts and the two accumulators the
    # tensor-core decode kernels use in turn
    # then the one-kernel TMA path's two sum sets, its control block (2 S
    # counters, the call and exit counters) and room for a plan (128-byte
    # header, 64 bytes per slot, 32 per CTA for up to 512 CTAs, T token ids)
    plan = (128 + 64 * 32 + 512 * 32 + 4 * 256 + 255) // 256 * 256
    tma = 2 * xa + (4 * (2 * 32 + 2) + 255) // 256 * 256 + plan
    assert nbytes >= 4 * xa + 2 * hl + tma
    assert nbytes - 4 * xa - 2 * hl - tma < 4 * (2 * 32 * 4 + 64) + 6 * 256
    # ranks above 64 have no bf16 hi/lo regions; up to 128 they keep the two
    # accumulators of the two-kernel decode paths
    big = L.lora_workspace_bytes(256, L.make_shape(32, 128, 4096, [4096]))
    assert 4 * 256 * 128 * 4 <= big < 4 * 256 * 128 * 4 + 4 * (2 * 32 * 4 + 64) + 6 * 256
    huge = L.lora_workspace_bytes(256, L.make_shape(32, 256, 4096, [4096]))
    assert 2 * 256 * 256 * 4 <= huge < 2 * 256 * 256 * 4 + 4 * (2 * 32 * 4 + 64) + 6 * 256
    with pytest.raises(L.LoraError) as e:
        L.lora_workspace_bytes(10, L.make_shape(0, 64, 4096, [4096]))
    assert e.value.status == 1
    with pytest.raises(L.LoraError) as e:
        L.lora_workspace_bytes(10, L.make_shape(4, 64, 4095, [4096]))
    assert e.value.status == 2


def test_moe_slot_pointers_follow_the_expert_offset(L):
    """Virtual slot a E + e gets adapter a's rank and scale, and A and B bases moved
    by e * dim * rank elements (TensorRT-LLM's per-expert layout), two bytes each."""
    n_ad, E, k, widths = 3, 4, 4096, [4096, 1024]
    sh = L.make_shape(n_ad * E, 64, k, widths)
    ranks = [16, 64, 0]
    a_base = [1 << 20, 2 << 20, 3 << 20, 4 << 20, 0, 0]
    b_base = [5 << 20, 6 << 20, 7 << 20, 8 << 20, 0, 0]
    vr, vs, ap, bp = L.lora_moe_slot_pointers(n_ad, E, sh, ranks, [0.5, 2.0, 1.0], a_base, b_base)
    for a in range(n_ad):
        for e in range(E):
            v = a * E + e
            assert vr[v] == ranks[a] and vs[v] == [0.5, 2.0, 1.0][a]
            for i, w in enumerate(widths):
                want_a = a_base[a * 2 + i] + e * ranks[a] * k * 2 if a_base[a * 2 + i] else 0
                want_b = b_base[a * 2 + i] + e * w * ranks[a] * 2 if b_base[a * 2 + i] else 0
                assert ap[v * 2 + i] == want_a and bp[v * 2 + i] == want_b
    with pytest.raises(L.LoraError):
        L.lora_moe_slot_pointers(n_ad, E + 1, sh, ranks, [1.0] * 3, a_base, b_base)


def test_rank_limit_is_512(L):
    """Ranks up to 512 (multiples of 8) are accepted by every host check; above it,
    LORA_ERR_RANK."""
    assert L.LORA_MAX_RANK == 512
    L.lora_workspace_bytes(64, L.make_shape(4, 512, 1024, [1024]))
    with pytest.raises(L.LoraError) as e:
        L.lora_workspace_bytes(64, L.make_shape(4, 520, 1024, [1024]))
    assert e.value.status == 3


def test_host_checks_of_the_plan_moe_and_activated_entry_points(L):
    """Argument errors are returned before anything is enqueued (no device is
    touched): null pointers, counts, unsupported paths, short buffers."""
    import ctypes
    from rank_adapter_gemm_gb300 import _lib
    lib = _lib.load()
    sh = L.make_shape(32, 64, 4096, [4096, 1024, 1024])
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: every call below fails its host checks first
    paths = _lib.PATHS
    # plan size: 0 for T < 1, two table images otherwise, growing with T
    assert lib.lora_plan_bytes(0, ctypes.byref(sh)) == 0
    b256, b512 = lib.lora_plan_bytes(256, ctypes.byref(sh)), lib.lora_plan_bytes(512, ctypes.byref(sh))
    assert 0 < b256 < b512 and b256 % 32 == 0
    # build: T < 1, unsupported path, short or null plan, misaligned plan
    assert lib.lora_build_plan(0, ctypes.byref(sh), fake, fake, fake, fake, paths["decode_direct"], fake, b256,
                               None, None) == 1
    assert lib.lora_build_plan(256, ctypes.byref(sh), fake, fake, fake, fake, paths["decode_split"], fake, b256,
                               None, None) == 9
    assert lib.lora_build_plan(256, ctypes.byref(sh), fake, fake, fake, fake, paths["decode_direct"], fake, 64,
                               None, None) == 6
    assert lib.lora_build_plan(256, ctypes.byref(sh), fake, fake, fake, fake, paths["decode_direct"], None, b256,
                               None, None) == 6
    assert lib.lora_build_plan(256, ctypes.byref(sh), fake, fake, fake, fake, paths["decode_direct"],
                               P((1 << 20) + 8), b256, None, None) == 2
    # FP8 plans need k % 16 == 0
    sh8 = L.make_shape(32, 64, 4104, [4096])
    assert lib.lora_build_plan(256, ctypes.byref(sh8), fake, fake, fake, fake, paths["decode_direct_fp8"], fake,
                               lib.lora_plan_bytes(256, ctypes.byref(sh8)), None, None) == 9
    # batched build: negative count, null arrays
    assert lib.lora_build_plans(256, ctypes.byref(sh), -1, None, None, b256, fake, fake, fake,
                                paths["decode_direct"], None, None) == 1
    assert lib.lora_build_plans(256, ctypes.byref(sh), 2, None, None, b256, fake, fake, fake,
                                paths["decode_direct"], None, None) == 1
    # MoE index: S not a multiple of E, T * K overflow
    assert lib.lora_build_index_moe(fake, fake, 10, 2, 3, 8, fake, fake, fake, fake, None, None) == 1
    assert lib.lora_build_index_moe(fake, fake, 1 << 30, 4, 2, 8, fake, fake, fake, fake, None, None) == 1
    # aLoRA index: negative counts, missing sequence arrays
    assert lib.lora_build_index_activated(fake, fake, -1, fake, fake, 2, 8, fake, fake, fake, fake, None, None) == 1
    assert lib.lora_build_index_activated(fake, fake, 4, None, None, 2, 8, fake, fake, fake, fake, None, None) == 1
    # MoE apply: K < 1; premultiply_e4m3: negative count
    assert lib.lora_apply_moe(fake, 4096, 1, fake, 6144, 4, 0, ctypes.byref(sh), fake, fake, fake, fake, fake, 0,
                              None, None) == 1
    assert lib.lora_premultiply_e4m3(fake, -1, ctypes.c_float(1.0), None) == 1


def test_host_checks_of_the_tma_entry_points(L):
    """The tensor-map table and the one-kernel TMA path: sizes and the argument
    errors returned before any device or driver call."""
    import ctypes
    from rank_adapter_gemm_gb300 import _lib
    lib = _lib.load()
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: every call below fails its host checks first
    sh = L.make_shape(32, 64, 4096, [4096, 1024, 1024])
    # the ordinary table, aligned to 128 bytes, a 128-byte block header, the
    # slot flags padded to 128 bytes, eight 128-byte tensor maps per slot
    base = (L.lora_slot_table_bytes(32, 3) + 127) // 128 * 128
    assert L.lora_slot_table_tma_bytes(32, sh) == base + 128 + 128 + 32 * 8 * 128
    assert L.lora_slot_table_tma_bytes(33, L.make_shape(33, 64, 4096, [4096, 1024, 1024])) == \
        (L.lora_slot_table_bytes(33, 3) + 127) // 128 * 128 + 128 + 256 + 33 * 8 * 128
    assert L.lora_slot_table_tma_bytes(31, sh) == 0  # S must match the shape
    assert L.lora_slot_table_tma_bytes(32, L.make_shape(32, 64, 4095, [4096])) == 0
    staging = np.zeros(L.lora_slot_table_tma_bytes(32, sh), np.uint8)
    ranks = np.full(32, 16, np.int32)
    scales = np.ones(32, np.float32)
    ptrs = np.full(96, 1 << 20, np.uint64)

    def setm(dev, rk=ranks, pa=ptrs):
        return lib.lora_set_slot_table_tma(dev, P(staging.ctypes.data), ctypes.byref(sh), P(rk.ctypes.data),
                                           P(scales.ctypes.data), P(pa.ctypes.data), P(pa.ctypes.data), None)

    assert lib.lora_set_slot_table_tma(None, P(staging.ctypes.data), ctypes.byref(sh), None, None, None, None,
                                       None) == 1
    assert setm(P((1 << 20) + 16)) == 2                      # table not 128-byte aligned
    assert setm(fake, rk=np.full(32, 12, np.int32)) == 3     # rank not a multiple of 8
    assert setm(fake, pa=np.zeros(96, np.uint64)) == 5       # null weight of a rank>0 slot
    # the path: unsupported shapes (rank above 64, n * r_max above 192, k % 64)
    b = lib.lora_plan_bytes(256, ctypes.byref(sh))
    assert b >= 128 + 64 * 32 + 512 * 32 + 4 * 256
    for bad in (L.make_shape(32, 128, 4096, [4096]), L.make_shape(32, 64, 4096, [1024] * 4),
                L.make_shape(32, 64, 4032 + 8, [4096])):
        nb = lib.lora_plan_bytes(256, ctypes.byref(bad))
        assert lib.lora_build_plan(256, ctypes.byref(bad), fake, fake, fake, fake, _lib.PATHS["decode_tma"], fake,
                                   nb, None, None) == 9
    assert lib.lora_build_plan(256, ctypes.byref(sh), fake, fake, fake, fake, _lib.PATHS["decode_tma"], fake,
                               128, None, None) == 6
    assert lib.lora_build_plan(256, ctypes.byref(sh), fake, fake, fake, fake, _lib.PATHS["decode_tma"],
                               P((1 << 20) + 8), b, None, None) == 2
    assert lib.lora_apply_plan(fake, 4096, fake, 6144, 256, ctypes.byref(sh), fake, 128, _lib.PATHS["decode_tma"],
                               fake, 1 << 30, None, None) == 6


def test_host_checks_of_the_cluster_path(L):
    """The one-cluster-per-slot decode path: AUTO's choice at 64 tokens and fewer,
    one launch per call, and the shapes it refuses before any device call (k or
    a slice offset not a multiple of 8, r_max above 256, tiles beyond a CTA's
    shared memory)."""
    import ctypes
    from rank_adapter_gemm_gb300 import _lib
    lib = _lib.load()
    assert L.lora_resolve_path("auto", 1) == ("decode_cluster", 1)
    assert L.lora_resolve_path("auto", 64) == ("decode_cluster", 1)
    assert L.lora_resolve_path("auto", 65)[0] == "decode_direct"
    assert L.lora_resolve_path("decode_cluster", 4096) == ("decode_cluster", 1)
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: every call below fails its host checks first
    cluster = _lib.PATHS["decode_cluster"]
    # k or a slice width not a multiple of 8: every path's shape check (alignment)
    for bad in (L.make_shape(8, 16, 4100, [4096]), L.make_shape(8, 16, 4096, [1028, 1020])):
        d = int(bad.slice_offsets[bad.n_slices])
        assert lib.lora_apply_ex(fake, 4104, fake, 4096, 64, ctypes.byref(bad), fake, fake, fake, fake, 0, cluster,
                                 fake, 1 << 30, None, None) == 2
    for bad in (L.make_shape(8, 264, 4096, [4096]),          # r_max above 256
                L.make_shape(8, 64, 4096, [14336, 14336])):  # B and y tiles beyond 227 KB
        d = int(bad.slice_offsets[bad.n_slices])
        ws = L.lora_workspace_bytes(64, bad)
        assert lib.lora_apply_ex(fake, bad.k, fake, d, 64, ctypes.byref(bad), fake, fake, fake, fake, 0, cluster,
                                 fake, ws, None, None) == 9
    # plans (also the routed-expert plan entry point) do not take it
    sh = L.make_shape(8, 16, 4096, [4096])
    assert lib.lora_build_plan(64, ctypes.byref(sh), fake, fake, fake, fake, cluster, fake,
                               lib.lora_plan_bytes(64, ctypes.byref(sh)), None, None) == 9
    assert lib.lora_apply_moe_plan_ex(fake, 4096, 1, fake, 4096, 32, 2, ctypes.byref(sh), fake, 1 << 20, cluster,
                                      fake, L.lora_workspace_bytes(64, sh), None, None) == 9
