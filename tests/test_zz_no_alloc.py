"""lora_apply_noalloc: the branch for callers that cannot allocate device memory.

Such callers (for example a plug-in inside an engine that owns all device memory
and offers no allocator, or code that must not call cudaMalloc because it
synchronises the device) cannot supply the workspace lora_apply needs.  The
no-allocation entry point keeps that scratch in a fixed array inside the
library.  It runs the same shrink and expand kernels as the decode_split path,
so its output must equal that path's bit for bit, and both must match the
oracle.  These tests check that on two calls in a row through the C ABI, and at
the largest size the fixed scratch holds.  The file is named so that pytest
collects it last.
"""
import numpy as np
import pytest

import workloads as W
from _parity import assert_y_close, oracle_y

pytestmark = pytest.mark.gpu


def _setup(cfg):
    import torch
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import ResidentProjection
    wl = W.config(cfg)
    rp = ResidentProjection.from_workload(wl)
    idx = L.TokenIndex(wl.T, wl.S)
    idx.build(torch.from_numpy(wl.slot_ids).cuda(), rp.table)
    return wl, rp, idx


def _run(wl, rp, idx, calls=2):
    """decode_split once, then lora_apply_noalloc `calls` times from the same y."""
    import torch
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import to_host_bits
    y0 = rp.y.clone()
    ws = L.Workspace(wl.T, rp.shape)
    L.lora_apply(rp.x, rp.y, rp.shape, rp.table.dev, idx.sorted_ids, idx.seg_offsets, idx.active, ws.buf,
                 idx.err, path="decode_split")
    torch.cuda.synchronize()
    split = to_host_bits(rp.y)
    outs = []
    for _ in range(calls):
        rp.y.copy_(y0)
        L.lora_apply_noalloc(rp.x, rp.y, rp.shape, rp.table.dev, idx.sorted_ids, idx.seg_offsets, idx.active,
                             idx.err)
        torch.cuda.synchronize()
        assert int(idx.err.item()) == 0
        outs.append(to_host_bits(rp.y))
    return split, outs


def test_noalloc_matches_split_bit_for_bit_and_the_oracle():
    for cfg in (2, 1):  # packed QKV (T=256, S=32, r up to 64), then q_proj (T=64, S=8, r=16)
        wl, rp, idx = _setup(cfg)
        split, outs = _run(wl, rp, idx)
        ref, _ = oracle_y(wl)
        for call, got in enumerate(outs):
            assert np.array_equal(got, split), f"config {cfg}, call {call + 1}: differs from decode_split"
            assert_y_close(got, ref, f"noalloc config {cfg}, call {call + 1}")


def test_noalloc_accepts_the_largest_size_its_scratch_holds():
    """n_slices * T * r_max * 4 bytes equal to the scratch: accepted, and correct."""
    import torch
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import ResidentProjection
    from test_gpu_parity import _small
    n, r_max, k = 4, 256, 64
    T = L.LORA_NOALLOC_WS_BYTES // (4 * n * r_max)  # exactly fits
    assert n * T * r_max * 4 == L.LORA_NOALLOC_WS_BYTES
    wl = _small(61, T, k, [8, 16, 8, 32], 4, [256, 8, 0, 64])
    assert wl.r_max == r_max
    rp = ResidentProjection.from_workload(wl)
    idx = L.TokenIndex(wl.T, wl.S)
    idx.build(torch.from_numpy(wl.slot_ids).cuda(), rp.table)
    split, outs = _run(wl, rp, idx, calls=1)
    assert np.array_equal(outs[0], split)
    ref, _ = oracle_y(wl)
    assert_y_close(outs[0], ref, "noalloc at the scratch's limit")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import torch
    import rank_adapter_gemm_gb300 as L
    S, r_max, k = 4, 256, 64
    T = L.LORA_NOALLOC_WS_BYTES // (4 * 4 * r_max) + 1   # 4 slices: one token too many
    shape = L.make_shape(S, r_max, k, [8, 8, 8, 8])
    tab = L.SlotTable(S, 4, r_max)
    x = torch.zeros(T, k, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(T, 32, dtype=torch.bfloat16, device="cuda")
    idx = L.TokenIndex(T, S)
    with pytest.raises(L.LoraError) as e:
        L.lora_apply_noalloc(x, y, shape, tab.dev, idx.sorted_ids, idx.seg_offsets, idx.active, idx.err)
    assert e.value.status == 6  # LORA_ERR_WORKSPACE
