"""lora_apply_noalloc: the branch for callers that cannot allocate device memory.

Such callers (for example a plug-in inside an engine that owns all device memory
and offers no allocator, or code that must not call cudaMalloc because it
synchronises the device) cannot supply the workspace lora_apply needs.  The
no-allocation entry point keeps that scratch in a fixed array inside the
library.  These tests check it against lora_apply on the same inputs, on two
calls in a row, through the C ABI.  The file is named so that pytest collects it
last.
"""
import numpy as np
import pytest

import workloads as W
from _parity import ATOL, RTOL

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


def _close(a_bits, b_bits):
    a = W.bf16_bits_to_f32(a_bits).astype(np.float64)
    b = W.bf16_bits_to_f32(b_bits).astype(np.float64)
    return bool(np.all(np.abs(a - b) <= ATOL + RTOL * np.abs(b)))


def test_noalloc_matches_lora_apply_on_two_calls_in_a_row():
    import torch
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import to_host_bits
    for cfg in (2, 1):  # packed QKV (T=256, S=32, r up to 64), then q_proj (T=64, S=8, r=16)
        wl, rp, idx = _setup(cfg)
        y0 = rp.y.clone()
        ws = L.Workspace(wl.T, rp.shape)
        L.lora_apply(rp.x, rp.y, rp.shape, rp.table.dev, idx.sorted_ids, idx.seg_offsets, idx.active, ws.buf,
                     idx.err, path="decode_split")
        torch.cuda.synchronize()
        want = to_host_bits(rp.y)
        for call in range(2):
            rp.y.copy_(y0)
            L.lora_apply_noalloc(rp.x, rp.y, rp.shape, rp.table.dev, idx.sorted_ids, idx.seg_offsets,
                                 idx.active, idx.err)
            torch.cuda.synchronize()
            got = to_host_bits(rp.y)
            assert int(idx.err.item()) == 0
            assert _close(got, want), f"config {cfg}, call {call + 1}"


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
