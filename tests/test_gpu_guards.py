"""Strided rows and guard bands: x and y as column windows of wider buffers
(ldx > k, ldy > d, the layout of a projection's output inside a fused
buffer), and canary regions around y, the workspace, the plan and the index
outputs.  After every call the window must match the oracle and every canary
byte must be unchanged: a write past a row, a slice or a buffer shows up as a
changed canary, with no device fault (plain host comparisons after a normal
run)."""
import numpy as np
import pytest

import oracle
import workloads as W
from _parity import assert_y_close, oracle_y, oracle_y_e4m3

pytestmark = pytest.mark.gpu

CANARY16 = 0x7F81           # a bf16 NaN payload no kernel writes
CANARY32 = np.int32(-777)   # index words
CANARYF = 0x7FC0DEAD        # workspace words (a float NaN payload)
XOFF, YOFF, PAD = 8, 16, 64  # window column offsets (16-byte aligned) and padding


def _torch():
    import torch
    return torch


def _window(t, rows_before, col_off, pad, fill):
    """t copied into a window of a larger buffer filled with `fill` (bit
    pattern); returns (big buffer, view)."""
    torch = _torch()
    T, w = t.shape
    big = torch.full((T + 2 * rows_before, w + pad), int(np.uint16(fill).view(np.int16)), dtype=torch.int16,
                     device=t.device)
    big = big.view(t.dtype)
    view = big[rows_before:rows_before + T, col_off:col_off + w]
    view.copy_(t)
    return big, view


def _guarded(n, dtype, fill, front=16, back=64):
    """A 1-D buffer of n elements with canary regions in front and behind."""
    torch = _torch()
    big = torch.empty(front + n + back, dtype=dtype, device="cuda")
    if dtype == torch.float32:
        big.view(torch.int32).fill_(int(np.int32(np.uint32(fill).view(np.int32))))
    else:
        big.fill_(int(fill))
    return big, big[front:front + n]


def _canaries_intact(big, view, what):
    """Everything of `big` outside `view` still holds its canary bits."""
    torch = _torch()
    mask = torch.ones(big.shape, dtype=torch.bool, device=big.device)
    if big.dim() == 2:
        r0 = (view.data_ptr() - big.data_ptr()) // big.element_size() // big.stride(0)
        c0 = ((view.data_ptr() - big.data_ptr()) // big.element_size()) % big.stride(0)
        mask[r0:r0 + view.shape[0], c0:c0 + view.shape[1]] = False
    else:
        o = (view.data_ptr() - big.data_ptr()) // big.element_size()
        mask[o:o + view.shape[0]] = False
    bits = big.view({1: torch.uint8, 2: torch.int16, 4: torch.int32}[big.element_size()])
    vals = bits[mask].cpu().numpy()
    first = vals[:1]
    assert vals.size == 0 or (vals == first).all(), f"{what}: canary changed"


class Guarded:
    """One projection's inputs and buffers placed in guarded, strided storage."""

    def __init__(self, wl, mod_idx=0):
        torch = _torch()
        import rank_adapter_gemm_gb300 as L
        from rank_adapter_gemm_gb300.resident import ResidentProjection
        self.wl, self.L = wl, L
        self.rp = ResidentProjection.from_workload(wl, mod_idx)
        T = wl.T
        self.xbig, self.x = _window(self.rp.x, 0, XOFF, PAD, CANARY16)
        self.ybig, self.y = _window(self.rp.y, 2, YOFF, PAD, CANARY16)
        self.y0 = self.y.clone()
        S = wl.S
        self.sbig, self.sorted_ids = _guarded(max(T, 1), torch.int32, CANARY32)
        self.gbig, self.seg = _guarded(S + 2, torch.int32, CANARY32)
        self.abig, self.active = _guarded(S + 1, torch.int32, CANARY32)
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        nws = (L.lora_workspace_bytes(T, self.rp.shape) + 3) // 4
        self.wbig, self.ws = _guarded(nws, torch.float32, CANARYF, front=64)
        self.ws.zero_()
        slots = torch.from_numpy(np.ascontiguousarray(wl.slot_ids, dtype=np.int32)).cuda()
        L.lora_build_index(slots, S, self.rp.table.dev, self.sorted_ids, self.seg, self.active, self.err)

    def check(self, what):
        torch = _torch()
        torch.cuda.synchronize()
        assert int(self.err.item()) == 0, what
        _canaries_intact(self.ybig, self.y, what + ": y")
        _canaries_intact(self.xbig, self.x, what + ": x")
        _canaries_intact(self.wbig, self.ws, what + ": workspace")
        _canaries_intact(self.sbig, self.sorted_ids, what + ": sorted_ids")
        _canaries_intact(self.gbig, self.seg, what + ": seg_offsets")
        _canaries_intact(self.abig, self.active, what + ": active")

    def y_bits(self):
        from rank_adapter_gemm_gb300.resident import to_host_bits
        return to_host_bits(self.y.contiguous())


@pytest.mark.parametrize("path", ["decode_split", "decode_fused", "decode_direct", "decode_tma", "decode_cluster",
                                  "prefill", "auto"])
def test_strided_rows_and_guard_bands(path):
    """The packed QKV decode config through every path, x and y column windows."""
    wl = W.config(2)
    g = Guarded(wl)
    ref, _ = oracle_y(wl)
    for call in range(2):
        g.y.copy_(g.y0)
        g.L.lora_apply(g.x, g.y, g.rp.shape, g.rp.table.dev, g.sorted_ids, g.seg, g.active, g.ws, g.err, path=path)
        g.check(f"{path} call {call}")
        assert_y_close(g.y_bits(), ref, f"strided {path}")


@pytest.mark.parametrize("path", ["decode_direct", "decode_tma"])
def test_strided_rows_through_plans(path):
    """Plans: the plan buffer guarded too; three calls back to back."""
    torch = _torch()
    wl = W.config(2)
    g = Guarded(wl)
    L = g.L
    nb = L.lora_plan_bytes(wl.T, g.rp.shape)
    pbig, plan = _guarded(nb, torch.uint8, 0xA5, front=256, back=256)
    L.lora_build_plan(wl.T, g.rp.shape, g.rp.table.dev, g.sorted_ids, g.seg, g.active, plan, g.err, path=path)
    ref, _ = oracle_y(wl)
    for call in range(3):
        g.y.copy_(g.y0)
        L.lora_apply_plan(g.x, g.y, g.rp.shape, plan, g.ws, g.err, path=path)
        g.check(f"plan {path} call {call}")
        _canaries_intact(pbig, plan, f"plan {path}: plan buffer")
        assert_y_close(g.y_bits(), ref, f"strided plan {path}")


def test_strided_rows_fp8():
    """FP8 adapters (packed QKV shapes): x and y column windows."""
    wl = W.config(6)
    g = Guarded(wl)
    ref, st = oracle_y_e4m3(wl)
    assert st == 0
    g.L.lora_apply(g.x, g.y, g.rp.shape, g.rp.table.dev, g.sorted_ids, g.seg, g.active, g.ws, g.err,
                   path="decode_direct_fp8")
    g.check("fp8")
    assert_y_close(g.y_bits(), ref, "strided fp8")


def test_strided_rows_prefill_long_segments():
    """The tensor-core prefill kernels on long segments with ragged tails."""
    from test_gpu_parity import _small
    wl = _small(33, 2100, 1024, [1536, 512], 6, [64, 16, 8, 64, 48, 32], slot_dist="zipf")
    g = Guarded(wl)
    ref, _ = oracle_y(wl)
    g.L.lora_apply(g.x, g.y, g.rp.shape, g.rp.table.dev, g.sorted_ids, g.seg, g.active, g.ws, g.err,
                   max_seg_hint=wl.T, path="prefill")
    g.check("prefill long")
    assert_y_close(g.y_bits(), ref, "strided prefill")


@pytest.mark.parametrize("path", ["decode_direct", "decode_tma", "decode_cluster"])
def test_strided_rows_moe(path):
    """Routed experts: y per (token, choice) pair in a column window, x per token
    in a column window, guarded pair index and workspace."""
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import ResidentMoeProjection, to_host_bits
    wl = W.moe_config()
    rp = ResidentMoeProjection(wl, 0)
    P, V = wl.T * wl.K, wl.n_adapters * wl.E
    xbig, x = _window(rp.x, 0, XOFF, PAD, CANARY16)
    ybig, y = _window(rp.y, 2, YOFF, PAD, CANARY16)
    sbig, sorted_ids = _guarded(P, torch.int32, CANARY32)
    gbig, seg = _guarded(V + 2, torch.int32, CANARY32)
    abig, active = _guarded(V + 1, torch.int32, CANARY32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    wbig, ws = _guarded((L.lora_workspace_bytes(P, rp.shape) + 3) // 4, torch.float32, CANARYF, front=64)
    ws.zero_()
    L.lora_build_index_moe(torch.from_numpy(wl.slot_ids).cuda(),
                           torch.from_numpy(wl.expert_ids.reshape(-1).copy()).cuda(), wl.K, wl.E, V, rp.table.dev,
                           sorted_ids, seg, active, err)
    L.lora_apply_moe(x, y, wl.K, rp.shape, rp.table.dev, sorted_ids, seg, active, ws, err,
                     x_per_token=rp.x_per_token, path=path)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for big, view, what in ((ybig, y, "y"), (xbig, x, "x"), (wbig, ws, "ws"), (sbig, sorted_ids, "sorted"),
                            (gbig, seg, "seg"), (abig, active, "active")):
        _canaries_intact(big, view, "moe " + what)
    m = wl.modules[0]
    scales = oracle.slot_scales(wl.ranks, wl.alphas, wl.scale_rule, False)
    ref, st = oracle.apply_moe(m.x, m.x_per_token, m.y_in, m.slice_widths, wl.slot_ids, wl.expert_ids, wl.E,
                               wl.ranks, scales, m.A, m.B)
    assert st == 0
    assert_y_close(to_host_bits(y.contiguous()), ref, f"strided moe {path}")


def test_strided_rows_prefill_request_major_tma_tiles():
    """Request-major prefill batch whose tiles mostly hold consecutive rows (the
    tensor-map copies of x and y and the per-warp tensor-map stores): ragged
    request lengths (tiles that end mid-buffer), adapters shared by several
    requests (tiles that straddle two requests gather row by row), k not a
    multiple of 64, slice widths not multiples of 64, x and y as column windows
    with canary bands, two calls in a row."""
    wl = W.generate(name="req_tma", seed=57, T=None, S=3, rank_choices=[16, 32, 64],
                    modules=[{"name": "m", "k": 1000, "slices": [200, 72, 328]}],
                    requests={"n": 7, "min_len": 100, "max_len": 700, "n_adapters": 3},
                    alpha=16.0, y_init="normal")
    assert wl.r_max <= 64
    g = Guarded(wl)
    ref, _ = oracle_y(wl)
    for call in range(2):
        g.y.copy_(g.y0)
        g.L.lora_apply(g.x, g.y, g.rp.shape, g.rp.table.dev, g.sorted_ids, g.seg, g.active, g.ws, g.err,
                       max_seg_hint=wl.T, path="prefill")
        g.check(f"prefill request-major call {call}")
        assert_y_close(g.y_bits(), ref, "strided request-major prefill")
