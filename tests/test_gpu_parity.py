"""GPU parity: the CUDA library against the CPU oracle on the same seeded inputs.

Index outputs must match bit for bit; y must lie within the y
tolerance |gpu - ref| <= 1e-2 + 2e-2 |ref| of the fp64 oracle; rows of tokens
without an active slot must keep their exact input bits.  Every call goes
through the C ABI (via the ctypes binding).
"""
import numpy as np
import pytest

import oracle
import workloads as W
from _parity import assert_y_close, cluster_ok, gpu_apply, oracle_y, untouched_rows

pytestmark = pytest.mark.gpu

DECODE_PATHS = ["decode_split", "decode_fused", "decode_direct", "decode_tma", "decode_cluster"]


def tma_ok(wl, mod_idx=0):
    """Shapes the one-kernel TMA decode path takes."""
    m = wl.modules[mod_idx]
    return wl.r_max <= 64 and len(m.slice_widths) * wl.r_max <= 192 and m.k % 64 == 0


def _torch():
    import torch
    return torch


def _small(seed, T, k, widths, S, ranks, frac_none=0.1, slot_dist="uniform", y_init="normal",
           scale_rule="alpha_over_r", premultiplied=False):
    wl = W.generate(name="case", seed=seed, T=T, S=S, rank=8, modules=[{"name": "m", "k": k, "slices": widths}],
                    slot_dist=slot_dist, frac_none=frac_none, alpha=16.0, y_init=y_init,
                    scale_rule=scale_rule, premultiplied=premultiplied)
    # per-slot ranks drawn with the same generator rules
    rng = np.random.Generator(np.random.PCG64(seed + 7))
    wl.ranks = np.asarray(ranks, dtype=np.int32)
    wl.r_max = max(8, int(max(ranks)))
    m = wl.modules[0]
    m.A = [[(W._normal_bf16(rng, (r, k), k ** -0.5) if r > 0 else None) for _ in widths] for r in wl.ranks]
    m.B = [[(W._normal_bf16(rng, (w, r), 0.02) if r > 0 else None) for w in widths] for r in wl.ranks]
    wl.alphas = np.full(S, 16.0)
    return wl


# ---------------------------------------------------------------------------
# Index
# ---------------------------------------------------------------------------
def _gpu_index(slot_ids, S, ranks):
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    T = len(slot_ids)
    tab = L.SlotTable(S, 1, 256)
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    ptrs = np.full(S, dummy.data_ptr(), dtype=np.uint64)
    tab.set(np.asarray(ranks, np.int32), np.ones(S, np.float32), ptrs, ptrs)
    idx = L.TokenIndex(T, S)
    sid = torch.from_numpy(np.ascontiguousarray(slot_ids, dtype=np.int32)).cuda()
    idx.build(sid, tab)
    torch.cuda.synchronize()
    return (idx.sorted_ids.cpu().numpy()[:T], idx.seg_offsets.cpu().numpy(), idx.active.cpu().numpy(),
            int(idx.err.cpu().item()))


def _check_index(slot_ids, S, ranks):
    so, seg, act, err = _gpu_index(slot_ids, S, ranks)
    so_r, seg_r, act_r, st_r = oracle.build_index(slot_ids, S, ranks)
    np.testing.assert_array_equal(so, so_r)
    np.testing.assert_array_equal(seg, seg_r)
    np.testing.assert_array_equal(act[:1 + act_r[0]], act_r[:1 + act_r[0]])
    assert (err == 4) == (st_r == oracle.ERR_SLOT_RANGE)
    assert err in (0, 4)


@pytest.mark.parametrize("cfg", range(5))
def test_index_bit_exact_on_configs(cfg):
    wl = W.config(cfg, y_init="zeros") if cfg != 3 else None
    if cfg == 3:  # the prefill config's slot ids only (avoid drawing 1 GB of y here)
        rng_wl = W.generate(name="ids", seed=1003, T=None, S=16, rank=16,
                            modules=[{"name": "m", "k": 8, "slices": [8]}],
                            requests={"n": 16, "min_len": 128, "max_len": 2048, "n_adapters": 16},
                            alpha=32.0)
        slot_ids, S, ranks = rng_wl.slot_ids, 16, rng_wl.ranks
    else:
        slot_ids, S, ranks = wl.slot_ids, wl.S, wl.ranks
    _check_index(slot_ids, S, ranks)


@pytest.mark.parametrize("T,S,seed", [(0, 1, 0), (1, 1, 1), (7, 3, 2), (33, 5, 3), (1024, 128, 4),
                                      (1025, 1, 5), (5000, 1024, 6), (40000, 17, 7), (100000, 300, 8)])
def test_index_fuzz(T, S, seed):
    rng = np.random.default_rng(seed)
    slot_ids = rng.integers(-1, S, size=T).astype(np.int32)
    ranks = rng.choice([0, 8, 16, 64], size=S).astype(np.int32)
    _check_index(slot_ids, S, ranks)


def _gpu_index_seq(seq_ids, tps, S, ranks):
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    T = len(seq_ids) * tps
    tab = L.SlotTable(S, 1, 256)
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    ptrs = np.full(S, dummy.data_ptr(), dtype=np.uint64)
    tab.set(np.asarray(ranks, np.int32), np.ones(S, np.float32), ptrs, ptrs)
    idx = L.TokenIndex(T, S)
    sid = torch.from_numpy(np.ascontiguousarray(seq_ids, dtype=np.int32)).cuda()
    idx.build_seq(sid, tps, tab)
    torch.cuda.synchronize()
    return (idx.sorted_ids.cpu().numpy()[:T], idx.seg_offsets.cpu().numpy(), idx.active.cpu().numpy(),
            int(idx.err.cpu().item()))


@pytest.mark.parametrize("n_seq,tps,S,seed", [(0, 4, 3, 0), (1, 1, 1, 1), (64, 4, 32, 2), (37, 3, 5, 3),
                                              (300, 8, 128, 4), (1024, 2, 17, 5), (5000, 3, 1024, 6)])
def test_speculative_index_bit_exact(n_seq, tps, S, seed):
    """Sequences of tps tokens (speculative decode): bit-exact against the oracle's
    token index of the repeated slot ids, out-of-range ids included."""
    rng = np.random.default_rng(seed)
    seq = rng.integers(-1, S, size=n_seq).astype(np.int32)
    if n_seq > 4:
        seq[3] = S + 2  # out of range: keyed with the no-adapter bucket, error reported
    ranks = rng.choice([0, 8, 16, 64], size=S).astype(np.int32)
    so, seg, act, err = _gpu_index_seq(seq, tps, S, ranks)
    so_r, seg_r, act_r, st_r = oracle.build_index_seq(seq, tps, S, ranks)
    np.testing.assert_array_equal(so, so_r)
    np.testing.assert_array_equal(seg, seg_r)
    np.testing.assert_array_equal(act[:1 + act_r[0]], act_r[:1 + act_r[0]])
    assert (err == 4) == (st_r == oracle.ERR_SLOT_RANGE)


@pytest.mark.parametrize("path", ["auto", "decode_direct", "decode_split"])
def test_apply_speculative_decode(path):
    """Packed QKV (Llama-3-8B shapes) for 64 sequences of 4 draft tokens each:
    index from the per-sequence slots, y against the oracle on the per-token slots."""
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import ResidentProjection, to_host_bits
    wl = W.config(5)
    tps = wl.tokens_per_seq
    seq = np.ascontiguousarray(wl.slot_ids[::tps])
    np.testing.assert_array_equal(np.repeat(seq, tps), wl.slot_ids)
    rp = ResidentProjection.from_workload(wl)
    idx = L.TokenIndex(wl.T, wl.S)
    idx.build_seq(torch.from_numpy(seq).cuda(), tps, rp.table)
    ws = L.Workspace(wl.T, rp.shape)
    counts = np.bincount(seq[seq >= 0], minlength=wl.S) * tps
    L.lora_apply(rp.x, rp.y, rp.shape, rp.table.dev, idx.sorted_ids, idx.seg_offsets, idx.active, ws.buf,
                 idx.err, max_seg_hint=int(counts.max()), path=path)
    torch.cuda.synchronize()
    assert int(idx.err.item()) == 0
    ref, _ = oracle_y(wl)
    assert_y_close(to_host_bits(rp.y), ref, "speculative decode")


def test_index_all_none_and_out_of_range():
    S = 4
    ranks = np.array([8, 8, 0, 16], np.int32)
    _check_index(np.full(50, -1, np.int32), S, ranks)
    ids = np.array([0, 5, -1, 3, -2, 2, 4, 1, 1, 0], np.int32)
    _check_index(ids, S, ranks)


def test_index_deterministic_over_runs():
    rng = np.random.default_rng(11)
    ids = rng.integers(-1, 64, size=3000).astype(np.int32)
    ranks = np.full(64, 16, np.int32)
    first = _gpu_index(ids, 64, ranks)
    for _ in range(20):
        again = _gpu_index(ids, 64, ranks)
        for a, b in zip(first[:3], again[:3]):
            np.testing.assert_array_equal(a, b)


# ---------------------------------------------------------------------------
# Branch on the named configs
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("path", DECODE_PATHS)
@pytest.mark.parametrize("cfg", [0, 1, 2])
@pytest.mark.parametrize("y_init", ["zeros", "normal"])
def test_apply_configs_full(cfg, y_init, path):
    wl = W.config(cfg, y_init=y_init)
    assert path != "decode_cluster" or cluster_ok(wl)
    y, err, *_ = gpu_apply(wl, path=path)
    assert err == 0
    ref, st = oracle_y(wl)
    assert st == 0
    assert_y_close(y, ref, f"config {cfg}")
    keep = untouched_rows(wl)
    np.testing.assert_array_equal(y[keep], wl.modules[0].y_in[keep])


@pytest.mark.parametrize("path", DECODE_PATHS)
def test_apply_large_decode_sampled(path):
    """T=1024, k=d=8192, r=64, S=128: all rows checked (the oracle takes seconds)."""
    wl = W.config(4)
    assert path != "decode_cluster" or cluster_ok(wl)
    y, err, *_ = gpu_apply(wl, path=path)
    assert err == 0
    rows = np.arange(wl.T, dtype=np.int32)
    ref, _ = oracle_y(wl, rows=rows)
    assert_y_close(y[rows], ref, "large decode")


@pytest.mark.parametrize("path", DECODE_PATHS)
@pytest.mark.parametrize("mod_idx", [0, 1, 2, 3])
def test_apply_layer_sweep_sampled(mod_idx, path):
    """The four packed projections of one Llama-3-8B layer at T=1024, r=64."""
    wl = W.config(4, sweep=True)
    if path == "decode_cluster" and not cluster_ok(wl, mod_idx):
        import rank_adapter_gemm_gb300 as L
        with pytest.raises(L.LoraError) as e:  # a CTA's B and y tiles exceed its shared memory
            gpu_apply(wl, mod_idx=mod_idx, path=path)
        assert e.value.status == 9
        return
    y, err, *_ = gpu_apply(wl, mod_idx=mod_idx, path=path)
    assert err == 0
    rng = np.random.default_rng(mod_idx)
    rows = np.sort(rng.choice(wl.T, size=96, replace=False)).astype(np.int32)
    ref, _ = oracle_y(wl, mod_idx=mod_idx, rows=rows)
    assert_y_close(y[rows], ref, wl.modules[mod_idx].name)
    keep = untouched_rows(wl)
    np.testing.assert_array_equal(y[keep], wl.modules[mod_idx].y_in[keep])


@pytest.mark.parametrize("path", ["auto", "decode_split"])
@pytest.mark.parametrize("mod_idx", [0, 1])
def test_apply_prefill_sampled(mod_idx, path):
    """Prefill MLP (about 17k tokens): sampled rows from every request, plus the
    first and last token of the batch.  "auto" takes the tensor-core prefill
    kernels here (segments far above LORA_DECODE_MAX_SEG)."""
    import rank_adapter_gemm_gb300 as L
    wl = W.config(3)
    if path == "auto":
        assert L.lora_resolve_path("auto", wl.T, wl.T)[0] == "prefill"
    y, err, *_ = gpu_apply(wl, mod_idx=mod_idx, path=path)
    assert err == 0
    rng = np.random.default_rng(100 + mod_idx)
    rows = np.unique(np.concatenate([[0, wl.T - 1], rng.choice(wl.T, size=190, replace=False)])).astype(np.int32)
    ref, _ = oracle_y(wl, mod_idx=mod_idx, rows=rows)
    assert_y_close(y[rows], ref, wl.modules[mod_idx].name)
    keep = untouched_rows(wl)
    np.testing.assert_array_equal(y[keep], wl.modules[mod_idx].y_in[keep])


def test_prefill_is_deterministic():
    """The prefill shrink reduces its split-K partials in cluster-rank order and
    the expand adds each product once: bit-identical over runs."""
    wl = _small(21, 1500, 2048, [1024, 512], 3, [16, 16, 8], frac_none=0.05)
    ys, err, *_ = gpu_apply(wl, repeat=3, path="prefill")
    assert err == 0
    for y in ys[1:]:
        np.testing.assert_array_equal(y, ys[0])


# ---------------------------------------------------------------------------
# Ragged shapes and edge cases
# ---------------------------------------------------------------------------
RAGGED = [
    # seed, T, k, widths, S, ranks
    (1, 33, 40, [8, 24], 5, [8, 24, 0, 72, 8]),
    (2, 1, 8, [8], 1, [8]),
    (3, 70, 264, [136, 8, 520], 3, [16, 256, 40]),
    (4, 300, 1000, [1000], 2, [64, 8]),
    (5, 129, 520, [512, 16, 8, 24], 7, [8, 16, 24, 32, 40, 48, 56]),
    (6, 257, 4096, [1024], 1, [128]),
    (7, 90, 272, [136, 8, 528], 5, [16, 128, 40, 0, 24]),
    (8, 200, 1040, [1040, 16], 9, [8, 8, 16, 32, 64, 120, 8, 16, 24]),
]


@pytest.mark.parametrize("path", DECODE_PATHS + ["prefill"])
@pytest.mark.parametrize("case", RAGGED, ids=[f"ragged{c[0]}" for c in RAGGED])
def test_apply_ragged(case, path):
    seed, T, k, widths, S, ranks = case
    wl = _small(seed, T, k, widths, S, ranks)
    if path == "prefill" and wl.r_max > 64:
        import rank_adapter_gemm_gb300 as L
        with pytest.raises(L.LoraError) as e:  # the tensor-core path pads ranks to at most 64
            gpu_apply(wl, path=path)
        assert e.value.status == 9
        return
    mma_ok = wl.r_max <= 128 and k % 16 == 0  # the fused warp-MMA kernel
    if ((path == "decode_fused" and not mma_ok) or (path == "decode_direct" and wl.r_max > 64)
            or (path == "decode_tma" and not tma_ok(wl)) or (path == "decode_cluster" and not cluster_ok(wl))):
        import rank_adapter_gemm_gb300 as L
        with pytest.raises(L.LoraError) as e:
            gpu_apply(wl, path=path)
        assert e.value.status == 9
        return
    y, err, *_ = gpu_apply(wl, path=path)
    assert err == 0
    ref, _ = oracle_y(wl)
    assert_y_close(y, ref, f"ragged {seed}")
    keep = untouched_rows(wl)
    np.testing.assert_array_equal(y[keep], wl.modules[0].y_in[keep])


# Long segments for the tensor-core path: several 128-token tiles per slot with
# ragged tails, gathered (non-contiguous) rows, k not a multiple of 64, slice
# widths not multiples of 256 or 64, and every rank padding (16, 32, 64).
PREFILL = [
    # seed, T, k, widths, S, ranks, slot_dist
    (31, 700, 4096, [4096], 2, [16, 16], "uniform"),
    (32, 1000, 520, [264, 8, 1000], 4, [32, 8, 0, 24], "uniform"),
    (33, 2100, 1024, [1536, 512], 6, [64, 16, 8, 64, 48, 32], "zipf"),
    (34, 513, 64, [72], 1, [16], "uniform"),
    (35, 3000, 8192, [512, 512, 512, 512], 5, [16, 8, 16, 0, 8], "uniform"),
    (36, 400, 4104, [4104], 3, [64, 64, 56], "uniform"),
]


@pytest.mark.parametrize("case", PREFILL, ids=[f"prefill{c[0]}" for c in PREFILL])
@pytest.mark.parametrize("y_init", ["zeros", "normal"])
def test_apply_prefill_long_segments(case, y_init):
    seed, T, k, widths, S, ranks, dist = case
    wl = _small(seed, T, k, widths, S, ranks, slot_dist=dist, y_init=y_init, frac_none=0.05)
    y, err, *_ = gpu_apply(wl, path="prefill")
    assert err == 0
    ref, _ = oracle_y(wl)
    assert_y_close(y, ref, f"prefill {seed}")
    keep = untouched_rows(wl)
    np.testing.assert_array_equal(y[keep], wl.modules[0].y_in[keep])


def test_prefill_request_major_batch():
    """Requests of 128..2048 tokens laid out one after another, each with one
    adapter (the prefill batch shape), reduced to k = 1024 so every row is checked."""
    wl = W.generate(name="req", seed=41, T=None, S=8, rank=16,
                    modules=[{"name": "m", "k": 1024, "slices": [2048, 2048]}],
                    requests={"n": 6, "min_len": 128, "max_len": 2048, "n_adapters": 8},
                    alpha=32.0, scale_rule="alpha_over_sqrt_r", y_init="normal")
    y, err, *_ = gpu_apply(wl, path="prefill")
    assert err == 0
    ref, _ = oracle_y(wl)
    assert_y_close(y, ref, "request-major prefill")


def test_apply_all_tokens_without_adapter():
    wl = _small(9, 64, 256, [256], 4, [16, 16, 16, 16], frac_none=1.0)
    y, err, *_ = gpu_apply(wl)
    assert err == 0
    np.testing.assert_array_equal(y, wl.modules[0].y_in)


def test_apply_zero_B_leaves_y_unchanged():
    wl = _small(10, 48, 512, [256, 128], 3, [16, 32, 8], frac_none=0.0)
    m = wl.modules[0]
    m.B = [[(np.zeros_like(b) if b is not None else None) for b in row] for row in m.B]
    y, err, *_ = gpu_apply(wl)
    assert err == 0
    np.testing.assert_array_equal(W.bf16_bits_to_f32(y), W.bf16_bits_to_f32(m.y_in))


def test_apply_out_of_range_slots_flag_error_and_skip_rows():
    wl = _small(12, 40, 256, [128], 3, [8, 16, 8], frac_none=0.0)
    wl.slot_ids[[0, 5, 9]] = [3, 100, -4]
    y, err, *_ = gpu_apply(wl)
    assert err == 4  # LORA_ERR_SLOT_RANGE
    ref, _ = oracle_y(wl)
    assert_y_close(y, ref, "out of range")
    np.testing.assert_array_equal(y[[0, 5, 9]], wl.modules[0].y_in[[0, 5, 9]])


def test_apply_rslora_and_premultiplied_configs():
    for rule, pre in [("alpha_over_sqrt_r", False), ("alpha_over_r", True), ("alpha_over_sqrt_r", True)]:
        wl = _small(13, 64, 512, [256, 256], 4, [16, 64, 8, 32], scale_rule=rule, premultiplied=pre)
        y, err, *_ = gpu_apply(wl)
        assert err == 0
        ref, _ = oracle_y(wl)
        assert_y_close(y, ref, f"{rule} premultiplied={pre}")


def test_apply_is_deterministic():
    """The split path reduces in a fixed order: bit-identical over runs."""
    wl = W.config(2)
    ys, err, *_ = gpu_apply(wl, repeat=5, path="decode_split")
    for y in ys[1:]:
        np.testing.assert_array_equal(y, ys[0])


@pytest.mark.parametrize("path", ["decode_fused", "decode_direct", "decode_tma", "decode_cluster"])
def test_fused_repeat_stays_within_tolerance(path):
    """The fused kernels add split-k partials with fp32 reductions, whose order
    varies; every repetition must still match the oracle."""
    wl = W.config(2)
    ys, err, *_ = gpu_apply(wl, repeat=5, path=path)
    assert err == 0
    ref, _ = oracle_y(wl)
    for y in ys:
        assert_y_close(y, ref, "fused repeat")


@pytest.mark.parametrize("path", ["decode_fused", "decode_direct"])
def test_decode_leaves_workspace_ready(path):
    """Each call leaves the workspace ready for the next one without a clearing
    launch: the fused kernel clears its accumulator rows and counters; the
    warp-streaming kernels add into one of their two accumulators, clear the
    other and advance the call counter g (the control word after the 8 S
    per-slot counters), so accumulator g & 1 is zero after every call."""
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import ResidentProjection, to_host_bits
    wl = W.config(2)
    rp = ResidentProjection.from_workload(wl)
    idx = L.TokenIndex(wl.T, wl.S)
    idx.build(torch.from_numpy(wl.slot_ids).cuda(), rp.table)
    ws = L.Workspace(wl.T, rp.shape)
    ref, _ = oracle_y(wl)
    y0 = rp.y.clone()
    n, T, r_max, S = wl.modules[0].n_slices, wl.T, wl.r_max, wl.S
    xa_floats = n * T * r_max
    region = (xa_floats + 63) // 64 * 64  # regions start on 256-byte boundaries
    hl_region = (n * T * 64 * 2 // 4 + 63) // 64 * 64  # bf16 hi or lo, rank padded to 64
    xa_off = L.lora_workspace_xa_offset(rp.shape) // 4
    acc_off = xa_off + region
    acc2_off = acc_off + region + 2 * hl_region
    gen_word = 2 * 4 * S
    for call in range(1, 4):
        rp.y.copy_(y0)
        L.lora_apply(rp.x, rp.y, rp.shape, rp.table.dev, idx.sorted_ids, idx.seg_offsets, idx.active, ws.buf,
                     idx.err, path=path)
        torch.cuda.synchronize()
        assert int(idx.err.item()) == 0
        assert_y_close(to_host_bits(rp.y), ref, path)
        buf = ws.buf.cpu().numpy()
        ctrl = buf[:xa_off].view(np.int32).copy()
        assert not buf[acc_off:acc_off + xa_floats].any(), "fused accumulator not cleared"
        if path == "decode_direct":
            assert ctrl[gen_word] == call, "call counter not advanced"
            ctrl[gen_word] = 0
            nxt = acc2_off + (call & 1) * region
            assert not buf[nxt:nxt + xa_floats].any(), "next accumulator not cleared"
        assert not ctrl.any(), "counters not reset"


@pytest.mark.parametrize("path", ["decode_fused"])
def test_fused_wait_timeout_reports_error_and_device_stays_usable(path):
    """Counters that can never reach their targets (a poisoned workspace) make the
    fused kernel's bounded cross-CTA wait give up: the call ends with
    LORA_ERR_TIMEOUT in the error word instead of hanging, and the next call on a
    clean workspace is correct."""
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import ResidentProjection, to_host_bits
    wl = W.config(2)
    rp = ResidentProjection.from_workload(wl)
    idx = L.TokenIndex(wl.T, wl.S)
    idx.build(torch.from_numpy(wl.slot_ids).cuda(), rp.table)
    ws = L.Workspace(wl.T, rp.shape)
    y0 = rp.y.clone()
    xa_off = L.lora_workspace_xa_offset(rp.shape) // 4
    ws.buf[:xa_off].view(torch.int32).fill_(-(1 << 30))
    L.lora_apply(rp.x, rp.y, rp.shape, rp.table.dev, idx.sorted_ids, idx.seg_offsets, idx.active, ws.buf,
                 idx.err, path=path)
    torch.cuda.synchronize()
    assert int(idx.err.item()) == 7  # LORA_ERR_TIMEOUT
    ws.buf.zero_()
    idx.err.zero_()
    rp.y.copy_(y0)
    L.lora_apply(rp.x, rp.y, rp.shape, rp.table.dev, idx.sorted_ids, idx.seg_offsets, idx.active, ws.buf,
                 idx.err, path=path)
    torch.cuda.synchronize()
    assert int(idx.err.item()) == 0
    ref, _ = oracle_y(wl)
    assert_y_close(to_host_bits(rp.y), ref, path + " after a timed-out call")


# ---------------------------------------------------------------------------
# Shrink and expand entry points on their own
# ---------------------------------------------------------------------------
def test_shrink_then_expand_entry_points():
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import ResidentProjection, to_host_bits
    wl = W.config(2)
    rp = ResidentProjection.from_workload(wl)
    idx = L.TokenIndex(wl.T, wl.S)
    idx.build(torch.from_numpy(wl.slot_ids).cuda(), rp.table)
    ws = L.Workspace(wl.T, rp.shape)
    L.lora_shrink(rp.x, rp.shape, rp.table.dev, idx.sorted_ids, idx.seg_offsets, idx.active, ws.buf, idx.err)
    torch.cuda.synchronize()
    # compare xa (float32 [n][T][r_max] in the workspace) with the oracle's shrink
    off = L.lora_workspace_xa_offset(rp.shape) // 4
    nxa = wl.modules[0].n_slices * wl.T * wl.r_max
    xa = ws.buf[off:off + nxa].view(wl.modules[0].n_slices, wl.T, wl.r_max).cpu().numpy().astype(np.float64)
    ref, _ = oracle.shrink(wl.modules[0].x, wl.slot_ids, wl.ranks, wl.modules[0].A, wl.r_max)
    for t in range(wl.T):
        r = wl.ranks[wl.slot_ids[t]]
        got = xa[:, t, :r]
        want = ref[t, :, :r]
        np.testing.assert_allclose(got, want, rtol=1e-4, atol=1e-4)
    L.lora_expand(ws.buf, rp.y, rp.shape, rp.table.dev, idx.sorted_ids, idx.seg_offsets, idx.active, idx.err)
    torch.cuda.synchronize()
    assert int(idx.err.cpu().item()) == 0
    y_ref, _ = oracle_y(wl)
    assert_y_close(to_host_bits(rp.y), y_ref, "shrink+expand")


def test_premultiply_kernel_matches_oracle():
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import to_device_bf16, to_host_bits
    rng = np.random.default_rng(3)
    b = W.f32_to_bf16_bits(rng.standard_normal(100000, dtype=np.float32))
    for s in (2.0, 0.25, 8.0):
        t = to_device_bf16(b)
        L.lora_premultiply(t, s)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(to_host_bits(t), oracle.premultiply(b, s))
    t = to_device_bf16(b)
    L.lora_premultiply(t, 0.3)
    torch.cuda.synchronize()
    got = W.bf16_bits_to_f32(to_host_bits(t)).astype(np.float64)
    want = W.bf16_bits_to_f32(oracle.premultiply(b, 0.3)).astype(np.float64)
    # fp32 product then one rounding vs the exact product rounded: at most one bf16 step apart
    np.testing.assert_allclose(got, want, rtol=2 ** -7, atol=0)


# ---------------------------------------------------------------------------
# Host-side argument checks (no kernel runs)
# ---------------------------------------------------------------------------
def test_host_validation_errors():
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    wl = _small(14, 16, 64, [64], 2, [8, 8])
    from rank_adapter_gemm_gb300.resident import ResidentProjection
    rp = ResidentProjection.from_workload(wl)
    idx = L.TokenIndex(wl.T, wl.S)
    idx.build(torch.from_numpy(wl.slot_ids).cuda(), rp.table)
    ws = L.Workspace(wl.T, rp.shape)
    args = (rp.shape, rp.table.dev, idx.sorted_ids, idx.seg_offsets, idx.active)
    with pytest.raises(L.LoraError) as e:
        L.lora_apply(rp.x, rp.y, *args, ws.buf[:4], idx.err)
    assert e.value.status == 6
    bad_x = torch.zeros(wl.T, 72, dtype=torch.bfloat16, device="cuda")[:, 1:65]
    with pytest.raises(L.LoraError) as e:
        L.lora_apply(bad_x, rp.y, *args, ws.buf, idx.err)
    assert e.value.status == 2
    bad_shape = L.make_shape(2, 8, 60, [64])
    with pytest.raises(L.LoraError) as e:
        L.lora_apply(rp.x, rp.y, bad_shape, *args[1:], ws.buf, idx.err)
    assert e.value.status == 2
    with pytest.raises(L.LoraError) as e:
        L.lora_apply(rp.x, rp.y, L.make_shape(2, 12, 64, [64]), *args[1:], ws.buf, idx.err)
    assert e.value.status == 3


def test_rank_above_r_max_is_rejected_on_device():
    """A table whose rank exceeds the shape's r_max (the workspace stride) is an
    error and the slot is skipped, never an out-of-bounds write."""
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import ResidentProjection, to_host_bits
    wl = _small(15, 32, 128, [128], 2, [32, 8], frac_none=0.0)
    rp = ResidentProjection.from_workload(wl)
    idx = L.TokenIndex(wl.T, wl.S)
    idx.build(torch.from_numpy(wl.slot_ids).cuda(), rp.table)
    small = L.make_shape(2, 16, 128, [128])
    ws = L.Workspace(wl.T, small)
    L.lora_apply(rp.x, rp.y, small, rp.table.dev, idx.sorted_ids, idx.seg_offsets, idx.active, ws.buf, idx.err)
    torch.cuda.synchronize()
    assert int(idx.err.cpu().item()) == 3
    y = to_host_bits(rp.y)
    rows0 = wl.slot_ids == 0
    np.testing.assert_array_equal(y[rows0], wl.modules[0].y_in[rows0])


@pytest.mark.parametrize("path", ["auto", "decode_split", "decode_fused"])
def test_apply_with_base_on_aux_stream(path):
    """y = x W0^T + branch with the branch on an auxiliary stream next to the base
    GEMM (TensorRT-LLM LoRA serving page, "与基座并行:forward_with_base"): the
    branch's x-only half overlaps the GEMM and its y half waits for the GEMM's
    event.  Reference: the oracle on top of the GPU's own base-GEMM output."""
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import ResidentProjection, to_host_bits
    wl = W.config(2)
    rp = ResidentProjection.from_workload(wl)
    d = sum(wl.modules[0].slice_widths)
    g = torch.Generator(device="cuda").manual_seed(5)
    w0 = (torch.randn(d, wl.modules[0].k, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    idx = L.TokenIndex(wl.T, wl.S)
    idx.build(torch.from_numpy(wl.slot_ids).cuda(), rp.table)
    ws = L.Workspace(wl.T, rp.shape)
    counts = np.bincount(wl.slot_ids[wl.slot_ids >= 0], minlength=wl.S)
    x = rp.x.view(torch.bfloat16)
    y = rp.y.view(torch.bfloat16)
    base = torch.matmul(x, w0.t())
    torch.cuda.synchronize()
    base_bits = to_host_bits(base)
    aux = torch.cuda.Stream()
    y.fill_(7.0)  # overwritten by the base GEMM before the branch touches it
    L.apply_with_base(x, w0, y, rp.shape, rp.table.dev, idx, ws.buf, aux, max_seg_hint=int(counts.max()), path=path)
    torch.cuda.synchronize()
    assert int(idx.err.item()) == 0
    ref, _ = oracle_y(wl, y_in=base_bits)
    assert_y_close(to_host_bits(rp.y), ref, f"with base ({path})")


# ---------------------------------------------------------------------------
# FP8 adapters (LORA_PATH_DECODE_DIRECT_FP8) against the e4m3 oracle
# ---------------------------------------------------------------------------
def _small_fp8(seed, T, k, widths, S, ranks, frac_none=0.1, slot_dist="uniform", premultiplied=False):
    wl = W.generate(name="case_fp8", seed=seed, T=T, S=S, rank=8, modules=[{"name": "m", "k": k, "slices": widths}],
                    slot_dist=slot_dist, frac_none=frac_none, alpha=1.0 / 32.0, premultiplied=premultiplied,
                    weights="e4m3")
    rng = np.random.Generator(np.random.PCG64(seed + 7))
    wl.ranks = np.asarray(ranks, dtype=np.int32)
    wl.r_max = max(8, int(max(ranks)))
    m = wl.modules[0]
    m.A = [[(W._e4m3_codes(rng, (r, k)) if r > 0 else None) for _ in widths] for r in wl.ranks]
    m.B = [[(W._e4m3_codes(rng, (w, r)) if r > 0 else None) for w in widths] for r in wl.ranks]
    wl.alphas = np.full(S, 1.0 / 32.0)
    return wl


def _check_fp8(wl, what, repeat=1, overlap=False):
    from _parity import oracle_y_e4m3
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import ResidentProjection, to_host_bits
    rp = ResidentProjection.from_workload(wl)
    assert rp.fp8
    idx = L.TokenIndex(wl.T, wl.S)
    idx.build(torch.from_numpy(np.ascontiguousarray(wl.slot_ids, dtype=np.int32)).cuda(), rp.table)
    ws = L.Workspace(wl.T, rp.shape)
    y0 = rp.y.clone()
    ref, st = oracle_y_e4m3(wl)
    assert st == 0
    keep = untouched_rows(wl)
    for _ in range(repeat):
        rp.y.copy_(y0)
        if overlap:
            ev = torch.cuda.Event()
            ev.record()
            L.lora_apply_overlap(rp.x, rp.y, rp.shape, rp.table.dev, idx.sorted_ids, idx.seg_offsets, idx.active,
                                 ws.buf, idx.err, y_ready=ev, path="decode_direct_fp8")
        else:
            L.lora_apply(rp.x, rp.y, rp.shape, rp.table.dev, idx.sorted_ids, idx.seg_offsets, idx.active, ws.buf,
                         idx.err, path="decode_direct_fp8")
        torch.cuda.synchronize()
        assert int(idx.err.item()) == 0
        y = to_host_bits(rp.y)
        assert_y_close(y, ref, what)
        np.testing.assert_array_equal(y[keep], wl.modules[0].y_in[keep])


@pytest.mark.parametrize("y_init", ["zeros", "normal"])
def test_apply_fp8_decode_qkv(y_init):
    """Packed QKV decode (T=256, Llama-3-8B shapes, S=32, Zipf) with e4m3 adapters."""
    _check_fp8(W.config(6, y_init=y_init), f"fp8 qkv {y_init}")


def test_apply_fp8_repeat_and_overlap():
    """The call counter and the two sum buffers stay consistent over calls, with
    and without the y-ready event split."""
    wl = W.config(6)
    _check_fp8(wl, "fp8 repeat", repeat=3)
    _check_fp8(wl, "fp8 overlap", repeat=2, overlap=True)


FP8_RAGGED = [
    # seed, T, k, widths, S, ranks
    (61, 37, 256, [256], 3, [8, 16, 64]),
    (62, 300, 4112, [4096, 1032, 520], 5, [64, 8, 0, 32, 24]),
    (63, 1, 1024, [2048], 1, [64]),
    (64, 700, 2048, [8, 136, 1000], 7, [8, 16, 24, 32, 40, 48, 56]),
    (65, 2048, 512, [512], 2, [64, 16]),
]


@pytest.mark.parametrize("case", FP8_RAGGED, ids=[f"fp8ragged{c[0]}" for c in FP8_RAGGED])
def test_apply_fp8_ragged(case):
    """Token groups of 24 with ragged tails, k not a multiple of 64, slice widths
    not multiples of 64, ranks 8..64, a single token and the 2048-token maximum."""
    seed, T, k, widths, S, ranks = case
    _check_fp8(_small_fp8(seed, T, k, widths, S, ranks), f"fp8 ragged {seed}")


def test_apply_fp8_premultiplied_and_clamped_x():
    """B scaled at load time by lora_premultiply_e4m3, and every x row heavily
    saturated: 64 of its 1024 entries beyond the e4m3 range (bf16 +-1000 and
    -464, clamped to +-448 before rounding; TensorRT-LLM LoRA serving page, the
    forward pass's clamp of the activation).  One slot's A also holds codes at
    +-448 in 32 of those columns, so its sums reach 32 * 448 * 448 (far past
    the f16 range): the sums enter the expand as bf16 hi and lo parts and every
    element must still meet the y tolerance."""
    wl = _small_fp8(66, 200, 1024, [1024, 256], 4, [16, 64, 32, 8], premultiplied=True)
    x = wl.modules[0].x
    rng = np.random.default_rng(66)
    big = np.array([0x447A, 0xC47A, 0xC3E8], np.uint16)  # bf16 1000, -1000, -464
    for t in range(wl.T):
        cols = rng.choice(1024, size=64, replace=False)
        x[t, cols] = big[rng.integers(0, 3, size=64)]
    hot = np.arange(0, 1024, 32)  # the columns the large A codes sit in
    x[:, hot] = np.uint16(0x447A)
    for Ai in wl.modules[0].A[1]:  # slot 1 (rank 64): codes 0x7E / 0xFE = +-448
        Ai[:, hot] = np.where(np.arange(Ai.shape[0])[:, None] % 2 == 0, 0x7E, 0xFE).astype(np.uint8)
    assert (wl.slot_ids == 1).any()
    _check_fp8(wl, "fp8 premultiplied, heavily clamped x, sums past 65504")


def test_apply_fp8_rejects_k_not_multiple_of_16():
    import rank_adapter_gemm_gb300 as L
    wl = _small_fp8(67, 40, 1032, [256], 2, [16, 16])
    with pytest.raises(L.LoraError) as e:
        _check_fp8(wl, "fp8 k % 16")
    assert e.value.status == 9


def test_premultiply_e4m3_kernel_bit_exact():
    """Every finite e4m3 code times scales that round, tie, clamp and underflow,
    against the oracle bit for bit; NaN codes become 0x7F."""
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    for s in (2.0, 0.3, 1.0 / 256.0, 100.0, 0.0078125, 3.0, -1.5, 1e-3):
        t = torch.from_numpy(np.tile(codes, 3)).cuda()
        L.lora_premultiply_e4m3(t, s)
        torch.cuda.synchronize()
        want = oracle.premultiply_e4m3(np.tile(codes, 3), float(np.float32(s)))
        np.testing.assert_array_equal(t.cpu().numpy(), want, err_msg=f"scale {s}")
    t = torch.tensor([0x7F, 0xFF, 0x01], dtype=torch.uint8, device="cuda")
    L.lora_premultiply_e4m3(t, 2.0)
    torch.cuda.synchronize()
    assert t.cpu().numpy().tolist()[:2] == [0x7F, 0x7F]


# ---------------------------------------------------------------------------
# Routed-expert (MoE) LoRA against the oracle's per-pair definition
# ---------------------------------------------------------------------------
def _gpu_moe_index(slot_ids, expert_ids, E, n_adapters, ranks):
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    T, K = expert_ids.shape
    V = n_adapters * E
    tab = L.SlotTable(V, 1, 256)
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    ptrs = np.full(V, dummy.data_ptr(), dtype=np.uint64)
    tab.set(np.repeat(np.asarray(ranks, np.int32), E), np.ones(V, np.float32), ptrs, ptrs)
    idx = L.TokenIndex(T * K, V)
    idx.build_moe(torch.from_numpy(np.ascontiguousarray(slot_ids, np.int32)).cuda(),
                  torch.from_numpy(np.ascontiguousarray(expert_ids, np.int32).reshape(-1)).cuda(), K, E, tab)
    torch.cuda.synchronize()
    return (idx.sorted_ids.cpu().numpy()[:T * K], idx.seg_offsets.cpu().numpy(), idx.active.cpu().numpy(),
            int(idx.err.cpu().item()))


@pytest.mark.parametrize("T,K,E,n_adapters,seed", [(128, 2, 8, 8, 1), (37, 3, 5, 2, 2), (1, 1, 1, 1, 3),
                                                   (1000, 2, 64, 8, 4), (64, 8, 64, 4, 5)])
def test_moe_index_bit_exact(T, K, E, n_adapters, seed):
    """Pair index against the oracle's pair slots sorted by its comparison sort,
    with no-adapter tokens, rank-0 adapters and out-of-range slot and expert ids."""
    rng = np.random.default_rng(seed)
    slots = rng.integers(-1, n_adapters, size=T).astype(np.int32)
    experts = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    if T > 10:
        slots[3] = n_adapters + 1
        experts[5, 0] = E + 2 if slots[5] >= 0 else experts[5, 0]
    ranks = rng.choice([0, 8, 16], size=n_adapters).astype(np.int32)
    so, seg, act, err = _gpu_moe_index(slots, experts, E, n_adapters, ranks)
    pair = oracle.moe_pair_slots(slots, experts, E, n_adapters)
    so_r, seg_r, act_r, st_r = oracle.build_index(pair, n_adapters * E, np.repeat(ranks, E))
    np.testing.assert_array_equal(so, so_r)
    np.testing.assert_array_equal(seg, seg_r)
    np.testing.assert_array_equal(act[:1 + act_r[0]], act_r[:1 + act_r[0]])
    assert (err == 4) == (st_r == oracle.ERR_SLOT_RANGE)


def _check_moe(wl, mod_idx, what, rows=None, path="decode_direct"):
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import ResidentMoeProjection, to_host_bits
    rp = ResidentMoeProjection(wl, mod_idx)
    P = wl.T * wl.K
    idx = L.TokenIndex(P, wl.n_adapters * wl.E)
    idx.build_moe(torch.from_numpy(wl.slot_ids).cuda(), torch.from_numpy(wl.expert_ids.reshape(-1).copy()).cuda(),
                  wl.K, wl.E, rp.table)
    ws = L.Workspace(P, rp.shape)
    L.lora_apply_moe(rp.x, rp.y, wl.K, rp.shape, rp.table.dev, idx.sorted_ids, idx.seg_offsets, idx.active, ws.buf,
                     idx.err, x_per_token=rp.x_per_token, path=path)
    torch.cuda.synchronize()
    assert int(idx.err.item()) == 0
    m = wl.modules[mod_idx]
    scales = oracle.slot_scales(wl.ranks, wl.alphas, wl.scale_rule, False)
    ref, st = oracle.apply_moe(m.x, m.x_per_token, m.y_in, m.slice_widths, wl.slot_ids, wl.expert_ids, wl.E,
                               wl.ranks, scales, m.A, m.B, rows=rows)
    assert st == 0
    y = to_host_bits(rp.y)
    sel = np.arange(P) if rows is None else rows
    assert_y_close(y[sel], ref, what)
    none = np.repeat(wl.slot_ids < 0, wl.K)
    np.testing.assert_array_equal(y[none], m.y_in[none])


MOE_PATHS = ["decode_direct", "decode_tma", "decode_cluster"]


@pytest.mark.parametrize("path", MOE_PATHS)
@pytest.mark.parametrize("mod_idx", [0, 1], ids=["w1_x_per_token", "w2_x_per_pair"])
def test_apply_moe_mixtral_decode(mod_idx, path):
    """128 tokens routed top-2 of 8 experts (Mixtral-8x7B expert shapes), 8 adapters."""
    _check_moe(W.moe_config(), mod_idx, f"moe module {mod_idx} {path}", path=path)


MOE_RAGGED = [
    # seed, T, K, E, n_adapters, k, widths, ranks, x_per_token
    (71, 37, 3, 5, 3, 264, [40, 16], [8, 24, 0], True),
    (72, 50, 2, 16, 2, 512, [1032], [64, 8], False),
    (73, 1, 1, 1, 1, 128, [64], [16], True),
    (74, 256, 8, 32, 2, 1024, [256], [16, 32], True),
]


@pytest.mark.parametrize("path", MOE_PATHS)
@pytest.mark.parametrize("case", MOE_RAGGED, ids=[f"moe{c[0]}" for c in MOE_RAGGED])
def test_apply_moe_ragged(case, path):
    seed, T, K, E, n_ad, k, widths, ranks, per_token = case
    wl = W.generate_moe(name="moe_case", seed=seed, T=T, K=K, E=E, n_adapters=n_ad, rank=8,
                        modules=[{"name": "m", "k": k, "slices": widths, "x_per_token": per_token}],
                        slot_dist="uniform", frac_none=0.1)
    rng = np.random.Generator(np.random.PCG64(seed + 7))
    wl.ranks = np.asarray(ranks, np.int32)
    wl.r_max = max(8, max(ranks))
    wl.alphas = 2.0 * np.maximum(wl.ranks, 1)
    m = wl.modules[0]
    m.A = [[W._normal_bf16(rng, (E * r, k), k ** -0.5).reshape(E, r, k) for _ in widths] for r in wl.ranks]
    m.B = [[W._normal_bf16(rng, (E * w, r), 0.02).reshape(E, w, r) for w in widths] for r in wl.ranks]
    if path == "decode_tma" and k % 64 != 0:
        # the tensor-map path streams x and A in 64-column boxes: k must be a multiple of 64
        import rank_adapter_gemm_gb300 as L
        with pytest.raises(L.LoraError) as e:
            _check_moe(wl, 0, f"moe ragged {seed} {path}", path=path)
        assert e.value.status == 9
        return
    _check_moe(wl, 0, f"moe ragged {seed} {path}", path=path)


def test_apply_moe_rejects_too_many_pairs():
    import rank_adapter_gemm_gb300 as L
    wl = W.generate_moe(name="moe_big", seed=75, T=1100, K=2, E=4, n_adapters=1, rank=8,
                        modules=[{"name": "m", "k": 128, "slices": [64], "x_per_token": True}])
    with pytest.raises(L.LoraError) as e:
        _check_moe(wl, 0, "moe too many pairs")
    assert e.value.status == 9


# ---------------------------------------------------------------------------
# Activated LoRA (aLoRA) enablement in the index
# ---------------------------------------------------------------------------
def _activation_case(seed, n_seq, S, max_len=40):
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, max_len + 1, size=n_seq)
    past = rng.integers(0, 100, size=n_seq)  # tokens already cached before this batch
    seq_ids = np.repeat(np.arange(n_seq), lens).astype(np.int32)
    positions = np.concatenate([p + np.arange(n) for p, n in zip(past, lens)]).astype(np.int32)
    seq_slot = rng.integers(-1, S, size=n_seq).astype(np.int32)
    start = rng.integers(0, 150, size=n_seq).astype(np.int32)
    start[::5] = 0  # plain LoRA sequences
    return seq_ids, positions, seq_slot, start


def _gpu_activated_index(seq_ids, positions, seq_slot, start, S, ranks, table=None):
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    T = len(seq_ids)
    if table is None:
        table = L.SlotTable(S, 1, 256)
        dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
        ptrs = np.full(S, dummy.data_ptr(), dtype=np.uint64)
        table.set(np.asarray(ranks, np.int32), np.ones(S, np.float32), ptrs, ptrs)
    idx = L.TokenIndex(T, S)
    dev = [torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda() for a in (seq_ids, positions, seq_slot, start)]
    idx.build_activated(*dev, table)
    torch.cuda.synchronize()
    return idx


@pytest.mark.parametrize("n_seq,S,seed", [(20, 8, 1), (64, 32, 2), (1, 1, 3), (300, 128, 4)])
def test_activated_index_bit_exact(n_seq, S, seed):
    seq_ids, positions, seq_slot, start = _activation_case(seed, n_seq, S)
    ranks = np.random.default_rng(seed).choice([0, 8, 16], size=S).astype(np.int32)
    idx = _gpu_activated_index(seq_ids, positions, seq_slot, start, S, ranks)
    T = len(seq_ids)
    slots = oracle.activated_token_slots(seq_ids, positions, seq_slot, start)
    so_r, seg_r, act_r, st_r = oracle.build_index(slots, S, ranks)
    np.testing.assert_array_equal(idx.sorted_ids.cpu().numpy()[:T], so_r)
    np.testing.assert_array_equal(idx.seg_offsets.cpu().numpy(), seg_r)
    np.testing.assert_array_equal(idx.active.cpu().numpy()[:1 + act_r[0]], act_r[:1 + act_r[0]])
    assert int(idx.err.item()) == 0 and st_r == 0


def test_activated_index_reports_unknown_sequence():
    seq_ids, positions, seq_slot, start = _activation_case(9, 10, 4)
    seq_ids[7] = 10
    idx = _gpu_activated_index(seq_ids, positions, seq_slot, start, 4, np.full(4, 8, np.int32))
    slots = oracle.activated_token_slots(seq_ids, positions, seq_slot, start)
    so_r, seg_r, _, st_r = oracle.build_index(slots, 4, np.full(4, 8, np.int32))
    assert int(idx.err.item()) == 4 and st_r == oracle.ERR_SLOT_RANGE
    np.testing.assert_array_equal(idx.sorted_ids.cpu().numpy()[:len(seq_ids)], so_r)


def test_apply_activated_decode_qkv():
    """Packed QKV shapes (config 2's weights and rows) for a batch of sequences of
    which some invoke their adapter mid-batch: y against the oracle on the
    per-token slots of the activation rule."""
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import ResidentProjection, to_host_bits
    wl = W.config(2)
    rng = np.random.default_rng(12)
    lens = np.full(16, 16)
    seq_ids = np.repeat(np.arange(16), lens).astype(np.int32)
    positions = np.tile(np.arange(16), 16).astype(np.int32) + 200
    seq_slot = rng.integers(-1, wl.S, size=16).astype(np.int32)
    start = (200 + rng.integers(0, 20, size=16)).astype(np.int32)
    rp = ResidentProjection.from_workload(wl)
    idx = _gpu_activated_index(seq_ids, positions, seq_slot, start, wl.S, wl.ranks, table=rp.table)
    ws = L.Workspace(wl.T, rp.shape)
    L.lora_apply(rp.x, rp.y, rp.shape, rp.table.dev, idx.sorted_ids, idx.seg_offsets, idx.active, ws.buf, idx.err)
    torch.cuda.synchronize()
    assert int(idx.err.item()) == 0
    wl.slot_ids = oracle.activated_token_slots(seq_ids, positions, seq_slot, start)
    assert (wl.slot_ids == -1).sum() > 0 and (wl.slot_ids >= 0).sum() > 0
    ref, st = oracle_y(wl)
    assert st == 0
    y = to_host_bits(rp.y)
    assert_y_close(y, ref, "activated")
    keep = untouched_rows(wl)
    np.testing.assert_array_equal(y[keep], wl.modules[0].y_in[keep])



@pytest.mark.parametrize("path", ["auto", "decode_split", "decode_fused", "decode_direct", "prefill", "decode_tma",
                                  "decode_cluster"])
def test_apply_ranks_up_to_512(path):
    """Ranks 512 and 264 next to 8: the split kernels (AUTO's choice above rank 128)
    take any rank in 64-wide chunks; the paths with a lower rank bound refuse."""
    wl = _small(81, 100, 1024, [1024, 256], 3, [512, 264, 8])
    if path in ("decode_fused", "decode_direct", "prefill", "decode_tma", "decode_cluster"):
        import rank_adapter_gemm_gb300 as L
        with pytest.raises(L.LoraError) as e:
            gpu_apply(wl, path=path)
        assert e.value.status == 9
        return
    y, err, *_ = gpu_apply(wl, path=path)
    assert err == 0
    ref, _ = oracle_y(wl)
    assert_y_close(y, ref, f"ranks to 512 ({path})")
    keep = untouched_rows(wl)
    np.testing.assert_array_equal(y[keep], wl.modules[0].y_in[keep])


# ---------------------------------------------------------------------------
# Degenerate batches through the FP8, MoE and aLoRA entry points
# ---------------------------------------------------------------------------
def test_empty_batches_of_the_newer_entry_points():
    """T = 0: the pair and activated indexes give zero offsets and no active slot,
    and the MoE branch returns without touching anything."""
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    S = 8
    tab = L.SlotTable(S, 1, 64)
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    ptrs = np.full(S, dummy.data_ptr(), dtype=np.uint64)
    tab.set(np.full(S, 16, np.int32), np.ones(S, np.float32), ptrs, ptrs)
    empty = torch.zeros(0, dtype=torch.int32, device="cuda")
    idx = L.TokenIndex(0, S)
    idx.seg_offsets.fill_(7)
    idx.active.fill_(7)
    idx.build_moe(empty, empty, 2, 4, tab)
    torch.cuda.synchronize()
    assert idx.seg_offsets.cpu().numpy().tolist() == [0] * (S + 2) and int(idx.active[0].item()) == 0
    idx.seg_offsets.fill_(7)
    idx.build_activated(empty, empty, torch.zeros(3, dtype=torch.int32, device="cuda"),
                        torch.zeros(3, dtype=torch.int32, device="cuda"), tab)
    torch.cuda.synchronize()
    assert idx.seg_offsets.cpu().numpy().tolist() == [0] * (S + 2) and int(idx.err.item()) == 0
    shape = L.make_shape(S, 64, 128, [64])
    ws = L.Workspace(0, shape)
    x = torch.zeros(0, 128, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    L.lora_apply_moe(x, y, 2, shape, tab.dev, idx.sorted_ids, idx.seg_offsets, idx.active, ws.buf, idx.err)
    torch.cuda.synchronize()


def test_no_adapter_batches_keep_y_fp8_and_moe():
    """Every token without an adapter: y keeps its input bits through the FP8 path
    and through the MoE branch."""
    wl = _small_fp8(91, 64, 256, [256], 2, [16, 8])
    wl.slot_ids[:] = -1
    _check_fp8(wl, "fp8 no adapter")
    wm = W.generate_moe(name="moe_none", seed=92, T=40, K=2, E=4, n_adapters=2, rank=8,
                        modules=[{"name": "m", "k": 128, "slices": [64], "x_per_token": True}])
    wm.slot_ids[:] = -1
    _check_moe(wm, 0, "moe no adapter")


def test_object_level_apply():
    """apply(x, y, table, index, ws, shape) is lora_apply on the objects' buffers."""
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import ResidentProjection, to_host_bits
    wl = W.config(0)
    rp = ResidentProjection.from_workload(wl)
    idx = L.TokenIndex(wl.T, wl.S)
    idx.build(torch.from_numpy(wl.slot_ids).cuda(), rp.table)
    ws = L.Workspace(wl.T, rp.shape)
    L.apply(rp.x, rp.y, rp.table, idx, ws, rp.shape)
    torch.cuda.synchronize()
    assert int(idx.err.item()) == 0
    ref, _ = oracle_y(wl)
    assert_y_close(to_host_bits(rp.y), ref, "object-level apply")


# ---------------------------------------------------------------------------
# Plans: the warp-streaming kernels' tables built once per batch and shape
# ---------------------------------------------------------------------------
def _plan_apply(wl, path="decode_direct", repeat=1, mod_idx=0):
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import ResidentProjection, to_host_bits
    rp = ResidentProjection.from_workload(wl, mod_idx)
    idx = L.TokenIndex(wl.T, wl.S)
    idx.build(torch.from_numpy(np.ascontiguousarray(wl.slot_ids, dtype=np.int32)).cuda(), rp.table)
    ws = L.Workspace(wl.T, rp.shape)
    plan = L.Plan(wl.T, rp.shape, path)
    plan.build(idx, rp.table)
    y0 = rp.y.clone()
    outs = []
    for _ in range(repeat):
        rp.y.copy_(y0)
        plan.apply(rp.x, rp.y, ws, idx.err)
        torch.cuda.synchronize()
        outs.append(to_host_bits(rp.y))
    return outs, int(idx.err.item()), (rp, idx, ws, plan)


@pytest.mark.parametrize("path", ["decode_direct", "decode_tma"])
@pytest.mark.parametrize("cfg", [0, 1, 2, 4, 5])
def test_apply_plan_configs(cfg, path):
    """Every call of a plan against the oracle, three calls in a row on one workspace."""
    wl = W.config(cfg)
    outs, err, _ = _plan_apply(wl, path=path, repeat=3)
    assert err == 0
    rows = None if wl.T <= 512 else np.arange(0, wl.T, 3, dtype=np.int32)
    ref, st = oracle_y(wl, rows=rows)
    assert st == 0
    for y in outs:
        assert_y_close(y if rows is None else y[rows], ref, f"plan config {cfg}")


@pytest.mark.parametrize("case", [c for c in RAGGED if max(c[5]) <= 64], ids=lambda c: f"plan_ragged{c[0]}")
def test_apply_plan_ragged(case):
    seed, T, k, widths, S, ranks = case
    wl = _small(seed, T, k, widths, S, ranks)
    outs, err, _ = _plan_apply(wl)
    assert err == 0
    ref, _ = oracle_y(wl)
    assert_y_close(outs[0], ref, f"plan ragged {seed}")
    keep = untouched_rows(wl)
    np.testing.assert_array_equal(outs[0][keep], wl.modules[0].y_in[keep])


def test_apply_plan_fp8():
    from _parity import oracle_y_e4m3
    wl = W.config(6)
    outs, err, _ = _plan_apply(wl, path="decode_direct_fp8", repeat=2)
    assert err == 0
    ref, st = oracle_y_e4m3(wl)
    assert st == 0
    for y in outs:
        assert_y_close(y, ref, "plan fp8")


def test_plan_for_another_batch_or_variant_does_nothing_and_reports():
    """A plan used with fewer tokens than it was built for, or for the other
    variant, leaves y unchanged and writes LORA_ERR_INVALID_ARG."""
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import to_host_bits
    wl = W.config(2)
    _, err, (rp, idx, ws, plan) = _plan_apply(wl)
    assert err == 0
    x, y = rp.x[:128], rp.y[:128]
    before = to_host_bits(y).copy()
    idx.err.zero_()
    L.lora_apply_plan(x, y, rp.shape, plan.buf, ws.buf, idx.err, path="decode_direct")
    torch.cuda.synchronize()
    assert int(idx.err.item()) == 1
    np.testing.assert_array_equal(to_host_bits(y), before)
    before = to_host_bits(rp.y).copy()
    idx.err.zero_()
    L.lora_apply_plan(rp.x, rp.y, rp.shape, plan.buf, ws.buf, idx.err, path="decode_direct_fp8")
    torch.cuda.synchronize()
    assert int(idx.err.item()) == 1
    np.testing.assert_array_equal(to_host_bits(rp.y), before)


def test_plans_of_several_layers_in_one_launch():
    """lora_build_plans for three layers with their own weights (one index): each
    layer's call through its plan matches the oracle on its own weights."""
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import ResidentProjection, to_host_bits
    wls = [W.config(2), W.config(2), W.config(2)]
    rng = np.random.default_rng(5)
    for wl in wls[1:]:  # same slots and ranks, other weights
        m = wl.modules[0]
        m.A = [[(W._normal_bf16(rng, a.shape, a.shape[1] ** -0.5) if a is not None else None) for a in row]
               for row in m.A]
        m.B = [[(W._normal_bf16(rng, b.shape, 0.02) if b is not None else None) for b in row] for row in m.B]
    rps = [ResidentProjection.from_workload(wl) for wl in wls]
    idx = L.TokenIndex(wls[0].T, wls[0].S)
    idx.build(torch.from_numpy(wls[0].slot_ids).cuda(), rps[0].table)
    plans = [L.Plan(wls[0].T, rp.shape) for rp in rps]
    L.lora_build_plans(plans, [rp.table for rp in rps], idx)
    ws = L.Workspace(wls[0].T, rps[0].shape)
    for wl, rp, plan in zip(wls, rps, plans):
        plan.apply(rp.x, rp.y, ws, idx.err)
        torch.cuda.synchronize()
        assert int(idx.err.item()) == 0
        ref, _ = oracle_y(wl)
        assert_y_close(to_host_bits(rp.y), ref, "batched plans")


@pytest.mark.parametrize("path", ["decode_direct", "decode_tma"])
@pytest.mark.parametrize("mod_idx", [0, 1], ids=["w1_x_per_token", "w2_x_per_pair"])
def test_apply_moe_with_plan(mod_idx, path):
    """The routed-expert branch through a plan built on the virtual table and the
    pair index (T*K rows)."""
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import ResidentMoeProjection, to_host_bits
    wl = W.moe_config()
    rp = ResidentMoeProjection(wl, mod_idx)
    P = wl.T * wl.K
    idx = L.TokenIndex(P, wl.n_adapters * wl.E)
    idx.build_moe(torch.from_numpy(wl.slot_ids).cuda(), torch.from_numpy(wl.expert_ids.reshape(-1).copy()).cuda(),
                  wl.K, wl.E, rp.table)
    plan = L.Plan(P, rp.shape, path=path)
    plan.build(idx, rp.table)
    ws = L.Workspace(P, rp.shape)
    for _ in range(2):
        L.lora_apply_moe(rp.x, rp.y, wl.K, rp.shape, None, None, None, None, ws.buf, idx.err,
                         x_per_token=rp.x_per_token, plan=plan)
    torch.cuda.synchronize()
    assert int(idx.err.item()) == 0
    m = wl.modules[mod_idx]
    scales = oracle.slot_scales(wl.ranks, wl.alphas, wl.scale_rule, False)
    # two calls: y_in + 2 * branch
    once, st = oracle.apply_moe(m.x, m.x_per_token, m.y_in, m.slice_widths, wl.slot_ids, wl.expert_ids, wl.E,
                                wl.ranks, scales, m.A, m.B)
    assert st == 0
    ref = 2 * once - W.bf16_bits_to_f32(m.y_in).astype(np.float64)
    assert_y_close(to_host_bits(rp.y), ref, f"moe plan {mod_idx} {path}")


def test_plan_for_other_slice_widths_does_nothing_and_reports():
    """A plan used with a shape of other slice widths (its offsets would place y
    writes elsewhere) is refused on the device: y unchanged, LORA_ERR_INVALID_ARG."""
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import to_host_bits
    wl = W.config(2)
    _, err, (rp, idx, ws, plan) = _plan_apply(wl)
    assert err == 0
    other = L.make_shape(wl.S, wl.r_max, 4096, [4096, 1024, 512])
    y = rp.y[:, :5632]
    before = to_host_bits(rp.y).copy()
    idx.err.zero_()
    L.lora_apply_plan(rp.x, y, other, plan.buf, ws.buf, idx.err, path="decode_direct")
    torch.cuda.synchronize()
    assert int(idx.err.item()) == 1
    np.testing.assert_array_equal(to_host_bits(rp.y), before)


# ---------------------------------------------------------------------------
# The one-kernel TMA decode path
# ---------------------------------------------------------------------------
# k a multiple of 64 with ragged slice widths (not multiples of 64), ranks of
# every multiple of 8 up to 64, slots with one token and slots with several
# token groups (more than 64 or 128 tokens), four slices, T = 1 and T = 2048.
TMA_RAGGED = [
    # seed, T, k, widths, S, ranks
    (41, 33, 64, [8, 24], 5, [8, 24, 0, 64, 8]),
    (42, 1, 64, [8], 1, [8]),
    (43, 300, 1024, [1000], 2, [64, 8]),
    (44, 129, 512, [512, 16, 8, 24], 7, [8, 16, 24, 32, 40, 48, 8]),
    (45, 700, 4096, [4096, 1024, 1024], 3, [64, 64, 32]),
    (46, 2048, 2048, [136, 520], 4, [16, 8, 64, 40]),
    (47, 90, 128, [72, 8, 528], 5, [16, 56, 40, 0, 24]),
    (48, 200, 192, [200], 9, [8, 8, 16, 32, 64, 56, 8, 16, 24]),
]


@pytest.mark.parametrize("case", [TMA_RAGGED[0], TMA_RAGGED[3], TMA_RAGGED[4], TMA_RAGGED[6]],
                         ids=lambda c: f"tma{c[0]}")
def test_tma_separate_a_slices(case):
    """A slot whose A slices are separate allocations (not one packed [n r][k]
    block) is copied slice by slice: same results as the oracle."""
    seed, T, k, widths, S, ranks = case
    wl = _small(seed, T, k, widths, S, ranks)
    outs, err, *_ = gpu_apply(wl, path="decode_tma", repeat=2, pack_a=False)
    assert err == 0
    ref, _ = oracle_y(wl)
    for y in outs:
        assert_y_close(y, ref, f"tma unpacked {seed}")


def test_tma_separate_a_slices_packed_qkv():
    """The packed QKV decode batch with every slot's A slices allocated apart."""
    wl = W.config(2)
    outs, err, *_ = gpu_apply(wl, path="decode_tma", repeat=2, pack_a=False)
    assert err == 0
    ref, _ = oracle_y(wl)
    for y in outs:
        assert_y_close(y, ref, "tma unpacked qkv")


@pytest.mark.parametrize("plan", [False, True], ids=["apply_ex", "plan"])
@pytest.mark.parametrize("case", TMA_RAGGED, ids=[f"tma{c[0]}" for c in TMA_RAGGED])
def test_tma_ragged(case, plan):
    seed, T, k, widths, S, ranks = case
    wl = _small(seed, T, k, widths, S, ranks)
    assert tma_ok(wl)
    if plan:
        outs, err, _ = _plan_apply(wl, path="decode_tma", repeat=2)
    else:
        outs, err, *_ = gpu_apply(wl, path="decode_tma", repeat=2)
    assert err == 0
    ref, _ = oracle_y(wl)
    keep = untouched_rows(wl)
    for y in outs:
        assert_y_close(y, ref, f"tma ragged {seed}")
        np.testing.assert_array_equal(y[keep], wl.modules[0].y_in[keep])


def test_tma_layer_plans_in_one_launch():
    """Plans of three layers (own weights, one index) in one launch; each layer's
    call through its plan matches the oracle, the calls back to back on one
    workspace (each call's kernel may start before the previous one ends)."""
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import ResidentProjection, to_host_bits
    wls = [W.config(2), W.config(2), W.config(2)]
    rng = np.random.default_rng(15)
    for wl in wls[1:]:
        m = wl.modules[0]
        m.A = [[(W._normal_bf16(rng, a.shape, a.shape[1] ** -0.5) if a is not None else None) for a in row]
               for row in m.A]
        m.B = [[(W._normal_bf16(rng, b.shape, 0.02) if b is not None else None) for b in row] for row in m.B]
    rps = [ResidentProjection.from_workload(wl) for wl in wls]
    idx = L.TokenIndex(wls[0].T, wls[0].S)
    idx.build(torch.from_numpy(wls[0].slot_ids).cuda(), rps[0].table)
    plans = [L.Plan(wls[0].T, rp.shape, "decode_tma") for rp in rps]
    L.lora_build_plans(plans, [rp.table for rp in rps], idx)
    ws = L.Workspace(wls[0].T, rps[0].shape)
    for rp, plan in zip(rps, plans):
        plan.apply(rp.x, rp.y, ws, idx.err)
    torch.cuda.synchronize()
    assert int(idx.err.item()) == 0
    for wl, rp in zip(wls, rps):
        ref, _ = oracle_y(wl)
        assert_y_close(to_host_bits(rp.y), ref, "tma layer plans")


def _tma_regions(L, T, shape):
    """Float offsets of the TMA path's two sum sets and its control block (the
    regions after the two-kernel decode paths' accumulators)."""
    n, r_max, S = shape.n_slices, shape.r_max, shape.S
    rp = 16 if r_max <= 16 else (32 if r_max <= 32 else 64)  # the prefill path's rank padding
    region = (n * T * r_max + 63) // 64 * 64
    hl_region = (n * T * rp * 2 // 4 + 63) // 64 * 64
    xa_off = L.lora_workspace_xa_offset(shape) // 4
    tacc0 = xa_off + region + region + 2 * hl_region + 2 * region
    return tacc0, tacc0 + region, tacc0 + 2 * region, n * T * r_max


def test_tma_leaves_workspace_ready():
    """Call g adds into sum set g & 1, clears set (g + 1) & 1 and advances the
    call counter (the word after the 2 S per-slot counters): after every call the
    set the next call adds into and its counters are zero."""
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import ResidentProjection, to_host_bits
    wl = W.config(2)
    rp = ResidentProjection.from_workload(wl)
    idx = L.TokenIndex(wl.T, wl.S)
    idx.build(torch.from_numpy(wl.slot_ids).cuda(), rp.table)
    ws = L.Workspace(wl.T, rp.shape)
    ref, _ = oracle_y(wl)
    y0 = rp.y.clone()
    tacc0, tacc1, tctrl, nfl = _tma_regions(L, wl.T, rp.shape)
    S = wl.S
    for call in range(1, 5):
        rp.y.copy_(y0)
        L.lora_apply(rp.x, rp.y, rp.shape, rp.table.dev, idx.sorted_ids, idx.seg_offsets, idx.active, ws.buf,
                     idx.err, path="decode_tma")
        torch.cuda.synchronize()
        assert int(idx.err.item()) == 0
        assert_y_close(to_host_bits(rp.y), ref, "tma")
        buf = ws.buf.cpu().numpy()
        ctrl = buf[tctrl:tctrl + 2 * S + 2].view(np.int32)
        assert ctrl[2 * S] == call, "call counter not advanced"
        assert ctrl[2 * S + 1] == 0, "exit counter not reset"
        nxt = call & 1
        assert not ctrl[nxt * S:(nxt + 1) * S].any(), "next counters not cleared"
        base = tacc1 if nxt else tacc0
        assert not buf[base:base + nfl].any(), "next sum set not cleared"


def test_tma_slot_wait_timeout_reports_error_and_device_stays_usable():
    """Per-slot counters that can never reach their targets (a poisoned
    workspace) make the expand's bounded wait give up: LORA_ERR_TIMEOUT in the
    error word, the affected y rows unchanged, and a call on a clean workspace
    afterwards is correct."""
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import ResidentProjection, to_host_bits
    wl = W.config(0)
    rp = ResidentProjection.from_workload(wl)
    idx = L.TokenIndex(wl.T, wl.S)
    idx.build(torch.from_numpy(wl.slot_ids).cuda(), rp.table)
    ws = L.Workspace(wl.T, rp.shape)
    y0 = rp.y.clone()
    tacc0, tacc1, tctrl, nfl = _tma_regions(L, wl.T, rp.shape)
    ws.buf[tctrl:tctrl + wl.S].view(torch.int32).fill_(-(1 << 30))  # call 0 counts into set 0
    L.lora_apply(rp.x, rp.y, rp.shape, rp.table.dev, idx.sorted_ids, idx.seg_offsets, idx.active, ws.buf,
                 idx.err, path="decode_tma")
    torch.cuda.synchronize()
    assert int(idx.err.item()) == 7  # LORA_ERR_TIMEOUT
    np.testing.assert_array_equal(to_host_bits(rp.y), to_host_bits(y0))
    ws.buf.zero_()
    idx.err.zero_()
    rp.y.copy_(y0)
    L.lora_apply(rp.x, rp.y, rp.shape, rp.table.dev, idx.sorted_ids, idx.seg_offsets, idx.active, ws.buf,
                 idx.err, path="decode_tma")
    torch.cuda.synchronize()
    assert int(idx.err.item()) == 0
    ref, _ = oracle_y(wl)
    assert_y_close(to_host_bits(rp.y), ref, "tma after a timed-out call")


def test_tma_refuses_a_table_without_maps_and_a_foreign_plan():
    """A table set without tensor maps, or a plan built for another T or for the
    warp-streaming kernels: LORA_ERR_INVALID_ARG in err, y unchanged."""
    torch = _torch()
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import ResidentProjection, to_host_bits
    wl = W.config(2)
    rp = ResidentProjection.from_workload(wl)
    plain = L.SlotTable(wl.S, rp.n, wl.r_max)
    plain.set(rp.ranks, rp.scales, *rp._ptrs)
    idx = L.TokenIndex(wl.T, wl.S)
    idx.build(torch.from_numpy(wl.slot_ids).cuda(), rp.table)
    ws = L.Workspace(wl.T, rp.shape)
    before = to_host_bits(rp.y).copy()
    L.lora_apply(rp.x, rp.y, rp.shape, plain.dev, idx.sorted_ids, idx.seg_offsets, idx.active, ws.buf, idx.err,
                 path="decode_tma")
    torch.cuda.synchronize()
    assert int(idx.err.item()) == 1
    np.testing.assert_array_equal(to_host_bits(rp.y), before)
    for path in ("decode_direct", "decode_tma"):
        plan = L.Plan(wl.T, rp.shape, path)
        plan.build(idx, rp.table)
        idx.err.zero_()
        x, y = (rp.x[:128], rp.y[:128]) if path == "decode_tma" else (rp.x, rp.y)
        L.lora_apply_plan(x, y, rp.shape, plan.buf, ws.buf, idx.err, path="decode_tma")
        torch.cuda.synchronize()
        assert int(idx.err.item()) == 1
        np.testing.assert_array_equal(to_host_bits(rp.y), before)
