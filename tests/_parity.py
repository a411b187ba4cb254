"""Helpers shared by the GPU parity tests: run the CUDA path and the oracle on
the same seeded inputs and compare them element by element."""
from __future__ import annotations

import numpy as np

import oracle
import workloads as W

# tolerance for bf16 y with fp32 accumulation: |gpu - ref| <= ATOL + RTOL |ref|,
# ref = the fp64 oracle value before rounding to bf16
ATOL = 1e-2
RTOL = 2e-2


def oracle_y(wl, mod_idx=0, rows=None, y_in="module"):
    """fp64 reference rows of projection mod_idx (pre-multiplied B handled as the pages say)."""
    m = wl.modules[mod_idx]
    rule = oracle.slot_scales(wl.ranks, wl.alphas, wl.scale_rule, False)
    if wl.premultiplied:
        scales = np.ones(wl.S)
        B = [[(oracle.premultiply(b, rule[s]) if b is not None else None) for b in row]
             for s, row in enumerate(m.B)]
    else:
        scales = rule
        B = m.B
    yi = m.y_in if isinstance(y_in, str) else y_in
    y, macs, st = oracle.apply(m.x, yi, m.slice_widths, wl.slot_ids, wl.ranks, scales, m.A, B, rows=rows)
    return y, st


def oracle_y_e4m3(wl, mod_idx=0, rows=None):
    """fp64 reference rows for FP8 adapters (A, B e4m3 codes; x rounded to e4m3),
    a pre-multiplied B scaled in bf16 and clamped back to e4m3 as the pages say."""
    m = wl.modules[mod_idx]
    rule = oracle.slot_scales(wl.ranks, wl.alphas, wl.scale_rule, False)
    if wl.premultiplied:
        scales = np.ones(wl.S)
        B = [[(oracle.premultiply_e4m3(b, rule[s]) if b is not None else None) for b in row]
             for s, row in enumerate(m.B)]
    else:
        scales = rule
        B = m.B
    return oracle.apply_e4m3(m.x, m.y_in, m.slice_widths, wl.slot_ids, wl.ranks, scales, m.A, B, rows=rows)


def cluster_ok(wl, mod_idx=0):
    """Shapes the one-cluster-per-slot decode path takes: k and every slice offset
    multiples of 8, r_max <= 256, and a CTA's tiles (A and x over 1/16 of k, the
    partial and sums tiles, B and y over 1/16 of the columns) within 227 KB."""
    m = wl.modules[mod_idx]
    k, widths, n = m.k, list(m.slice_widths), len(m.slice_widths)
    offs = np.concatenate([[0], np.cumsum(widths)])
    if k % 8 or any(int(o) % 8 for o in offs) or wl.r_max > 256:
        return False
    rp8, rp16 = -(-wl.r_max // 8) * 8, -(-wl.r_max // 16) * 16
    for ks in (16,):
        kcw = -(-(k // 8) // ks) * 8
        ars = -(-kcw // 16) * 16 + 8
        ncol = sum(-(-(-(-w // ks)) // 8) * 8 for w in widths)
        srs, yrs = n * rp16 + 8, ncol + 8
        size = (n * rp8 * ars * 2 + 16 * ars * 2 + 16 * n * rp8 * 4 + 2 * 16 * srs * 2 + ncol * (rp16 + 8) * 2
                + 16 * yrs * 2 + 16 * 4)
        if size <= 227 * 1024:
            return True
    return False


def gpu_apply(wl, mod_idx=0, path="auto", max_seg_hint=0, repeat=1, pack_a=True):
    import torch
    import rank_adapter_gemm_gb300 as L
    from rank_adapter_gemm_gb300.resident import ResidentProjection, to_host_bits
    rp = ResidentProjection.from_workload(wl, mod_idx, pack_a=pack_a)
    slot_dev = torch.from_numpy(np.ascontiguousarray(wl.slot_ids, dtype=np.int32)).cuda()
    idx = L.TokenIndex(wl.T, wl.S)
    idx.build(slot_dev, rp.table)
    ws = L.Workspace(wl.T, rp.shape)
    y0 = rp.y.clone()
    outs = []
    for _ in range(repeat):
        rp.y.copy_(y0)
        L.lora_apply(rp.x, rp.y, rp.shape, rp.table.dev, idx.sorted_ids, idx.seg_offsets, idx.active, ws.buf,
                     idx.err, max_seg_hint=max_seg_hint, path=path)
        torch.cuda.synchronize()
        outs.append(to_host_bits(rp.y))
    err = int(idx.err.cpu().item())
    return outs if repeat > 1 else outs[0], err, idx, rp, ws


def untouched_rows(wl):
    s = wl.slot_ids
    bad = (s < 0) | (s >= wl.S)
    rank0 = np.zeros_like(bad)
    ok = ~bad
    rank0[ok] = wl.ranks[s[ok]] == 0
    return bad | rank0


def assert_y_close(y_gpu_bits, y_ref, what=""):
    g = W.bf16_bits_to_f32(y_gpu_bits).astype(np.float64)
    diff = np.abs(g - y_ref)
    tol = ATOL + RTOL * np.abs(y_ref)
    bad = diff > tol
    if bad.any():
        idx = np.unravel_index(np.argmax(diff - tol), diff.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements outside tolerance; worst at {idx}: "
                             f"gpu {g[idx]!r} ref {y_ref[idx]!r}")
    return float(diff.max()) if diff.size else 0.0
