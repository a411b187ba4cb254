"""Put one packed projection's adapters, activations and slot table on the device.

Marshalling only: numpy bf16 bit patterns become torch bf16 device tensors
(numpy uint8 float8_e4m3fn codes become torch uint8 tensors), per-slot scales
come from the library's lora_scale, a pre-multiplied scale is folded into B by
the library's lora_premultiply (or lora_premultiply_e4m3) kernel, and the
pointer table is uploaded with lora_set_slot_table.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np

from . import SlotTable, lora_premultiply, lora_premultiply_e4m3, lora_scale, make_shape


def _to_dev(bits: np.ndarray, device):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def _w_to_dev(w: np.ndarray, device):
    """A weight matrix: bf16 bits (uint16) or e4m3 codes (uint8, kept as bytes)."""
    if w.dtype == np.uint8:
        import torch
        return torch.from_numpy(np.ascontiguousarray(w)).to(device)
    return _to_dev(w, device)


class ResidentProjection:
    """Adapter weights of S slots for one projection plus its x and y rows.

    A[s][i] is [r_s, k], B[s][i] is [d_i, r_s] (bf16 bit patterns, or uint8
    float8_e4m3fn codes for every matrix: then ``fp8`` is True and the table
    serves the FP8 path); rank-0 slots have None.  ``scale_rule`` is "alpha_over_r" or "alpha_over_sqrt_r";
    with ``premultiplied`` the rule's scale is folded into B and the table
    carries scale 1.  With ``pack_a`` (the default) a slot's A slices are views
    of one [n, r_s, k] block, the layout the one-kernel TMA path copies with a
    single tensor-map copy per stage.
    """

    def __init__(self, *, S: int, r_max: int, ranks: Sequence[int], alphas: Sequence[float], scale_rule: str,
                 premultiplied: bool, k: int, slice_widths: Sequence[int],
                 A: Sequence[Sequence[Optional[np.ndarray]]], B: Sequence[Sequence[Optional[np.ndarray]]],
                 x: Optional[np.ndarray] = None, y_in: Optional[np.ndarray] = None, device="cuda",
                 pack_a: bool = True):
        self.S, self.r_max, self.k = int(S), int(r_max), int(k)
        self.slice_widths = [int(w) for w in slice_widths]
        self.n = len(self.slice_widths)
        self.d = sum(self.slice_widths)
        self.ranks = np.asarray(ranks, dtype=np.int32)
        rslora = scale_rule == "alpha_over_sqrt_r"
        rule_scales = np.array([lora_scale(alphas[s], int(self.ranks[s]), rslora) for s in range(S)])
        self.A: List[List] = []
        self.B: List[List] = []
        a_ptrs = np.zeros(S * self.n, dtype=np.uint64)
        b_ptrs = np.zeros(S * self.n, dtype=np.uint64)
        mats = [m for row in A for m in row if m is not None]
        self.fp8 = bool(mats) and mats[0].dtype == np.uint8
        premul = lora_premultiply_e4m3 if self.fp8 else lora_premultiply
        self.pack_a = pack_a
        for s in range(S):
            rowA, rowB = [], []
            packed = (_w_to_dev(np.stack([np.asarray(A[s][i]) for i in range(self.n)]), device)
                      if pack_a and self.ranks[s] > 0 else None)
            for i in range(self.n):
                if self.ranks[s] > 0:
                    ta = packed[i] if packed is not None else _w_to_dev(A[s][i], device)
                    tb = _w_to_dev(B[s][i], device)
                    if premultiplied:
                        premul(tb, float(rule_scales[s]))
                    a_ptrs[s * self.n + i] = ta.data_ptr()
                    b_ptrs[s * self.n + i] = tb.data_ptr()
                else:
                    ta = tb = None
                rowA.append(ta)
                rowB.append(tb)
            self.A.append(rowA)
            self.B.append(rowB)
        self.scales = np.ones(S, dtype=np.float32) if premultiplied else rule_scales.astype(np.float32)
        self.shape = make_shape(S, r_max, k, self.slice_widths)
        self.table = SlotTable(S, self.n, r_max, device=device, shape=self._table_shape())
        self.table.set(self.ranks, self.scales, a_ptrs, b_ptrs)
        self._ptrs = (a_ptrs, b_ptrs)
        self.x = _to_dev(x, device) if x is not None else None
        self.y = _to_dev(y_in, device) if y_in is not None else None

    def clone(self, device="cuda") -> "ResidentProjection":
        """Same values in fresh device buffers (weights, rows and slot table)."""
        import copy
        other = copy.copy(self)
        n = self.n
        a_ptrs = np.zeros(self.S * n, dtype=np.uint64)
        b_ptrs = np.zeros(self.S * n, dtype=np.uint64)
        import torch

        def clone_row(row):
            if row and row[0] is not None and self.pack_a:
                block = torch.stack(row)  # a fresh [n, r, k] block
                return [block[i] for i in range(len(row))]
            return [(t.clone() if t is not None else None) for t in row]
        other.A = [clone_row(row) for row in self.A]
        other.B = [[(t.clone() if t is not None else None) for t in row] for row in self.B]
        for s in range(self.S):
            for i in range(n):
                if other.A[s][i] is not None:
                    a_ptrs[s * n + i] = other.A[s][i].data_ptr()
                    b_ptrs[s * n + i] = other.B[s][i].data_ptr()
        other.table = SlotTable(self.S, n, self.r_max, device=device, shape=self._table_shape())
        other.table.set(self.ranks, self.scales, a_ptrs, b_ptrs)
        other._ptrs = (a_ptrs, b_ptrs)
        other.x = self.x.clone() if self.x is not None else None
        other.y = self.y.clone() if self.y is not None else None
        return other

    def _table_shape(self):
        """bf16 adapters of a shape the one-kernel TMA path takes (r_max <= 64,
        n_slices * r_max <= 192, k % 64 == 0) get the table with tensor maps."""
        tma = not self.fp8 and self.r_max <= 64 and self.n * self.r_max <= 192 and self.k % 64 == 0
        return self.shape if tma else None

    def refresh_table(self, stream=None) -> None:
        """Re-upload the slot table (what a change of slot ownership costs)."""
        self.table.set(self.ranks, self.scales, *self._ptrs, stream=stream)

    @classmethod
    def from_workload(cls, wl, module_index: int = 0, device="cuda", with_rows: bool = True, pack_a: bool = True):
        m = wl.modules[module_index]
        return cls(S=wl.S, r_max=wl.r_max, ranks=wl.ranks, alphas=wl.alphas, scale_rule=wl.scale_rule,
                   premultiplied=wl.premultiplied, k=m.k, slice_widths=m.slice_widths, A=m.A, B=m.B,
                   x=m.x if with_rows else None, y_in=m.y_in if with_rows else None, device=device, pack_a=pack_a)


def to_device_bf16(bits: np.ndarray, device="cuda"):
    """uint16 bf16 bit patterns -> torch bf16 tensor on the device."""
    return _to_dev(bits, device)


def to_host_bits(t) -> np.ndarray:
    """torch bf16 tensor -> numpy uint16 bit patterns."""
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


class ResidentMoeProjection:
    """One routed-expert projection on the device: each adapter's A [E, r, k] and
    B [E, d_i, r] as one bf16 tensor per slice, the virtual slot table of
    n_adapters * E slots (lora_moe_slot_pointers + lora_set_slot_table), x and
    the per-pair y rows."""

    def __init__(self, wl, module_index: int = 0, device="cuda"):
        from . import lora_moe_slot_pointers
        m = wl.modules[module_index]
        self.K, self.E, self.n_adapters = wl.K, wl.E, wl.n_adapters
        self.x_per_token = m.x_per_token
        self.slice_widths = list(m.slice_widths)
        n = len(self.slice_widths)
        rslora = wl.scale_rule == "alpha_over_sqrt_r"
        scales = np.array([lora_scale(wl.alphas[s], int(wl.ranks[s]), rslora) for s in range(wl.n_adapters)],
                          dtype=np.float32)
        self.A = [[_to_dev(a.reshape(-1), device) for a in row] for row in m.A]
        self.B = [[_to_dev(b.reshape(-1), device) for b in row] for row in m.B]
        a_base = np.array([t.data_ptr() for row in self.A for t in row], dtype=np.uint64)
        b_base = np.array([t.data_ptr() for row in self.B for t in row], dtype=np.uint64)
        V = wl.n_adapters * wl.E
        self.shape = make_shape(V, wl.r_max, m.k, self.slice_widths)
        v_ranks, v_scales, a_ptrs, b_ptrs = lora_moe_slot_pointers(wl.n_adapters, wl.E, self.shape, wl.ranks, scales,
                                                                   a_base, b_base)
        self.ranks, self.scales = np.asarray(wl.ranks, np.int32), scales
        self.table = SlotTable(V, n, wl.r_max, device=device, shape=self._table_shape())
        self.table.set(v_ranks, v_scales, a_ptrs, b_ptrs)
        self.x = _to_dev(m.x, device)
        self.y = _to_dev(m.y_in, device)

    def _table_shape(self):
        """Shapes the one-kernel TMA path takes (r_max <= 64, n_slices * r_max <= 192,
        k % 64 == 0) get the virtual table with tensor maps."""
        tma = (self.shape.r_max <= 64 and self.shape.n_slices * self.shape.r_max <= 192
               and self.shape.k % 64 == 0)
        return self.shape if tma else None


def clone_moe(rp: ResidentMoeProjection, device="cuda") -> ResidentMoeProjection:
    """Same values in fresh device buffers (weights, rows and virtual slot table)."""
    import copy
    from . import lora_moe_slot_pointers
    other = copy.copy(rp)
    other.A = [[t.clone() for t in row] for row in rp.A]
    other.B = [[t.clone() for t in row] for row in rp.B]
    a_base = np.array([t.data_ptr() for row in other.A for t in row], dtype=np.uint64)
    b_base = np.array([t.data_ptr() for row in other.B for t in row], dtype=np.uint64)
    v_ranks, v_scales, a_ptrs, b_ptrs = lora_moe_slot_pointers(rp.n_adapters, rp.E, rp.shape, rp.ranks, rp.scales,
                                                               a_base, b_base)
    other.table = SlotTable(rp.table.S, rp.table.n_slices, rp.table.r_max, device=device, shape=rp._table_shape())
    other.table.set(v_ranks, v_scales, a_ptrs, b_ptrs)
    other.x = rp.x.clone()
    other.y = rp.y.clone()
    return other
