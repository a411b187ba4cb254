"""Pins for the CPU oracle: checks against what the pages and mathematics fix.

None of these re-types the oracle's formula.  Each compares it with something
else: numpy's fp64 matmul (a library routine), the merged-weight identity,
closed forms, values the pages print (tests/golden/), or brute force over all
permutations of tiny inputs.  Chosen so that a dropped term, a wrong sign or
index, or a transposed operand in the oracle fails at least one of them
(tests/test_oracle_mutants.py plants such mistakes and checks that they do).
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def _small_workload(seed=7, T=40, k=48, widths=(32, 16, 24), S=5, ranks=(8, 16, 0, 24, 8),
                    frac_none=0.15, y_init="normal"):
    wl = W.generate(name="pin", seed=seed, T=T, S=S, rank=8,
                    modules=[{"name": "m", "k": k, "slices": list(widths)}],
                    slot_dist="uniform", frac_none=frac_none, alpha=16.0, y_init=y_init)
    # re-draw weights for the requested ranks (per-slot ranks), same generator rules
    rng = np.random.Generator(np.random.PCG64(seed + 100))
    mod = wl.modules[0]
    wl.ranks = np.asarray(ranks, dtype=np.int32)
    mod.A = [[(W.f32_to_bf16_bits(rng.standard_normal((r, k), dtype=np.float32) / np.float32(math.sqrt(k)))
               if r > 0 else None) for _ in widths] for r in ranks]
    mod.B = [[(W.f32_to_bf16_bits(0.02 * rng.standard_normal((w, r), dtype=np.float32)) if r > 0 else None)
              for w in widths] for r in ranks]
    wl.r_max = max(ranks)
    return wl


def _run(wl, scales, y_in="module", rows=None):
    mod = wl.modules[0]
    yi = mod.y_in if isinstance(y_in, str) else y_in
    return oracle.apply(mod.x, yi, mod.slice_widths, wl.slot_ids, wl.ranks, scales, mod.A, mod.B, rows=rows)


# ---------------------------------------------------------------------------
# Index
# ---------------------------------------------------------------------------
def _brute_force_sorted(slot_ids, S):
    """The unique permutation whose (key, token) sequence is strictly increasing,
    found by searching all permutations (TensorRT-LLM LoRA serving page, step 2:
    rows of one slot made contiguous; ties kept in request order)."""
    T = len(slot_ids)
    key = [s if 0 <= s < S else S for s in slot_ids]
    hits = []
    for perm in itertools.permutations(range(T)):
        seq = [(key[p], p) for p in perm]
        if all(seq[q] < seq[q + 1] for q in range(T - 1)):
            hits.append(list(perm))
    assert len(hits) == 1
    return hits[0], key


@pytest.mark.parametrize("ranks", [(8, 8), (0, 16)])
def test_index_brute_force_all_tiny_inputs(ranks):
    S = 2
    alphabet = (-1, 0, 1, 2, -3)   # 2 and -3 are outside [-1, S)
    for T in range(0, 5):
        for ids in itertools.product(alphabet, repeat=T):
            ids = np.array(ids, dtype=np.int32)
            sorted_ids, seg, active, st = oracle.build_index(ids, S, np.array(ranks, np.int32))
            perm, key = _brute_force_sorted(list(ids), S)
            assert list(sorted_ids) == perm
            skeys = np.sort(np.array(key, dtype=np.int64))
            assert list(seg) == [int(np.searchsorted(skeys, b, side="left")) for b in range(S + 2)]
            present = {k for k in key if k < S}
            want = sorted(s for s in present if ranks[s] > 0)
            assert active[0] == len(want) and list(active[1:1 + len(want)]) == want
            bad = any(not (-1 <= s < S) for s in ids)
            assert st == (oracle.ERR_SLOT_RANGE if bad else oracle.ERR_OK)


@pytest.mark.parametrize("seed", range(6))
def test_index_matches_library_stable_sort(seed):
    rng = np.random.default_rng(seed)
    S = int(rng.integers(1, 300))
    T = int(rng.integers(0, 6000))
    ids = rng.integers(-1, S, size=T).astype(np.int32)
    ranks = rng.choice([0, 8, 16, 64], size=S).astype(np.int32)
    sorted_ids, seg, active, st = oracle.build_index(ids, S, ranks)
    key = np.where(ids < 0, S, ids)
    assert st == oracle.ERR_OK
    np.testing.assert_array_equal(sorted_ids, np.argsort(key, kind="stable"))
    counts = np.bincount(key, minlength=S + 1)
    np.testing.assert_array_equal(seg, np.concatenate([[0], np.cumsum(counts)]))
    want = [s for s in range(S) if counts[s] > 0 and ranks[s] > 0]
    assert active[0] == len(want)
    np.testing.assert_array_equal(active[1:1 + len(want)], want)


def test_index_layout_matches_pages():
    rows = {r[0]: r for r in _golden("index_layout.txt")}
    for S, T in [(1, 0), (8, 64), (32, 256), (128, 1024)]:
        ids = np.random.default_rng(S).integers(-1, S, size=T).astype(np.int32)
        _, seg, active, _ = oracle.build_index(ids, S, np.full(S, 16, np.int32))
        assert rows["seg_offsets"][1] == "S+2" and len(seg) == S + 2
        assert seg[0] == 0 and seg[-1] == T
        assert rows["active"][1] == "S+1" and len(active) == S + 1


@pytest.mark.parametrize("seed,tps", [(0, 1), (1, 2), (2, 4), (3, 5), (4, 8)])
def test_speculative_index_matches_pages_expansion(seed, tps):
    """TensorRT-LLM LoRA serving page, "一次 decode 批次的路由": with tokens_per_seq
    > 1 the sequence-level order is expanded to tokens as sorted * tps +
    arange(tps), and the per-slot counts scale by tps.  The oracle's speculative
    index (the token index of the repeated slot ids) must equal that expansion of
    its sequence-level index."""
    rng = np.random.default_rng(100 + seed)
    S = int(rng.integers(1, 40))
    n_seq = int(rng.integers(0, 300))
    seq = rng.integers(-1, S, size=n_seq).astype(np.int32)
    ranks = rng.choice([0, 8, 16, 64], size=S).astype(np.int32)
    so_s, seg_s, act_s, st_s = oracle.build_index(seq, S, ranks)
    so_t, seg_t, act_t, st_t = oracle.build_index_seq(seq, tps, S, ranks)
    assert st_s == st_t == oracle.ERR_OK
    want = (so_s.astype(np.int64)[:, None] * tps + np.arange(tps)).ravel()
    np.testing.assert_array_equal(so_t, want)
    np.testing.assert_array_equal(seg_t, seg_s * tps)
    np.testing.assert_array_equal(act_t, act_s)


def test_speculative_index_one_token_per_sequence_is_the_token_index():
    rng = np.random.default_rng(7)
    ids = rng.integers(-1, 16, size=500).astype(np.int32)
    ranks = np.full(16, 8, np.int32)
    for a, b in zip(oracle.build_index(ids, 16, ranks), oracle.build_index_seq(ids, 1, 16, ranks)):
        np.testing.assert_array_equal(a, b)


# ---------------------------------------------------------------------------
# Branch value
# ---------------------------------------------------------------------------
def test_branch_matches_library_matmul():
    """Per slot, y = y_in + s * (X_s A^T) B^T with numpy's fp64 matmul (vLLM book
    ch. 16, §16.1.3: Y = xW + s (xA)B in row-vector form)."""
    wl = _small_workload()
    mod = wl.modules[0]
    scales = np.array([2.0, 0.5, 3.0, 1.25, -1.5])
    y, _, st = _run(wl, scales)
    assert st == oracle.ERR_OK
    X = _f64(mod.x)
    want = _f64(mod.y_in).copy()
    offs = mod.slice_offsets
    for s in range(wl.S):
        rows = np.nonzero(wl.slot_ids == s)[0]
        if len(rows) == 0 or wl.ranks[s] == 0:
            continue
        for i in range(mod.n_slices):
            A = _f64(mod.A[s][i])
            B = _f64(mod.B[s][i])
            want[np.ix_(rows, range(offs[i], offs[i + 1]))] += scales[s] * ((X[rows] @ A.T) @ B.T)
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)


def test_shrink_matches_library_matmul():
    wl = _small_workload(seed=11)
    mod = wl.modules[0]
    xa, macs = oracle.shrink(mod.x, wl.slot_ids, wl.ranks, mod.A, wl.r_max)
    X = _f64(mod.x)
    n_checked = 0
    for t in range(wl.T):
        s = wl.slot_ids[t]
        if s < 0 or wl.ranks[s] == 0:
            assert np.all(np.isnan(xa[t]))
            continue
        for i in range(mod.n_slices):
            np.testing.assert_allclose(xa[t, i, :wl.ranks[s]], _f64(mod.A[s][i]) @ X[t], rtol=1e-12, atol=1e-13)
            n_checked += 1
    assert n_checked > 0
    lora_tokens = [t for t in range(wl.T) if wl.slot_ids[t] >= 0 and wl.ranks[wl.slot_ids[t]] > 0]
    assert macs == sum(int(wl.ranks[wl.slot_ids[t]]) * mod.n_slices * mod.k for t in lora_tokens)


def test_merged_weight_identity():
    """x (W0 + s B A)^T == x W0^T + branch: the branch need not be merged
    (llama.cpp LoRA adapter page, §"为什么低秩增量可以「后加」"; export-lora merges
    delta = scale * B A into the base)."""
    wl = _small_workload(seed=3, frac_none=0.0)
    mod = wl.modules[0]
    rng = np.random.default_rng(5)
    W0 = rng.standard_normal((mod.d, mod.k))
    scales = np.array([2.0, 0.25, 1.0, 4.0, 0.5])
    branch, _, _ = _run(wl, scales, y_in=None)
    X = _f64(mod.x)
    offs = mod.slice_offsets
    for t in range(wl.T):
        s = wl.slot_ids[t]
        Wm = W0.copy()
        if wl.ranks[s] > 0:
            for i in range(mod.n_slices):
                Wm[offs[i]:offs[i + 1]] += scales[s] * (_f64(mod.B[s][i]) @ _f64(mod.A[s][i]))
        merged = Wm @ X[t]
        unmerged = W0 @ X[t] + branch[t]
        np.testing.assert_allclose(unmerged, merged, rtol=1e-11, atol=1e-11)


def test_orientation_matches_printed_shapes():
    """lora_a is (r, k) and lora_b is (d, r), as printed for q_proj."""
    (mod_name, k, d, r, ar, ac, br, bc), = _golden("adapter_shapes.txt")
    k, d, r, ar, ac, br, bc = map(int, (k, d, r, ar, ac, br, bc))
    assert (ar, ac, br, bc) == (r, k, d, r)
    # a one-token, one-slot check at those shapes, reduced to a closed form:
    # A = first r rows of the identity, B = first r columns of the identity
    x = W.f32_to_bf16_bits(np.random.default_rng(0).standard_normal((1, k), dtype=np.float32))
    A = np.zeros((ar, ac), np.uint16)
    B = np.zeros((br, bc), np.uint16)
    one = oracle.round_bf16(1.0)
    for j in range(r):
        A[j, j] = one
        B[j, j] = one
    y, _, _ = oracle.apply(x, None, [d], np.array([0], np.int32), np.array([r], np.int32),
                           np.array([1.0]), [[A]], [[B]])
    want = np.zeros(d)
    want[:r] = _f64(x[0, :r])
    np.testing.assert_array_equal(y[0], want)


def test_closed_form_one_hot_rank1():
    """Rank-1 one-hot adapter: A picks input column c, B writes output column m,
    so the branch adds exactly s * x[t, c] at y[t, m] and nothing elsewhere."""
    T, k, d = 6, 40, 24
    rng = np.random.default_rng(1)
    x = W.f32_to_bf16_bits(rng.standard_normal((T, k), dtype=np.float32))
    y_in = W.f32_to_bf16_bits(rng.standard_normal((T, d), dtype=np.float32))
    one = oracle.round_bf16(1.0)
    c, m, s = 17, 5, 0.5
    A = np.zeros((8, k), np.uint16)
    A[0, c] = one          # rank padded to 8 with zero rows
    B = np.zeros((d, 8), np.uint16)
    B[m, 0] = one
    ids = np.array([0, -1, 0, 0, -1, 0], np.int32)
    y, _, _ = oracle.apply(x, y_in, [d], ids, np.array([8], np.int32), np.array([s]), [[A]], [[B]])
    want = _f64(y_in).copy()
    for t in range(T):
        if ids[t] == 0:
            want[t, m] += s * _f64(x[t, c])
    np.testing.assert_array_equal(y, want)


def test_zero_B_and_no_adapter_rows_are_unchanged():
    """B = 0 (the training initialisation) adds nothing, and slot -1 rows are
    untouched (llama.cpp LoRA adapter page, same section; vLLM book ch. 16,
    §16.4.2: -1 = no LoRA)."""
    wl = _small_workload(seed=9)
    mod = wl.modules[0]
    scales = np.full(wl.S, 3.0)
    y, _, _ = _run(wl, scales)
    none = wl.slot_ids == -1
    assert none.any()
    np.testing.assert_array_equal(y[none], _f64(mod.y_in[none]))
    mod.B = [[(np.zeros_like(b) if b is not None else None) for b in row] for row in mod.B]
    y0, _, _ = _run(wl, scales)
    np.testing.assert_array_equal(y0, _f64(mod.y_in))


def test_token_permutation_invariance():
    """Sorting tokens by slot and restoring the order is a permutation
    (TensorRT-LLM LoRA serving page, index_copy_ restore): permuting (x, slot,
    y_in) rows permutes the output rows."""
    wl = _small_workload(seed=21)
    mod = wl.modules[0]
    scales = np.linspace(0.5, 2.0, wl.S)
    y, _, _ = _run(wl, scales)
    perm = np.random.default_rng(2).permutation(wl.T)
    yp, _, _ = oracle.apply(mod.x[perm], mod.y_in[perm], mod.slice_widths, wl.slot_ids[perm],
                            wl.ranks, scales, mod.A, mod.B)
    np.testing.assert_array_equal(yp, y[perm])


def test_rslora_versus_standard_scale():
    """alpha/r vs alpha/sqrt(r) (vLLM LoRA deep-dive page, §1 "rsLoRA 变体"): at
    r=16, alpha=32 the scales are 2 and 8, so the rsLoRA delta is exactly 4x."""
    assert oracle.scale(32, 16) == 2.0
    assert oracle.scale(32, 16, rslora=True) == 8.0
    assert oracle.scale(32, 64, rslora=True) == 4.0
    assert oracle.scale(16, 64, rslora=True) == 2.0
    wl = _small_workload(seed=4, ranks=(16, 16, 16, 16, 16), y_init="zeros")
    std = np.array([oracle.scale(32, 16)] * wl.S)
    rs = np.array([oracle.scale(32, 16, rslora=True)] * wl.S)
    d_std, _, _ = _run(wl, std)
    d_rs, _, _ = _run(wl, rs)
    np.testing.assert_array_equal(d_rs, 4.0 * d_std)


def test_scale_values_printed_on_pages():
    for rule, alpha, rank, adapter_scale, expected in _golden("scale_values.txt"):
        got = oracle.scale(float(alpha), int(rank), rule == "alpha_over_sqrt_r", float(adapter_scale))
        assert got == float(expected), (rule, alpha, rank)


def test_premultiplied_scale_equals_runtime_scale():
    """vLLM folds the scale into lora_b on load (optimize(): lora_b *= scaling,
    scaling = 1); llama.cpp applies it to the branch output.  With a power-of-two
    scale both are exact, so the results agree to the last bit."""
    wl = _small_workload(seed=13)
    mod = wl.modules[0]
    s = oracle.scale(32, 16)          # 2.0
    y_rt, _, _ = _run(wl, np.full(wl.S, s))
    B_pre = [[(oracle.premultiply(b, s) if b is not None else None) for b in row] for row in mod.B]
    for row, row_pre in zip(mod.B, B_pre):
        for b, bp in zip(row, row_pre):
            if b is not None:
                np.testing.assert_array_equal(_f64(bp), 2.0 * _f64(b))
    y_pre, _, _ = oracle.apply(mod.x, mod.y_in, mod.slice_widths, wl.slot_ids, wl.ranks,
                               np.ones(wl.S), mod.A, B_pre)
    np.testing.assert_array_equal(y_pre, y_rt)


def test_rank_concatenation_identity():
    """Two adapters on the same tokens equal one adapter of rank r1+r2 with A
    stacked along rank and B side by side (llama.cpp LoRA adapter page,
    §"从读源码到改源码:几个可以落地的扩展点": merging adapters into one branch by
    concatenating A along the rank and aligning B blocks)."""
    T, k, d, r1, r2 = 10, 64, 40, 8, 16
    rng = np.random.default_rng(8)
    x = W.f32_to_bf16_bits(rng.standard_normal((T, k), dtype=np.float32))
    A1 = W.f32_to_bf16_bits(rng.standard_normal((r1, k), dtype=np.float32) * 0.1)
    A2 = W.f32_to_bf16_bits(rng.standard_normal((r2, k), dtype=np.float32) * 0.1)
    B1 = W.f32_to_bf16_bits(rng.standard_normal((d, r1), dtype=np.float32) * 0.1)
    B2 = W.f32_to_bf16_bits(rng.standard_normal((d, r2), dtype=np.float32) * 0.1)
    ids = np.zeros(T, np.int32)
    y1, _, _ = oracle.apply(x, None, [d], ids, np.array([r1], np.int32), np.array([0.75]), [[A1]], [[B1]])
    y2, _, _ = oracle.apply(x, None, [d], ids, np.array([r2], np.int32), np.array([0.75]), [[A2]], [[B2]])
    Ac = np.concatenate([A1, A2], axis=0)
    Bc = np.concatenate([B1, B2], axis=1)
    yc, _, _ = oracle.apply(x, None, [d], ids, np.array([r1 + r2], np.int32), np.array([0.75]), [[Ac]], [[Bc]])
    np.testing.assert_allclose(yc, y1 + y2, rtol=1e-12, atol=1e-13)


def test_packed_slices_equal_separate_projections():
    """A packed QKV output is the three projections side by side (vLLM LoRA
    deep-dive page, §5.4 packed modules; TensorRT-LLM attn_qkv)."""
    wl = _small_workload(seed=17)
    mod = wl.modules[0]
    scales = np.linspace(0.25, 2.0, wl.S)
    y, _, _ = _run(wl, scales)
    offs = mod.slice_offsets
    for i, w in enumerate(mod.slice_widths):
        yi, _, _ = oracle.apply(mod.x, np.ascontiguousarray(mod.y_in[:, offs[i]:offs[i + 1]]), [w],
                                wl.slot_ids, wl.ranks, scales,
                                [[row[i]] for row in mod.A], [[row[i]] for row in mod.B])
        np.testing.assert_array_equal(yi, y[:, offs[i]:offs[i + 1]])


def test_mac_count_matches_pages():
    """2dr multiply-adds per token against dk for the base, about 0.8% at
    d=k=4096, r=16; adapter parameters 2r/d = 0.78%."""
    rows = {r[0]: r for r in _golden("cost_ratios.txt")}
    _, d, k, r, pct, prec = rows["branch_macs_over_base"]
    d, k, r, pct, prec = int(d), int(k), int(r), float(pct), float(prec)
    rng = np.random.default_rng(0)
    x = W.f32_to_bf16_bits(rng.standard_normal((3, k), dtype=np.float32))
    A = W.f32_to_bf16_bits(rng.standard_normal((r, k), dtype=np.float32))
    B = W.f32_to_bf16_bits(rng.standard_normal((d, r), dtype=np.float32))
    ids = np.array([0, -1, 0], np.int32)
    _, macs, _ = oracle.apply(x, None, [d], ids, np.array([r], np.int32), np.array([1.0]), [[A]], [[B]])
    per_token = macs / 2            # two LoRA tokens
    assert per_token == 2 * d * r
    assert abs(100.0 * per_token / (d * k) - pct) <= prec
    _, d2, _, r2, pct2, prec2 = rows["adapter_params_over_base"]
    d2, r2 = int(d2), int(r2)
    assert abs(100.0 * (A.size + B.size) / (d2 * d2) - float(pct2)) <= float(prec2)


def test_mac_count_packed_module():
    wl = _small_workload(seed=30)
    mod = wl.modules[0]
    _, macs, _ = _run(wl, np.ones(wl.S))
    want = sum(int(wl.ranks[s]) * (mod.n_slices * mod.k + mod.d)
               for s in wl.slot_ids if s >= 0 and wl.ranks[s] > 0)
    assert macs == want


def test_rank0_slot_and_out_of_range_slot():
    """A rank-0 slot contributes nothing (TensorRT-LLM's base sentinel slot has
    rank 0); an out-of-range slot id is an error and its row is left alone."""
    wl = _small_workload(seed=12)
    mod = wl.modules[0]
    ids = wl.slot_ids.copy()
    ids[0] = 2                       # rank-0 slot
    ids[1] = wl.S + 3                # out of range
    ids[2] = -7                      # out of range
    y, _, st = oracle.apply(mod.x, mod.y_in, mod.slice_widths, ids, wl.ranks, np.ones(wl.S), mod.A, mod.B)
    assert st == oracle.ERR_SLOT_RANGE
    np.testing.assert_array_equal(y[:3], _f64(mod.y_in[:3]))
    sorted_ids, seg, active, st = oracle.build_index(ids, wl.S, wl.ranks)
    assert st == oracle.ERR_SLOT_RANGE
    tail = set(sorted_ids[seg[wl.S]:seg[wl.S + 1]])
    assert {1, 2} <= tail
    assert 0 in set(sorted_ids[seg[2]:seg[3]])
    assert 2 not in set(active[1:1 + active[0]])


# ---------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------
def _bf16_neighbours(v):
    """Brute force: the two bf16 values bracketing v, by walking the bit patterns."""
    f = np.float32(v)
    b = int(W.f32_to_bf16_bits(np.array([f]))[0])
    cands = []
    for bb in range(max(0, b - 2), min(0xFFFF, b + 2) + 1):
        cands.append(bb)
    if v < 0:
        cands = [c | 0x8000 for c in cands if c & 0x8000] or cands
    return cands


def test_round_bf16_against_brute_force():
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000),
                           [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 2.0 ** -130, 0.0]])
    for v in vals:
        got = oracle.round_bf16(v)
        best = None
        for c in _bf16_neighbours(v):
            cv = float(W.bf16_bits_to_f32(np.array([c], np.uint16))[0])
            if not np.isfinite(cv):
                continue
            key = (abs(cv - v), c & 1)          # nearest, then even significand
            if best is None or key < best[0]:
                best = (key, c)
        gv = float(W.bf16_bits_to_f32(np.array([got], np.uint16))[0])
        bv = float(W.bf16_bits_to_f32(np.array([best[1]], np.uint16))[0])
        assert abs(gv - v) == abs(bv - v), v
        if abs(gv - v) == abs(bv - v) and gv != bv:
            assert got & 1 == 0, v


def test_round_bf16_agrees_with_input_rounding_on_float32_values():
    v = np.random.default_rng(1).standard_normal(20000).astype(np.float32)
    want = W.f32_to_bf16_bits(v)
    got = np.array([oracle.round_bf16(float(a)) for a in v], dtype=np.uint16)
    np.testing.assert_array_equal(got, want)


# ---------------------------------------------------------------------------
# FP8 adapters (TensorRT-LLM LoRA serving page, "第五步:FP8 特判" and the
# forward-pass data_type check: weights stay float8_e4m3fn, x is clamped to the
# FP8 range and converted)
# ---------------------------------------------------------------------------
def test_e4m3_decode_matches_library_on_every_code():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_double(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(lib))
    np.testing.assert_array_equal(ours[~np.isnan(ours)], lib[~np.isnan(lib)])
    assert oracle.e4m3_to_double(np.array([0x7E], np.uint8))[0] == 448.0  # fp8_max on the page


def test_e4m3_round_matches_library_clamp_and_convert():
    """x.clamp(-fp8_max, fp8_max).to(float8_e4m3fn), including ties and the clamp."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    v = rng.standard_normal(4000) * np.exp(rng.uniform(-12, 8, 4000))
    pos = oracle.e4m3_to_double(np.arange(0x7F, dtype=np.uint8))
    mids = (pos[:-1] + pos[1:]) / 2  # exact ties between neighbouring codes
    v = np.concatenate([v, mids, -mids, [500.0, -1e6, 448.0, 0.0]])
    ours = oracle.e4m3_round(v)
    lib = torch.from_numpy(v).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, lib)


def test_e4m3_premultiply_matches_pages_expression():
    """(t_out.to(bf16) * scale).clamp(-fp8_max, fp8_max).to(t_out.dtype)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(4)
    codes = rng.integers(0, 256, size=3000).astype(np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]  # no NaN codes
    for s in (0.25, 2.0, 1.0 / 3.0, 8.0):
        ours = oracle.premultiply_e4m3(codes, s)
        t = torch.from_numpy(codes).view(torch.float8_e4m3fn)
        lib = (t.to(torch.bfloat16) * s).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        np.testing.assert_array_equal(ours, lib)


def test_fp8_branch_equals_bf16_branch_on_decoded_values():
    """Every e4m3 value is a bf16 value, so the FP8 branch is the bf16 branch run
    on x rounded through e4m3 and on the decoded weights."""
    rng = np.random.default_rng(5)
    T, k, widths, S = 12, 64, [24, 8], 3
    ranks = np.array([8, 0, 16], np.int32)
    x = W.f32_to_bf16_bits(rng.standard_normal((T, k)).astype(np.float32))
    y_in = W.f32_to_bf16_bits(rng.standard_normal((T, sum(widths))).astype(np.float32))
    ids = np.array([0, 2, -1, 1, 2, 0, 0, 2, -1, 2, 1, 0], np.int32)
    A8 = [[(rng.integers(0, 256, size=(r, k)).astype(np.uint8) & 0xF7 if r else None) for _ in widths] for r in ranks]
    B8 = [[(rng.integers(0, 256, size=(w, r)).astype(np.uint8) & 0xF7 if r else None) for w in widths] for r in ranks]
    scales = np.array([0.5, 1.0, 2.0])
    got, st = oracle.apply_e4m3(x, y_in, widths, ids, ranks, scales, A8, B8)
    assert st == oracle.ERR_OK

    def bf16_of(codes):
        return W.f32_to_bf16_bits(oracle.e4m3_to_double(codes).astype(np.float32))

    xq = bf16_of(oracle.e4m3_round(W.bf16_bits_to_f32(x).astype(np.float64)))
    A = [[bf16_of(a) if a is not None else None for a in row] for row in A8]
    B = [[bf16_of(b) if b is not None else None for b in row] for row in B8]
    ref, _, _ = oracle.apply(xq, y_in, widths, ids, ranks, scales, A, B)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# Routed-expert (MoE) LoRA: llama.cpp's build_lora_mm_id routes A and B by the
# token's expert ids; TensorRT-LLM's per-expert layout is A [E, r, k], B [E, d, r]
# with expert e's pair e * dim * rank elements in.
# ---------------------------------------------------------------------------
ONE_BF16 = np.uint16(0x3F80)


def _moe_case(seed, T=6, K=2, E=3, k=16, widths=(8,), r=8, x_per_token=True):
    rng = np.random.default_rng(seed)
    x = W.f32_to_bf16_bits(rng.standard_normal((T if x_per_token else T * K, k), dtype=np.float32))
    y_in = W.f32_to_bf16_bits(rng.standard_normal((T * K, sum(widths)), dtype=np.float32))
    experts = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    return x, y_in, experts


@pytest.mark.parametrize("x_per_token", [True, False])
def test_moe_one_hot_at_the_pages_expert_offset(x_per_token):
    """A single 1 in A at flat index e0*r*k + j0*k + c0 and in B at e0*d*r + m0*r + j0
    (the pages' expert * dim * rank offset): pairs routed to e0 gain s * x[row][c0]
    at column m0, exactly; every other entry keeps y."""
    T, K, E, k, d, r = 6, 2, 3, 16, 8, 8
    e0, j0, c0, m0, s = 1, 5, 11, 6, 0.5
    x, y_in, experts = _moe_case(3, T, K, E, k, (d,), r, x_per_token)
    A = np.zeros(E * r * k, np.uint16)
    A[e0 * r * k + j0 * k + c0] = ONE_BF16
    B = np.zeros(E * d * r, np.uint16)
    B[e0 * d * r + m0 * r + j0] = ONE_BF16
    slots = np.array([0, -1, 0, 0, 0, -1], np.int32)
    y, st = oracle.apply_moe(x, x_per_token, y_in, [d], slots, experts, E, np.array([r]), np.array([s]),
                             [[A]], [[B]])
    assert st == 0
    want = _f64(y_in).copy()
    for p in range(T * K):
        t = p // K
        if slots[t] == 0 and experts[t, p % K] == e0:
            want[p, m0] += s * _f64(x[t if x_per_token else p, c0])
    np.testing.assert_array_equal(y, want)
    assert any(slots[t] == 0 and e0 in experts[t] for t in range(T))


def test_moe_single_expert_reduces_to_dense_branch():
    """E = 1, K = 1 is the dense branch; K = 1 with every token on expert e is the
    dense branch with each adapter's expert-e slices as its A and B."""
    wl = _small_workload(seed=21, T=24, k=32, widths=(16, 8), S=3, ranks=(8, 16, 8))
    mod = wl.modules[0]
    scales = np.array([0.5, 2.0, 1.5])
    dense, _, st0 = _run(wl, scales)
    ids1 = np.zeros((wl.T, 1), np.int32)
    y1, st1 = oracle.apply_moe(mod.x, True, mod.y_in, mod.slice_widths, wl.slot_ids, ids1, 1, wl.ranks, scales,
                               mod.A, mod.B)
    assert st0 == st1
    np.testing.assert_array_equal(y1, dense)
    E, e = 3, 2
    rng = np.random.default_rng(5)
    A3 = [[(W.f32_to_bf16_bits(rng.standard_normal((E, r, 32), dtype=np.float32)) if a is not None else None)
           for a in row] for r, row in zip(wl.ranks, mod.A)]
    B3 = [[(W.f32_to_bf16_bits(rng.standard_normal((E, w, r), dtype=np.float32) * np.float32(0.02))
            if b is not None else None) for w, b in zip(mod.slice_widths, row)] for r, row in zip(wl.ranks, mod.B)]
    ye, _ = oracle.apply_moe(mod.x, True, mod.y_in, mod.slice_widths, wl.slot_ids, np.full((wl.T, 1), e, np.int32),
                             E, wl.ranks, scales, A3, B3)
    Ae = [[(a[e] if a is not None else None) for a in row] for row in A3]
    Be = [[(b[e] if b is not None else None) for b in row] for row in B3]
    yd, _, _ = oracle.apply(mod.x, mod.y_in, mod.slice_widths, wl.slot_ids, wl.ranks, scales, Ae, Be)
    np.testing.assert_array_equal(ye, yd)


def test_moe_choice_order_and_shared_rows():
    """Permuting a token's K choices permutes its K output rows; x shared per
    token equals per-pair rows that repeat it; tokens without an adapter keep y."""
    T, K, E, k, widths = 7, 3, 4, 24, (16, 8)
    rng = np.random.default_rng(9)
    x, y_in, experts = _moe_case(11, T, K, E, k, widths)
    ranks = np.array([8, 16])
    A = [[W.f32_to_bf16_bits(rng.standard_normal((E, r, k), dtype=np.float32)) for _ in widths] for r in ranks]
    B = [[W.f32_to_bf16_bits(rng.standard_normal((E, w, r), dtype=np.float32)) for w in widths] for r in ranks]
    slots = np.array([0, 1, -1, 1, 0, 0, -1], np.int32)
    sc = np.array([0.25, 1.0])
    y, st = oracle.apply_moe(x, True, y_in, widths, slots, experts, E, ranks, sc, A, B)
    assert st == 0
    perm = np.array([2, 0, 1])
    y_in_p = y_in.reshape(T, K, -1)[:, perm].reshape(T * K, -1)
    yp, _ = oracle.apply_moe(x, True, y_in_p, widths, slots, experts[:, perm], E, ranks, sc, A, B)
    np.testing.assert_array_equal(yp.reshape(T, K, -1), y.reshape(T, K, -1)[:, perm])
    yr, _ = oracle.apply_moe(np.repeat(x, K, axis=0), False, y_in, widths, slots, experts, E, ranks, sc, A, B)
    np.testing.assert_array_equal(yr, y)
    none = np.repeat(slots == -1, K)
    np.testing.assert_array_equal(y[none], _f64(y_in[none]))
    assert not np.array_equal(y[~none], _f64(y_in[~none]))


def test_moe_out_of_range_ids_and_pair_slots():
    """Pair slots of a hand-worked routing (E = 3, 2 adapters): s E + e, -1 without
    an adapter, and 6 (out of range, reported) for a bad slot or expert id; the
    branch leaves such pairs unchanged and reports them."""
    slots = np.array([1, -1, 0, 5], np.int32)
    experts = np.array([[2, 0], [1, 1], [0, 3], [0, 1]], np.int32)
    np.testing.assert_array_equal(oracle.moe_pair_slots(slots, experts, 3, 2), [5, 3, -1, -1, 0, 6, 6, 6])
    k, E = 8, 4
    rng = np.random.default_rng(4)
    x = W.f32_to_bf16_bits(rng.standard_normal((4, k), dtype=np.float32))
    y_in = W.f32_to_bf16_bits(rng.standard_normal((8, 8), dtype=np.float32))
    A = [[W.f32_to_bf16_bits(rng.standard_normal((E, 8, k), dtype=np.float32))] for _ in range(2)]
    B = [[W.f32_to_bf16_bits(rng.standard_normal((E, 8, 8), dtype=np.float32))] for _ in range(2)]
    bad_e = np.array([[0, 1], [2, 4], [0, -2], [3, 3]], np.int32)
    y, st = oracle.apply_moe(x, True, y_in, [8], np.array([0, 1, 1, -1], np.int32), bad_e, E, np.array([8, 8]),
                             np.ones(2), A, B)
    assert st == oracle.ERR_SLOT_RANGE
    np.testing.assert_array_equal(y[[3, 5, 6, 7]], _f64(y_in[[3, 5, 6, 7]]))
    assert not np.array_equal(y[[0, 1, 2, 4]], _f64(y_in[[0, 1, 2, 4]]))


# ---------------------------------------------------------------------------
# Activated LoRA (llama.cpp's aLoRA): no adapter before the invocation point
# ---------------------------------------------------------------------------
def test_activated_slots_hand_worked():
    """Sequence 0 (slot 3) invoked at position 2, sequence 1 without an adapter,
    sequence 2 (slot 1) invoked at 7, past its tokens (the pages' "not found" case):
    worked out by hand.  Start 0 everywhere is the plain per-sequence slot; an
    unknown sequence id gives an out-of-range slot."""
    seq = np.array([0, 0, 0, 0, 1, 1, 2, 2, 0], np.int32)
    pos = np.array([0, 1, 2, 3, 0, 1, 5, 6, 4], np.int32)
    slot = np.array([3, -1, 1], np.int32)
    start = np.array([2, 0, 7], np.int32)
    np.testing.assert_array_equal(oracle.activated_token_slots(seq, pos, slot, start),
                                  [-1, -1, 3, 3, -1, -1, -1, -1, 3])
    np.testing.assert_array_equal(oracle.activated_token_slots(seq, pos, slot, np.zeros(3, np.int32)),
                                  [3, 3, 3, 3, -1, -1, 1, 1, 3])
    bad = oracle.activated_token_slots(np.array([3], np.int32), np.array([0], np.int32), slot, start)
    assert bad[0] >= 3
