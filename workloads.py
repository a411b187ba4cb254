"""Seeded synthetic inputs for the batched multi-adapter LoRA branch.

Both sides of every parity check read their inputs from here: the CUDA library
(through its Python binding) and the CPU oracle.  The module only draws random
numbers and lays them out.  It holds none of the branch arithmetic: there is no
product, no scale rule and no index here.  Ranks, alphas, the scale rule's name
and the "pre-multiplied into B" flag are returned as plain data, and each
consumer derives the per-slot scale (and any pre-multiplied B) with its own code.

Layouts (PEFT orientation, row-major, bf16 stored as uint16 bit patterns; FP8
weights as uint8 float8_e4m3fn codes):
  x    [T, k]        one row per token
  A    [r_s, k]      per slot s and output slice i (``mod.A[s][i]``)
  B    [d_i, r_s]    per slot s and output slice i (``mod.B[s][i]``)
  y_in [T, d]        d = sum of the slice widths, slices side by side

Generation rules (all configs): numpy PCG64, seed ``1000 + config index``;
draw order slot_ids, ranks, then per module x, A (slot-major, slice-minor),
B (same order), y_in; values drawn in fp32 and rounded to bf16 with
round-to-nearest-even.  A ~ N(0, 1/k) (variance 1/k), B ~ N(0, 0.02^2)
(standard deviation 0.02), x ~ N(0, 1), y_in ~ N(0, 1) (or zeros).  FP8
weights (``weights="e4m3"``) are drawn as codes, not rounded from values: sign
uniform, exponent field uniform in {3..7} (magnitudes 2^-4 .. 1.875), mantissa
field uniform in {0..7}; the adapters' real magnitude then lives in the scale.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence

import numpy as np

RANK_CHOICES = (8, 16, 32, 64)


# ----------------------------------------------------------------------------
# bf16 bit patterns (input preparation only)
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return uint16 bits.

    Inputs are finite by construction (normal draws), so NaN handling is not
    needed here.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounded = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _e4m3_codes(rng: np.random.Generator, shape: Sequence[int]) -> np.ndarray:
    """float8_e4m3fn codes: sign, exponent field in {3..7}, mantissa field in {0..7}."""
    sign = rng.integers(0, 2, size=shape, dtype=np.uint8)
    expo = rng.integers(3, 8, size=shape, dtype=np.uint8)
    mant = rng.integers(0, 8, size=shape, dtype=np.uint8)
    return ((sign << np.uint8(7)) | (expo << np.uint8(3)) | mant).astype(np.uint8)


def _normal_bf16(rng: np.random.Generator, shape: Sequence[int], std: float,
                 chunk_rows: int = 2048) -> np.ndarray:
    """Draw N(0, std^2) in fp32 row-chunk by row-chunk and round to bf16 bits."""
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.uint16)
    if out.size == 0:
        return out
    rows = shape[0]
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        v = rng.standard_normal((r1 - r0,) + shape[1:], dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        out[r0:r1] = f32_to_bf16_bits(v)
    return out


# ----------------------------------------------------------------------------
# Containers
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class Module:
    """One packed projection: one x, one y, per-slot per-slice A and B."""
    name: str
    k: int
    slice_widths: List[int]
    x: np.ndarray                                  # uint16 [T, k]
    y_in: np.ndarray                               # uint16 [T, d]
    A: List[List[Optional[np.ndarray]]]            # [S][n] uint16 (uint8 for e4m3) [r_s, k] (None if r_s == 0)
    B: List[List[Optional[np.ndarray]]]            # [S][n] uint16 (uint8 for e4m3) [d_i, r_s]

    @property
    def n_slices(self) -> int:
        return len(self.slice_widths)

    @property
    def d(self) -> int:
        return int(sum(self.slice_widths))

    @property
    def slice_offsets(self) -> List[int]:
        offs = [0]
        for w in self.slice_widths:
            offs.append(offs[-1] + int(w))
        return offs


@dataclasses.dataclass
class Workload:
    name: str
    T: int
    S: int
    r_max: int
    slot_ids: np.ndarray          # int32 [T], -1 = no adapter
    ranks: np.ndarray             # int32 [S]
    alphas: np.ndarray            # float64 [S] (lora_alpha per slot)
    scale_rule: str               # "alpha_over_r" or "alpha_over_sqrt_r"
    premultiplied: bool           # scale folded into B on load (runtime scale 1)
    modules: List[Module]
    seed: int
    description: str = ""
    tokens_per_seq: int = 1       # speculative decode: sequences of this many tokens, sequence-major
    weights: str = "bf16"         # "bf16" or "e4m3" (A and B as float8_e4m3fn codes)


# ----------------------------------------------------------------------------
# Slot-id draws
# ----------------------------------------------------------------------------
def zipf_probabilities(S: int, exponent: float) -> np.ndarray:
    """Finite Zipf popularity over S slots: slot s has weight (s+1)^-exponent."""
    w = np.arange(1, S + 1, dtype=np.float64) ** (-float(exponent))
    return w / w.sum()


def _draw_slot_ids(rng: np.random.Generator, T: int, S: int, dist: str,
                   frac_none: float, zipf_exponent: float = 1.1) -> np.ndarray:
    if dist == "uniform_with_none":          # uniform over {-1, 0, .., S-1}
        ids = rng.integers(-1, S, size=T)
    elif dist == "uniform":
        ids = rng.integers(0, S, size=T)
    elif dist == "zipf":
        ids = rng.choice(S, size=T, p=zipf_probabilities(S, zipf_exponent))
    else:
        raise ValueError(f"unknown slot distribution {dist!r}")
    ids = ids.astype(np.int32)
    n_none = int(round(frac_none * T))
    if n_none > 0 and dist != "uniform_with_none":
        pos = rng.choice(T, size=n_none, replace=False)
        ids[pos] = -1
    return ids


# ----------------------------------------------------------------------------
# Generic generator
# ----------------------------------------------------------------------------
def generate(*, name: str, seed: int, T: Optional[int], S: int,
             modules: Sequence[Dict], rank: Optional[int] = None,
             rank_choices: Optional[Sequence[int]] = None, r_max: Optional[int] = None,
             slot_dist: str = "uniform", frac_none: float = 0.0,
             zipf_exponent: float = 1.1, alpha: Optional[float] = None,
             alpha_times_rank: Optional[float] = None, scale_rule: str = "alpha_over_r",
             premultiplied: bool = False, requests: Optional[Dict] = None,
             y_init: str = "normal", description: str = "", tokens_per_seq: int = 1,
             weights: str = "bf16") -> Workload:
    """Draw one workload.

    ``modules`` is a list of ``{"name", "k", "slices"}`` dicts.  Slots get either
    one ``rank`` for all, or a rank drawn per slot from ``rank_choices``.  The
    alpha of a slot is ``alpha`` or ``alpha_times_rank * r_s``.  ``requests``
    (``{"n", "min_len", "max_len", "n_adapters"}``) makes a request-major
    prefill batch: lengths uniform in [min_len, max_len], one adapter per request
    drawn uniformly.  ``tokens_per_seq`` > 1 draws one slot per sequence of that
    many consecutive tokens (speculative decode; T must be a multiple).
    ``weights="e4m3"`` draws A and B as float8_e4m3fn codes (module docstring).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    # 1. slot ids
    if requests is not None:
        lens = rng.integers(requests["min_len"], requests["max_len"] + 1, size=requests["n"])
        adapters = rng.integers(0, requests["n_adapters"], size=requests["n"])
        slot_ids = np.repeat(adapters, lens).astype(np.int32)
        T = int(slot_ids.shape[0])
    else:
        assert T is not None and T % tokens_per_seq == 0
        seq_ids = _draw_slot_ids(rng, T // tokens_per_seq, S, slot_dist, frac_none, zipf_exponent)
        slot_ids = np.repeat(seq_ids, tokens_per_seq).astype(np.int32)
    # 2. ranks
    if rank_choices is not None:
        ranks = rng.choice(np.asarray(rank_choices), size=S).astype(np.int32)
    else:
        ranks = np.full(S, int(rank), dtype=np.int32)
    if r_max is None:
        r_max = int(ranks.max()) if S > 0 else 0
    if alpha_times_rank is not None:
        alphas = alpha_times_rank * ranks.astype(np.float64)
    else:
        alphas = np.full(S, float(alpha), dtype=np.float64)
    # 3. per module: x, A, B, y_in
    mods = []
    for m in modules:
        k = int(m["k"])
        widths = [int(w) for w in m["slices"]]
        d = sum(widths)
        x = _normal_bf16(rng, (T, k), 1.0)
        if weights == "e4m3":
            A = [[(_e4m3_codes(rng, (int(ranks[s]), k)) if ranks[s] > 0 else None)
                  for _ in widths] for s in range(S)]
            B = [[(_e4m3_codes(rng, (w, int(ranks[s]))) if ranks[s] > 0 else None)
                  for w in widths] for s in range(S)]
        else:
            A = [[(_normal_bf16(rng, (int(ranks[s]), k), float(k) ** -0.5) if ranks[s] > 0 else None)
                  for _ in widths] for s in range(S)]
            B = [[(_normal_bf16(rng, (w, int(ranks[s])), 0.02) if ranks[s] > 0 else None)
                  for w in widths] for s in range(S)]
        if y_init == "normal":
            y_in = _normal_bf16(rng, (T, d), 1.0)
        elif y_init == "zeros":
            y_in = np.zeros((T, d), dtype=np.uint16)
        else:
            raise ValueError(y_init)
        mods.append(Module(name=m["name"], k=k, slice_widths=widths, x=x, y_in=y_in, A=A, B=B))
    return Workload(name=name, T=int(T), S=S, r_max=int(r_max), slot_ids=slot_ids, ranks=ranks,
                    alphas=alphas, scale_rule=scale_rule, premultiplied=premultiplied,
                    modules=mods, seed=seed, description=description, tokens_per_seq=int(tokens_per_seq),
                    weights=weights)


# ----------------------------------------------------------------------------
# The five named workloads
# ----------------------------------------------------------------------------
LLAMA3_8B_LAYER = [
    {"name": "qkv", "k": 4096, "slices": [4096, 1024, 1024]},
    {"name": "o", "k": 4096, "slices": [4096]},
    {"name": "gate_up", "k": 4096, "slices": [14336, 14336]},
    {"name": "down", "k": 14336, "slices": [4096]},
]

CONFIG_NAMES = ("tiny", "decode_q_proj", "decode_qkv", "prefill_mlp", "large_decode", "decode_qkv_spec",
                "decode_qkv_fp8")


def config(index: int, y_init: str = "normal", sweep: bool = False, n_requests: int = 16) -> Workload:
    """Config ``index`` (0..6) of the benchmark suite, drawn at seed 1000+index.

    0 tiny: T=8, k=d=256, one slice, S=2, r=8, slot ids uniform over {-1,0,1},
      alpha=16 (scale alpha/r applied at run time).
    1 decode q_proj: T=64, k=d=4096, S=8, r=16, 8 tokens at -1, the rest uniform
      over the 8 slots, alpha=32, scale pre-multiplied into B.
    2 decode packed QKV (Llama-3-8B shapes): T=256, k=4096, slices 4096/1024/1024,
      S=32, ranks drawn from {8,16,32,64} (r_max 64), Zipf(1.1) slot popularity,
      alpha=2r.
    3 prefill MLP: 16 requests (``n_requests``, a smaller batch of the same
      recipe for profiling) of uniform length in [128, 2048], request-major,
      adapter per request uniform over 16 slots; gate_up (k=4096, 14336+14336)
      then down (k=14336, d=4096); r=16; rsLoRA alpha/sqrt(r) with alpha=32.
    4 large multi-tenant decode: T=1024, k=d=8192, r=64, S=128, Zipf(1.1) with 5%
      of tokens at -1, alpha=2r.  ``sweep=True`` instead draws the four packed
      projections of one Llama-3-8B layer (qkv, o, gate_up, down) on the same
      slot draw.
    5 speculative decode, packed QKV (Llama-3-8B shapes): 64 sequences of 4
      tokens (one verified plus three draft tokens, T=256), one slot per sequence
      with Zipf(1.1) popularity over S=32, ranks from {8,16,32,64}, alpha=2r.
    6 decode packed QKV with FP8 adapters: config 2's shapes and slot draw recipe,
      A and B as float8_e4m3fn codes, alpha = r / 256 (scale 1/256 at run time).
    """
    seed = 1000 + index
    if index == 0:
        return generate(name="tiny", seed=seed, T=8, S=2, rank=8,
                        modules=[{"name": "proj", "k": 256, "slices": [256]}],
                        slot_dist="uniform_with_none", alpha=16.0, y_init=y_init,
                        description="T=8, k=d=256, S=2, r=8, slots uniform over {-1,0,1}")
    if index == 1:
        return generate(name="decode_q_proj", seed=seed, T=64, S=8, rank=16,
                        modules=[{"name": "q_proj", "k": 4096, "slices": [4096]}],
                        slot_dist="uniform", frac_none=1.0 / 8.0, alpha=32.0,
                        premultiplied=True, y_init=y_init,
                        description="T=64, k=d=4096, S=8, r=16, 1/8 of tokens at -1")
    if index == 2:
        return generate(name="decode_qkv", seed=seed, T=256, S=32, rank_choices=RANK_CHOICES,
                        r_max=64, modules=[LLAMA3_8B_LAYER[0]], slot_dist="zipf",
                        alpha_times_rank=2.0, y_init=y_init,
                        description="T=256, k=4096, slices 4096/1024/1024, S=32, "
                                    "r in {8,16,32,64}, Zipf(1.1)")
    if index == 3:
        return generate(name="prefill_mlp", seed=seed, T=None, S=16, rank=16,
                        modules=[{"name": "gate_up", "k": 4096, "slices": [14336, 14336]},
                                 {"name": "down", "k": 14336, "slices": [4096]}],
                        requests={"n": n_requests, "min_len": 128, "max_len": 2048, "n_adapters": 16},
                        alpha=32.0, scale_rule="alpha_over_sqrt_r", y_init=y_init,
                        description=f"{n_requests} requests, lengths U[128,2048], gate_up 4096->2x14336, "
                                    "down 14336->4096, r=16, rsLoRA")
    if index == 4:
        mods = LLAMA3_8B_LAYER if sweep else [{"name": "qo_8192", "k": 8192, "slices": [8192]}]
        return generate(name="large_decode_sweep" if sweep else "large_decode", seed=seed,
                        T=1024, S=128, rank=64, modules=mods, slot_dist="zipf",
                        frac_none=0.05, alpha_times_rank=2.0, y_init=y_init,
                        description="T=1024, r=64, S=128, Zipf(1.1), 5% at -1")
    if index == 5:
        return generate(name="decode_qkv_spec", seed=seed, T=256, S=32, rank_choices=RANK_CHOICES,
                        r_max=64, modules=[LLAMA3_8B_LAYER[0]], slot_dist="zipf",
                        alpha_times_rank=2.0, y_init=y_init, tokens_per_seq=4,
                        description="64 sequences x 4 tokens (speculative decode), k=4096, "
                                    "slices 4096/1024/1024, S=32, r in {8,16,32,64}, Zipf(1.1) per sequence")
    if index == 6:
        return generate(name="decode_qkv_fp8", seed=seed, T=256, S=32, rank_choices=RANK_CHOICES,
                        r_max=64, modules=[LLAMA3_8B_LAYER[0]], slot_dist="zipf",
                        alpha_times_rank=1.0 / 256.0, y_init=y_init, weights="e4m3",
                        description="T=256, k=4096, slices 4096/1024/1024, S=32, r in {8,16,32,64}, "
                                    "Zipf(1.1), float8_e4m3fn adapters")
    raise IndexError(index)


# ----------------------------------------------------------------------------
# Routed-expert (MoE) LoRA workloads
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class MoeModule:
    """One expert projection: per adapter and slice, A [E, r, k] and B [E, d_i, r]."""
    name: str
    k: int
    slice_widths: List[int]
    x_per_token: bool                              # x rows per token (shared by its experts) or per pair
    x: np.ndarray                                  # uint16 [T, k] or [T*K, k]
    y_in: np.ndarray                               # uint16 [T*K, d], one row per (token, choice) pair
    A: List[List[Optional[np.ndarray]]]            # [n_adapters][n] uint16 [E, r_s, k]
    B: List[List[Optional[np.ndarray]]]            # [n_adapters][n] uint16 [E, d_i, r_s]

    @property
    def d(self) -> int:
        return int(sum(self.slice_widths))


@dataclasses.dataclass
class MoeWorkload:
    name: str
    T: int                        # tokens
    K: int                        # experts per token
    E: int                        # experts
    n_adapters: int
    r_max: int
    slot_ids: np.ndarray          # int32 [T], adapter per token, -1 = none
    expert_ids: np.ndarray        # int32 [T, K], distinct per token
    ranks: np.ndarray             # int32 [n_adapters]
    alphas: np.ndarray            # float64 [n_adapters]
    scale_rule: str
    modules: List[MoeModule]
    seed: int
    description: str = ""


def generate_moe(*, name: str, seed: int, T: int, K: int, E: int, n_adapters: int, rank: int,
                 modules: Sequence[Dict], slot_dist: str = "zipf", frac_none: float = 0.0,
                 zipf_exponent: float = 1.1, alpha_times_rank: float = 2.0, y_init: str = "normal",
                 description: str = "") -> MoeWorkload:
    """Draw one routed-expert workload.  Draw order: adapter per token, K distinct
    experts per token (uniform), then per module x, A (adapter-major, slice-minor;
    each [E, r, k] ~ N(0, 1/k)), B ([E, d_i, r] ~ N(0, 0.02^2)), y_in.  ``modules``
    holds ``{"name", "k", "slices", "x_per_token"}`` dicts."""
    rng = np.random.Generator(np.random.PCG64(seed))
    slot_ids = _draw_slot_ids(rng, T, n_adapters, slot_dist, frac_none, zipf_exponent).astype(np.int32)
    expert_ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    ranks = np.full(n_adapters, int(rank), dtype=np.int32)
    alphas = alpha_times_rank * ranks.astype(np.float64)
    mods = []
    for m in modules:
        k = int(m["k"])
        widths = [int(w) for w in m["slices"]]
        per_token = bool(m["x_per_token"])
        x = _normal_bf16(rng, (T if per_token else T * K, k), 1.0)
        A = [[_normal_bf16(rng, (E * int(ranks[s]), k), float(k) ** -0.5).reshape(E, int(ranks[s]), k)
              for _ in widths] for s in range(n_adapters)]
        B = [[_normal_bf16(rng, (E * w, int(ranks[s])), 0.02).reshape(E, w, int(ranks[s])) for w in widths]
             for s in range(n_adapters)]
        d = sum(widths)
        y_in = _normal_bf16(rng, (T * K, d), 1.0) if y_init == "normal" else np.zeros((T * K, d), np.uint16)
        mods.append(MoeModule(name=m["name"], k=k, slice_widths=widths, x_per_token=per_token, x=x, y_in=y_in,
                              A=A, B=B))
    return MoeWorkload(name=name, T=int(T), K=int(K), E=int(E), n_adapters=int(n_adapters), r_max=int(rank),
                       slot_ids=slot_ids, expert_ids=expert_ids, ranks=ranks, alphas=alphas,
                       scale_rule="alpha_over_r", modules=mods, seed=seed, description=description)


MIXTRAL_EXPERT = [
    {"name": "w1", "k": 4096, "slices": [14336], "x_per_token": True},
    {"name": "w2", "k": 14336, "slices": [4096], "x_per_token": False},
]


def moe_config(T: int = 128, y_init: str = "normal") -> MoeWorkload:
    """Decode through one routed-expert layer with Mixtral-8x7B expert shapes: T
    tokens (default 128) routed top-2 of 8 experts (T*2 pairs), 8 adapters with
    Zipf(1.1) popularity, r = 16, alpha = 2r; modules w1 (hidden 4096 -> 14336,
    x per token) and w2 (14336 -> 4096, x per pair); seed 1007."""
    return generate_moe(name="decode_moe", seed=1007, T=T, K=2, E=8, n_adapters=8, rank=16,
                        modules=MIXTRAL_EXPERT, y_init=y_init,
                        description=f"routed-expert decode, Mixtral-8x7B expert shapes: T={T} tokens, top-2 of "
                                    "8 experts, 8 adapters Zipf(1.1), r=16, w1 4096->14336 and w2 14336->4096")
