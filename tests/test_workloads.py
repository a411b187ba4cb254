"""The seeded input generators: deterministic, with the documented structure."""
import numpy as np

import workloads as W


def test_moe_config_is_seeded_and_routes_distinct_experts():
    a, b = W.moe_config(T=32), W.moe_config(T=32)
    np.testing.assert_array_equal(a.slot_ids, b.slot_ids)
    np.testing.assert_array_equal(a.expert_ids, b.expert_ids)
    np.testing.assert_array_equal(a.modules[0].A[0][0], b.modules[0].A[0][0])
    assert a.expert_ids.shape == (32, 2)
    assert all(len(set(row)) == 2 for row in a.expert_ids.tolist())
    assert a.expert_ids.min() >= 0 and a.expert_ids.max() < a.E
    up, down = a.modules
    assert up.x_per_token and up.x.shape == (32, 4096) and up.y_in.shape == (64, 14336)
    assert not down.x_per_token and down.x.shape == (64, 14336) and down.y_in.shape == (64, 4096)
    assert up.A[0][0].shape == (8, 16, 4096) and up.B[0][0].shape == (8, 14336, 16)


def test_fp8_codes_follow_the_documented_fields():
    """Sign any, exponent field 3..7, mantissa any: never NaN (0x7F, 0xFF), never
    zero or subnormal."""
    wl = W.config(6)
    codes = np.concatenate([a.reshape(-1) for row in wl.modules[0].A for a in row if a is not None])
    exp = (codes >> 3) & 15
    assert codes.dtype == np.uint8
    assert exp.min() == 3 and exp.max() == 7
    assert not np.isin(codes, [0x7F, 0xFF]).any()
    assert len(np.unique(codes & 7)) == 8 and len(np.unique(codes >> 7)) == 2


def test_speculative_config_repeats_each_sequence_slot():
    wl = W.config(5)
    tps = wl.tokens_per_seq
    assert tps == 4 and wl.T == 256
    seq = wl.slot_ids.reshape(-1, tps)
    assert (seq == seq[:, :1]).all()
