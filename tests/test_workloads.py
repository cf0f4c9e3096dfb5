"""The input builder and the workload generators (CPU only).

The datum helpers are pinned by the worked examples of the Deep Dive - Tinker
page (tests/golden/); the generators by their stated structure.
"""
import math

import numpy as np
import pytest

import workloads as wl
from _util import golden


def test_shift_and_mean_reduction_worked_example():
    g = golden("datum_shift.json")
    inputs, targets, weights = wl.shift_sequence(g["full_tokens"], g["role_weight"])
    assert inputs == g["inputs"] and targets == g["targets"] and weights == g["weights"]
    assert wl.mean_reduction(weights) == g["mean_weights"]
    # masking by the input role instead would drop the first answer token
    assert weights[targets.index(20)] == 1


def test_group_centering_worked_example():
    g = golden("group_centering.json")
    assert wl.center_group(g["rewards"]) == tuple(g["advantages"])
    assert wl.group_has_signal(g["rewards"])
    assert not wl.group_has_signal(g["constant_group"])
    assert wl.center_group(g["constant_group"]) == (0.0,) * 4


def test_rl_datum_rules_reject_nine_inputs():
    g = golden("rl_datum_rules.json")
    good = g["valid"]
    wl.check_rl_datum(**good)
    assert good["target_tokens"][1] == g["first_action_target"] and good["mask"][1] == 1
    rejected = 0
    for var in g["invalid_variants"]:
        d = dict(good)
        for k, v in var.items():
            if k != "why":
                d[k] = [float(x) if isinstance(x, str) else x for x in v]
        with pytest.raises(ValueError):
            wl.check_rl_datum(**d)
        rejected += 1
    for rewards in g["invalid_reward_groups"]:
        with pytest.raises(ValueError):
            wl.center_group([float(x) for x in rewards])
        rejected += 1
    assert rejected == 9


def test_bf16_rounding():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, -2.5, 0.0, 3.0e38], np.float32)
    b = wl.f32_to_bf16_bits(x)
    y = wl.bf16_bits_to_f32(b)
    assert y[0] == 1.0
    assert y[1] == 1.0                        # tie -> even
    assert y[2] == 1.0 + 2 ** -7              # above the tie -> up
    assert y[3] == -2.5 and y[4] == 0.0
    assert np.all(wl.f32_to_bf16_bits(y) == b)


@pytest.mark.parametrize("name", wl.CONFIG_NAMES)
def test_batch_structure(name):
    cfg = wl.get_config(name)
    n = 128 if name == "tiny_fp32" else 2048
    b = wl.make_batch(cfg, n)
    N = len(b["tokens"])
    assert abs(N - n) <= 64 and N == b["seq_lens"].sum()
    assert b["tokens"].min() >= 0 and b["tokens"].max() < cfg.vocab
    assert b["targets"].min() >= 0 and b["targets"].max() < cfg.vocab
    assert b["adapter_ids"].min() >= 0 and b["adapter_ids"].max() < cfg.n_adapters
    # targets are the inputs shifted by one inside each sequence
    off = 0
    for T in b["seq_lens"]:
        assert np.array_equal(b["tokens"][off + 1:off + T], b["targets"][off:off + T - 1])
        off += T
    b2 = wl.make_batch(cfg, n)
    assert all(np.array_equal(b[k], b2[k]) for k in ("tokens", "targets", "adapter_ids"))
    if name == "tiny_fp32":
        assert b["weights"].reshape(4, 32)[:, :16].sum() == 0
        assert b["weights"].reshape(4, 32)[:, 16:].min() == 1
    if name == "qwen3_4b_is":
        A = b["advantages"].reshape(64, -1)
        T = A.shape[1]
        assert (A[:, :T // 4] == 0).all()
        for gidx in range(8):
            grp = A[gidx * 8:(gidx + 1) * 8, -1].astype(np.float64)
            assert abs(grp.mean()) < 1e-6 and abs(grp.std() - 1) < 1e-5
    if name == "long_custom":
        g = b["dloss"].reshape(4, -1)
        assert (g[:, :int(0.3 * g.shape[1])] == 0).all()


def test_weights_deterministic_and_bf16():
    cfg = wl.get_config("tiny_fp32", dtype="bf16", vocab=64, d_model=16, d_ffn=32)
    w1 = wl.make_base_weights(cfg)
    w2 = wl.make_base_weights(cfg)
    assert w1["E"].dtype == np.uint16 and np.array_equal(w1["E"], w2["E"])
    x = wl.bf16_bits_to_f32(w1["W1"][0])
    assert 0.015 < float(np.std(x)) < 0.025
    ad = wl.make_adapters(cfg)
    assert ad["A1"][0][0].shape == (4, 16) and ad["B2"][2][1].shape == (16, 4)
