"""Client-side datum construction, restated from the Tinker deep-dive page.

These transforms run on the client before a batch reaches the training
worker; the worker itself only sees flattened per-token arrays.  They are
used to build synthetic workloads and are pinned by the worked examples the
page prints (tests/golden/).

* shift_sequence  -- "SFT first: a token-level contract": a full sequence
  becomes inputs (all but the last id) and targets (all but the first id);
  the weight of each position follows the role of its *target* token.
* mean_reduction  -- same section: the cookbook's reduction="mean" rescales
  a datum's positive weights to sum to one.
* center_group    -- "RL: preserve tokens, logprobs, and credit": group
  relative advantages A_i = R_i - mean(R).
* standardize_group -- centring followed by division by the group's standard
  deviation (the group normalisation of the 4B-width workload).
* check_rl_datum  -- "A runnable contract check": the validation rules an RL
  datum must satisfy before submission.
"""
from __future__ import annotations

import math
from typing import Sequence

import numpy as np


def shift_sequence(full_tokens: Sequence[int], role_weight: Sequence[float]):
    """Return (inputs, targets, weights) for one datum.

    ``role_weight[j]`` is the weight token j receives when it is a target
    (0 for prompt/observation tokens, 1 or a fraction for answer tokens).
    Weights follow the target role, so the first answer token is trained.
    """
    full = list(full_tokens)
    rw = list(role_weight)
    if len(full) != len(rw):
        raise ValueError("one role weight per token is required")
    if len(full) < 2:
        raise ValueError("a datum needs at least two tokens")
    inputs = full[: len(full) - 1]
    targets = full[1:]
    weights = rw[1:]
    return inputs, targets, weights


def mean_reduction(weights: Sequence[float]):
    """Scale weights so that a positive total becomes 1 (else unchanged)."""
    w = [float(x) for x in weights]
    total = sum(w)
    if total > 0:
        return [x / total for x in w]
    return w


def _finite_nonempty(rewards):
    r = [float(x) for x in rewards]
    if len(r) == 0 or any(not math.isfinite(x) for x in r):
        raise ValueError("a reward group must be non-empty and finite")
    return r


def center_group(rewards: Sequence[float]):
    """Group-relative advantages: each reward minus the group mean."""
    r = _finite_nonempty(rewards)
    mu = sum(r) / len(r)
    return tuple(x - mu for x in r)


def group_has_signal(rewards: Sequence[float]) -> bool:
    """A group whose rewards are all equal carries no reward contrast."""
    return len(set(float(x) for x in rewards)) > 1


def standardize_group(rewards) -> np.ndarray:
    """Centred rewards divided by the group's (population) standard deviation.

    A constant group returns zeros.
    """
    r = np.asarray(rewards, dtype=np.float64)
    c = r - r.mean()
    s = r.std()
    return c / s if s > 0 else np.zeros_like(c)


def check_rl_datum(input_tokens, target_tokens, sampled_logprobs, advantages, mask):
    """Raise ValueError unless the RL datum obeys the page's contract.

    Rules: all five arrays non-empty and of one length; every token id a
    non-negative integer; logprobs and advantages finite; mask entries 0 or
    1; at least one action position; no positive logprob at an action
    position; zero advantage wherever the mask is 0.
    """
    arrays = (input_tokens, target_tokens, sampled_logprobs, advantages, mask)
    lens = {len(x) for x in arrays}
    if len(lens) != 1 or 0 in lens:
        raise ValueError("arrays must be non-empty and equally long")
    for t in list(input_tokens) + list(target_tokens):
        if isinstance(t, bool) or not isinstance(t, (int, np.integer)) or t < 0:
            raise ValueError("token ids must be non-negative integers")
    for x in list(sampled_logprobs) + list(advantages):
        if not math.isfinite(float(x)):
            raise ValueError("logprobs and advantages must be finite")
    for m in mask:
        if float(m) not in (0.0, 1.0):
            raise ValueError("mask entries must be 0 or 1")
    if not any(float(m) == 1.0 for m in mask):
        raise ValueError("datum has no action position")
    for m, lp in zip(mask, sampled_logprobs):
        if float(m) == 1.0 and float(lp) > 0.0:
            raise ValueError("an action logprob cannot be positive")
    for m, a in zip(mask, advantages):
        if float(m) == 0.0 and float(a) != 0.0:
            raise ValueError("masked positions need zero advantage")
