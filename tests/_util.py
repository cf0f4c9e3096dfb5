"""Helpers shared by the test modules (no method arithmetic here)."""
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


def tiny_problem(seed_shift=0, n_adapters=3, ranks=(4, 4, 4), alphas=(8.0, 8.0, 8.0),
                 d=16, f=24, V=40, L=2, n_tokens=24, b_std=0.3, w_std=0.3):
    """A very small fp32 problem with O(1) weights, for finite differences.

    Weights are larger than the workloads' N(0, 0.02) so that every term of
    the gradient is well above rounding noise.
    """
    rng = np.random.Generator(np.random.PCG64([7, seed_shift]))
    base = {
        "E": rng.standard_normal((V, d)).astype(np.float32) * w_std,
        "Wout": rng.standard_normal((V, d)).astype(np.float32) * w_std,
        "W1": [rng.standard_normal((f, d)).astype(np.float32) * w_std for _ in range(L)],
        "W2": [rng.standard_normal((d, f)).astype(np.float32) * w_std for _ in range(L)],
    }
    ad = {"A1": [], "B1": [], "A2": [], "B2": []}
    for a in range(n_adapters):
        r = ranks[a]
        ad["A1"].append([rng.standard_normal((r, d)).astype(np.float32) * w_std for _ in range(L)])
        ad["B1"].append([rng.standard_normal((f, r)).astype(np.float32) * b_std for _ in range(L)])
        ad["A2"].append([rng.standard_normal((r, f)).astype(np.float32) * w_std for _ in range(L)])
        ad["B2"].append([rng.standard_normal((d, r)).astype(np.float32) * b_std for _ in range(L)])
    batch = {
        "tokens": rng.integers(0, V, n_tokens).astype(np.int32),
        "targets": rng.integers(0, V, n_tokens).astype(np.int32),
        "adapter_ids": rng.integers(0, n_adapters, n_tokens).astype(np.int32),
        "weights": rng.random(n_tokens).astype(np.float32),
        "advantages": rng.standard_normal(n_tokens).astype(np.float32),
        "noise": (rng.standard_normal(n_tokens) * 0.3).astype(np.float32),
        "dloss": rng.standard_normal(n_tokens).astype(np.float32),
    }
    return base, ad, list(ranks), list(alphas), batch
