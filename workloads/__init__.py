"""Seeded synthetic inputs for the multi-tenant LoRA training step.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle. It holds no arithmetic of the method itself: it only draws random
numbers, lays out token sequences, and rounds fp32 draws to bf16 bit patterns
(the storage format of the frozen base).

Workloads (Tinker deep dive pages; the base model is a token embedding, L
residual SiLU-MLP blocks with per-adapter LoRA on both projections, and an
untied LM head):

* ``tiny_fp32``        V=512, d=64, f=256, L=2, 3 adapters rank 4 alpha 8,
                        4 sequences x 32 tokens, first 16 target positions
                        weighted 0, cross entropy.  fp32 weights.
* ``qwen3_4b_is``      Qwen3-4B widths, 8 adapters rank 32, 8 groups x 8
                        completions x 1024 tokens, 25 % prompt, importance
                        sampling with group-normalised advantages.
* ``qwen3_8b_ppo``     Qwen3-8B widths, 32 adapters rank 32, 65,536 tokens in
                        sequences of 512-2048 tokens, Zipf(1.1) adapter choice,
                        PPO clip 0.2.
* ``many_tenant_ce``   8B widths with L=2, 128 adapters, ranks from
                        {8,16,32,64}, alpha = 2 rank, 262,144 tokens in
                        sequences of 256-4096 tokens, Bernoulli(0.6) weights.
* ``long_custom``      d=5120, f=25600, L=2, 4 adapters rank 64, 4 x 22,528
                        tokens, 30 % prompt masked, caller-supplied dL/dlogprob.

Every draw comes from numpy ``PCG64`` streams keyed by (config seed, tensor
id, block index); a tensor is drawn in independent row blocks so that it can
be generated on several host threads and still be the same on every machine.
The base weights are drawn N(0, 0.02) in fp32 and rounded to bf16 (round to
nearest even); adapters are fp32 masters, A ~ N(0, 0.02), B ~ N(0, 0.01).
Token ids are uniform on [0, V).  Sequences are laid out contiguously in
generation order, so tokens of different adapters interleave.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace
from typing import Dict, List, Optional

import numpy as np

from .datum import (center_group, check_rl_datum, group_has_signal,  # noqa: F401
                    mean_reduction, shift_sequence, standardize_group)

__all__ = [
    "Config", "CONFIG_NAMES", "get_config", "make_base_weights",
    "make_adapters", "make_batch", "f32_to_bf16_bits", "bf16_bits_to_f32",
    "shift_sequence", "mean_reduction", "center_group", "group_has_signal",
    "standardize_group", "check_rl_datum",
]

_BLOCK_ELEMS = 1 << 22


@dataclass(frozen=True)
class Config:
    name: str
    vocab: int
    d_model: int
    d_ffn: int
    n_layers: int
    dtype: str                 # "bf16" (frozen base stored as bf16) or "fp32"
    n_adapters: int
    ranks: tuple
    alphas: tuple
    n_tokens: int              # tokens of the full-size workload
    loss: str                  # cross_entropy | importance_sampling | ppo | custom
    seed: int
    clip_eps: float = 0.2
    sampler_sigma: float = 0.0  # std of sampler-logprob noise (IS / PPO)
    lr: float = 1e-4
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    description: str = ""
    extra: dict = field(default_factory=dict)


def _cfg_many_tenant_ranks(seed: int, n: int) -> tuple:
    rng = np.random.Generator(np.random.PCG64([seed, 9]))
    return tuple(int(x) for x in rng.choice(np.array([8, 16, 32, 64]), size=n))


def _build_configs() -> Dict[str, Config]:
    cfgs = {}
    cfgs["tiny_fp32"] = Config(
        name="tiny_fp32", vocab=512, d_model=64, d_ffn=256, n_layers=2,
        dtype="fp32", n_adapters=3, ranks=(4, 4, 4), alphas=(8.0, 8.0, 8.0),
        n_tokens=128, loss="cross_entropy", seed=1001,
        description="tiny fp32: V=512 d=64 f=256 L=2, 3 adapters r=4 a=8, "
                    "4 seqs x 32 tokens, first 16 target positions masked, CE")
    cfgs["qwen3_4b_is"] = Config(
        name="qwen3_4b_is", vocab=151936, d_model=2560, d_ffn=9728, n_layers=4,
        dtype="bf16", n_adapters=8, ranks=(32,) * 8, alphas=(32.0,) * 8,
        n_tokens=65536, loss="importance_sampling", seed=1002,
        sampler_sigma=0.05,
        description="Qwen3-4B widths bf16: V=151936 d=2560 f=9728 L=4, 8 adapters "
                    "r=32 a=32, 8 groups x 8 completions x 1024 tokens, 25% prompt, "
                    "importance sampling")
    cfgs["qwen3_8b_ppo"] = Config(
        name="qwen3_8b_ppo", vocab=151936, d_model=4096, d_ffn=12288, n_layers=4,
        dtype="bf16", n_adapters=32, ranks=(32,) * 32, alphas=(32.0,) * 32,
        n_tokens=65536, loss="ppo", seed=1003, clip_eps=0.2, sampler_sigma=0.1,
        description="Qwen3-8B widths bf16: V=151936 d=4096 f=12288 L=4, 32 adapters "
                    "r=32 a=32, 65536 tokens in seqs of 512-2048, Zipf(1.1) adapters, "
                    "PPO clip 0.2")
    r4 = _cfg_many_tenant_ranks(1004, 128)
    cfgs["many_tenant_ce"] = Config(
        name="many_tenant_ce", vocab=151936, d_model=4096, d_ffn=12288, n_layers=2,
        dtype="bf16", n_adapters=128, ranks=r4, alphas=tuple(2.0 * r for r in r4),
        n_tokens=262144, loss="cross_entropy", seed=1004,
        description="many-tenant bf16: V=151936 d=4096 f=12288 L=2, 128 adapters "
                    "r in {8,16,32,64} a=2r, 262144 tokens in seqs of 256-4096, "
                    "Bernoulli(0.6) weights, CE + Adam")
    cfgs["long_custom"] = Config(
        name="long_custom", vocab=151936, d_model=5120, d_ffn=25600, n_layers=2,
        dtype="bf16", n_adapters=4, ranks=(64,) * 4, alphas=(64.0,) * 4,
        n_tokens=4 * 22528, loss="custom", seed=1005,
        description="long-context bf16: V=151936 d=5120 f=25600 L=2, 4 adapters "
                    "r=64 a=64, 4 seqs x 22528 tokens, 30% prompt masked, "
                    "forward_backward_custom + Adam")
    return cfgs


_CONFIGS = _build_configs()
CONFIG_NAMES = list(_CONFIGS)


def get_config(name: str, **overrides) -> Config:
    """Return a workload config by name; keyword overrides replace fields."""
    cfg = _CONFIGS[name]
    return replace(cfg, **overrides) if overrides else cfg


# ----------------------------------------------------------------------------
# bf16 storage format
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to the fp32 values they encode (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ----------------------------------------------------------------------------
# block-parallel normal draws
# ----------------------------------------------------------------------------

def _n_threads() -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        n = os.cpu_count() or 1
    return max(1, min(32, n))


def _normal_matrix(key: tuple, rows: int, cols: int, std: float, to_bf16: bool,
                   pool: Optional[ThreadPoolExecutor] = None) -> np.ndarray:
    """rows x cols matrix of N(0, std^2) draws, fp32 or bf16 bits.

    Row block i (``rows_per_block`` rows) is drawn from PCG64([*key, i]).
    """
    rows_per_block = max(1, _BLOCK_ELEMS // max(1, cols))
    n_blocks = (rows + rows_per_block - 1) // rows_per_block
    out = np.empty((rows, cols), dtype=np.uint16 if to_bf16 else np.float32)

    def fill(i):
        r0 = i * rows_per_block
        r1 = min(rows, r0 + rows_per_block)
        rng = np.random.Generator(np.random.PCG64([*key, i]))
        blk = rng.standard_normal((r1 - r0) * cols, dtype=np.float32)
        blk *= np.float32(std)
        blk = blk.reshape(r1 - r0, cols)
        out[r0:r1] = f32_to_bf16_bits(blk) if to_bf16 else blk

    if pool is None or n_blocks == 1:
        for i in range(n_blocks):
            fill(i)
    else:
        list(pool.map(fill, range(n_blocks)))
    return out


def make_base_weights(cfg: Config, std: float = 0.02) -> dict:
    """Frozen base: E [V,d], W1[l] [f,d], W2[l] [d,f], Wout [V,d].

    bf16 configs return uint16 bit patterns, fp32 configs return float32.
    """
    bf = cfg.dtype == "bf16"
    V, d, f, L = cfg.vocab, cfg.d_model, cfg.d_ffn, cfg.n_layers
    with ThreadPoolExecutor(_n_threads()) as pool:
        E = _normal_matrix((cfg.seed, 0, 0), V, d, std, bf, pool)
        Wout = _normal_matrix((cfg.seed, 0, 1), V, d, std, bf, pool)
        W1 = [_normal_matrix((cfg.seed, 0, 10 + l), f, d, std, bf, pool) for l in range(L)]
        W2 = [_normal_matrix((cfg.seed, 0, 100 + l), d, f, std, bf, pool) for l in range(L)]
    return {"E": E, "W1": W1, "W2": W2, "Wout": Wout, "dtype": cfg.dtype}


def make_adapters(cfg: Config, std_a: float = 0.02, std_b: float = 0.01) -> dict:
    """fp32 LoRA masters per adapter a and layer l.

    A1[a][l] [r,d], B1[a][l] [f,r], A2[a][l] [r,f], B2[a][l] [d,r].
    """
    d, f, L = cfg.d_model, cfg.d_ffn, cfg.n_layers
    out = {"A1": [], "B1": [], "A2": [], "B2": []}
    for a in range(cfg.n_adapters):
        r = cfg.ranks[a]
        row = {k: [] for k in out}
        for l in range(L):
            row["A1"].append(_normal_matrix((cfg.seed, 1, a, l, 0), r, d, std_a, False))
            row["B1"].append(_normal_matrix((cfg.seed, 1, a, l, 1), f, r, std_b, False))
            row["A2"].append(_normal_matrix((cfg.seed, 1, a, l, 2), r, f, std_a, False))
            row["B2"].append(_normal_matrix((cfg.seed, 1, a, l, 3), d, r, std_b, False))
        for k in out:
            out[k].append(row[k])
    return out


# ----------------------------------------------------------------------------
# batches
# ----------------------------------------------------------------------------

def _scaled(lo: int, hi: int, scale: float) -> tuple:
    return max(1, int(round(lo * scale))), max(1, int(round(hi * scale)))


def _lengths_fill(rng, total: int, lo: int, hi: int) -> List[int]:
    """Uniform integer lengths in [lo, hi] until ``total``; last one trimmed."""
    lens, acc = [], 0
    while acc < total:
        n = int(rng.integers(lo, hi + 1))
        n = min(n, total - acc)
        lens.append(n)
        acc += n
    return lens


def make_batch(cfg: Config, n_tokens: Optional[int] = None, stream: int = 0) -> dict:
    """Token batch of the config's structure with about ``n_tokens`` tokens.

    Each sequence draws T+1 ids; its inputs are the first T ids and its
    targets the last T ids (the one-token shift of the pages' datum layout).
    A smaller ``n_tokens`` scales the sequence lengths by n_tokens/full.

    Returned arrays (length N): tokens, targets, adapter_ids (int32);
    weights (CE), advantages (IS/PPO), sampler_noise (the sampler logprob of
    token t is the current logprob plus this noise), dloss (custom loss
    dL/dlogprob); plus seq_lens and seq_adapters describing the layout.
    """
    full = cfg.n_tokens
    n = full if n_tokens is None else int(n_tokens)
    scale = n / full
    rng = np.random.Generator(np.random.PCG64([cfg.seed, 2, n, stream]))
    V = cfg.vocab
    seq_lens: List[int] = []
    seq_ad: List[int] = []
    toks, tgts, w, adv, dl = [], [], [], [], []

    def new_seq(T, a, prompt_ids=None):
        if prompt_ids is None:
            ids = rng.integers(0, V, T + 1)
        else:
            ids = np.concatenate([prompt_ids, rng.integers(0, V, T + 1 - len(prompt_ids))])
        toks.append(ids[:-1])
        tgts.append(ids[1:])
        seq_lens.append(T)
        seq_ad.append(a)

    if cfg.name == "tiny_fp32":
        n_seq, T = 4, 32
        for i in range(n_seq):
            new_seq(T, i % cfg.n_adapters)
            ww = np.ones(T, np.float32)
            ww[:16] = 0.0
            w.append(ww)
    elif cfg.name == "qwen3_4b_is":
        groups, comps = 8, 8
        T = max(2, n // (groups * comps))
        P = T // 4                      # masked prompt target positions
        for g in range(groups):
            prompt = rng.integers(0, V, P + 1)
            raw = rng.standard_normal(comps)
            A = standardize_group(raw)
            for c in range(comps):
                new_seq(T, g % cfg.n_adapters, prompt)
                aa = np.zeros(T, np.float32)
                aa[P:] = A[c]
                adv.append(aa)
    elif cfg.name == "qwen3_8b_ppo":
        lo, hi = _scaled(512, 2048, scale)
        k = np.arange(1, cfg.n_adapters + 1, dtype=np.float64)
        p = k ** -1.1
        p /= p.sum()
        for T in _lengths_fill(rng, n, lo, hi):
            a = int(rng.choice(cfg.n_adapters, p=p))
            new_seq(T, a)
            adv.append(np.full(T, rng.standard_normal(), np.float32))
    elif cfg.name == "many_tenant_ce":
        lo, hi = _scaled(256, 4096, scale)
        for T in _lengths_fill(rng, n, lo, hi):
            a = int(rng.integers(0, cfg.n_adapters))
            new_seq(T, a)
            w.append((rng.random(T) < 0.6).astype(np.float32))
    elif cfg.name == "long_custom":
        n_seq = 4
        T = max(2, n // n_seq)
        P = int(0.3 * T)
        for i in range(n_seq):
            new_seq(T, i % cfg.n_adapters)
            mask = np.ones(T, np.float32)
            mask[:P] = 0.0
            dl.append((rng.standard_normal(T).astype(np.float32) * mask).astype(np.float32))
    else:
        raise KeyError(cfg.name)

    tokens = np.concatenate(toks).astype(np.int32)
    N = len(tokens)
    out = {
        "tokens": tokens,
        "targets": np.concatenate(tgts).astype(np.int32),
        "adapter_ids": np.repeat(np.array(seq_ad, np.int32), seq_lens).astype(np.int32),
        "seq_lens": np.array(seq_lens, np.int64),
        "seq_adapters": np.array(seq_ad, np.int32),
        "weights": np.concatenate(w).astype(np.float32) if w else np.zeros(N, np.float32),
        "advantages": np.concatenate(adv).astype(np.float32) if adv else np.zeros(N, np.float32),
        "dloss": np.concatenate(dl).astype(np.float32) if dl else np.zeros(N, np.float32),
        "sampler_noise": (rng.standard_normal(N) * cfg.sampler_sigma).astype(np.float32),
        "loss": cfg.loss,
        "clip_eps": cfg.clip_eps,
    }
    return out
