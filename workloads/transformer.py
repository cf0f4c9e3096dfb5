"""Seeded synthetic inputs for the transformer-block variant of the step.

Shared by the CUDA path's tests and benchmark and by the CPU oracle; holds no
arithmetic of the method (random draws, sequence layout, bf16 rounding only).

The block is a pre-norm decoder layer: RMSNorm, grouped-head causal
attention with rotary positions, RMSNorm, gated SiLU MLP; every one of the
seven projections q, k, v, o, gate, up, down carries per-adapter LoRA
(tinker-ticks, "How the SGMV kernel works": seven adapted projections per
layer).  Workloads:

* ``tf_small``        V=1000, d=256, 4 query / 2 key-value heads of 128,
                       f=512, L=2, 3 adapters ranks 8/16/32; sequences of
                       20-300 tokens, adapters uniform.  Parity size.
* ``qwen3_8b_tf_ppo`` Qwen3-8B widths (d=4096, 32 query / 8 key-value heads
                       of 128, f=12288, V=151936), L=4, 32 adapters rank 32,
                       65,536 tokens in sequences of 512-2048 tokens,
                       Zipf(1.1) adapter choice, PPO clip 0.2: the 8B-width
                       workload of the MLP model with the real block.

Draws follow the MLP workloads: numpy PCG64 streams keyed by (seed, tensor
id, block); base weights N(0, w_std) rounded to bf16; norm gains 1 + N(0,
0.1) rounded to bf16; adapters fp32 masters, A ~ N(0, 0.02), B ~ N(0, 0.01);
token ids uniform; sequences laid out contiguously in generation order, each
token's position its index inside its sequence.  qk_std > 0 draws the q and k
weights at that scale instead (at d = 256, 0.08 makes the attention scores
spread like those of the 8B widths at 0.02: query entries of standard
deviation ~1.3).
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace
from typing import Dict, Optional

import numpy as np

from . import _lengths_fill, _n_threads, _normal_matrix, _scaled, f32_to_bf16_bits

PROJ = ("q", "k", "v", "o", "gate", "up", "down")


@dataclass(frozen=True)
class TfConfig:
    name: str
    vocab: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    d_ffn: int
    n_layers: int
    n_adapters: int
    ranks: tuple
    alphas: tuple
    n_tokens: int
    loss: str
    seed: int
    seq_lo: int
    seq_hi: int
    adapter_dist: str = "uniform"     # uniform | zipf
    w_std: float = 0.02
    qk_std: float = 0.0                # q / k weights (0: w_std)
    clip_eps: float = 0.2
    sampler_sigma: float = 0.1
    rope_theta: float = 1e6
    rms_eps: float = 1e-6
    lr: float = 1e-4
    dtype: str = "bf16"
    description: str = ""


def proj_shapes(cfg: TfConfig) -> dict:
    """(out, in) of each projection's frozen weight [out x in]."""
    q, kv = cfg.n_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    d, f = cfg.d_model, cfg.d_ffn
    return {"q": (q, d), "k": (kv, d), "v": (kv, d), "o": (d, q),
            "gate": (f, d), "up": (f, d), "down": (d, f)}


_TF = {
    "tf_small": TfConfig(
        name="tf_small", vocab=1000, d_model=256, n_heads=4, n_kv_heads=2, head_dim=128,
        d_ffn=512, n_layers=2, n_adapters=3, ranks=(8, 16, 32), alphas=(16.0, 16.0, 32.0),
        n_tokens=1024, loss="ppo", seed=2001, seq_lo=20, seq_hi=300,
        description="small transformer bf16: V=1000 d=256 4q/2kv heads x 128 f=512 L=2, "
                    "3 adapters r=8/16/32, seqs of 20-300 tokens"),
    "qwen3_8b_tf_ppo": TfConfig(
        name="qwen3_8b_tf_ppo", vocab=151936, d_model=4096, n_heads=32, n_kv_heads=8,
        head_dim=128, d_ffn=12288, n_layers=4, n_adapters=32, ranks=(32,) * 32,
        alphas=(32.0,) * 32, n_tokens=65536, loss="ppo", seed=2003, seq_lo=512,
        seq_hi=2048, adapter_dist="zipf",
        description="Qwen3-8B widths transformer bf16: V=151936 d=4096 32q/8kv heads x 128 "
                    "f=12288 L=4, 32 adapters r=32 a=32, 65536 tokens in seqs of 512-2048, "
                    "Zipf(1.1) adapters, PPO clip 0.2"),
}
TF_CONFIG_NAMES = list(_TF)


def get_tf_config(name: str, **overrides) -> TfConfig:
    cfg = _TF[name]
    return replace(cfg, **overrides) if overrides else cfg


def make_tf_base_weights(cfg: TfConfig) -> dict:
    """Frozen base as bf16 bit patterns: E, Wout [V x d]; final_norm [d];
    attn_norm[l], mlp_norm[l] [d]; W[p][l] [out x in]."""
    V, d, L = cfg.vocab, cfg.d_model, cfg.n_layers
    shapes = proj_shapes(cfg)
    with ThreadPoolExecutor(_n_threads()) as pool:
        E = _normal_matrix((cfg.seed, 0, 0), V, d, cfg.w_std, True, pool)
        Wout = _normal_matrix((cfg.seed, 0, 1), V, d, cfg.w_std, True, pool)
        std = {p: (cfg.qk_std if p in ("q", "k") and cfg.qk_std > 0 else cfg.w_std) for p in PROJ}
        W = {p: [_normal_matrix((cfg.seed, 0, 10 + 10 * i, l), *shapes[p], std[p], True, pool)
                 for l in range(L)] for i, p in enumerate(PROJ)}

    def gain(key):
        g = 1.0 + _normal_matrix((cfg.seed, 3) + key, 1, d, 0.1, False)[0]
        return f32_to_bf16_bits(g)

    return {"E": E, "Wout": Wout, "W": W, "final_norm": gain((0,)),
            "attn_norm": [gain((1, l)) for l in range(L)],
            "mlp_norm": [gain((2, l)) for l in range(L)], "dtype": "bf16"}


def make_tf_adapters(cfg: TfConfig, std_a: float = 0.02, std_b: float = 0.01) -> dict:
    """fp32 masters: A[p][a][l] [r x in], B[p][a][l] [out x r]."""
    shapes = proj_shapes(cfg)
    A = {p: [] for p in PROJ}
    B = {p: [] for p in PROJ}
    for a in range(cfg.n_adapters):
        r = cfg.ranks[a]
        for i, p in enumerate(PROJ):
            out, inp = shapes[p]
            A[p].append([_normal_matrix((cfg.seed, 1, a, l, 2 * i), r, inp, std_a, False)
                         for l in range(cfg.n_layers)])
            B[p].append([_normal_matrix((cfg.seed, 1, a, l, 2 * i + 1), out, r, std_b, False)
                         for l in range(cfg.n_layers)])
    return {"A": A, "B": B}


def make_tf_batch(cfg: TfConfig, n_tokens: Optional[int] = None, stream: int = 0) -> dict:
    """Token batch with per-token positions.  Each sequence draws T+1 ids
    (inputs the first T, targets the last T).  A smaller n_tokens scales the
    sequence lengths by n_tokens / full.  Every loss kind's inputs are drawn:
    weights Bernoulli(0.7), advantages N(0,1) per sequence, dloss N(0,1),
    sampler_noise N(0, sampler_sigma) (the sampler logprob is the current
    logprob plus this noise)."""
    n = cfg.n_tokens if n_tokens is None else int(n_tokens)
    scale = n / cfg.n_tokens
    lo, hi = _scaled(cfg.seq_lo, cfg.seq_hi, scale)
    rng = np.random.Generator(np.random.PCG64([cfg.seed, 2, n, stream]))
    if cfg.adapter_dist == "zipf":
        k = np.arange(1, cfg.n_adapters + 1, dtype=np.float64)
        pz = k ** -1.1
        pz /= pz.sum()
    toks, tgts, pos, ads, adv = [], [], [], [], []
    for T in _lengths_fill(rng, n, lo, hi):
        if cfg.adapter_dist == "zipf":
            a = int(rng.choice(cfg.n_adapters, p=pz))
        else:
            a = int(rng.integers(0, cfg.n_adapters))
        ids = rng.integers(0, cfg.vocab, T + 1)
        toks.append(ids[:-1])
        tgts.append(ids[1:])
        pos.append(np.arange(T))
        ads.append(np.full(T, a))
        adv.append(np.full(T, rng.standard_normal()))
    N = sum(len(t) for t in toks)
    return {
        "tokens": np.concatenate(toks).astype(np.int32),
        "targets": np.concatenate(tgts).astype(np.int32),
        "positions": np.concatenate(pos).astype(np.int32),
        "adapter_ids": np.concatenate(ads).astype(np.int32),
        "weights": (rng.random(N) < 0.7).astype(np.float32),
        "advantages": np.concatenate(adv).astype(np.float32),
        "dloss": rng.standard_normal(N).astype(np.float32),
        "sampler_noise": (rng.standard_normal(N) * cfg.sampler_sigma).astype(np.float32),
        "loss": cfg.loss,
        "clip_eps": cfg.clip_eps,
    }
