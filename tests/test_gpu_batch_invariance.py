"""Batch invariance and the deterministic mode, on the GPU.

tinker-ticks, "Why RL needs batch-invariant kernels": the logprob of a token
must not depend on how many other tokens (of other tenants) share the
flattened batch, and the rollout (sampler) and training logprobs of the same
tokens must agree bit for bit.  With mlora_set_deterministic(h, 1) the
adapter gradients, losses and post-Adam weights must also repeat bit for bit
and must not depend on which other adapters share the batch.

The problem is mid-sized (V=4096, d=512, f=1536, L=2, four adapters of ranks
8-64) so that it runs the same kernels as the full workloads (CTA-pair GEMMs
for the dense products, grouped gradient GEMMs) while adapter 0 owns more
than 1024 padded rows, i.e. several 1024-row gradient chunks in the default
mode.  Every input is seeded; bitwise checks compare the CUDA path with
itself, and the one parity check compares it with the oracle.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from _gpu_util import create_handle, dev, grad_errors

pytestmark = pytest.mark.gpu

N_Y = 4655          # the mixed batch
N_X = 47            # one short sequence of adapter 0 inside it


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _cfg(dtype):
    return wl.Config(name="mid_" + dtype, vocab=4096, d_model=512, d_ffn=1536, n_layers=2,
                     dtype=dtype, n_adapters=4, ranks=(32, 16, 64, 8),
                     alphas=(32.0, 32.0, 64.0, 16.0), n_tokens=N_Y, loss="ppo",
                     seed=2001 if dtype == "bf16" else 2002)


def _sequences(cfg, n_total, x_seq, key):
    """Sequences of random adapters (adapter 0 the most frequent) filling
    n_total tokens, with the sequence x_seq (adapter 0) in the middle."""
    rng = np.random.Generator(np.random.PCG64([cfg.seed, 7, key]))
    V = cfg.vocab
    seqs, ads, advs = [], [], []
    n = 0
    target = n_total - (len(x_seq) - 1)
    while n < target:
        T = int(min(rng.integers(40, 600), target - n))
        seqs.append(rng.integers(0, V, T + 1))
        ads.append(int(rng.choice(4, p=[0.55, 0.15, 0.15, 0.15])))
        advs.append(float(rng.standard_normal()))
        n += T
    mid = len(seqs) // 2
    seqs.insert(mid, x_seq)
    ads.insert(mid, 0)
    advs.insert(mid, 0.75)
    tokens = np.concatenate([s[:-1] for s in seqs]).astype(np.int32)
    targets = np.concatenate([s[1:] for s in seqs]).astype(np.int32)
    ids = np.concatenate([np.full(len(s) - 1, a, np.int32) for s, a in zip(seqs, ads)])
    adv = np.concatenate([np.full(len(s) - 1, v, np.float32) for s, v in zip(seqs, advs)])
    x0 = sum(len(s) - 1 for s in seqs[:mid])
    x_pos = np.arange(x0, x0 + len(x_seq) - 1)
    noise = (0.1 * rng.standard_normal(len(tokens))).astype(np.float32)
    sampler = (noise - np.float32(np.log(V))).astype(np.float32)
    return {"tokens": tokens, "targets": targets, "adapter_ids": ids, "advantages": adv,
            "sampler": sampler, "x_pos": x_pos}


def _problem(dtype):
    cfg = _cfg(dtype)
    base = wl.make_base_weights(cfg)
    ad = wl.make_adapters(cfg)
    rng = np.random.Generator(np.random.PCG64([cfg.seed, 8]))
    x_seq = rng.integers(0, cfg.vocab, N_X + 1)
    Y = _sequences(cfg, N_Y, x_seq, 0)
    Y2 = _sequences(cfg, N_Y + 3000, x_seq, 1)     # another mix of another size
    return cfg, base, ad, x_seq, Y, Y2


def _subset(b, rows):
    return {k: (v[rows] if k != "x_pos" else v) for k, v in b.items()}


def _bits(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32)


def _fwd(h, b):
    import rl_step_gb300 as m
    return m.mlora_forward(h, dev(b["tokens"]), dev(b["targets"]),
                           dev(b["adapter_ids"])).cpu().numpy()


def _fwd_bwd(h, b, cfg):
    import rl_step_gb300 as m
    lp, loss = m.mlora_forward_backward(h, dev(b["tokens"]), dev(b["targets"]),
                                        dev(b["adapter_ids"]), "ppo",
                                        advantages=dev(b["advantages"]),
                                        sampler_logprobs=dev(b["sampler"]), clip_eps=0.2)
    assert m.mlora_check_status(h) == 0
    return lp.cpu().numpy(), loss.cpu().numpy()


def _adapter_state(h, cfg, a, prefixes):
    import rl_step_gb300 as m
    return {(p, l, k): m.mlora_read_adapter(h, a, l, p + k).cpu().numpy()
            for p in prefixes for l in range(cfg.n_layers) for k in oracle.TENSORS}


def _assert_same_bits(s1, s2):
    for key in s1:
        assert np.array_equal(_bits(s1[key]), _bits(s2[key])), key


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_logprobs_do_not_depend_on_the_batch(dtype):
    """Sampler-side and training-side logprobs of the same 47 tokens are bitwise
    equal alone, inside a 4655-token mixed batch and inside a 7655-token one."""
    cfg, base, ad, x_seq, Y, Y2 = _problem(dtype)
    h = create_handle(cfg, base, ad, len(Y2["tokens"]))
    X = _subset(Y, Y["x_pos"])
    assert np.array_equal(X["tokens"], x_seq[:-1]) and (X["adapter_ids"] == 0).all()
    lp_x = _fwd(h, X)
    lp_y = _fwd(h, Y)
    lp_y2 = _fwd(h, Y2)
    assert np.isfinite(lp_x).all()
    assert np.array_equal(_bits(lp_y[Y["x_pos"]]), _bits(lp_x))
    assert np.array_equal(_bits(lp_y2[Y2["x_pos"]]), _bits(lp_x))
    # the training pass reports the very same logprobs (rollout == training)
    lp_train, _ = _fwd_bwd(h, Y, cfg)
    assert np.array_equal(_bits(lp_train), _bits(lp_y))
    lp_train_x, _ = _fwd_bwd(h, X, cfg)
    assert np.array_equal(_bits(lp_train_x), _bits(lp_x))
    # a single token too
    one = _subset(X, np.arange(1))
    assert np.array_equal(_bits(_fwd(h, one)), _bits(lp_x[:1]))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_deterministic_mode_repeats_and_ignores_other_tenants(dtype):
    """Deterministic mode: adapter 0's loss, gradients and post-Adam state are
    bitwise equal over two runs of the mixed batch and a run of adapter 0's
    tokens alone; the other adapters repeat bitwise across the two runs."""
    import rl_step_gb300 as m
    cfg, base, ad, _, Y, _ = _problem(dtype)
    rows0 = np.nonzero(Y["adapter_ids"] == 0)[0]
    assert len(rows0) > 1024                       # several chunks in the default mode
    Z = _subset(Y, rows0)
    hs = [create_handle(cfg, base, ad, len(Y["tokens"])) for _ in range(3)]
    for h in hs:
        m.mlora_set_deterministic(h, True)
    lp1, loss1 = _fwd_bwd(hs[0], Y, cfg)
    lp2, loss2 = _fwd_bwd(hs[1], Y, cfg)
    lpz, lossz = _fwd_bwd(hs[2], Z, cfg)
    assert np.array_equal(_bits(lp1), _bits(lp2))
    assert np.array_equal(_bits(lp1[rows0]), _bits(lpz))
    assert np.array_equal(loss1.view(np.uint64), loss2.view(np.uint64))
    assert loss1[0] == lossz[0]
    g = [_adapter_state(h, cfg, 0, ["g"]) for h in hs]
    _assert_same_bits(g[0], g[1])
    _assert_same_bits(g[0], g[2])
    for a in range(1, cfg.n_adapters):
        _assert_same_bits(_adapter_state(hs[0], cfg, a, ["g"]), _adapter_state(hs[1], cfg, a, ["g"]))
    for h in hs:
        m.mlora_optim_step(h, lr=1e-3, adapters=[0])
    s = [_adapter_state(h, cfg, 0, ["", "m", "v"]) for h in hs]
    _assert_same_bits(s[0], s[1])
    _assert_same_bits(s[0], s[2])


def test_deterministic_mode_matches_the_oracle():
    """The one-chunk-per-adapter reduction is the same sum: gradients within
    the parity tolerance of the oracle, and close to the default mode's."""
    import rl_step_gb300 as m
    cfg, base, ad, _, Y, _ = _problem("bf16")
    o = oracle.Oracle(base, ad, cfg.ranks, cfg.alphas)
    b = dict(Y)
    b["sampler"] = (o.forward(Y["tokens"], Y["targets"], Y["adapter_ids"])
                    + 0.1 * Y["sampler"] + 0.1 * np.log(cfg.vocab)).astype(np.float32)
    hd = create_handle(cfg, base, ad, len(Y["tokens"]))
    m.mlora_set_deterministic(hd, True)
    hn = create_handle(cfg, base, ad, len(Y["tokens"]))
    _fwd_bwd(hd, b, cfg)
    _fwd_bwd(hn, b, cfg)
    o.forward_backward(Y["tokens"], Y["targets"], Y["adapter_ids"], "ppo",
                       advantages=Y["advantages"], sampler_logprobs=b["sampler"], clip_eps=0.2)
    err, where = grad_errors(hd, o, range(cfg.n_adapters))
    print(f"\n[deterministic, mid bf16] grad rel Fro max={err:.3e} at {where}")
    assert err <= 1e-2
    worst = 0.0
    for a in range(cfg.n_adapters):
        gd = _adapter_state(hd, cfg, a, ["g"])
        gn = _adapter_state(hn, cfg, a, ["g"])
        for key in gd:
            nr = np.linalg.norm(gn[key])
            worst = max(worst, float(np.linalg.norm(gd[key] - gn[key]) / nr))
    print(f"[deterministic vs default] grad rel Fro max={worst:.3e}")
    assert worst <= 1e-5
