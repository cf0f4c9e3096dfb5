"""Sampler side on the GPU: scoring and one-token decode with pinned adapter
snapshots, against the training path and the oracle.

OpenTinker ("Multi-LoRA rollout"): rows are batched by pinned adapter
version over the shared base.  tinker-ticks ("Why RL needs batch-invariant
kernels"): rollout and training logprobs must agree bit for bit.  So the
sampler's logprobs are compared bitwise with the training handle's
mlora_forward on the same tokens and adapter weights, and within the bf16
tolerance with the oracle; sampled tokens are checked against the oracle's
inverse CDF (exactly where the distribution's rounding leaves no doubt).
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from _gpu_util import create_handle, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _bits(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32)


def _cfg(dtype, V=4096, d=512, f=1536, L=2, ranks=(32, 16, 64, 8), seed=4001):
    return wl.Config(name="mid_" + dtype, vocab=V, d_model=d, d_ffn=f, n_layers=L, dtype=dtype,
                     n_adapters=len(ranks), ranks=tuple(ranks),
                     alphas=tuple(float(2 * r) for r in ranks), n_tokens=512,
                     loss="cross_entropy", seed=seed)


def _rows(cfg, n, key):
    rng = np.random.Generator(np.random.PCG64([cfg.seed, 11, key]))
    return {"tokens": rng.integers(0, cfg.vocab, n).astype(np.int32),
            "targets": rng.integers(0, cfg.vocab, n).astype(np.int32),
            "adapter_ids": rng.integers(0, cfg.n_adapters, n).astype(np.int32),
            "u": rng.random(n).astype(np.float32)}


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_scoring_is_bitwise_the_training_forward(dtype):
    """Slot a = snapshot of adapter a: the sampler's logprobs of mixed-slot
    rows equal mlora_forward's bitwise, at 1, 77 and 700 rows (block GEMMs on
    the single-CTA kernel) and 2048 rows (on the CTA-pair kernel)."""
    import rl_step_gb300 as m
    cfg = _cfg(dtype, seed=4001 if dtype == "bf16" else 4002)
    base = wl.make_base_weights(cfg)
    ad = wl.make_adapters(cfg, std_a=0.05, std_b=0.05)
    h = create_handle(cfg, base, ad, 2048)
    smp = m.mlora_sampler_create(h, 6, 2048)
    for a in range(cfg.n_adapters):
        assert m.mlora_sampler_publish(smp, a, a) == 0
    o = oracle.Oracle(base, ad, cfg.ranks, cfg.alphas)
    for n in (1, 77, 700, 2048):
        b = _rows(cfg, n, n)
        tok, tgt, ids = dev(b["tokens"]), dev(b["targets"]), dev(b["adapter_ids"])
        lp_s = m.mlora_sampler_logprobs(smp, tok, tgt, ids).cpu().numpy()
        assert m.mlora_sampler_check_status(smp) == 0
        lp_t = m.mlora_forward(h, tok, tgt, ids).cpu().numpy()
        assert np.array_equal(_bits(lp_s), _bits(lp_t)), n
        ref = o.forward(b["tokens"], b["targets"], b["adapter_ids"])
        tol = 2e-2 if dtype == "bf16" else 1e-4
        assert np.max(np.abs(lp_s - ref)) <= tol


def test_snapshot_is_pinned_until_republished():
    """Training adapter 0 after publishing leaves slot 0's logprobs bitwise
    unchanged; publishing again gives the trained weights' logprobs (the
    training handle's, bitwise) and the new version number."""
    import rl_step_gb300 as m
    cfg = _cfg("bf16", seed=4003)
    base = wl.make_base_weights(cfg)
    ad = wl.make_adapters(cfg, std_a=0.05, std_b=0.05)
    h = create_handle(cfg, base, ad, 1024)
    smp = m.mlora_sampler_create(h, 2, 512)
    assert m.mlora_sampler_publish(smp, 0, 0) == 0
    b = _rows(cfg, 300, 1)
    slots = np.zeros(300, np.int32)
    tok, tgt, sl = dev(b["tokens"]), dev(b["targets"]), dev(slots)
    before = m.mlora_sampler_logprobs(smp, tok, tgt, sl).cpu().numpy()
    lp_t0 = m.mlora_forward(h, tok, tgt, sl).cpu().numpy()
    assert np.array_equal(_bits(before), _bits(lp_t0))
    # one training step of adapter 0
    m.mlora_forward_backward(h, tok, tgt, sl, "cross_entropy",
                             weights=dev(np.ones(300, np.float32)))
    m.mlora_optim_step(h, lr=1e-2)
    lp_t1 = m.mlora_forward(h, tok, tgt, sl).cpu().numpy()
    assert not np.array_equal(_bits(lp_t1), _bits(lp_t0))
    pinned = m.mlora_sampler_logprobs(smp, tok, tgt, sl).cpu().numpy()
    assert np.array_equal(_bits(pinned), _bits(before))
    assert m.mlora_sampler_publish(smp, 0, 0) == 1
    after = m.mlora_sampler_logprobs(smp, tok, tgt, sl).cpu().numpy()
    assert np.array_equal(_bits(after), _bits(lp_t1))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_sampling_uniform_distribution_is_floor_uV(dtype):
    """Wout = 0: every next-token distribution is uniform, so the token is
    floor(u V) wherever u V is not within rounding of an integer; V = 1000
    leaves a ragged last vocabulary tile."""
    import rl_step_gb300 as m
    cfg = _cfg(dtype, V=1000, d=256, f=512, L=1, ranks=(16, 8), seed=4004)
    base = wl.make_base_weights(cfg)
    base = dict(base)
    base["Wout"] = np.zeros_like(base["Wout"])
    ad = wl.make_adapters(cfg)
    h = create_handle(cfg, base, ad, 512)
    smp = m.mlora_sampler_create(h, 2, 512)
    m.mlora_sampler_publish(smp, 0, 0)
    m.mlora_sampler_publish(smp, 1, 1)
    rng = np.random.Generator(np.random.PCG64([4004, 3]))
    n = 500
    u = rng.random(n).astype(np.float32)
    u[:6] = np.array([0.0, 1e-7, 0.2561, 0.7689, 0.9995, 0.99999994], np.float32)
    tok = rng.integers(0, cfg.vocab, n).astype(np.int32)
    sl = rng.integers(0, 2, n).astype(np.int32)
    nxt, lp = m.mlora_sampler_sample(smp, dev(tok), dev(sl), dev(u))
    assert m.mlora_sampler_check_status(smp) == 0
    nxt, lp = nxt.cpu().numpy(), lp.cpu().numpy()
    x = u.astype(np.float64) * cfg.vocab
    frac = x - np.floor(x)
    clear = (frac > 1e-3) & (frac < 1 - 1e-3)
    assert np.array_equal(nxt[clear], np.floor(x[clear]).astype(np.int32))
    assert (np.abs(nxt - np.floor(x)) <= 1).all()
    assert np.max(np.abs(lp + np.log(cfg.vocab))) <= 1e-5


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_sampling_against_oracle_inverse_cdf(dtype):
    """Mixed slots: each sampled token's oracle CDF interval contains u up to
    the logprob tolerance carried into the CDF, most tokens equal the
    oracle's, and the returned logprob is bitwise the sampler's score of that
    token (and within tolerance of the oracle's)."""
    import rl_step_gb300 as m
    cfg = _cfg(dtype, V=2000, d=256, f=768, L=2, ranks=(16, 32, 8), seed=4005)
    base = dict(wl.make_base_weights(cfg, std=0.08))
    # a wide LM head makes the next-token distributions peaked (logit std ~2)
    wout = np.random.Generator(np.random.PCG64([cfg.seed, 12])).standard_normal(
        (cfg.vocab, cfg.d_model)).astype(np.float32) * 1.5
    base["Wout"] = wl.f32_to_bf16_bits(wout) if dtype == "bf16" else wout
    ad = wl.make_adapters(cfg, std_a=0.05, std_b=0.05)
    h = create_handle(cfg, base, ad, 512)
    smp = m.mlora_sampler_create(h, 3, 512)
    for a in range(3):
        m.mlora_sampler_publish(smp, a, a)
    b = _rows(cfg, 400, 7)
    ids = b["adapter_ids"] % 3
    tok, sl, u = dev(b["tokens"]), dev(ids.astype(np.int32)), dev(b["u"])
    nxt, lp = m.mlora_sampler_sample(smp, tok, sl, u)
    assert m.mlora_sampler_check_status(smp) == 0
    nxt_n, lp_n = nxt.cpu().numpy(), lp.cpu().numpy()
    again = m.mlora_sampler_logprobs(smp, tok, nxt, sl).cpu().numpy()
    assert np.array_equal(_bits(again), _bits(lp_n))
    o = oracle.Oracle(base, ad, cfg.ranks, cfg.alphas)
    cdf = o.next_token_cdf(b["tokens"], ids)
    v = nxt_n.astype(np.int64)
    lo = np.where(v > 0, cdf[np.arange(len(v)), np.maximum(v - 1, 0)], 0.0)
    hi = cdf[np.arange(len(v)), v]
    # Logprob error bound per row.  The wide LM head scales the logits (|z| up
    # to ~10), so besides the workloads' tolerance the bf16 rounding of the
    # final hidden state (2^-9 per element, then the log-sum-exp) counts:
    # |dz_v| <= 2^-9 sum_i |h_i W_vi| for every v, twice for z_y - lse.
    hid = o.forward_hidden(b["tokens"], ids)[0]
    wabs = np.abs(wl.bf16_bits_to_f32(base["Wout"]) if dtype == "bf16" else base["Wout"]).astype(np.float64)
    zmag = (np.abs(hid) @ wabs.T).max(axis=1)
    lp_tol = (2e-2 + 2.0 ** -8 * zmag) if dtype == "bf16" else np.full(len(zmag), 1e-4)
    # CDF(v) = sum_w p_w exp(d_w) with |d_w| <= lp_tol moves by at most ~lp_tol
    slack = lp_tol
    uu = b["u"].astype(np.float64)
    assert ((lo - slack <= uu) & (uu <= hi + slack)).all()
    ref_next, ref_lp, _, _ = o.sample(b["tokens"], ids, uu)
    same = nxt_n == ref_next
    print(f"\n[{dtype}] sampled tokens equal to the oracle's: {same.mean():.3f}")
    assert same.mean() >= (0.8 if dtype == "bf16" else 0.99)
    err = np.abs(lp_n - np.log(hi - lo))
    print(f"[{dtype}] sampled-token logprob error max {err.max():.3e} (bound {lp_tol.min():.3e}-{lp_tol.max():.3e})")
    assert (err <= lp_tol).all()


def test_bad_rows_are_flagged():
    import torch
    import rl_step_gb300 as m
    cfg = _cfg("bf16", V=1000, d=256, f=512, L=1, ranks=(16, 8), seed=4006)
    base = wl.make_base_weights(cfg)
    ad = wl.make_adapters(cfg)
    h = create_handle(cfg, base, ad, 64)
    smp = m.mlora_sampler_create(h, 3, 64)
    m.mlora_sampler_publish(smp, 0, 1)
    tok = np.array([1, 2, 3, 4, 5], np.int32)
    tgt = np.array([1, 2000, 3, 4, 5], np.int32)      # row 1: target out of range
    sl = np.array([0, 0, 2, 7, 0], np.int32)          # row 2 unpublished, row 3 out of range
    lp = m.mlora_sampler_logprobs(smp, dev(tok), dev(tgt), dev(sl)).cpu().numpy()
    assert m.mlora_sampler_check_status(smp) == -2
    assert np.isfinite(lp[[0, 4]]).all() and np.isnan(lp[[1, 2, 3]]).all()
    u = np.array([0.5, 0.5, 0.5, 0.5, 1.5], np.float32)   # row 4: u out of range
    nxt, lps = m.mlora_sampler_sample(smp, dev(tok), dev(sl), dev(u))
    assert m.mlora_sampler_check_status(smp) == -2
    nxt = nxt.cpu().numpy()
    assert nxt[0] >= 0 and nxt[1] >= 0 and (nxt[2:] == -1).all()
    with pytest.raises(m.MLoRAError):
        m.mlora_sampler_logprobs(smp, dev(np.zeros(65, np.int32)), dev(np.zeros(65, np.int32)),
                                 dev(np.zeros(65, np.int32)))
    e = torch.empty(0, dtype=torch.int32, device="cuda")
    assert m.mlora_sampler_logprobs(smp, e, e, e).numel() == 0
