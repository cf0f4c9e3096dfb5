"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Tolerances (fixed by the method's specification): logprobs max abs error
<= 1e-4 for the fp32 base and <= 2e-2 for the bf16 base; adapter gradients
and post-Adam adapter weights relative Frobenius error <= 1e-2; routing
bit-exact.  Every input is seeded; the oracle alone produces expected values
(sampler logprobs of the IS / PPO workloads come from an oracle forward).
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from _gpu_util import (create_handle, dev, grad_errors, rel_fro, run_gpu_step,
                       run_oracle_step)

pytestmark = pytest.mark.gpu

LP_TOL = {"fp32": 1e-4, "bf16": 2e-2}
GRAD_TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


# --------------------------------------------------------------------- routing

@pytest.mark.parametrize("n,n_ad,seed", [(1, 1, 0), (127, 3, 1), (129, 3, 2), (1000, 17, 3),
                                         (5000, 128, 4), (4096, 4, 5), (3000, 1, 6)])
def test_routing_bit_exact(n, n_ad, seed):
    import rl_step_gb300 as m
    cfg = wl.get_config("tiny_fp32", n_adapters=n_ad, ranks=(4,) * n_ad, alphas=(8.0,) * n_ad)
    base = wl.make_base_weights(cfg)
    ad = wl.make_adapters(cfg)
    h = create_handle(cfg, base, ad, max(n, 1))
    rng = np.random.Generator(np.random.PCG64([17, seed]))
    ids = rng.integers(0, n_ad, n).astype(np.int32)
    if n_ad > 2:
        ids[ids == 1] = 0                       # an empty segment
    perm, seg, pad, tiles = m.mlora_get_routing(h, dev(ids))
    ref = oracle.routing(ids, n_ad, m.TILE_M)
    assert m.mlora_check_status(h) == 0
    assert np.array_equal(perm.cpu().numpy(), ref["perm"])
    assert np.array_equal(seg.cpu().numpy(), ref["seg_off"])
    assert np.array_equal(pad.cpu().numpy(), ref["pad_off"])
    t = tiles.cpu().numpy()
    nt = len(ref["tile_ad"])
    assert np.array_equal(t[:nt], ref["tile_ad"]) and (t[nt:] == -1).all()


def test_routing_flags_out_of_range_ids():
    import rl_step_gb300 as m
    cfg = wl.get_config("tiny_fp32")
    h = create_handle(cfg, wl.make_base_weights(cfg), wl.make_adapters(cfg), 64)
    ids = np.array([0, 1, 7, 2, -1, 0], np.int32)
    perm, seg, pad, tiles = m.mlora_get_routing(h, dev(ids))
    assert m.mlora_check_status(h) == -2
    ok = ids[(ids >= 0) & (ids < 3)]
    ref = oracle.routing(ok, 3, m.TILE_M)
    assert seg.cpu().numpy().tolist() == ref["seg_off"].tolist()
    assert m.mlora_check_status(h) == 0          # status cleared


# --------------------------------------------------------------- full steps

# Odd widths: d = 320 and f = 704 are 5 and 11 blocks of 64 along K, so the CTA-pair
# GEMMs (two K blocks per pipeline stage) end every tile on a half-filled stage.
ODD_K = {"d_model": 320, "d_ffn": 704, "vocab": 4000}

CASES = [("tiny_fp32", None, None), ("qwen3_4b_is", 1024, None), ("qwen3_8b_ppo", 1024, None),
         ("many_tenant_ce", 2048, None), ("long_custom", 512, None), ("qwen3_8b_ppo", 1024, ODD_K)]


def _setup(name, n, overrides=None):
    cfg = wl.get_config(name, **(overrides or {}))
    base = wl.make_base_weights(cfg)
    ad = wl.make_adapters(cfg)
    b = wl.make_batch(cfg, n)
    o = oracle.Oracle(base, ad, cfg.ranks, cfg.alphas)
    s = None
    if cfg.loss in ("importance_sampling", "ppo"):
        s = o.forward(b["tokens"], b["targets"], b["adapter_ids"]) + b["sampler_noise"]
    return cfg, base, ad, b, o, s


@pytest.mark.parametrize("lm", ["recompute", "keep_logits"])
@pytest.mark.parametrize("name,n,overrides", CASES,
                         ids=[c[0] + ("_odd_k_blocks" if c[2] else "") for c in CASES])
def test_step_parity(name, n, overrides, lm):
    import rl_step_gb300 as m
    cfg, base, ad, b, o, s = _setup(name, n, overrides)
    kind = cfg.loss
    N = len(b["tokens"])
    h = create_handle(cfg, base, ad, N, lm_backward=lm)
    lp, loss = run_gpu_step(h, b, kind, s)
    assert m.mlora_check_status(h) == 0
    ref = run_oracle_step(o, b, kind, s)
    lp_err = float(np.max(np.abs(lp - ref["logprobs"])))
    dev_gpu = lp + np.log(cfg.vocab)
    dev_ref = ref["logprobs"] + np.log(cfg.vocab)
    present = np.unique(b["adapter_ids"])
    g_err, g_where = grad_errors(h, o, present)
    # per-adapter loss sums cancel (centred advantages): scale by sum |value|
    val, _ = oracle.token_loss(kind if kind != "custom" else "custom", ref["logprobs"],
                               **({"dloss": b["dloss"]} if kind == "custom" else
                                  {"weights": b["weights"]} if kind == "cross_entropy" else
                                  {"advantages": b["advantages"], "sampler_logprobs": s,
                                   "clip_eps": b["clip_eps"]}))
    scale = np.array([np.abs(val[b["adapter_ids"] == a]).sum() for a in present])
    loss_err = float(np.max(np.abs(loss[present] - ref["loss_per_adapter"][present]) /
                            np.maximum(scale, 1e-30)))
    print(f"\n[{name} N={N} {lm}] logprob max|err|={lp_err:.3e} (signal {np.max(np.abs(dev_ref)):.3e}, "
          f"rel {rel_fro(dev_gpu, dev_ref):.3e}); loss rel={loss_err:.3e}; "
          f"grad rel Fro max={g_err:.3e} at {g_where}")
    assert lp_err <= LP_TOL[cfg.dtype]
    assert g_err <= GRAD_TOL
    assert loss_err <= GRAD_TOL

    # Adam on the touched adapters
    m.mlora_optim_step(h, lr=cfg.lr, beta1=cfg.beta1, beta2=cfg.beta2, eps=cfg.eps,
                       weight_decay=cfg.weight_decay)
    P0 = {k: [[x.copy() for x in row] for row in o.P[k]] for k in oracle.TENSORS}
    skipped = o.optim_step(lr=cfg.lr, beta1=cfg.beta1, beta2=cfg.beta2, eps=cfg.eps,
                           weight_decay=cfg.weight_decay)
    assert skipped == []
    p_err, p_where = grad_errors(h, o, range(cfg.n_adapters), which_prefix="p")
    # the update itself (reported; it is sign-like at t = 1, see the design notes)
    upd = []
    for a in present:
        for l in range(o.L):
            for k in oracle.TENSORS:
                x = m.mlora_read_adapter(h, a, l, k).cpu().numpy().astype(np.float64)
                upd.append(rel_fro(x - P0[k][a][l], o.P[k][a][l] - P0[k][a][l]))
    steps = m.mlora_get_steps(h)
    print(f"[{name}] post-Adam weights rel Fro max={p_err:.3e} at {p_where}; "
          f"update rel Fro median={np.median(upd):.3e} max={np.max(upd):.3e}")
    assert steps == o.step
    assert p_err <= GRAD_TOL
    g_after, _ = grad_errors(h, o, present)
    assert g_after == 0.0                            # gradients consumed


@pytest.mark.parametrize("dtype", ["bf16", "bf16_wide", "fp32"])
def test_lm_backward_modes_bitwise_equal(dtype):
    """Recomputing each chunk's logits and keeping them from the forward give
    bitwise the same logprobs, losses and gradients (the recompute GEMM's
    accumulator is the forward's and dz is formed by the same arithmetic), over
    a batch of three LM-head chunks; "bf16_wide" (V = 65,536, d = 512) runs dh
    on its 256 x 512 tiles and the forward on the full-size tile layout of the
    kept fp16 e.  Deterministic mode makes the gradient reductions themselves
    repeatable (by default they meet in fp32 atomics in arrival order).  The
    recompute handle holds less memory: no kept-logit chunks (fp16 e = exp(z -
    tile max) on the bf16 engine, fp32 logits on the fp32 one) and one dz chunk
    buffer instead of two."""
    import rl_step_gb300 as m
    over = {"bf16": {"d_model": 256, "d_ffn": 512, "vocab": 1000},
            "bf16_wide": {"d_model": 512, "d_ffn": 1024, "vocab": 65536},
            "fp32": {"d_model": 64, "d_ffn": 128, "vocab": 520, "dtype": "fp32"}}[dtype]
    cfg = wl.get_config("qwen3_8b_ppo", **over)
    base = wl.make_base_weights(cfg)
    ad = wl.make_adapters(cfg)
    b = wl.make_batch(cfg, 40000)
    N = len(b["tokens"])
    s = (np.full(N, -np.log(cfg.vocab)) + b["sampler_noise"]) if cfg.loss == "ppo" else None
    res = {}
    for lm in ("keep_logits", "recompute"):
        h = create_handle(cfg, base, ad, N, lm_backward=lm)
        m.mlora_set_deterministic(h, True)
        lp, loss = run_gpu_step(h, b, cfg.loss, s)
        assert m.mlora_check_status(h) == 0
        grads = {(a, l, k): m.mlora_read_adapter(h, a, l, "g" + k).cpu().numpy()
                 for a in range(cfg.n_adapters) for l in range(cfg.n_layers) for k in oracle.TENSORS}
        res[lm] = (lp, loss, grads, h.device_bytes)
        del h
    lp_k, loss_k, g_k, bytes_k = res["keep_logits"]
    lp_r, loss_r, g_r, bytes_r = res["recompute"]
    assert np.array_equal(lp_k, lp_r)
    assert np.array_equal(loss_k, loss_r)
    assert any(x.any() for x in g_k.values())
    for key in g_k:
        assert np.array_equal(g_k[key], g_r[key]), key
    es = 2 if cfg.dtype == "bf16" else 4
    tiles = -(-(N + 127 * min(N, cfg.n_adapters)) // 128)
    assert tiles > 2 * 128                               # three LM-head chunks
    rows, vpad = 128 * 128, (cfg.vocab + 63) // 64 * 64
    zes = 2 if cfg.dtype == "bf16" else 4                # kept fp16 e (bf16 engine) or fp32 logits
    assert bytes_k - bytes_r == rows * vpad * (es + 2 * zes)


def test_lm_backward_mode_switch_frees_and_rejects():
    """Switching modes allocates / frees the kept-logit buffers; an unknown mode
    is E_ARG and leaves the handle as it was."""
    import rl_step_gb300 as m
    cfg, base, ad, b, o, _ = _setup("tiny_fp32", None)
    h = create_handle(cfg, base, ad, len(b["tokens"]))
    b0 = h.device_bytes
    m.mlora_set_lm_backward(h, "keep_logits")
    b1 = h.device_bytes
    assert b1 > b0
    m.mlora_set_lm_backward(h, "keep_logits")
    assert h.device_bytes == b1
    rc = m.load_library().mlora_set_lm_backward(h.ptr, 7)
    assert rc == -1 and h.device_bytes == b1
    m.mlora_set_lm_backward(h, "recompute")
    assert h.device_bytes == b0
    lp, _ = run_gpu_step(h, b, "cross_entropy")
    ref = run_oracle_step(o, b, "cross_entropy")
    assert np.max(np.abs(lp - ref["logprobs"])) <= 1e-4


def test_tiny_two_steps_accumulate_and_custom_equals_ce():
    """Gradients accumulate over calls; custom(g=-w) equals CE(w) on the GPU."""
    import rl_step_gb300 as m
    cfg, base, ad, b, o, _ = _setup("tiny_fp32", None)
    N = len(b["tokens"])
    h1 = create_handle(cfg, base, ad, N)
    run_gpu_step(h1, b, "cross_entropy")
    run_gpu_step(h1, b, "cross_entropy")
    o.forward_backward(b["tokens"], b["targets"], b["adapter_ids"], "cross_entropy", weights=b["weights"])
    o.forward_backward(b["tokens"], b["targets"], b["adapter_ids"], "cross_entropy", weights=b["weights"])
    err, _ = grad_errors(h1, o, range(3))
    assert err <= 1e-4
    h2 = create_handle(cfg, base, ad, N)
    b2 = dict(b)
    b2["dloss"] = -b["weights"]
    run_gpu_step(h2, b2, "custom")
    run_gpu_step(h2, b2, "custom")
    for a in range(3):
        for l in range(cfg.n_layers):
            for k in oracle.TENSORS:
                x = m.mlora_read_adapter(h1, a, l, "g" + k).cpu().numpy()
                y = m.mlora_read_adapter(h2, a, l, "g" + k).cpu().numpy()
                assert rel_fro(y, x) <= 1e-6


def test_edge_cases_empty_single_and_bad_ids():
    import torch
    import rl_step_gb300 as m
    cfg, base, ad, b, o, _ = _setup("tiny_fp32", None)
    h = create_handle(cfg, base, ad, 256)
    # empty batch
    e = torch.empty(0, dtype=torch.int32, device="cuda")
    lp, loss = m.mlora_forward_backward(h, e, e, e, "cross_entropy",
                                        weights=torch.empty(0, device="cuda"))
    assert m.mlora_check_status(h) == 0 and not loss.cpu().numpy().any()
    # a single token
    one = {k: v[:1] if hasattr(v, "__len__") and not isinstance(v, str) else v for k, v in b.items()}
    lp1 = m.mlora_forward(h, dev(one["tokens"]), dev(one["targets"]), dev(one["adapter_ids"]))
    ref1 = o.forward(one["tokens"], one["targets"], one["adapter_ids"])
    assert abs(float(lp1.cpu()[0]) - ref1[0]) <= 1e-4
    # out-of-range token, target and adapter ids: flagged, NaN logprobs, others exact
    tok, tgt, ids = b["tokens"][:8].copy(), b["targets"][:8].copy(), b["adapter_ids"][:8].copy()
    tok[1] = cfg.vocab
    tgt[3] = -5
    ids[5] = 3
    lp = m.mlora_forward(h, dev(tok), dev(tgt), dev(ids)).cpu().numpy()
    assert m.mlora_check_status(h) == -2
    bad = np.zeros(8, bool)
    bad[[1, 3, 5]] = True
    assert np.isnan(lp[bad]).all() and np.isfinite(lp[~bad]).all()
    ref = o.forward(tok[~bad], tgt[~bad], ids[~bad])
    assert np.max(np.abs(lp[~bad] - ref)) <= 1e-4


def test_nonfinite_gradient_skips_adapter():
    """An adapter whose gradient is not finite is skipped and reported; the
    others step as the oracle does (inf factor planted on both sides)."""
    import rl_step_gb300 as m
    cfg, base, ad, b, o, _ = _setup("tiny_fp32", None)
    N = len(b["tokens"])
    h = create_handle(cfg, base, ad, N)
    bad = np.full(o.P["A1"][1][0].shape, np.inf, np.float32)
    m.mlora_write_adapter(h, 1, 0, "A1", dev(bad))
    o.P["A1"][1][0][...] = np.inf
    lp, _ = run_gpu_step(h, b, "cross_entropy")
    with np.errstate(all="ignore"):
        ref = run_oracle_step(o, b, "cross_entropy")
    rows1 = b["adapter_ids"] == 1
    assert np.isnan(lp[rows1]).all() and np.isnan(ref["logprobs"][rows1]).all()
    assert np.max(np.abs(lp[~rows1] - ref["logprobs"][~rows1])) <= 1e-4
    skipped = m.mlora_optim_step(h, lr=1e-3).cpu().numpy()
    assert o.optim_step(lr=1e-3) == [1]
    assert skipped.tolist() == [0, 1, 0]
    assert m.mlora_get_steps(h) == [1, 0, 1] == o.step
    p_err, _ = grad_errors(h, o, [0, 2], which_prefix="p")
    assert p_err <= 1e-4
    assert np.isinf(m.mlora_read_adapter(h, 1, 0, "A1").cpu().numpy()).all()
    assert not m.mlora_read_adapter(h, 1, 0, "gB1").cpu().numpy().any()


def test_save_state_round_trip(tmp_path):
    import rl_step_gb300 as m
    cfg, base, ad, b, o, _ = _setup("tiny_fp32", None)
    h = create_handle(cfg, base, ad, len(b["tokens"]))
    run_gpu_step(h, b, "cross_entropy")
    m.mlora_optim_step(h, lr=1e-3, adapters=[0, 2])
    path = str(tmp_path / "state.bin")
    m.mlora_save_state(h, path)
    st = oracle.read_state_file(path)
    assert st["n_adapters"] == 3 and st["n_layers"] == cfg.n_layers
    for a, rec in enumerate(st["adapters"]):
        assert rec["rank"] == cfg.ranks[a] and rec["alpha"] == cfg.alphas[a]
        assert rec["step"] == (1 if a in (0, 2) else 0)
        for l in range(cfg.n_layers):
            for k in oracle.TENSORS:
                assert np.array_equal(rec["P"][k][l], m.mlora_read_adapter(h, a, l, k).cpu().numpy())
                assert np.array_equal(rec["M"][k][l], m.mlora_read_adapter(h, a, l, "m" + k).cpu().numpy())
                assert np.array_equal(rec["V"][k][l], m.mlora_read_adapter(h, a, l, "v" + k).cpu().numpy())


def _state(h, cfg, prefixes=("", "m", "v")):
    import rl_step_gb300 as m
    return {(p, a, l, k): m.mlora_read_adapter(h, a, l, p + k).cpu().numpy()
            for p in prefixes for a in range(cfg.n_adapters) for l in range(cfg.n_layers)
            for k in oracle.TENSORS}


def test_load_state_with_and_without_optimizer(tmp_path):
    """load_state_with_optimizer restores weights, moments and step counts
    bitwise and the resumed run takes the uninterrupted run's next step;
    load_state restores the weights only, and the next step matches the
    oracle restarted from the same file."""
    import rl_step_gb300 as m
    cfg, base, ad, b, o, _ = _setup("tiny_fp32", None)
    N = len(b["tokens"])
    ha = create_handle(cfg, base, ad, N)
    for _ in range(2):
        run_gpu_step(ha, b, "cross_entropy")
        m.mlora_optim_step(ha, lr=1e-3)
    path = str(tmp_path / "state.bin")
    m.mlora_save_state(ha, path)
    saved = _state(ha, cfg)
    # resume with the optimizer in a handle that holds a pending gradient
    hb = create_handle(cfg, base, ad, N)
    run_gpu_step(hb, b, "cross_entropy")
    m.mlora_load_state(hb, path, with_optimizer=True)
    assert m.mlora_get_steps(hb) == [2, 2, 2]
    got = _state(hb, cfg, ("", "m", "v", "g"))
    for key, x in saved.items():
        assert np.array_equal(got[key], x), key
    assert not any(got[("g",) + key[1:]].any() for key in saved if key[0] == "")
    for h in (ha, hb):
        run_gpu_step(h, b, "cross_entropy")
        m.mlora_optim_step(h, lr=1e-3)
    sa, sb = _state(ha, cfg), _state(hb, cfg)
    for key in sa:
        assert np.array_equal(sa[key], sb[key]), key
    # weights only: moments and steps reset; next step as the oracle's
    hc = create_handle(cfg, base, ad, N)
    m.mlora_load_state(hc, path, with_optimizer=False)
    assert m.mlora_get_steps(hc) == [0, 0, 0]
    got = _state(hc, cfg)
    for key, x in saved.items():
        if key[0] == "":
            assert np.array_equal(got[key], x), key
        else:
            assert not got[key].any(), key
    oracle.load_state_file(path, o, with_optimizer=False)
    run_gpu_step(hc, b, "cross_entropy")
    run_oracle_step(o, b, "cross_entropy")
    m.mlora_optim_step(hc, lr=1e-3)
    o.optim_step(lr=1e-3)
    assert m.mlora_get_steps(hc) == o.step == [1, 1, 1]
    p_err, _ = grad_errors(hc, o, range(3), which_prefix="p")
    assert p_err <= 1e-4


def test_load_state_rejects_bad_files(tmp_path):
    """A file of other shapes is E_ARG, a missing, foreign or truncated file
    E_IO; none of them changes the handle."""
    import rl_step_gb300 as m
    cfg, base, ad, b, o, _ = _setup("tiny_fp32", None)
    h = create_handle(cfg, base, ad, len(b["tokens"]))
    before = _state(h, cfg)
    good = str(tmp_path / "good.bin")
    m.mlora_save_state(h, good)
    other = oracle.Oracle(base, ad, cfg.ranks, [2.0 * x for x in cfg.alphas])
    bad_alpha = str(tmp_path / "alpha.bin")
    oracle.write_state_file(bad_alpha, other)
    raw = open(good, "rb").read()
    trunc = str(tmp_path / "trunc.bin")
    open(trunc, "wb").write(raw[:-4])
    extra = str(tmp_path / "extra.bin")
    open(extra, "wb").write(raw + b"\0")
    foreign = str(tmp_path / "foreign.bin")
    open(foreign, "wb").write(b"NOTMLORA" + raw[8:])
    cases = [(bad_alpha, "E_ARG"), (str(tmp_path / "missing.bin"), "E_IO"), (trunc, "E_IO"),
             (extra, "E_IO"), (foreign, "E_IO")]
    for path, code in cases:
        with pytest.raises(m.MLoRAError) as ei:
            m.mlora_load_state(h, path, with_optimizer=True)
        assert code in str(ei.value), (path, str(ei.value))
        now = _state(h, cfg)
        for key in before:
            assert np.array_equal(now[key], before[key])
