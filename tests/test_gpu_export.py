"""Export merge W' = W + gamma B A on the GPU against the oracle.

Deep Dive - Tinker, "Checkpoints and export paths": merging the adapter into
the base gives a standalone model.  The oracle computes W + gamma B A in
fp64 from the same fp32 master factors.  For a bf16 base the export is the
bf16 rounding of that sum: element by element it must equal the oracle's
round-to-nearest-even, except where the exact sum lies within the kernel's
error bound of a rounding midpoint, where either neighbour is valid (the
number of such elements is reported; it is the band width over the bf16
spacing, of the order of 10 %).  For an fp32 base
the export must agree within fp32 rounding.  A model built from the
exported matrices (with zero adapters) must reproduce the adapter's
logprobs within the usual logprob tolerance.
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


def _cfg(name, V, d, f, L, dtype, ranks, seed):
    return wl.Config(name=name, vocab=V, d_model=d, d_ffn=f, n_layers=L, dtype=dtype,
                     n_adapters=len(ranks), ranks=tuple(ranks),
                     alphas=tuple(float(2 * r) for r in ranks), n_tokens=256,
                     loss="cross_entropy", seed=seed)


def _bf16_check(got_bits, exact, mag):
    """got_bits (uint16) against the fp64 exact sum with error bound tol:
    the oracle's rounding where [exact - tol, exact + tol] rounds to one
    bf16 value, else a bf16 value between the roundings of the two ends."""
    # kernel error: each factor is hi + lo to within 2^-18 of itself, so the
    # three-term product misses B A by at most 3 * 2^-18 mag (the two factor
    # residuals and the dropped B_lo A_lo); fp32 accumulation of 192
    # products adds about 2^-19 mag and the final fma 2^-24 |exact|.
    tol = 2.0 ** -15 * mag + 2.0 ** -23 * np.abs(exact)
    ref = wl.f32_to_bf16_bits(exact.astype(np.float32))
    lo = wl.f32_to_bf16_bits((exact - tol).astype(np.float32))
    hi = wl.f32_to_bf16_bits((exact + tol).astype(np.float32))
    unique = lo == hi
    assert np.array_equal(got_bits[unique], ref[unique])
    amb = ~unique
    g = wl.bf16_bits_to_f32(got_bits[amb])
    assert ((wl.bf16_bits_to_f32(lo[amb]) <= g) & (g <= wl.bf16_bits_to_f32(hi[amb]))).all()
    return int(amb.sum())


CASES = [
    # Qwen3-8B widths, one layer: the CTA-pair GEMM over a 12288 x 4096 output
    ("w8b", 1024, 4096, 12288, 1, "bf16", (32, 64), 3001),
    # mid widths, ragged against the 256-column tiles (d = 320, f = 960)
    ("mid", 512, 320, 960, 2, "bf16", (8, 64, 20), 3002),
    # fp32 base through the FFMA engine
    ("f32", 512, 128, 384, 2, "fp32", (4, 16), 3003),
]


@pytest.mark.parametrize("name,V,d,f,L,dtype,ranks,seed", CASES)
def test_export_merged_matches_oracle(name, V, d, f, L, dtype, ranks, seed):
    import rl_step_gb300 as m
    cfg = _cfg(name, V, d, f, L, dtype, ranks, seed)
    base = wl.make_base_weights(cfg)
    # factors of trained size: B is zero at init in practice, so draw it like A
    ad = wl.make_adapters(cfg, std_a=0.05, std_b=0.05)
    o = oracle.Oracle(base, ad, cfg.ranks, cfg.alphas)
    h = create_handle(cfg, base, ad, 256)
    worst_amb = 0
    for a in range(cfg.n_adapters):
        for l in range(L):
            for which, (Bk, Ak) in (("W1", ("B1", "A1")), ("W2", ("B2", "A2"))):
                got = m.mlora_export_merged(h, a, l, which)
                exact = o.merged_weight(a, l, which)
                mag = o.gamma[a] * (np.abs(o.P[Bk][a][l]) @ np.abs(o.P[Ak][a][l]))
                if dtype == "bf16":
                    bits = got.view(__import__("torch").int16).cpu().numpy().view(np.uint16)
                    amb = _bf16_check(bits, exact, mag)
                    worst_amb = max(worst_amb, amb)
                    # band width 2 tol against the bf16 spacing of |W'| ~ 0.02-0.1
                    # (2^-13 .. 2^-11): of the order of 10 % of the elements
                    assert amb <= 0.25 * exact.size
                else:
                    g = got.cpu().numpy().astype(np.float64)
                    err = np.abs(g - exact)
                    assert (err <= 2.0 ** -22 * np.abs(exact) + 2.0 ** -20 * mag).all()
    print(f"\n[{name}] export: elements within the rounding band at most {worst_amb} "
          f"({worst_amb / exact.size:.2%})")


def test_exported_model_reproduces_adapter_logprobs():
    """Replace every W1, W2 by adapter 1's export and run with zero adapters:
    the logprobs match the adapter's own (bf16 tolerance)."""
    import rl_step_gb300 as m
    cfg = _cfg("mid", 2048, 512, 1536, 2, "bf16", (16, 32), 3004)
    base = wl.make_base_weights(cfg)
    ad = wl.make_adapters(cfg, std_a=0.05, std_b=0.05)
    h = create_handle(cfg, base, ad, 1024)
    rng = np.random.Generator(np.random.PCG64([cfg.seed, 5]))
    tok = rng.integers(0, cfg.vocab, 1000).astype(np.int32)
    tgt = rng.integers(0, cfg.vocab, 1000).astype(np.int32)
    ids = np.full(1000, 1, np.int32)
    lp_ad = m.mlora_forward(h, dev(tok), dev(tgt), dev(ids)).cpu().numpy()
    mb = dict(base)
    mb["W1"] = [m.mlora_export_merged(h, 1, l, "W1").view(__import__("torch").int16).cpu().numpy()
                .view(np.uint16) for l in range(cfg.n_layers)]
    mb["W2"] = [m.mlora_export_merged(h, 1, l, "W2").view(__import__("torch").int16).cpu().numpy()
                .view(np.uint16) for l in range(cfg.n_layers)]
    zero = {k: [[np.zeros_like(x) for x in row] for row in ad[k]] for k in ("A1", "B1", "A2", "B2")}
    h2 = create_handle(cfg, mb, zero, 1024)
    lp_m = m.mlora_forward(h2, dev(tok), dev(tgt), dev(ids)).cpu().numpy()
    o = oracle.Oracle(base, ad, cfg.ranks, cfg.alphas)
    ref = o.forward(tok, tgt, ids)
    print(f"\nexported model: max|lp - oracle| = {np.max(np.abs(lp_m - ref)):.3e}, "
          f"adapter path {np.max(np.abs(lp_ad - ref)):.3e}")
    assert np.max(np.abs(lp_m - ref)) <= 2e-2
    assert np.max(np.abs(lp_ad - ref)) <= 2e-2
