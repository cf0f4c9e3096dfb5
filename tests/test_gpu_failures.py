"""Failure detection on the GPU without a GPU fault.

* A bounded device wait that runs out: a test hook makes one tensor-core GEMM
  leave one pipeline stage unloaded (nothing is in flight for it) and shortens
  the MMA thread's wait for it to 1 ms.  The kernel must raise the timeout
  status bit, drain what it issued, free its tensor memory and return;
  mlora_check_status reports MLORA_E_TIMEOUT, and the same handle then takes
  a normal step that matches the oracle.
* Allocation failure in the create calls: a test hook makes the k-th device
  allocation fail (without calling the driver).  For every k over all the
  allocations of mlora_create, mlora_tf_create and mlora_sampler_create the
  call must return MLORA_E_NOMEM and give back every byte it had allocated.

Both hooks are exported by the library but are not part of its public
headers.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads as wl
from _gpu_util import create_handle, dev, grad_errors, run_gpu_step, run_oracle_step

pytestmark = pytest.mark.gpu

E_NOMEM, E_TIMEOUT = -4, -5
SMALL_BF16 = {"d_model": 320, "d_ffn": 704, "vocab": 4000}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _hooks():
    import rl_step_gb300 as m
    lib = m.load_library()
    lib.mlk_test_gemm_withhold.restype = ctypes.c_int32
    lib.mlk_test_gemm_withhold.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64]
    lib.mlk_test_alloc_calls.restype = ctypes.c_int64
    lib.mlk_test_alloc_calls.argtypes = []
    lib.mlk_test_fail_alloc_at.restype = None
    lib.mlk_test_fail_alloc_at.argtypes = [ctypes.c_int64]
    return lib


def test_bounded_wait_runs_out_and_handle_recovers():
    import time

    import torch
    import rl_step_gb300 as m
    lib = _hooks()
    cfg = wl.get_config("qwen3_8b_ppo", **SMALL_BF16)
    base, ad = wl.make_base_weights(cfg), wl.make_adapters(cfg)
    b = wl.make_batch(cfg, 512)
    o = oracle.Oracle(base, ad, cfg.ranks, cfg.alphas)
    h = create_handle(cfg, base, ad, len(b["tokens"]))
    tok, tgt, ids = dev(b["tokens"]), dev(b["targets"]), dev(b["adapter_ids"])
    # K block 2 of 5 (d = 320) of the step's first LoRA shrink is never loaded
    assert lib.mlk_test_gemm_withhold(h.ptr, 2, 1_000_000) == 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    m.mlora_forward(h, tok, tgt, ids)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert m.mlora_check_status(h) == E_TIMEOUT
    assert m.mlora_check_status(h) == 0                 # the status word was cleared
    assert elapsed < 2.0                                 # the 1 ms bound, not the default ~4 s
    # the context and the handle are intact: a normal step matches the oracle
    s = o.forward(b["tokens"], b["targets"], b["adapter_ids"]) + b["sampler_noise"]
    lp, _ = run_gpu_step(h, b, cfg.loss, s)
    assert m.mlora_check_status(h) == 0
    ref = run_oracle_step(o, b, cfg.loss, s)
    assert np.max(np.abs(lp - ref["logprobs"])) <= 2e-2
    err, where = grad_errors(h, o, np.unique(b["adapter_ids"]))
    assert err <= 1e-2, where


def _sweep(lib, create, what):
    """Fail each allocation of create() in turn; every attempt returns E_NOMEM
    and leaves the device's free memory where it was.  Garbage collection is
    off meanwhile, so that no earlier test's handle is freed inside a
    measurement."""
    import gc

    import torch
    import rl_step_gb300 as m
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    gc.disable()
    try:
        c0 = lib.mlk_test_alloc_calls()
        obj = create()                           # a full create: counts its allocations
        n_alloc = lib.mlk_test_alloc_calls() - c0
        del obj
        torch.cuda.synchronize()
        assert n_alloc > 5, what
        for k in range(1, n_alloc + 1):
            torch.cuda.synchronize()
            free0 = torch.cuda.mem_get_info()[0]
            lib.mlk_test_fail_alloc_at(lib.mlk_test_alloc_calls() + k)
            try:
                with pytest.raises(m.MLoRAError) as ei:
                    create()
            finally:
                lib.mlk_test_fail_alloc_at(0)
            assert ei.value.code == E_NOMEM, (what, k, str(ei.value))
            torch.cuda.synchronize()
            assert torch.cuda.mem_get_info()[0] == free0, (what, k)
    finally:
        gc.enable()
    return n_alloc


def test_create_calls_release_everything_on_allocation_failure():
    import rl_step_gb300 as m
    import rl_step_gb300.transformer as t
    import workloads.transformer as wt
    lib = _hooks()
    # the MLP model's handle (bf16: tensor-core engine, all buffers)
    cfg = wl.get_config("qwen3_8b_ppo", **SMALL_BF16)
    base, ad = wl.make_base_weights(cfg), wl.make_adapters(cfg)
    dbase = {"E": dev(base["E"]), "W1": [dev(w) for w in base["W1"]],
             "W2": [dev(w) for w in base["W2"]], "Wout": dev(base["Wout"])}
    dad = [[[dev(x) for x in row] for row in ad[k]] for k in ("A1", "B1", "A2", "B2")]

    def make_mlp():
        return m.mlora_create(cfg.vocab, cfg.d_model, cfg.d_ffn, cfg.n_layers, cfg.dtype, cfg.ranks,
                              cfg.alphas, 700, dbase["E"], dbase["W1"], dbase["W2"], dbase["Wout"], *dad)
    n1 = _sweep(lib, make_mlp, "mlora_create")

    # the sampler over a training handle
    trainer = make_mlp()
    n2 = _sweep(lib, lambda: m.mlora_sampler_create(trainer, 4, 300), "mlora_sampler_create")
    del trainer

    # the transformer-block handle
    tcfg = wt.get_tf_config("tf_small")
    tbase, tad = wt.make_tf_base_weights(tcfg), wt.make_tf_adapters(tcfg)
    tb = {"E": dev(tbase["E"]), "Wout": dev(tbase["Wout"]), "final_norm": dev(tbase["final_norm"]),
          "attn_norm": [dev(g) for g in tbase["attn_norm"]], "mlp_norm": [dev(g) for g in tbase["mlp_norm"]],
          "W": {p: [dev(w) for w in tbase["W"][p]] for p in t.PROJ}}
    A = {p: [[dev(x) for x in row] for row in tad["A"][p]] for p in t.PROJ}
    B = {p: [[dev(x) for x in row] for row in tad["B"][p]] for p in t.PROJ}

    def make_tf():
        return t.tf_create(tcfg.vocab, tcfg.d_model, tcfg.n_heads, tcfg.n_kv_heads, tcfg.d_ffn,
                           tcfg.n_layers, tcfg.ranks, tcfg.alphas, 600, tb, A, B,
                           rope_theta=tcfg.rope_theta, rms_eps=tcfg.rms_eps)
    n3 = _sweep(lib, make_tf, "mlora_tf_create")
    print(f"\nallocation failures injected: mlora_create {n1}, mlora_sampler_create {n2}, "
          f"mlora_tf_create {n3}; each returned E_NOMEM and released all it held")
