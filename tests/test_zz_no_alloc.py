"""The allocation-free routing entry point (mlora_routing_noalloc).

It serves callers that cannot call cudaMalloc -- their device memory is
owned by another allocator, or their loop must not pay for cudaMalloc's
possible device synchronisation -- by keeping the routing scratch in a fixed
device array inside the library.  Its results must equal those of the
handle-based mlora_get_routing, bit for bit (integer outputs), on two calls
in a row: the second call reuses the array the first one left behind.

This file is collected last so that a run stopping at its first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import workloads as wl


def _lib():
    import __graft_entry__
    __graft_entry__.build()
    import rl_step_gb300
    return rl_step_gb300.load_library()


def test_noalloc_rejects_sizes_beyond_its_limits():
    """Checked on the host before any CUDA call (runs without a GPU)."""
    lib = _lib()
    dummy = ctypes.c_void_p(16)
    rc = lib.mlora_routing_noalloc(dummy, 65537, 4, dummy, dummy, dummy, dummy, None)
    assert rc == -1 and b"MLORA_NOALLOC_MAX_TOKENS" in lib.mlora_last_error()
    rc = lib.mlora_routing_noalloc(dummy, 16, 129, dummy, dummy, dummy, dummy, None)
    assert rc == -1 and b"MLORA_NOALLOC_MAX_ADAPTERS" in lib.mlora_last_error()


@pytest.mark.gpu
def test_noalloc_routing_equals_get_routing_on_two_calls():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _lib()
    import rl_step_gb300 as m
    from _gpu_util import create_handle, dev

    n_ad = 37
    cfg = wl.get_config("tiny_fp32", n_adapters=n_ad, ranks=(4,) * n_ad, alphas=(8.0,) * n_ad)
    h = create_handle(cfg, wl.make_base_weights(cfg), wl.make_adapters(cfg), 20000)
    rng = np.random.Generator(np.random.PCG64([2024]))
    # the second call is smaller than the first: stale scratch must not leak
    for n in (20000, 3001):
        ids = rng.integers(0, n_ad, n).astype(np.int32)
        ids[ids == 5] = 6                                # one empty segment
        ids_d = dev(ids)
        ref = m.mlora_get_routing(h, ids_d)
        out = m.mlora_routing_noalloc(ids_d, n_ad)
        torch.cuda.synchronize()
        for name, a, b in zip(("perm", "seg_off", "pad_off", "tile_ad"), out, ref):
            assert torch.equal(a, b), name
        assert m.mlora_check_status(h) == 0
