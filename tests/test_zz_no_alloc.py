"""The allocation-free routing entry point (mlora_routing_noalloc).

It serves callers that cannot call cudaMalloc -- their device memory is
owned by another allocator, or their loop must not pay for cudaMalloc's
possible device synchronisation -- by keeping the routing scratch in a fixed
device array inside the library.  Its results must equal, bit for bit
(integer outputs), both the oracle's routing and the handle-based
mlora_get_routing, on two calls in a row: the second call reuses the array
the first one left behind.  The cases reach the documented limits (65,536
tokens over 128 adapters, every segment one row past a tile boundary, which
gives the largest padded layout the scratch is sized for), an empty batch,
and out-of-range ids (left out of the routing).

This file is collected last so that a run stopping at its first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads as wl

TILE_M = 128
MAX_TOKENS, MAX_ADAPTERS = 65536, 128


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


def _cases():
    """(name, adapter ids, n_adapters): seeded, from the largest to the smallest."""
    rng = np.random.Generator(np.random.PCG64([2024]))
    out = []
    # the limits: 128 adapters, 65,536 tokens, every segment of length 1 mod 128
    lens = np.full(MAX_ADAPTERS, 4 * TILE_M + 1)
    lens[-1] = MAX_TOKENS - lens[:-1].sum()
    assert lens[-1] % TILE_M == 1 and lens.sum() == MAX_TOKENS
    ids = np.repeat(np.arange(MAX_ADAPTERS, dtype=np.int32), lens)
    out.append(("limits_max_padding", rng.permutation(ids).astype(np.int32), MAX_ADAPTERS))
    # random ids over 37 adapters with one empty segment; a smaller second call
    for n in (20000, 3001):
        x = rng.integers(0, 37, n).astype(np.int32)
        x[x == 5] = 6
        out.append((f"random_{n}", x, 37))
    # out-of-range ids (== n_adapters, negative) are left out
    x = rng.integers(0, 9, 1000).astype(np.int32)
    x[rng.choice(1000, 12, replace=False)] = 9
    x[rng.choice(1000, 5, replace=False)] = -3
    out.append(("out_of_range", x, 9))
    out.append(("empty", np.zeros(0, np.int32), 5))
    return out


def _oracle_routing(ids, n_ad):
    """The oracle's routing of the in-range ids, with perm in batch positions."""
    ok = (ids >= 0) & (ids < n_ad)
    ref = oracle.routing(ids[ok], n_ad, TILE_M)
    ref = dict(ref)
    ref["perm"] = np.nonzero(ok)[0][ref["perm"]].astype(np.int64)
    return ref


@pytest.mark.gpu
def test_noalloc_routing_equals_oracle_and_get_routing_on_two_calls():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _lib()
    import rl_step_gb300 as m
    from _gpu_util import create_handle, dev

    handles = {}
    for name, ids, n_ad in _cases():
        if n_ad not in handles:
            cfg = wl.get_config("tiny_fp32", n_adapters=n_ad, ranks=(4,) * n_ad, alphas=(8.0,) * n_ad)
            handles[n_ad] = create_handle(cfg, wl.make_base_weights(cfg), wl.make_adapters(cfg),
                                          MAX_TOKENS)
        h = handles[n_ad]
        n = len(ids)
        ref = _oracle_routing(ids, n_ad)
        nv = int(ref["seg_off"][-1])                     # tokens routed (in-range ids)
        ids_d = dev(ids) if n else torch.zeros(0, dtype=torch.int32, device="cuda")
        via_handle = m.mlora_get_routing(h, ids_d)
        for call in range(2):                            # two calls in a row
            out = m.mlora_routing_noalloc(ids_d, n_ad)
            torch.cuda.synchronize()
            perm, seg, pad, tiles = (x.cpu().numpy() for x in out)
            assert np.array_equal(perm[:nv], ref["perm"]), (name, call)
            assert np.array_equal(seg, ref["seg_off"]), (name, call)
            assert np.array_equal(pad, ref["pad_off"]), (name, call)
            nt = len(ref["tile_ad"])
            assert len(tiles) == n // TILE_M + n_ad + 1
            assert np.array_equal(tiles[:nt], ref["tile_ad"]), (name, call)
            assert (tiles[nt:] == -1).all(), (name, call)
            for what, a, b in zip(("perm", "seg_off", "pad_off", "tile_ad"), out, via_handle):
                if what == "perm":
                    a, b = a[:nv], b[:nv]
                assert torch.equal(a, b), (name, call, what)
        if name == "limits_max_padding":
            # the largest padded layout: every segment one row past a tile boundary
            assert pad[-1] == MAX_TOKENS + (TILE_M - 1) * MAX_ADAPTERS
        expect = -2 if name == "out_of_range" else 0     # the handle flags bad ids, noalloc cannot
        assert m.mlora_check_status(h) == expect, name
