"""Python binding of libmlora.so: the multi-tenant LoRA training step on sm_103a.

Argument marshalling only.  Every step of the computation runs in the
library's CUDA kernels; PyTorch provides device memory and streams.  Loading
fails loudly if the compiled library is missing -- there is no fallback.

The functions mirror the C entry points of include/mlora.h:

    h = mlora_create(V, d, f, L, "bf16"|"fp32", ranks, alphas, max_tokens,
                     E, W1s, W2s, Wout, A1, B1, A2, B2)     # A1[a][l] ... fp32 factors
    mlora_forward(h, tokens, targets, adapter_ids)              -> logprobs
    mlora_forward_backward(h, tokens, targets, adapter_ids, kind, ...)
                                                                -> (logprobs, loss per adapter)
    mlora_forward_backward_custom(h, tokens, targets, adapter_ids, dloss)
    mlora_optim_step(h, lr=..., ...)                            -> skipped flags
    mlora_save_state(h, path) / mlora_load_state(h, path, with_optimizer)
    mlora_destroy(h)

Tensors passed in must be CUDA tensors of the documented dtype (int32 ids,
float32 loss inputs); the current torch stream is used unless one is given.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_double, c_float, c_int32, c_int64, c_void_p
from typing import Optional, Sequence

__all__ = [
    "LIB_PATH", "load_library", "MLoRAError", "Handle",
    "mlora_create", "mlora_destroy", "mlora_forward", "mlora_forward_backward",
    "mlora_forward_backward_custom", "mlora_optim_step", "mlora_save_state", "mlora_load_state", "mlora_export_merged",
    "mlora_read_adapter", "mlora_write_adapter", "mlora_get_steps", "mlora_get_routing",
    "mlora_check_status", "mlora_routing_noalloc", "Sampler", "mlora_sampler_create",
    "mlora_sampler_publish", "mlora_sampler_logprobs", "mlora_sampler_sample",
    "mlora_sampler_check_status", "mlora_set_deterministic", "mlora_set_lm_backward",
    "mlora_profile_enable", "mlora_profile_read", "PROF_CLASSES",
    "LOSS_KINDS", "LM_BACKWARD_MODES", "TENSOR_IDS", "TILE_M", "MAX_RANK",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmlora.so")
TILE_M = 128
MAX_RANK = 64
LOSS_KINDS = {"cross_entropy": 0, "importance_sampling": 1, "ppo": 2}
LM_BACKWARD_MODES = {"recompute": 0, "keep_logits": 1}
TENSOR_IDS = {n: i for i, n in enumerate(
    ["A1", "B1", "A2", "B2", "gA1", "gB1", "gA2", "gB2",
     "mA1", "mB1", "mA2", "mB2", "vA1", "vB1", "vA2", "vB2"])}
PROF_CLASSES = ["routing", "embed", "shrink", "w1_fwd", "w2_fwd", "lm_fwd", "loss", "lm_dz",
                "lm_dh", "w2_bwd", "w1_bwd", "grad", "adam", "other"]
_ERRORS = {-1: "E_ARG", -2: "E_RANGE", -3: "E_CUDA", -4: "E_NOMEM", -5: "E_TIMEOUT",
           -6: "E_IO", -7: "E_UNSUPPORTED"}


class MLoRAError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_ERRORS.get(code, code)}: {msg}")
        self.code = code


class _Config(ctypes.Structure):
    _fields_ = [("vocab", c_int32), ("d_model", c_int32), ("d_ffn", c_int32),
                ("n_layers", c_int32), ("dtype", c_int32), ("n_adapters", c_int32),
                ("ranks", POINTER(c_int32)), ("alphas", POINTER(c_float)),
                ("max_tokens", c_int64)]


class _Init(ctypes.Structure):
    _fields_ = [("E", c_void_p), ("W1", POINTER(c_void_p)), ("W2", POINTER(c_void_p)),
                ("Wout", c_void_p), ("A1", POINTER(c_void_p)), ("B1", POINTER(c_void_p)),
                ("A2", POINTER(c_void_p)), ("B2", POINTER(c_void_p))]


class _Batch(ctypes.Structure):
    _fields_ = [("n_tokens", c_int64), ("tokens", c_void_p), ("targets", c_void_p),
                ("adapter_ids", c_void_p)]


class _LossInputs(ctypes.Structure):
    _fields_ = [("weights", c_void_p), ("advantages", c_void_p),
                ("sampler_logprobs", c_void_p), ("clip_eps", c_float)]


class _Adam(ctypes.Structure):
    _fields_ = [("lr", c_float), ("beta1", c_float), ("beta2", c_float), ("eps", c_float),
                ("weight_decay", c_float)]


_SIGNATURES = {
    "mlora_create": (c_int32, [POINTER(_Config), POINTER(_Init), POINTER(c_void_p)]),
    "mlora_destroy": (c_int32, [c_void_p]),
    "mlora_forward": (c_int32, [c_void_p, POINTER(_Batch), c_void_p, c_void_p]),
    "mlora_forward_backward": (c_int32, [c_void_p, POINTER(_Batch), c_int32, POINTER(_LossInputs),
                                         c_void_p, c_void_p, c_void_p]),
    "mlora_forward_backward_custom": (c_int32, [c_void_p, POINTER(_Batch), c_void_p, c_void_p,
                                                c_void_p, c_void_p]),
    "mlora_optim_step": (c_int32, [c_void_p, POINTER(_Adam), POINTER(c_int32), c_int32, c_void_p,
                                   c_void_p]),
    "mlora_save_state": (c_int32, [c_void_p, c_char_p, c_void_p]),
    "mlora_load_state": (c_int32, [c_void_p, c_char_p, c_int32, c_void_p]),
    "mlora_export_merged": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p]),
    "mlora_sampler_create": (c_int32, [c_void_p, c_int32, c_int64, POINTER(c_void_p)]),
    "mlora_sampler_destroy": (c_int32, [c_void_p]),
    "mlora_sampler_publish": (c_int32, [c_void_p, c_int32, c_int32, POINTER(c_int64), c_void_p]),
    "mlora_sampler_logprobs": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_void_p,
                                         c_void_p]),
    "mlora_sampler_sample": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_void_p,
                                       c_void_p, c_void_p]),
    "mlora_sampler_check_status": (c_int32, [c_void_p, c_void_p]),
    "mlora_sampler_kernel_launches": (c_int64, [c_void_p]),
    "mlora_read_adapter": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p]),
    "mlora_write_adapter": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p]),
    "mlora_get_steps": (c_int32, [c_void_p, POINTER(c_int64), c_void_p]),
    "mlora_get_routing": (c_int32, [c_void_p, c_void_p, c_int64, c_void_p, c_void_p, c_void_p,
                                    c_void_p, c_void_p]),
    "mlora_check_status": (c_int32, [c_void_p, c_void_p]),
    "mlora_routing_noalloc": (c_int32, [c_void_p, c_int64, c_int32, c_void_p, c_void_p, c_void_p,
                                        c_void_p, c_void_p]),
    "mlora_set_deterministic": (c_int32, [c_void_p, c_int32]),
    "mlora_set_lm_backward": (c_int32, [c_void_p, c_int32]),
    "mlora_profile_enable": (c_int32, [c_void_p, c_int32]),
    "mlora_profile_read": (c_int32, [c_void_p, POINTER(c_double), POINTER(c_int64), c_int32]),
    "mlora_kernel_launches": (c_int64, [c_void_p]),
    "mlora_device_bytes": (c_int64, [c_void_p]),
    "mlora_last_error": (c_char_p, []),
}

_lib: Optional[ctypes.CDLL] = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmlora.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build the CUDA library first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(rc: int):
    if rc != 0:
        msg = _lib.mlora_last_error().decode(errors="replace")
        raise MLoRAError(rc, msg)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return c_void_p(stream.cuda_stream)


class Handle:
    """Owns one mlora_t*; keeps the config it was created with."""

    def __init__(self, ptr: int, n_adapters: int, ranks, d: int, f: int, n_layers: int,
                 dtype: str = "bf16"):
        self.ptr = c_void_p(ptr)
        self.dtype = dtype
        self.n_adapters = n_adapters
        self.ranks = list(ranks)
        self.d, self.f, self.n_layers = d, f, n_layers

    @property
    def kernel_launches(self) -> int:
        return int(_lib.mlora_kernel_launches(self.ptr))

    @property
    def device_bytes(self) -> int:
        return int(_lib.mlora_device_bytes(self.ptr))

    def shape_of(self, which: str, adapter: int):
        r = self.ranks[adapter]
        k = which[-2:]
        return {"A1": (r, self.d), "B1": (self.f, r), "A2": (r, self.f), "B2": (self.d, r)}[k]

    def __del__(self):
        try:
            if self.ptr and _lib is not None:
                _lib.mlora_destroy(self.ptr)
                self.ptr = c_void_p(0)
        except Exception:  # pragma: no cover - interpreter shutdown
            pass


def mlora_create(vocab: int, d_model: int, d_ffn: int, n_layers: int, dtype: str,
                 ranks: Sequence[int], alphas: Sequence[float], max_tokens: int,
                 E, W1, W2, Wout, A1=None, B1=None, A2=None, B2=None) -> Handle:
    """Create a handle.  Base tensors: CUDA tensors (bf16 or float32); adapter
    factors: nested lists [a][l] of CUDA float32 tensors (or None)."""
    load_library()
    n_ad, L = len(ranks), n_layers
    cfg = _Config(vocab, d_model, d_ffn, n_layers, 0 if dtype == "bf16" else 1, n_ad,
                  (c_int32 * n_ad)(*ranks), (c_float * n_ad)(*alphas), max_tokens)
    w1 = (c_void_p * L)(*[w.data_ptr() for w in W1])
    w2 = (c_void_p * L)(*[w.data_ptr() for w in W2])

    def table(x):
        if x is None:
            return None
        return (c_void_p * (n_ad * L))(*[x[a][l].data_ptr() if x[a][l] is not None else None
                                         for a in range(n_ad) for l in range(L)])
    tabs = [table(x) for x in (A1, B1, A2, B2)]
    init = _Init(E.data_ptr(), ctypes.cast(w1, POINTER(c_void_p)), ctypes.cast(w2, POINTER(c_void_p)),
                 Wout.data_ptr(),
                 *[ctypes.cast(t, POINTER(c_void_p)) if t is not None else None for t in tabs])
    out = c_void_p()
    _check(_lib.mlora_create(ctypes.byref(cfg), ctypes.byref(init), ctypes.byref(out)))
    return Handle(out.value, n_ad, ranks, d_model, d_ffn, n_layers, dtype)


def mlora_destroy(h: Handle):
    if h.ptr:
        _check(_lib.mlora_destroy(h.ptr))
        h.ptr = c_void_p(0)


def _batch(tokens, targets, adapter_ids) -> _Batch:
    n = int(tokens.numel())
    assert targets.numel() == n and adapter_ids.numel() == n
    return _Batch(n, _ptr(tokens), _ptr(targets), _ptr(adapter_ids))


def mlora_forward(h: Handle, tokens, targets, adapter_ids, logprobs_out=None, stream=None):
    import torch
    if logprobs_out is None:
        logprobs_out = torch.empty(tokens.numel(), dtype=torch.float32, device=tokens.device)
    b = _batch(tokens, targets, adapter_ids)
    _check(_lib.mlora_forward(h.ptr, ctypes.byref(b), _ptr(logprobs_out), _stream(stream)))
    return logprobs_out


def mlora_forward_backward(h: Handle, tokens, targets, adapter_ids, loss_kind: str, weights=None,
                           advantages=None, sampler_logprobs=None, clip_eps: float = 0.2,
                           logprobs_out=None, loss_out=None, stream=None):
    """Returns (logprobs [N] float32, loss per adapter [n_adapters] float64)."""
    import torch
    dev = tokens.device
    if logprobs_out is None:
        logprobs_out = torch.empty(tokens.numel(), dtype=torch.float32, device=dev)
    if loss_out is None:
        loss_out = torch.empty(h.n_adapters, dtype=torch.float64, device=dev)
    b = _batch(tokens, targets, adapter_ids)
    li = _LossInputs(_ptr(weights), _ptr(advantages), _ptr(sampler_logprobs), clip_eps)
    _check(_lib.mlora_forward_backward(h.ptr, ctypes.byref(b), LOSS_KINDS[loss_kind],
                                       ctypes.byref(li), _ptr(logprobs_out), _ptr(loss_out),
                                       _stream(stream)))
    return logprobs_out, loss_out


def mlora_forward_backward_custom(h: Handle, tokens, targets, adapter_ids, dloss_dlogprobs,
                                  logprobs_out=None, loss_out=None, stream=None):
    import torch
    dev = tokens.device
    if logprobs_out is None:
        logprobs_out = torch.empty(tokens.numel(), dtype=torch.float32, device=dev)
    if loss_out is None:
        loss_out = torch.empty(h.n_adapters, dtype=torch.float64, device=dev)
    b = _batch(tokens, targets, adapter_ids)
    _check(_lib.mlora_forward_backward_custom(h.ptr, ctypes.byref(b), _ptr(dloss_dlogprobs),
                                              _ptr(logprobs_out), _ptr(loss_out), _stream(stream)))
    return logprobs_out, loss_out


def mlora_optim_step(h: Handle, lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0,
                     adapters: Optional[Sequence[int]] = None, skipped_out=None, stream=None):
    """Adam step; returns the device int32 [n_adapters] skipped flags."""
    import torch
    if skipped_out is None:
        skipped_out = torch.empty(h.n_adapters, dtype=torch.int32, device="cuda")
    p = _Adam(lr, beta1, beta2, eps, weight_decay)
    if adapters is None:
        arr, n = None, 0
    else:
        n = len(adapters)
        arr = (c_int32 * max(1, n))(*adapters)
    _check(_lib.mlora_optim_step(h.ptr, ctypes.byref(p), arr, n, _ptr(skipped_out),
                                 _stream(stream)))
    return skipped_out


def mlora_save_state(h: Handle, path: str, stream=None):
    _check(_lib.mlora_save_state(h.ptr, os.fsencode(path), _stream(stream)))


def mlora_load_state(h: Handle, path: str, with_optimizer: bool = False, stream=None):
    """load_state (weights; optimizer reset) or load_state_with_optimizer."""
    _check(_lib.mlora_load_state(h.ptr, os.fsencode(path), 1 if with_optimizer else 0,
                                 _stream(stream)))


def mlora_export_merged(h: Handle, adapter: int, layer: int, which: str, out=None, stream=None):
    """W' = W + gamma B A of W1 (which="W1", [f, d]) or W2 ("W2", [d, f]) in the base dtype."""
    import torch
    idx = {"W1": 0, "W2": 1}[which]
    shape = (h.f, h.d) if idx == 0 else (h.d, h.f)
    if out is None:
        dt = torch.bfloat16 if h.dtype == "bf16" else torch.float32
        out = torch.empty(shape, dtype=dt, device="cuda")
    assert tuple(out.shape) == shape and out.is_contiguous()
    _check(_lib.mlora_export_merged(h.ptr, adapter, layer, idx, _ptr(out), _stream(stream)))
    return out


class Sampler:
    """Owns one mlora_sampler_t*; keeps its training handle alive."""

    def __init__(self, ptr: int, trainer: Handle, n_slots: int, max_rows: int):
        self.ptr = c_void_p(ptr)
        self.trainer = trainer
        self.n_slots, self.max_rows = n_slots, max_rows

    @property
    def kernel_launches(self) -> int:
        return int(_lib.mlora_sampler_kernel_launches(self.ptr))

    def __del__(self):
        try:
            if self.ptr and _lib is not None:
                _lib.mlora_sampler_destroy(self.ptr)
                self.ptr = c_void_p(0)
        except Exception:  # pragma: no cover - interpreter shutdown
            pass


def mlora_sampler_create(h: Handle, n_slots: int, max_rows: int) -> Sampler:
    out = c_void_p()
    _check(_lib.mlora_sampler_create(h.ptr, n_slots, max_rows, ctypes.byref(out)))
    return Sampler(out.value, h, n_slots, max_rows)


def mlora_sampler_publish(s: Sampler, slot: int, adapter: int, stream=None) -> int:
    """Snapshot adapter's current weights into slot; returns its optimizer step count."""
    ver = c_int64(0)
    _check(_lib.mlora_sampler_publish(s.ptr, slot, adapter, ctypes.byref(ver), _stream(stream)))
    return int(ver.value)


def mlora_sampler_logprobs(s: Sampler, tokens, targets, slots, stream=None):
    import torch
    n = int(tokens.numel())
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    _check(_lib.mlora_sampler_logprobs(s.ptr, _ptr(tokens), _ptr(targets), _ptr(slots), n, _ptr(out),
                                       _stream(stream)))
    return out


def mlora_sampler_sample(s: Sampler, tokens, slots, uniforms, stream=None):
    """One decode step: (next tokens int32, their logprobs fp32)."""
    import torch
    n = int(tokens.numel())
    nxt = torch.empty(n, dtype=torch.int32, device="cuda")
    lp = torch.empty(n, dtype=torch.float32, device="cuda")
    _check(_lib.mlora_sampler_sample(s.ptr, _ptr(tokens), _ptr(slots), _ptr(uniforms), n, _ptr(nxt),
                                     _ptr(lp), _stream(stream)))
    return nxt, lp


def mlora_sampler_check_status(s: Sampler, stream=None) -> int:
    """0, or the negative MLORA_E_* code of the sampler's status word (cleared)."""
    return int(_lib.mlora_sampler_check_status(s.ptr, _stream(stream)))


def mlora_read_adapter(h: Handle, adapter: int, layer: int, which: str, stream=None):
    import torch
    out = torch.empty(h.shape_of(which, adapter), dtype=torch.float32, device="cuda")
    _check(_lib.mlora_read_adapter(h.ptr, adapter, layer, TENSOR_IDS[which], _ptr(out),
                                   _stream(stream)))
    return out


def mlora_write_adapter(h: Handle, adapter: int, layer: int, which: str, src, stream=None):
    assert tuple(src.shape) == h.shape_of(which, adapter)
    _check(_lib.mlora_write_adapter(h.ptr, adapter, layer, TENSOR_IDS[which], _ptr(src),
                                    _stream(stream)))


def mlora_get_steps(h: Handle, stream=None):
    arr = (c_int64 * h.n_adapters)()
    _check(_lib.mlora_get_steps(h.ptr, arr, _stream(stream)))
    return list(arr)


def mlora_get_routing(h: Handle, adapter_ids, stream=None):
    """Returns (perm, seg_off, pad_off, tile_ad) as CUDA int32 tensors."""
    import torch
    n = int(adapter_ids.numel())
    dev = adapter_ids.device
    perm = torch.empty(max(1, n), dtype=torch.int32, device=dev)
    seg = torch.empty(h.n_adapters + 1, dtype=torch.int32, device=dev)
    pad = torch.empty(h.n_adapters + 1, dtype=torch.int32, device=dev)
    tiles = torch.empty(n // TILE_M + h.n_adapters + 1, dtype=torch.int32, device=dev)
    _check(_lib.mlora_get_routing(h.ptr, _ptr(adapter_ids), n, _ptr(perm), _ptr(seg), _ptr(pad),
                                  _ptr(tiles), _stream(stream)))
    return perm[:n], seg, pad, tiles


def mlora_routing_noalloc(adapter_ids, n_adapters: int, stream=None):
    """Routing with no handle and no device allocation by the library.

    For callers that cannot call cudaMalloc; the library keeps its scratch in
    a fixed device array.  The output tensors here are allocated by torch on
    the caller's side.  Returns (perm, seg_off, pad_off, tile_ad) like
    mlora_get_routing.
    """
    import torch
    load_library()
    n = int(adapter_ids.numel())
    dev = adapter_ids.device
    perm = torch.empty(max(1, n), dtype=torch.int32, device=dev)
    seg = torch.empty(n_adapters + 1, dtype=torch.int32, device=dev)
    pad = torch.empty(n_adapters + 1, dtype=torch.int32, device=dev)
    tiles = torch.empty(n // TILE_M + n_adapters + 1, dtype=torch.int32, device=dev)
    _check(_lib.mlora_routing_noalloc(_ptr(adapter_ids), n, n_adapters, _ptr(perm), _ptr(seg),
                                      _ptr(pad), _ptr(tiles), _stream(stream)))
    return perm[:n], seg, pad, tiles


def mlora_check_status(h: Handle, stream=None) -> int:
    """Synchronise and return the device status code (0, -2 E_RANGE, -5 E_TIMEOUT)."""
    return int(_lib.mlora_check_status(h.ptr, _stream(stream)))


def mlora_set_deterministic(h: Handle, on: bool = True):
    """One gradient chunk per adapter: bitwise-reproducible gradients."""
    _check(_lib.mlora_set_deterministic(h.ptr, 1 if on else 0))


def mlora_set_lm_backward(h: Handle, mode: str):
    """LM-head backward mode: "recompute" (default) or "keep_logits"."""
    _check(_lib.mlora_set_lm_backward(h.ptr, LM_BACKWARD_MODES[mode]))


def mlora_profile_enable(h: Handle, on: bool = True):
    _check(_lib.mlora_profile_enable(h.ptr, 1 if on else 0))


def mlora_profile_read(h: Handle, reset: bool = True) -> dict:
    """{class: (milliseconds, launches)} accumulated since the last reset."""
    n = len(PROF_CLASSES)
    ms = (c_double * n)()
    cnt = (c_int64 * n)()
    _check(_lib.mlora_profile_read(h.ptr, ms, cnt, 1 if reset else 0))
    return {PROF_CLASSES[i]: (float(ms[i]), int(cnt[i])) for i in range(n)}
