#!/usr/bin/env python
"""Benchmark: trained tokens/s of one forward_backward + optim_step.

A step is one pass of the whole hot path over one synthetic batch: routing,
embedding, L LoRA-MLP blocks, LM head with the loss epilogue, the backward
(LM head chunk by chunk, the blocks in reverse, per-adapter gradient GEMMs)
and the per-adapter Adam update.  Default workload: Qwen3-8B widths
(V=151936, d=4096, f=12288, L=4), 32 rank-32 adapters with Zipf(1.1)
traffic, 65,536 tokens in sequences of 512-2048 tokens, PPO clip 0.2.

The LM-head backward has two modes (mlora_set_lm_backward): "keep_logits"
(each chunk's logits kept from the forward as fp16 exp(z - tile max) beside
the tile maxima; the headline by default,
--lm-backward) and "recompute" (a second GEMM recomputes each chunk's
logits; the library's default).  Both are timed; `lm_backward` reports the
step time and device memory of each.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is device-timed throughput with the
inputs resident in HBM (CUDA events on the launch stream, max over ranks);
`e2e` is the same metric through the C-ABI with host buffers, the copies
inside the timed region.  The headline loop runs without instrumentation; a
second loop of the same length records the library's per-launch CUDA events,
from which `roofline` (the tcgen05 GEMM kernel family, algorithmic FLOPs
only) and `kernels` (per-class breakdown) are taken.  `cpu_baseline` is the
CPU oracle on a bounded sample.
`--impl reference` times the CPU oracle itself (the reference arm).
With N > 1 (torchrun) every rank runs an independent replica of the
workload on its own GPU: the path has no cross-replica exchange in this
build, so scaling is weak and no collective touches the data path.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as wl  # noqa: E402

PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GB300 datasheet dense bf16 tensor-core peak (no sparsity), TFLOP/s, and the
# dense bf16 rate of one SM's tensor cores per clock (FLOP), for the
# clock-adjusted peak = SMs x rate x sampled median SM clock
DATASHEET_BF16_TFLOPS = 2250.0
BF16_FLOP_PER_CLK_SM = 8192
TC_CLASSES = ("w1_fwd", "w2_fwd", "lm_fwd", "lm_dh", "w2_bwd", "w1_bwd")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="qwen3_8b_ppo", choices=wl.CONFIG_NAMES)
    ap.add_argument("--tokens", type=int, default=None, help="override the batch size (tokens)")
    ap.add_argument("--cpu-sample", type=int, default=256,
                    help="tokens of the oracle's bounded CPU sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the sampler-decode and export-merge measurements")
    ap.add_argument("--no-tf", action="store_true",
                    help="skip the transformer-block row (next_rows.transformer_step)")
    ap.add_argument("--tf-only", action="store_true",
                    help="run only the transformer-block row and print it (profiling)")
    ap.add_argument("--tf-tokens", type=int, default=None,
                    help="override the transformer row's batch size (profiling; not a bench value)")
    ap.add_argument("--tf-prefix", type=int, default=None,
                    help="profiling: the first N tokens of the full-size batch (sequences keep "
                         "their 512-2048 lengths; not a bench value)")
    ap.add_argument("--tf-vocab", type=int, default=None,
                    help="override the transformer row's vocabulary (profiling; not a bench value)")
    ap.add_argument("--tf-layers", type=int, default=None,
                    help="override the transformer row's layer count (profiling; not a bench value)")
    ap.add_argument("--tf-attn-bwd", default="stored_ds", choices=["stored_ds", "recompute"],
                    help="attention backward of the transformer row's timed loop: dS blocks stored "
                         "for the workload's longest sequence, or S and dP recomputed on the query "
                         "side (the other mode's per-class times are reported too)")
    ap.add_argument("--deterministic", action="store_true",
                    help="batch-invariant mode: one gradient chunk per adapter")
    ap.add_argument("--lm-backward", default="keep_logits", choices=["keep_logits", "recompute"],
                    help="LM-head backward mode of the headline loop (the other mode is timed too)")
    ap.add_argument("--no-other-lm-mode", action="store_true",
                    help="skip timing the LM-head backward mode the headline does not use")
    ap.add_argument("--layers", type=int, default=None,
                    help="profiling only: override the block count (not a bench value)")
    ap.add_argument("--vocab", type=int, default=None,
                    help="profiling only: override the vocabulary size (not a bench value)")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    except (OSError, ValueError):
        return dict(PEAKS_FALLBACK), "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.first = 0
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def mark(self):
        """The timed region starts: later summaries use the samples from here on
        (and the one just before, so that a short region has one)."""
        self.first = max(0, len(self.lines) - 1)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines[self.first:]:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# the workload
# ---------------------------------------------------------------------------
def flop_model(cfg, b):
    """Algorithmic FLOPs of one step, per kernel family (no recompute, no padding)."""
    d, f, L, V = cfg.d_model, cfg.d_ffn, cfg.n_layers, cfg.vocab
    N = len(b["tokens"])
    ranks = np.array(cfg.ranks)[b["adapter_ids"]]
    sr = float(ranks.sum())                         # sum over tokens of r
    base = 8.0 * N * d * f * L
    lora_ext = 4.0 * sr * (d + f) * L               # expand in fwd + dgrad through A in bwd
    lm = 4.0 * N * V * d                            # LM head forward + dh
    small = 8.0 * sr * (d + f) * L                  # shrinks (fwd+bwd) and dA/dB reductions
    return {"tc256": base + lora_ext + lm, "tc64": small, "total": base + lora_ext + lm + small,
            "mean_rank": sr / max(1, N)}


def adam_bytes(cfg, b):
    present = np.unique(b["adapter_ids"])
    n = sum(cfg.n_layers * 2 * cfg.ranks[a] * (cfg.d_model + cfg.d_ffn) for a in present)
    return 28.0 * n, n


# Sources that determine the GEMM kernels and their launches: the kernel and
# header files whole, and of the host code the span that builds the step's
# launch descriptors (from the GEMM descriptor helpers to the first entry
# point), so that a change elsewhere in the host code (create, checkpoints)
# does not void the committed counters.
KERNEL_SOURCES = ("gemm_tc.cu", "gemm_common.cuh", "tc_ptx.cuh", "common.cuh", "internal.h",
                  "kernels_misc.cu")
LAUNCH_SPAN = ("mlora_api.cu", "// GEMM descriptor helpers", 'extern "C" int mlora_forward(')


def kernel_source_hash(read=None) -> str:
    """Hash of the sources that determine the GEMM kernels and their launches.
    `read(name) -> bytes` reads a file of the kernel directory (default: the tree)."""
    import hashlib
    if read is None:
        def read(name):
            with open(os.path.join(ROOT, "rl_step_gb300", "csrc", name), "rb") as fh:
                return fh.read()
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        h.update(read(name))
    text = read(LAUNCH_SPAN[0])
    a = text.index(LAUNCH_SPAN[1].encode())
    b = text.index(LAUNCH_SPAN[2].encode(), a)
    h.update(text[a:b])
    return h.hexdigest()


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic_tc_gemm_pair_kernel_small_case.json")
BLOCK_KINDS = ("w1_fwd", "w2_fwd", "w2_bwd", "w1_bwd")


def scaled_traffic(cfg, rows: int, launches_per_step: float, lm_mode: str, path: str = TRAFFIC_FILE):
    """Per-launch DRAM bytes of the CTA-pair GEMM at this workload's size, from
    the committed small-case capture: each launch kind's bytes scaled by the
    padded rows (and, for the LM-head launches, by the vocabulary), summed
    over the step's launches and divided by their number.  None when the
    capture is missing, was taken at other widths or on other kernel sources."""
    try:
        with open(path) as fh:
            rec = json.load(fh)
        current = kernel_source_hash()
    except (OSError, ValueError):          # no capture, or a source / span marker is gone
        return None
    if rec.get("kernel_source_sha256") != current:
        return None
    if (rec.get("d_model"), rec.get("d_ffn")) != (cfg.d_model, cfg.d_ffn) or launches_per_step <= 0:
        return None
    kinds = rec.get("bytes_per_launch", {}).get(lm_mode)
    if not kinds:
        return None
    r = rows / rec["rows"]
    v = cfg.vocab / rec["vocab"]
    total = cfg.n_layers * sum(kinds[k] for k in BLOCK_KINDS) * r
    total += sum(b for k, b in kinds.items() if k not in BLOCK_KINDS) * r * v
    return total / launches_per_step


def padded_rows(cfg, b):
    counts = np.bincount(b["adapter_ids"], minlength=cfg.n_adapters)
    return int(((counts + 127) // 128 * 128).sum())


def loss_epilogue_bytes(cfg, b, bn=256):
    """Bytes the loss epilogue must move: per padded row the vocabulary-tile
    log-sum-exp partials (4 B each) and five scalars; per token its loss
    inputs and the logprob it returns."""
    n_nt = (cfg.vocab + bn - 1) // bn
    rows = padded_rows(cfg, b)
    per_tok_in = {"cross_entropy": 4, "importance_sampling": 8, "ppo": 8, "custom": 4}[cfg.loss]
    return rows * (4.0 * n_nt + 20.0) + len(b["tokens"]) * (per_tok_in + 4.0)


def lora_hbm_bytes(cfg, b):
    """Bytes the LoRA shrinks (and, equally, the per-adapter gradient GEMMs)
    must move per step: each reads one activation per launch once -- per
    layer h and act forward, dh and du backward, [tokens x d or f] in the
    base dtype -- and its [tokens x 64] factor operand."""
    es = 2 if cfg.dtype == "bf16" else 4
    N = len(b["tokens"])
    return cfg.n_layers * (2.0 * N * (cfg.d_model + cfg.d_ffn) * es + 4.0 * N * 64 * es)


def lm_dz_bytes(cfg, b):
    """Bytes the LM-head dz pass must move: per token its kept logits read and
    its dz row written -- on the bf16 engine the fp16 e = exp(z - tile max)
    (2 B x V) and bf16 dz (2 B x V), on the fp32 one fp32 logits and dz."""
    return len(b["tokens"]) * cfg.vocab * (4.0 if cfg.dtype == "bf16" else 8.0)


def run_ours(args, rank, world):
    import torch

    import rl_step_gb300 as m
    from rl_step_gb300 import _build

    _build.build()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = wl.get_config(args.config)
    over = {k: v for k, v in (("n_layers", args.layers), ("vocab", args.vocab)) if v}
    if over:
        cfg = wl.get_config(args.config, **over)
    N_req = args.tokens or cfg.n_tokens
    b = wl.make_batch(cfg, N_req)
    N = len(b["tokens"])
    base = wl.make_base_weights(cfg)
    ad = wl.make_adapters(cfg)

    def T(x):
        x = np.ascontiguousarray(x)
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(x).to(dev)

    dbase = {"E": T(base["E"]), "W1": [T(w) for w in base["W1"]],
             "W2": [T(w) for w in base["W2"]], "Wout": T(base["Wout"])}
    dad = [[[T(x) for x in row] for row in ad[k]] for k in ("A1", "B1", "A2", "B2")]
    h = m.mlora_create(cfg.vocab, cfg.d_model, cfg.d_ffn, cfg.n_layers, cfg.dtype, cfg.ranks,
                       cfg.alphas, N, dbase["E"], dbase["W1"], dbase["W2"], dbase["Wout"], *dad)
    if args.deterministic:
        m.mlora_set_deterministic(h, True)
    m.mlora_set_lm_backward(h, args.lm_backward)
    torch.cuda.synchronize()
    del dbase, dad                      # the library holds its own copies
    torch.cuda.empty_cache()
    tok, tgt, ids = T(b["tokens"]), T(b["targets"]), T(b["adapter_ids"])
    stream = torch.cuda.current_stream()
    kind = cfg.loss
    # sampler logprobs of the policy-gradient losses: the current policy's
    # logprobs (one untimed forward) plus the workload's noise
    s_dev = None
    if kind in ("importance_sampling", "ppo"):
        ell = m.mlora_forward(h, tok, tgt, ids)
        s_dev = (ell + T(b["sampler_noise"])).contiguous()
    w_dev, a_dev, g_dev = T(b["weights"]), T(b["advantages"]), T(b["dloss"])
    lp_out = torch.empty(N, dtype=torch.float32, device=dev)
    loss_out = torch.empty(cfg.n_adapters, dtype=torch.float64, device=dev)
    skipped = torch.empty(cfg.n_adapters, dtype=torch.int32, device=dev)

    def step(tk=tok, tg=tgt, ai=ids, w=w_dev, av=a_dev, sl=s_dev, gd=g_dev):
        if kind == "custom":
            m.mlora_forward_backward_custom(h, tk, tg, ai, gd, logprobs_out=lp_out, loss_out=loss_out)
        else:
            m.mlora_forward_backward(h, tk, tg, ai, kind, weights=w, advantages=av,
                                     sampler_logprobs=sl, clip_eps=cfg.clip_eps,
                                     logprobs_out=lp_out, loss_out=loss_out)
        m.mlora_optim_step(h, lr=cfg.lr, beta1=cfg.beta1, beta2=cfg.beta2, eps=cfg.eps,
                           weight_decay=cfg.weight_decay, skipped_out=skipped)

    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist = dist_mod

    def barrier():
        if dist is not None:
            dist.barrier()

    def timed_steps(n):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    # ---- device-timed region (no instrumentation) ----------------------------
    # The clock sampler starts first; the warm-up steps then run right before
    # the timed ones, so the timed steps follow steps as in training, not an
    # idle GPU (whose power controller overshoots on the first busy second).
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.5)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = m.mlora_check_status(h)
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up")
    launches0 = h.kernel_launches
    barrier()
    torch.cuda.synchronize()
    clocks.mark()
    ms = timed_steps(args.steps)
    barrier()
    clk = clocks.stop()
    launches = h.kernel_launches - launches0
    ms_max = max_over_ranks(ms, dev)
    status = m.mlora_check_status(h)
    if status != 0:
        raise RuntimeError(f"device status {status} in the timed region")

    # ---- per-class timing: a second loop with the library's per-launch events
    m.mlora_profile_read(h, reset=True)
    m.mlora_profile_enable(h, True)
    ms_prof = timed_steps(args.steps)
    m.mlora_profile_enable(h, False)
    prof = m.mlora_profile_read(h, reset=True)

    # ---- end-to-end through host buffers -------------------------------------
    e2e = None
    if not args.no_e2e:
        pin = lambda x: torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
        hs = {"tok": pin(b["tokens"]), "tgt": pin(b["targets"]), "ids": pin(b["adapter_ids"])}
        dev_bufs = {k: torch.empty_like(v, device=dev) for k, v in hs.items()}
        loss_in = {}
        if kind == "cross_entropy":
            loss_in["w"] = pin(b["weights"])
        elif kind == "custom":
            loss_in["g"] = pin(b["dloss"])
        else:
            loss_in["av"] = pin(b["advantages"])
            loss_in["sl"] = s_dev.cpu().pin_memory()
        dev_loss = {k: torch.empty_like(v, device=dev) for k, v in loss_in.items()}
        lp_host = torch.empty(N, dtype=torch.float32).pin_memory()
        loss_host = torch.empty(cfg.n_adapters, dtype=torch.float64).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in list(hs.values()) + list(loss_in.values()))
        d2h = lp_host.numel() * 4 + loss_host.numel() * 8

        def e2e_step():
            for k, v in hs.items():
                dev_bufs[k].copy_(v, non_blocking=True)
            for k, v in loss_in.items():
                dev_loss[k].copy_(v, non_blocking=True)
            step(dev_bufs["tok"], dev_bufs["tgt"], dev_bufs["ids"], dev_loss.get("w", w_dev),
                 dev_loss.get("av", a_dev), dev_loss.get("sl", s_dev), dev_loss.get("g", g_dev))
            lp_host.copy_(lp_out, non_blocking=True)
            loss_host.copy_(loss_out, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        barrier()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            e2e_step()
        torch.cuda.synchronize()
        t_e2e = max_over_ranks(time.perf_counter() - t0, dev)
        e2e = {"value": job_throughput(N, args.steps, world, 1e3 * t_e2e), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": 1e3 * t_e2e / args.steps,
               "note": ("timed after the headline and per-class loops, so later in the SM clock's "
                        "rise over the first seconds of load; the copies cost well under 1 % of a step")}

    # ---- tokens whose dL/dl is non-zero (from this run's logprobs) ----------
    nz_g = count_nonzero_g(cfg, b, lp_out.cpu().numpy(),
                           s_dev.cpu().numpy() if s_dev is not None else None)

    # ---- custom-loss protocol: the client's forward, then the custom step ----
    protocol = None
    if kind == "custom" and not args.no_extras:
        torch.cuda.synchronize()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        for _ in range(args.steps):
            m.mlora_forward(h, tok, tgt, ids, logprobs_out=lp_out)
            step()
        p1.record(stream)
        torch.cuda.synchronize()
        pms = p0.elapsed_time(p1) / args.steps
        protocol = {"what": "mlora_forward + mlora_forward_backward_custom + mlora_optim_step",
                    "ms_per_step": pms, "tokens_per_s": N / (pms * 1e-3),
                    "cost_vs_step": pms / (ms / args.steps)}

    # ---- the other LM-head backward mode --------------------------------------
    fl = flop_model(cfg, b)
    lm_modes = {args.lm_backward: {"ms_per_step": ms_max / args.steps,
                                   "tokens_per_s": job_throughput(N, args.steps, world, ms_max),
                                   "device_bytes": h.device_bytes, "headline": True}}
    if not args.no_other_lm_mode:
        other = "recompute" if args.lm_backward == "keep_logits" else "keep_logits"
        m.mlora_set_lm_backward(h, other)
        for _ in range(2):
            step()
        torch.cuda.synchronize()
        barrier()
        oms = max_over_ranks(timed_steps(args.steps), dev)
        if m.mlora_check_status(h) != 0:
            raise RuntimeError(f"device status set in the {other} timing")
        m.mlora_profile_read(h, reset=True)
        m.mlora_profile_enable(h, True)
        timed_steps(1)
        m.mlora_profile_enable(h, False)
        oprof = m.mlora_profile_read(h, reset=True)
        lm_modes[other] = {"ms_per_step": oms / args.steps,
                           "tokens_per_s": job_throughput(N, args.steps, world, oms),
                           "device_bytes": h.device_bytes, "headline": False,
                           "lm_ms_per_step": {c: oprof[c][0] for c in ("lm_fwd", "lm_dz", "lm_dh", "loss")}}
        m.mlora_set_lm_backward(h, args.lm_backward)
    for v in lm_modes.values():
        v["frac_of_bf16_peak"] = fl["total"] / (v["ms_per_step"] * 1e-3) / 1e12 / \
            load_peaks()[0]["bf16_tflops"]
    lm_modes["note"] = ("recompute: a second LM-head GEMM per chunk (2 N V d executed FLOPs, not "
                        "credited) and one dz chunk buffer; keep_logits: each chunk's logits kept from "
                        "the forward (fp16 exp(z - tile max) on the bf16 engine), dz by an "
                        "elementwise pass on a side stream")

    # ---- rows beyond the step (outside the timed region) ---------------------
    extras = None if args.no_extras else measure_next_rows(m, h, cfg, b, dev, stream)

    # ---- derived numbers -----------------------------------------------------
    peaks, peak_src = load_peaks()
    if extras is not None:
        del h
        torch.cuda.empty_cache()
        extras["loss_epilogue_scaled"] = measure_loss_epilogue_scaled(dev, stream, peaks)
        if not args.no_tf:
            extras["transformer_step"] = measure_transformer_row(args, dev, stream, peaks)
    if extras:
        for k in ("sampler_decode", "export_merge"):
            extras[k]["frac_of_hbm"] = extras[k]["achieved_gbs"] / peaks["hbm_gbs"]
    K = args.steps
    # dominant kernel: the CTA-pair tcgen05 GEMM, which carries every base and
    # LM-head GEMM (22 launches per step at L=4: 16 block GEMMs and 3 + 3
    # LM-head chunks).  Algorithmic FLOPs credit the base and LoRA-extension
    # GEMMs, the LM-head forward and dh; padding rows are executed work only.
    tc_classes = TC_CLASSES + (("lm_dz",) if args.lm_backward == "recompute" else ())
    tc_ms = sum(prof[c][0] for c in tc_classes)
    tc_launch = sum(prof[c][1] for c in tc_classes)
    achieved = fl["tc256"] * K / (tc_ms * 1e-3) / 1e12 if tc_ms > 0 else None
    rows = padded_rows(cfg, b)
    exec_flops = fl["tc256"] * rows / max(1, N)
    executed = exec_flops * K / (tc_ms * 1e-3) / 1e12 if tc_ms > 0 else None
    peak_tc = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    traffic = scaled_traffic(cfg, padded_rows(cfg, b), tc_launch / K, args.lm_backward)
    step_ms = ms_max / K
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    adam_b, n_ad_params = adam_bytes(cfg, b)
    kernels = {c: {"ms_per_step": v[0] / K, "launches_per_step": v[1] / K} for c, v in prof.items()
               if v[1] > 0}
    if prof["adam"][0] > 0:
        kernels["adam"]["achieved_gbs"] = adam_b * K / (prof["adam"][0] * 1e-3) / 1e9
        kernels["adam"]["frac_of_hbm"] = kernels["adam"]["achieved_gbs"] / peaks["hbm_gbs"]
        kernels["adam"]["bytes_per_step"] = adam_b
    if prof["lm_dz"][0] > 0 and args.lm_backward == "keep_logits":
        zb = lm_dz_bytes(cfg, b)
        kernels["lm_dz"]["achieved_gbs"] = zb * K / (prof["lm_dz"][0] * 1e-3) / 1e9
        kernels["lm_dz"]["frac_of_hbm"] = kernels["lm_dz"]["achieved_gbs"] / peaks["hbm_gbs"]
        kernels["lm_dz"]["bytes_per_step"] = zb
        kernels["lm_dz"]["note"] = ("side stream, concurrent with the next chunk's LM-head GEMM: "
                                    "ms_per_step is the span of its events under that overlap, "
                                    "not its exclusive time (see the serialised ncu launch list)")
    lb_lora = lora_hbm_bytes(cfg, b)
    for c in ("shrink", "grad"):
        if prof[c][0] > 0:
            kernels[c]["achieved_gbs"] = lb_lora * K / (prof[c][0] * 1e-3) / 1e9
            kernels[c]["frac_of_hbm"] = kernels[c]["achieved_gbs"] / peaks["hbm_gbs"]
            kernels[c]["bytes_per_step"] = lb_lora
    if prof["loss"][0] > 0:
        lb = loss_epilogue_bytes(cfg, b)
        kernels["loss"]["achieved_gbs"] = lb * K / (prof["loss"][0] * 1e-3) / 1e9
        kernels["loss"]["frac_of_hbm"] = kernels["loss"]["achieved_gbs"] / peaks["hbm_gbs"]
        kernels["loss"]["bytes_per_step"] = lb
    out = {
        "metric": "trained tokens/sec per forward_backward+optim_step",
        "value": job_throughput(N, K, world, ms_max),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if cfg.dtype == "bf16" else "f32",
        "data": "synthetic (seeded), random-init weights",
        "config": {"workload": cfg.description, "name": cfg.name, "tokens_per_gpu": N,
                   "adapters": cfg.n_adapters, "loss": cfg.loss,
                   "l2": "inputs larger than L2 (frozen base %.1f GB)" %
                         ((2 * cfg.vocab * cfg.d_model + 2 * cfg.n_layers * cfg.d_model * cfg.d_ffn)
                          * (2 if cfg.dtype == "bf16" else 4) / 1e9),
                   "parallelism": f"replicas x{world}",
                   "deterministic": bool(args.deterministic)},
        "tflops_algorithmic": fl["total"] * K * world / (ms_max * 1e-3) / 1e12,
        "frac_of_bf16_peak": fl["total"] / (step_ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
        "frac_of_bf16_peak_basis": {
            "measured_burst": fl["total"] / (step_ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
            "measured_sustained": fl["total"] / (step_ms * 1e-3) / 1e12 /
                                  peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]),
            "datasheet_dense_2250": fl["total"] / (step_ms * 1e-3) / 1e12 / DATASHEET_BF16_TFLOPS,
            "clock_adjusted": (fl["total"] / (step_ms * 1e-3) / 1e12 /
                               (BF16_FLOP_PER_CLK_SM * n_sms * clk["sm_mhz"] * 1e6 / 1e12))
                              if clk.get("sm_mhz") else None,
            "clock_adjusted_peak_tflops": (BF16_FLOP_PER_CLK_SM * n_sms * clk["sm_mhz"] * 1e6 / 1e12)
                                          if clk.get("sm_mhz") else None},
        "lm_backward": lm_modes,
        "roofline": {"kernel": "the CTA-pair tcgen05 GEMM: tc_gemm_pair_kernel<256,3,2,2> (base, LoRA-extension "
                               "and LM-head forward GEMMs) and <512,4,1,1> (LM-head dh)",
                     "bound": "tensor", "achieved": achieved, "peak": peak_tc,
                     "peak_kind": f"bf16_tflops_sustained ({peak_src})", "unit": "TFLOP/s",
                     "frac": (achieved / peak_tc) if achieved else None, "traffic": traffic,
                     "traffic_unit": "bytes per launch (DRAM read + write, ncu): small-case capture "
                                     "scaled by padded rows (and vocabulary for the LM head)",
                     "launches_per_step": tc_launch / K,
                     "timed_in": "a second loop of the same steps with per-launch CUDA events "
                                 f"({ms_prof / K:.2f} ms per step there, {step_ms:.2f} without)",
                     "algorithmic_flops_per_launch": fl["tc256"] / max(1.0, tc_launch / K),
                     "executed_tflops": executed},
        "kernels": kernels,
        "clocks": clk,
        "gpu_launches": int(launches),
        "e2e": e2e,
    }
    out["config"]["tokens_nonzero_g"] = nz_g
    if over:
        out["config"]["profiling_override"] = over      # not a bench value
    if protocol:
        out["custom_protocol"] = protocol
    if extras:
        out["next_rows"] = extras
    return out, (cfg, base, ad, b)


TF_TC_CLASSES = ("qkv", "o", "gateup", "down", "lm_fwd", "lm_dh", "down_bwd", "gateup_bwd", "o_bwd",
                 "qkv_bwd")


def tf_flop_model(cfg, b):
    """Algorithmic FLOPs of one transformer-block step (no recompute, no
    padding rows, no masked attention pairs): the seven projections forward
    and their dgrad backward, the LoRA shrink / expand and gradient GEMMs,
    causal attention (QK^T and PV forward; dV, dP, dQ, dK backward) over the
    (query, key) pairs of each sequence, and the LM head (forward + dh)."""
    d, f, L, V = cfg.d_model, cfg.d_ffn, cfg.n_layers, cfg.vocab
    q, kv, hd = cfg.n_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim, cfg.head_dim
    N = len(b["tokens"])
    io = [(q, d), (kv, d), (kv, d), (d, q), (f, d), (f, d), (d, f)]
    macs = sum(o * i for o, i in io)
    sr = float(np.array(cfg.ranks)[b["adapter_ids"]].sum())
    proj = 4.0 * N * macs * L                                  # forward + dgrad
    lora = 6.0 * sr * sum(o + i for o, i in io) * L            # 2 r(in+out) forward, twice that backward
    pairs = float((b["positions"].astype(np.int64) + 1).sum())  # causal (query, key) pairs
    attn_fwd = 4.0 * pairs * hd * cfg.n_heads * L
    attn_bwd = 2.0 * attn_fwd
    lm = 4.0 * N * V * d
    return {"proj_lm": proj + lm, "lora": lora, "attn_fwd": attn_fwd, "attn_bwd": attn_bwd,
            "total": proj + lora + attn_fwd + attn_bwd + lm}


def measure_transformer_row(args, dev, stream, peaks):
    """One forward_backward + optim_step of the transformer-block model at the
    Qwen3-8B widths (qwen3_8b_tf_ppo: 32 / 8 heads of 128, L = 4, 32 adapters,
    65,536 tokens in sequences of 512-2048, PPO), device-timed with CUDA
    events on the launch stream after warm-up; per-class times from the
    library's per-launch events."""
    import torch

    import rl_step_gb300.transformer as t
    import workloads.transformer as wt
    over = {k: v for k, v in (("n_layers", args.tf_layers), ("vocab", args.tf_vocab)) if v}
    cfg = wt.get_tf_config("qwen3_8b_tf_ppo", **over)
    b = wt.make_tf_batch(cfg, args.tf_tokens)
    if args.tf_prefix:
        b = {k: (v[:args.tf_prefix] if isinstance(v, np.ndarray) else v) for k, v in b.items()}
    N = len(b["tokens"])
    base = wt.make_tf_base_weights(cfg)
    ad = wt.make_tf_adapters(cfg)

    def T(x):
        x = np.ascontiguousarray(x)
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(x).to(dev)

    dbase = {"E": T(base["E"]), "Wout": T(base["Wout"]), "final_norm": T(base["final_norm"]),
             "attn_norm": [T(g) for g in base["attn_norm"]], "mlp_norm": [T(g) for g in base["mlp_norm"]],
             "W": {p: [T(w) for w in base["W"][p]] for p in t.PROJ}}
    A = {p: [[T(x) for x in row] for row in ad["A"][p]] for p in t.PROJ}
    B = {p: [[T(x) for x in row] for row in ad["B"][p]] for p in t.PROJ}
    del base, ad
    h = t.tf_create(cfg.vocab, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.d_ffn, cfg.n_layers, cfg.ranks,
                    cfg.alphas, N, dbase, A, B, rope_theta=cfg.rope_theta, rms_eps=cfg.rms_eps)
    t.tf_set_lm_backward(h, args.lm_backward)     # the MLP step's mode
    # stored dS blocks: sequences of at most the workload's longest (2,048 tokens)
    attn_seq = {"stored_ds": cfg.seq_hi, "recompute": 0}
    t.tf_set_attention_backward(h, attn_seq[args.tf_attn_bwd])
    mode_bytes = {args.tf_attn_bwd: h.device_bytes}
    torch.cuda.synchronize()
    del dbase, A, B
    torch.cuda.empty_cache()
    tok, tgt, pos, ids = T(b["tokens"]), T(b["targets"]), T(b["positions"]), T(b["adapter_ids"])
    s_dev = (t.tf_forward(h, tok, tgt, pos, ids) + T(b["sampler_noise"])).contiguous()
    a_dev = T(b["advantages"])
    lp_out = torch.empty(N, dtype=torch.float32, device=dev)
    loss_out = torch.empty(cfg.n_adapters, dtype=torch.float64, device=dev)
    skipped = torch.empty(cfg.n_adapters, dtype=torch.int32, device=dev)

    def step():
        t.tf_forward_backward(h, tok, tgt, pos, ids, "ppo", advantages=a_dev, sampler_logprobs=s_dev,
                              clip_eps=cfg.clip_eps, logprobs_out=lp_out, loss_out=loss_out)
        t.tf_optim_step(h, lr=cfg.lr, skipped_out=skipped)

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    if t.tf_check_status(h) != 0:
        raise RuntimeError("transformer row: device status after warm-up")
    K = max(1, min(args.steps, 5))

    def timed(profile):
        """ms per step over K steps; with per-launch events (per-class times) when profile."""
        t.tf_profile_read(h, reset=True)
        t.tf_profile_enable(h, profile)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        t.tf_profile_enable(h, False)
        if t.tf_check_status(h) != 0:
            raise RuntimeError("transformer row: device status in the timed region")
        return e0.elapsed_time(e1) / K, t.tf_profile_read(h, reset=True)

    launches0 = h.kernel_launches
    ms, _ = timed(False)                 # the row's step time: no per-launch events
    launches = (h.kernel_launches - launches0) / K
    ms_prof, prof = timed(True)          # per-class times, a second loop
    device_bytes = h.device_bytes
    # the other attention backward mode: per-class times of its own loop
    other = "recompute" if args.tf_attn_bwd == "stored_ds" else "stored_ds"
    t.tf_set_attention_backward(h, attn_seq[other])
    mode_bytes[other] = h.device_bytes
    step()
    torch.cuda.synchronize()
    ms_other, prof_other = timed(True)
    fl = tf_flop_model(cfg, b)
    peak_tc = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    kern = {c: {"ms_per_step": v[0] / K, "launches_per_step": v[1] / K} for c, v in prof.items() if v[1] > 0}

    def rate(flops, classes):
        tms = sum(prof[c][0] for c in classes) / K
        return (flops / (tms * 1e-3) / 1e12) if tms > 0 else None
    att_f, att_b = rate(fl["attn_fwd"], ("attn_fwd",)), rate(fl["attn_bwd"], ("attn_bwd",))
    gemm = rate(fl["proj_lm"], TF_TC_CLASSES)
    attn_modes = {}
    for mode, (msm, pr) in ((args.tf_attn_bwd, (ms_prof, prof)), (other, (ms_other, prof_other))):
        tb = pr["attn_bwd"][0] / K
        attn_modes[mode] = {"attn_bwd_ms_per_step": tb,
                            "bwd_tflops": fl["attn_bwd"] / (tb * 1e-3) / 1e12 if tb > 0 else None,
                            "bwd_frac": fl["attn_bwd"] / (tb * 1e-3) / 1e12 / peak_tc if tb > 0 else None,
                            "step_ms_with_per_launch_events": msm,
                            "max_seq_len": attn_seq[mode],
                            "device_bytes": mode_bytes[mode]}
    row = {
        "workload": cfg.description + (f" (override {over})" if over else ""),
        "tokens": N, "ms_per_step": ms, "tokens_per_s": N / (ms * 1e-3),
        "tflops_algorithmic": fl["total"] / (ms * 1e-3) / 1e12,
        "frac_of_bf16_peak": fl["total"] / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
        "flops_per_step": fl,
        "attention": {"fwd_tflops": att_f, "bwd_tflops": att_b, "peak": peak_tc,
                      "fwd_frac": att_f / peak_tc if att_f else None,
                      "bwd_frac": att_b / peak_tc if att_b else None,
                      "bound": "tensor", "unit": "TFLOP/s (algorithmic, causal pairs only; backward "
                                                "includes its rowsum pass; the recompute mode's second S "
                                                "and dP are not credited)",
                      "backward_mode": args.tf_attn_bwd, "backward_modes": attn_modes},
        "projection_and_lm_gemms": {"tflops": gemm, "frac": gemm / peak_tc if gemm else None},
        "kernels": kern, "gpu_launches_per_step": launches,
        "device_bytes": device_bytes, "lm_backward": args.lm_backward,
        "timing": "step time from a loop without per-launch events; per-class times from a second loop "
                  "with them",
    }
    del h
    torch.cuda.empty_cache()
    return row


def measure_loss_epilogue_scaled(dev, stream, peaks, n_tokens=1 << 24, reps=3):
    """The LM-head partial combine + loss epilogue as one launch over many rows.

    Inside the step the kernel runs per chunk of at most 16,384 rows (~39 MB
    each), too little work per launch to reach HBM bandwidth.  Here the same
    kernel runs once over n_tokens rows through mlora_forward (whose LM head
    keeps no logits and combines all rows at once) on a handle of the same
    vocabulary (V = 151,936, so 594 vocabulary-tile partials per row) whose
    model is shrunk to d = f = 64, L = 1, so that the rows are cheap to
    produce.  Bytes per padded row: 4 B per partial + 20 B of per-row scalars;
    per token the 4-byte logprob written.  Timed by the library's per-launch
    events (class "loss")."""
    import torch

    import rl_step_gb300 as m
    cfg = wl.get_config("qwen3_8b_ppo", d_model=64, d_ffn=64, n_layers=1, n_adapters=1, ranks=(32,),
                        alphas=(32.0,))
    base = wl.make_base_weights(cfg)
    ad = wl.make_adapters(cfg)

    def T(x):
        x = np.ascontiguousarray(x)
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(x).to(dev)

    h = m.mlora_create(cfg.vocab, cfg.d_model, cfg.d_ffn, cfg.n_layers, cfg.dtype, cfg.ranks, cfg.alphas,
                       n_tokens, T(base["E"]), [T(w) for w in base["W1"]], [T(w) for w in base["W2"]],
                       T(base["Wout"]), *[[[T(x) for x in row] for row in ad[k]] for k in ("A1", "B1", "A2", "B2")])
    rng = np.random.Generator(np.random.PCG64([cfg.seed, 41]))
    tok = T(rng.integers(0, cfg.vocab, n_tokens).astype(np.int32))
    tgt = T(rng.integers(0, cfg.vocab, n_tokens).astype(np.int32))
    ids = torch.zeros(n_tokens, dtype=torch.int32, device=dev)
    lp = torch.empty(n_tokens, dtype=torch.float32, device=dev)
    m.mlora_forward(h, tok, tgt, ids, logprobs_out=lp)
    torch.cuda.synchronize()
    m.mlora_profile_read(h, reset=True)
    m.mlora_profile_enable(h, True)
    for _ in range(reps):
        m.mlora_forward(h, tok, tgt, ids, logprobs_out=lp)
    torch.cuda.synchronize()
    m.mlora_profile_enable(h, False)
    prof = m.mlora_profile_read(h, reset=True)
    if m.mlora_check_status(h) != 0 or not bool(torch.isfinite(lp).all()):
        raise RuntimeError("scaled loss-epilogue run: bad status or logprobs")
    ms, n = prof["loss"]
    rows = (n_tokens + 127) // 128 * 128
    byt = rows * (4.0 * ((cfg.vocab + 255) // 256) + 20.0) + 4.0 * n_tokens
    del h
    torch.cuda.empty_cache()
    gbs = byt / (ms / n * 1e-3) / 1e9
    return {"kernel": "combine_loss_kernel", "tokens": n_tokens, "launches": n / reps, "ms": ms / n,
            "bytes": byt, "achieved_gbs": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"],
            "what": "one launch over all rows of a forward (V = 151,936; model shrunk to d = f = 64, L = 1)"}


def count_nonzero_g(cfg, b, lp, s):
    """Tokens whose dL/dl is non-zero for this batch (reported beside the
    trained-token count): CE w != 0, IS A != 0, custom g != 0; PPO A != 0 and
    the unclipped branch active at the run's logprobs."""
    if cfg.loss == "cross_entropy":
        return int(np.count_nonzero(b["weights"]))
    if cfg.loss == "custom":
        return int(np.count_nonzero(b["dloss"]))
    A = b["advantages"].astype(np.float64)
    if cfg.loss == "importance_sampling":
        return int(np.count_nonzero(A))
    r = np.exp(lp.astype(np.float64) - s.astype(np.float64))
    un = r * A
    cl = np.clip(r, 1 - cfg.clip_eps, 1 + cfg.clip_eps) * A
    return int(np.count_nonzero((A != 0) & (un <= cl)))


def measure_next_rows(m, h, cfg, b, dev, stream, reps=20):
    """Time the sampler's decode step and the export merge on the benchmark's
    handle (CUDA events on the launch stream, after a warm-up call).

    decode: one mlora_sampler_sample over `rows` rows spread over every
    adapter (one slot each); algorithmic bytes = the frozen base it streams
    (W1, W2 of every layer and Wout, base dtype) + every slot's factors + the
    rows' fp32 logits written and read.  export: one W1' = W1 + gamma B A;
    algorithmic bytes = W1 read + W1' written."""
    import torch
    es = 2 if cfg.dtype == "bf16" else 4
    d, f, L, V = cfg.d_model, cfg.d_ffn, cfg.n_layers, cfg.vocab
    out = {}
    n_slots = min(cfg.n_adapters, 64)
    rows = 256
    smp = m.mlora_sampler_create(h, n_slots, rows)
    for a in range(n_slots):
        m.mlora_sampler_publish(smp, a, a)
    rng = np.random.Generator(np.random.PCG64([cfg.seed, 31]))
    tok = torch.from_numpy(rng.integers(0, V, rows).astype(np.int32)).to(dev)
    sl = torch.from_numpy(rng.integers(0, n_slots, rows).astype(np.int32)).to(dev)
    u = torch.from_numpy(rng.random(rows).astype(np.float32)).to(dev)

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    launches0 = smp.kernel_launches
    ms = timed(lambda: m.mlora_sampler_sample(smp, tok, sl, u, stream=stream))
    if m.mlora_sampler_check_status(smp) != 0:
        raise RuntimeError("sampler status after the decode timing")
    vpad = (V + 63) // 64 * 64
    byt = (2 * L * d * f + V * d) * es + n_slots * 64 * 2 * (d + f) * L * es + rows * vpad * 8
    out["sampler_decode"] = {"rows": rows, "slots": n_slots, "ms_per_step": ms,
                             "tokens_per_s": rows / (ms * 1e-3),
                             "bytes_per_step": byt, "achieved_gbs": byt / (ms * 1e-3) / 1e9,
                             "gpu_launches_per_step": (smp.kernel_launches - launches0) / (reps + 1)}
    del smp
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    buf = torch.empty((f, d), dtype=dt, device=dev)
    ms = timed(lambda: m.mlora_export_merged(h, 0, 0, "W1", out=buf, stream=stream))
    byt = 2 * f * d * es
    out["export_merge"] = {"matrix": f"W1' [{f} x {d}]", "ms": ms, "bytes": byt,
                           "achieved_gbs": byt / (ms * 1e-3) / 1e9}
    return out


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of x over all ranks (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, steps: int, world: int, ms_max: float) -> float:
    """Whole-job tokens/s: all ranks' tokens over the slowest rank's time."""
    return tokens_per_rank * steps * world / (ms_max * 1e-3)


def make_oracle(cfg, base, ad):
    import oracle
    return oracle.Oracle(base, ad, cfg.ranks, cfg.alphas)


def oracle_sample_rate(cfg, o, b, n_sample, s_full=None):
    """Time the oracle's step on the first n_sample tokens; returns (tokens/s, seconds)."""
    sl = slice(0, n_sample)
    tok, tgt, ids = b["tokens"][sl], b["targets"][sl], b["adapter_ids"][sl]
    kw = {}
    if cfg.loss == "cross_entropy":
        kw["weights"] = b["weights"][sl]
    elif cfg.loss in ("importance_sampling", "ppo"):
        ell = o.forward(tok, tgt, ids) if s_full is None else s_full[sl]
        kw = {"advantages": b["advantages"][sl], "sampler_logprobs": ell + b["sampler_noise"][sl],
              "clip_eps": cfg.clip_eps}
    t0 = time.perf_counter()
    if cfg.loss == "custom":
        o.forward_backward_custom(tok, tgt, ids, b["dloss"][sl])
    else:
        o.forward_backward(tok, tgt, ids, cfg.loss, **kw)
    o.optim_step(lr=cfg.lr, beta1=cfg.beta1, beta2=cfg.beta2, eps=cfg.eps,
                 weight_decay=cfg.weight_decay)
    dt = time.perf_counter() - t0
    return n_sample / dt, dt


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count()


def run_reference(args):
    """The reference arm: the CPU oracle, timed as it stands, on a bounded
    sample of the same workload per step."""
    cfg = wl.get_config(args.config)
    b = wl.make_batch(cfg, args.tokens or cfg.n_tokens)
    base = wl.make_base_weights(cfg)
    ad = wl.make_adapters(cfg)
    n = min(64, len(b["tokens"]))
    o = make_oracle(cfg, base, ad)
    for _ in range(args.warmup):
        oracle_sample_rate(cfg, o, b, n)
    total = 0.0
    for _ in range(args.steps):
        total += oracle_sample_rate(cfg, o, b, n)[1]
    value = n * args.steps / total
    return {
        "metric": "trained tokens/sec per forward_backward+optim_step", "impl": "reference",
        "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded), random-init weights",
        "config": {"workload": cfg.description, "name": cfg.name,
                   "tokens_per_step": n, "sample": f"first {n} tokens of the batch per step"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores(), "kind": "oracle",
                         "sample": f"{n} tokens per step at full widths (numpy fp64)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if args.tf_only:
        import torch

        from rl_step_gb300 import _build
        _build.build()
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        row = measure_transformer_row(args, torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0"))),
                                      torch.cuda.current_stream(), load_peaks()[0])
        if rank == 0:
            print(json.dumps({"transformer_step": row}), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    out, ctx = run_ours(args, rank, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cfg, base, ad, b = ctx
        n = min(args.cpu_sample, len(b["tokens"]))
        rate, dt = oracle_sample_rate(cfg, make_oracle(cfg, base, ad), b, n)
        out["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": cores(),
                               "kind": "oracle",
                               "sample": f"first {n} tokens of the batch, forward_backward + "
                                         f"optim_step at full widths (numpy fp64, {dt:.1f} s)"}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
