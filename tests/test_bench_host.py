"""Host-side pieces of the benchmark that need no GPU: the hash that ties the
committed DRAM-traffic counters to the kernel sources they were taken on."""
import json
import os

import bench


def test_kernel_source_hash_finds_its_launch_span():
    h = bench.kernel_source_hash()
    assert len(h) == 64
    name, start, end = bench.LAUNCH_SPAN
    with open(os.path.join(bench.ROOT, "rl_step_gb300", "csrc", name)) as fh:
        text = fh.read()
    a = text.index(start)
    span = text[a:text.index(end, a)]
    # the span holds the step's launch sequence and the GEMM descriptor builders
    for marker in ("static int step_impl", "dense_params", "grad_params", "band_for_k"):
        assert marker in span, marker


def test_hash_follows_the_kernel_sources_and_ignores_other_host_code():
    files = {}

    def read(name):
        if name not in files:
            with open(os.path.join(bench.ROOT, "rl_step_gb300", "csrc", name), "rb") as fh:
                files[name] = fh.read()
        return files[name]

    h0 = bench.kernel_source_hash(read)
    api = read("mlora_api.cu")
    start = api.index(bench.LAUNCH_SPAN[1].encode())
    files["mlora_api.cu"] = b"// an edit outside the span\n" + api
    assert bench.kernel_source_hash(read) == h0
    files["mlora_api.cu"] = api[:start + 40] + b" " + api[start + 40:]
    assert bench.kernel_source_hash(read) != h0
    files["mlora_api.cu"] = api
    files["gemm_tc.cu"] = read("gemm_tc.cu") + b"\n"
    assert bench.kernel_source_hash(read) != h0


def test_scaled_traffic_scales_rows_and_vocabulary(tmp_path):
    import workloads as wl
    cfg = wl.get_config("qwen3_8b_ppo")
    rec = {"kernel_source_sha256": bench.kernel_source_hash(), "rows": 1000, "vocab": cfg.vocab // 2,
           "d_model": cfg.d_model, "d_ffn": cfg.d_ffn,
           "bytes_per_launch": {"keep_logits": {"w1_fwd": 1.0, "w2_fwd": 2.0, "w2_bwd": 3.0, "w1_bwd": 4.0,
                                                "lm_fwd": 5.0, "lm_dh": 6.0}}}
    path = tmp_path / "t.json"
    path.write_text(json.dumps(rec))
    got = bench.scaled_traffic(cfg, 3000, 10.0, "keep_logits", str(path))
    want = (cfg.n_layers * 10.0 * 3 + 11.0 * 3 * 2) / 10.0
    assert abs(got - want) < 1e-9
    # other widths, another mode, or other kernel sources: no figure
    assert bench.scaled_traffic(wl.get_config("qwen3_4b_is"), 3000, 10.0, "keep_logits", str(path)) is None
    assert bench.scaled_traffic(cfg, 3000, 10.0, "recompute", str(path)) is None
    rec["kernel_source_sha256"] = "0" * 64
    path.write_text(json.dumps(rec))
    assert bench.scaled_traffic(cfg, 3000, 10.0, "keep_logits", str(path)) is None
