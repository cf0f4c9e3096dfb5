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


def test_committed_traffic_is_void_when_launch_count_differs():
    with open(os.path.join(bench.ROOT, "profiles", "dram_traffic_qwen3_8b_ppo.json")) as fh:
        rec = json.load(fh)
    n = rec["kernels"]["tc_gemm_pair_kernel"]["launches_per_step"]
    assert bench.committed_traffic("qwen3_8b_ppo", "tc_gemm_pair_kernel", n + 1) is None
    assert bench.committed_traffic("no_such_workload", "tc_gemm_pair_kernel", n) is None
