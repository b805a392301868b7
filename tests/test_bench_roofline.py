"""Host logic of the benchmark's roofline object (no GPU)."""
import bench
from exact_attention_17_gb300 import inputs

PEAKS = {"hbm_gbs": 6689.5, "bf16_tflops": 1955.1, "bf16_tflops_sustained": 1727.8}


def entry(name, ms):
    w = inputs.workload(name)
    b = bench.algorithmic_bytes(w)
    balance = PEAKS["bf16_tflops"] * 1e12 / (PEAKS["hbm_gbs"] * 1e9)
    tf = w.flops / (ms * 1e-3) / 1e12
    return bench.roofline_entry(w.flops / b < balance, tf, PEAKS["bf16_tflops"], "measured",
                                PEAKS, None, w.flops, b, ms), w, b


def test_long_causal_sequence_is_tensor_bound():
    r, w, _ = entry("b1_h32_n16384_d128_causal", 1.7)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - w.flops / 1.7e-3 / 1e12) < 0.01
    assert abs(r["frac"] - r["achieved"] / PEAKS["bf16_tflops"]) < 1e-4


def test_short_query_long_key_is_hbm_bound():
    # Nq = 128 against Nk = 8192: about 128 FLOPs per byte, below the ~292 balance
    r, w, b = entry("b16_h32_nq128_nk8192_d128", 0.347)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - b / 0.347e-3 / 1e9) < 0.1
    assert 0.9 < r["frac"] < 1.0
    assert r["tensor_frac"] < 0.5


def test_algorithmic_bytes_count_each_tensor_once():
    w = inputs.workload("b2_h8_n1000_d64")
    q = kv = 2 * 8 * 1000 * 64 * 2
    o32, lse = 2 * 8 * 1000 * 64 * 4, 2 * 8 * 1000 * 4
    assert bench.algorithmic_bytes(w) == q + 2 * kv + o32 + lse
    assert bench.algorithmic_bytes(w, 2) == q + 2 * kv + o32 // 2 + lse


def test_traffic_records_follow_the_kernel_source():
    """A recorded DRAM figure is reported only for the translation unit it was
    taken on and only while the kernel sources hash to the recorded value."""
    import json
    import os

    sources = bench.fwd_kernel_sources(128)
    assert sources[-1].endswith("fa2_tc_d128_bf16.cu")
    assert bench.fwd_kernel_sources(256, fp16=True)[-1].endswith("fa2_tc_d256_f16.cu")
    with open(os.path.join(bench.ROOT, "profiles", "dram_traffic.json")) as f:
        rec = json.load(f)
    for name, entry in rec.items():
        if name.endswith(":backward"):
            srcs = bench.BWD_KERNEL_SOURCES
        else:
            srcs = bench.fwd_kernel_sources(inputs.workload(name).d)
        if entry["kernel_source_hash"] == bench.kernel_source_hash(srcs):
            assert bench.recorded_traffic(name, srcs) == entry["dram_bytes_per_launch"]
        # another translation unit (fp16) never picks up a bf16 record
        if not name.endswith(":backward"):
            assert bench.recorded_traffic(name, bench.fwd_kernel_sources(inputs.workload(name).d, True)) is None
    assert bench.recorded_traffic("no_such_workload", sources) is None
