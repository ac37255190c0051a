"""CPU checks of the benchmark's roofline arithmetic and of its ncu traffic record.

The algorithmic work per launch is fixed by the layer's definition: the gate/up GEMM does 4*P*d*I
FLOP (two projections of every (token, expert) row), and at decode it must at least stream the
gate and up weights of every touched expert (2*I*d bf16 values each) plus its row input (P*d) and
h output (P*I).  The traffic recorder sums a stage's kernels (the CTA-pair launch and the
small-expert launch) and divides by the stage's launches.
"""
import json

import numpy as np

import bench
from synth import WORKLOADS

PK = {"hbm_gbs": 6479.9, "bf16_tflops": 1793.3, "bf16_tflops_sustained": 1362.7}


def test_prefill_roofline_is_flops_over_the_launch_time():
    w = WORKLOADS["prefill_t8192"]
    counts = np.full(w.N, w.P // w.N, dtype=np.int32)
    rl = bench.gate_up_roofline(w, counts, 2.5, PK, "measured")
    flop = 4.0 * 131072 * 4096 * 1408
    assert rl["bound"] == "tensor" and rl["algorithmic_per_launch"]["flop"] == flop
    assert abs(rl["achieved"] - flop / 2.5e-3 / 1e12) < 0.01
    assert rl["peak"] == 1793.3 and rl["frac"] == round(rl["achieved"] / 1793.3, 4)   # burst is the denominator
    assert rl["frac_sustained"] == round(rl["achieved"] / 1362.7, 4)
    assert rl["launch_ms"] == 2.5


def test_decode_roofline_counts_only_touched_experts():
    w = WORKLOADS["decode_t32"]
    counts = np.zeros(w.N, dtype=np.int32)
    counts[:51] = 1                          # 51 of 64 experts touched
    rl = bench.gate_up_roofline(w, counts, 0.2, PK, "measured")
    per_expert = 2 * 1408 * 4096 * 2         # W_gate + W_up rows of one expert, bf16
    want = 51 * per_expert + 512 * 4096 * 2 + 512 * 1408 * 2
    assert per_expert == 23068672 and want == 1182138368
    assert rl["bound"] == "hbm" and rl["algorithmic_per_launch"]["bytes"] == want
    assert rl["algorithmic_per_launch"]["touched_experts"] == 51
    assert abs(rl["achieved"] - want / 0.2e-3 / 1e9) < 0.1


def test_layer_roofline_and_job_throughput():
    w = WORKLOADS["decode_t32"]
    counts = np.zeros(w.N, dtype=np.int32)
    counts[:51] = 1
    lr = bench.layer_roofline(w, counts, 0.3, PK)
    assert lr["touched_experts"] == 51
    wbytes = 51 * 3 * 1408 * 4096 * 2
    assert abs(lr["weight_gbs"] - wbytes / 0.3e-3 / 1e9) < 0.1
    # decode: the HBM time of the touched weights is the roofline
    assert lr["roofline_ms"] == round(wbytes / 6479.9e9 * 1e3, 4)
    assert bench.job_tokens_per_s(8192, 4, 4.0) == 8192 * 4 / 4e-3


def test_stress_layer_roofline_takes_the_larger_of_tensor_and_hbm_time():
    """The stress layer (T=4096, d=7680, N=256, K=8, I=2048): 6*P*d*I + 2*T*d*N FLOP = 3.108 TFLOP
    and the weights of the touched experts (3*d*I bf16 values each); the roofline time is the
    larger of the two times at the measured peaks."""
    w = WORKLOADS["stress_n256"]
    counts = np.zeros(w.N, dtype=np.int32)
    counts[:89] = 1
    lr = bench.layer_roofline(w, counts, 3.0, PK)
    flop = 6.0 * 32768 * 7680 * 2048 + 2.0 * 4096 * 7680 * 256
    wbytes = 89 * 3 * 7680 * 2048 * 2
    assert lr["flop"] == flop and lr["weight_bytes"] == wbytes and wbytes == 8_399_093_760
    t_roof = max(flop / 1793.3e12, wbytes / 6479.9e9)
    assert lr["roofline_ms"] == round(t_roof * 1e3, 4) and lr["roofline_frac"] == round(t_roof / 3e-3, 4)
    assert lr["tc_frac"] == round(flop / 3e-3 / 1e12 / 1793.3, 4)


def test_both_arms_report_the_same_config():
    w = WORKLOADS["prefill_t8192"]
    c = bench.workload_config(w, 1)
    assert c["workload"] == "prefill_t8192" and (c["T"], c["K"], c["I"]) == (8192, 16, 1408)
    assert c == bench.workload_config(WORKLOADS["prefill_t8192"], 1)


def test_traffic_record_sums_the_stage_kernels(tmp_path, monkeypatch):
    hdr = ["ID", "Kernel Name", "Metric Name", "Metric Unit", "Metric Value", "a", "b", "c", "d", "e", "f"]
    rows = [hdr]

    def add(i, name, rd, wr):
        rows.append([str(i), name, "dram__bytes_read.sum", "byte", f"{rd:,}", *"......"])
        rows.append([str(i), name, "dram__bytes_write.sum", "byte", f"{wr:,}", *"......"])
        rows.append([str(i), name, "gpu__time_duration.sum", "ns", "1", *"......"])

    pair, small = "void tc::ffn_tc_pair_kernel<1, 2>(CUtensorMap_st, ...)", "void tc::ffn_tc_kernel<2, 32, 0>(...)"
    pair_dn, small_dn = "void tc::ffn_tc_pair_kernel<0, 1>(CUtensorMap_st, ...)", "void tc::ffn_tc_kernel<3, 32, 0>(...)"
    for k in range(3):                       # three prefill layers: gate/up and down stages
        add(10 * k, pair, 3_000_000_000, 300_000_000)
        add(10 * k + 1, small, 800_000_000, 100_000_000)
        add(10 * k + 2, pair_dn, 1_500_000_000, 500_000_000)
        add(10 * k + 3, small_dn, 200_000_000, 10_000_000)
    add(99, "void tc::ffn_tc_kernel<2, 32, 1>(...)", 1_100_000_000, 80_000_000)
    add(100, "void tc::ffn_tc_kernel<3, 32, 0>(...)", 550_000_000, 40_000_000)   # decode down: same name
    csv_path = tmp_path / "launches.csv"
    csv_path.write_text("\n".join(",".join(f'"{c}"' for c in r) for r in rows) + "\n")
    out = tmp_path / "ncu_traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_PATH", str(out))
    bench.record_traffic(str(csv_path), "ncu ...")
    rec = json.loads(out.read_text())
    assert rec["prefill_t8192:gate_up"]["launches"] == 3
    assert rec["prefill_t8192:gate_up"]["dram_bytes_per_launch"] == 4_200_000_000
    assert rec["prefill_t8192:down"]["dram_bytes_per_launch"] == 2_210_000_000
    assert rec["decode_t32:gate_up"]["dram_bytes_per_launch"] == 1_180_000_000
    assert rec["decode_t32:down"]["launches"] == 1 and rec["decode_t32:down"]["dram_bytes_per_launch"] == 590_000_000
    assert rec["prefill_t8192:gate_up"]["kernel_sha256_16"] == bench.kernel_hash()
