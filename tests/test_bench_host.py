"""Host-side arithmetic of bench.py: the algorithmic byte counts behind the reported HBM
figures and roofline fractions (no GPU needed)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_glm_decode_step_bytes():
    # 9 experts x 18,915,328 B + router 256 x 6144 x 4 + bias 256 x 4 + x and y (2 x 6144 x 4)
    wl = synth.WORKLOADS["glm_decode"]
    assert bench.expert_bytes(6144, 2048) == 18_915_328
    assert bench.step_bytes(wl, 1, 8) == 9 * 18_915_328 + 6_291_456 + 1_024 + 2 * 24_576
    assert bench.step_bytes(wl, 1, 8) == 176_579_584


def test_gateup_bytes_are_two_thirds_of_an_expert_plus_their_scales():
    # gate and up: 2 x 2048 rows of 3072 bytes, 2 x 2048 float32 scales
    assert bench.gateup_bytes(6144, 2048) == 2 * 2048 * 3072 + 8 * 2048
    # int8 rows: one byte per value
    assert bench.gateup_bytes(6144, 2048, 1) == 2 * 2048 * 6144 + 8 * 2048


def test_stack_bytes_per_token():
    # 40 layers x (4 routed + 1 shared expert of 1,585,152 B + router 256 x 2048 x 4 + bias + x, y)
    wl = synth.WORKLOADS["stack35b"]
    per_layer = 5 * 1_585_152 + 256 * 2048 * 4 + 256 * 4 + 2 * 2048 * 4
    assert bench.step_bytes(wl, 1, wl.K) == per_layer
    assert wl.n_layers * per_layer == 401_612_800


def test_batched_step_counts_each_touched_expert_once():
    wl = synth.WORKLOADS["glm_batched"]
    one = bench.step_bytes(wl, 512, 1)
    two = bench.step_bytes(wl, 512, 2)
    assert two - one == bench.expert_bytes(6144, 2048)


def test_workload_description_names_the_shapes():
    d = bench.workload_desc(synth.WORKLOADS["glm_decode"])
    for part in ("T=1", "H=6144", "E=256", "top-8", "moe_inter=2048", "routed_scale=2.5"):
        assert part in d, part


def test_binding_roofline_is_the_nearer_roof():
    # T=512 on tcgen05: 0.18 of the tensor peak, 0.10 of the copy bandwidth
    assert bench.binding_roofline(0.10, 0.18) == "tensor"
    # T=2 on mma.sync: weights streamed at 0.45 of the copy bandwidth, 0.007 of the tensor peak
    assert bench.binding_roofline(0.45, 0.007) == "hbm"


def test_cpu_baseline_times_all_cores_and_one():
    import oracle
    oracle.build()
    wl = synth.WORKLOADS["tiny"]
    li = synth.layer_inputs(wl)
    xs = [synth.tokens(wl, T=1, stream=s) for s in range(4)]
    cores = oracle.threads()
    out = bench.cpu_baseline(wl, li, xs, 0.4)
    assert out["kind"] == "oracle" and out["cores"] == cores and out["value"] > 0
    assert out["single_core"]["cores"] == 1 and out["single_core"]["value"] > 0
    assert oracle.threads() == cores          # the thread count is restored


def test_recorded_traffic_is_per_workload():
    """A committed DRAM summary is used only for the workload and token count it was
    captured on, and only while the kernel source is the captured one."""
    import bench
    assert bench.recorded_traffic("fused", "group8", 1) is None
    assert bench.recorded_traffic("gate_up", "glm_batched_t16", 16) is None
    for (kind, wl, T), (name, _) in bench.TRAFFIC_FILES.items():
        v = bench.recorded_traffic(kind, wl, T)
        assert v is None or v > 0, (kind, wl, T, name)
