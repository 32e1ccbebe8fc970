"""Host-side checks of bench.py: the recorded DRAM traffic of the logits
kernel belongs to the logits sources as they are (the bench reports it only
then), the default run is the headline workload on one GPU, and every
workload of the scope table can be selected."""

import bench


def test_recorded_traffic_matches_the_logits_sources():
    assert bench.TRAFFIC["source_sha1"] == bench.kernel_sha1(), \
        "logits sources changed: re-capture the traffic (application replay) and update TRAFFIC"
    # about the key bytes of one launch: the keys are read once
    k_bytes = 6 * 2 * 32768 * 256 * 2
    assert 1.0 <= bench.TRAFFIC["bytes_per_launch"]["draft2b"] / k_bytes < 1.02


def test_default_run_is_one_gpu_with_a_long_timed_region():
    args = bench.parse([])
    assert args.gpus == 1 and args.warmup >= 3 and args.steps >= 200
    assert args.workload == "draft2b" and args.impl == "ours"


def test_every_workload_is_selectable():
    from synth import WORKLOADS
    for name in WORKLOADS:
        assert bench.parse(["--workload", name]).workload == name


def test_workload_description_names_the_shape():
    from synth import get_workload
    text = bench.describe(get_workload("serving"), 169000)
    assert "16 prompts" in text and "head_dim 256" in text and "mass 0.85" in text
    text = bench.describe(get_workload("draft2b"), 32768)
    assert "N=32768" in text and "fixed p=0.15" in text and "boost" in text
