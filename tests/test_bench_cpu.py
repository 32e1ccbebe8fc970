"""Host-side checks of bench.py: the recorded DRAM traffic of the logits
kernel belongs to the logits sources as they are (the bench reports it only
then), and the reference arm is the oracle on a bounded sample."""

import bench


def test_recorded_traffic_matches_the_logits_sources():
    assert bench.TRAFFIC["source_sha1"] == bench.kernel_sha1(), \
        "logits sources changed: re-capture the traffic (application replay) and update TRAFFIC"
    # about the key bytes of one launch: the keys are read once
    k_bytes = 6 * 2 * 32768 * 256 * 2
    assert 1.0 <= bench.TRAFFIC["bytes_per_launch"] / k_bytes < 1.02


def test_default_run_is_one_gpu_with_a_long_timed_region():
    import sys
    argv = sys.argv
    sys.argv = ["bench.py"]
    try:
        args = bench.parse()
    finally:
        sys.argv = argv
    assert args.gpus == 1 and args.warmup >= 3 and args.steps >= 200
