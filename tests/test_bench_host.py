"""Host-side logic of bench.py that needs no GPU: the committed traffic
record and its source-hash guard, the kernel instance each workload's line
names, the roofline denominator and its fallback, and the sizes the line's
throughput is computed from."""
import json

import pytest

import bench
import workloads


def test_traffic_record_covers_the_timed_workloads_on_this_source():
    est = bench.recorded_traffic("estimator_B256_K8_V128256_bf16")
    fly = bench.recorded_traffic("fly_B128_K15_V152064_bf16")
    if est is None and fly is None:
        # the bench then reports traffic as null, as it should
        pytest.skip("the traffic record predates the current kernel sources")
    assert est is not None and fly is not None
    # every logit byte is read at least once; the excess stays small
    for name, t in (("estimator_B256_K8_V128256_bf16", est), ("fly_B128_K15_V152064_bf16", fly)):
        w = workloads.WORKLOADS[name]
        alg = w.logit_bytes(w.mode == "stochastic" or w.with_confidence)
        assert alg <= t < 1.2 * alg, name
    assert bench.recorded_traffic("no_such_workload") is None


def test_traffic_record_is_ignored_once_the_source_changes(tmp_path, monkeypatch):
    f = tmp_path / "traffic.txt"
    f.write_text("# a comment with = in it\nsource_sha256=0000000000000000\n"
                 "dram_bytes_per_launch.estimator_B256_K8_V128256_bf16=123\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic("estimator_B256_K8_V128256_bf16") is None
    f.write_text(f"source_sha256={bench.source_hash()}\n"
                 "dram_bytes_per_launch.estimator_B256_K8_V128256_bf16=123\n")
    assert bench.recorded_traffic("estimator_B256_K8_V128256_bf16") == 123.0
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.txt"))
    assert bench.recorded_traffic("estimator_B256_K8_V128256_bf16") is None


def test_kernel_instance_names():
    W = workloads.WORKLOADS
    assert bench.verify_kernel_name(W["estimator_B256_K8_V128256_bf16"]) == "verify_kernel<__nv_bfloat16, 0, 0>"
    assert bench.verify_kernel_name(W["fly_B128_K15_V152064_bf16"]) == "verify_kernel<__nv_bfloat16, 0, 1>"
    assert bench.verify_kernel_name(W["tiny_B4_K4_V1024_f32"]) == "verify_kernel<float, 0, 0>"


def test_measured_peak_and_fallback(tmp_path, monkeypatch):
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6500.5}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peak, src = bench.measured_hbm_peak()
    assert peak == 6500.5 and src.startswith("measured")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path / "nowhere"))
    peak, src = bench.measured_hbm_peak()
    assert peak == 6800.0 and src.startswith("fallback")


@pytest.mark.parametrize("name", sorted(workloads.WORKLOADS))
def test_algorithmic_bytes(name):
    """B(2K+1)V·s with the draft rows, B(K+1)V·s without them."""
    w = workloads.WORKLOADS[name]
    s = 2 if w.dtype == "bf16" else 4
    assert w.logit_bytes(True) == w.B * (2 * w.K + 1) * w.V * s
    assert w.logit_bytes(False) == w.B * (w.K + 1) * w.V * s
