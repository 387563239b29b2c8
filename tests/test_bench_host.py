"""Host-side pieces of bench.py that need no GPU: the DRAM traffic record applies only to the
kernel sources and the configuration it was captured on."""

import importlib.util
import json
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def test_traffic_record_matches_sources_and_configuration():
    b = _bench()
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    cfg = dict(rec["config"])
    got = b.traffic_record(cfg)
    if rec["source_sha256"] != b.kernel_source_hash():
        assert got is None  # taken with other kernel sources: never reported
        return
    assert got is not None and got["per_launch_bytes"] == rec["per_launch_bytes"]
    for k, other in (("workload", "tiny_fp32"), ("n_labelled", cfg["n_labelled"] // 2),
                     ("chunk_rows", cfg["chunk_rows"] // 2), ("dtype", "f16")):
        assert b.traffic_record(dict(cfg, **{k: other})) is None, k


def test_every_workload_has_a_title():
    from linear_cross_entropy_logits_gb300 import inputs as I
    b = _bench()
    assert set(b.WORKLOAD_TITLES) == set(I.WORKLOADS)
