"""Host logic of bench.py (no GPU): the kernel labels of the default bench line
name the DRAM-traffic records in profiles/traffic.json (so every GEMM roofline
of the line can carry its measured traffic), and each record is close to the
algorithmic bytes of the launch it names."""
import json
import os

import bench


def _names():
    return [bench.DEFAULT_HEADLINE] + bench.DEFAULT_EXTRA.split(",")


def _records():
    with open(os.path.join(bench.HERE, "profiles", "traffic.json")) as f:
        return json.load(f)


def _launches():
    for name in _names():
        wl = bench.host_workload(name)
        alg = bench.algorithmic_counts(wl)
        yield name, "gemm1", bench.gemm1_variant(wl), alg["g1_bytes"]
        yield name, "gemm2", bench.gemm2_variant(wl), alg["g2_bytes"]


def test_every_default_gemm_names_a_traffic_record():
    rec = _records()
    missing = [f"{label}@{bench.traffic_name(name)}:{which}" for name, which, label, _ in _launches()
               if f"{label}@{bench.traffic_name(name)}:{which}" not in rec]
    assert not missing, f"no traffic record for {missing}"


def test_traffic_records_are_close_to_the_algorithmic_bytes():
    # measured DRAM bytes within [0.8, 1.2] of the algorithmic count: nothing
    # re-read in bulk, and each label points at the right launch
    rec = _records()
    for name, which, label, ab in _launches():
        r = rec[f"{label}@{bench.traffic_name(name)}:{which}"]
        ratio = (r["dram_read_bytes"] + r["dram_write_bytes"]) / ab
        assert 0.8 <= ratio <= 1.2, (name, which, ratio)
        assert r["src"] == bench.kernel_source(label)
