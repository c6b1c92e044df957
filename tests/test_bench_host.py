"""Host-side rules of bench.py (CPU): the committed DRAM counters are attached
to a roofline only while the kernel sources still hash to the ones they were
captured on."""
import hashlib
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _summary(path, sha, traffic):
    path.write_text("# capture\n\n"
                    f"source_sha256_16: {sha}\n"
                    f"traffic_bytes_per_launch_full: {traffic}\n")


def _sha(*paths):
    h = hashlib.sha256()
    for p in paths:
        h.update(p.read_bytes())
    return h.hexdigest()[:16]


@pytest.fixture
def capture(tmp_path, monkeypatch):
    src_a, src_b = tmp_path / "a.cu", tmp_path / "b.cuh"
    src_a.write_text("kernel a\n")
    src_b.write_text("kernel b\n")
    summary = tmp_path / "summary.md"
    monkeypatch.setattr(bench, "PROFILES", {False: (str(summary), [str(src_a), str(src_b)]),
                                            True: (str(summary), [str(src_a)])})
    return summary, src_a, src_b


def test_counters_attached_while_sources_match(capture):
    summary, a, b = capture
    _summary(summary, _sha(a, b), 123456789)
    traffic, sha = bench.committed_traffic(False)
    assert traffic == 123456789.0 and sha == _sha(a, b)


def test_counters_dropped_once_a_source_changes(capture):
    summary, a, b = capture
    _summary(summary, _sha(a, b), 123456789)
    b.write_text("kernel b, changed\n")
    traffic, sha = bench.committed_traffic(False)
    assert traffic is None and sha == _sha(a, b)


def test_hash_covers_every_listed_source_in_order(capture):
    summary, a, b = capture
    _summary(summary, _sha(b, a), 1)  # right files, wrong order
    assert bench.committed_traffic(False)[0] is None
    _summary(summary, _sha(a), 7)     # the fp8 entry lists one source
    assert bench.committed_traffic(True)[0] == 7.0
    assert bench.committed_traffic(False)[0] is None


def test_missing_or_malformed_summary(capture):
    summary, a, b = capture
    assert bench.committed_traffic(False)[0] is None  # no summary file
    summary.write_text(f"source_sha256_16: {_sha(a, b)}\n")  # no traffic line
    assert bench.committed_traffic(False)[0] is None
    summary.write_text(f"source_sha256_16: {_sha(a, b)}\ntraffic_bytes_per_launch_full: n/a\n")
    assert bench.committed_traffic(False)[0] is None


def test_committed_profiles_name_existing_sources():
    for fp8 in (False, True):
        summary, sources = bench.PROFILES[fp8]
        assert os.path.isfile(summary), summary
        for rel in sources:
            assert os.path.isfile(os.path.join(bench.ROOT, rel)), rel


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the reference arm (the oracle on the host cores) runs on
    rank 0 alone; every other rank exits 0 at once and prints nothing."""
    import subprocess
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1",
               MASTER_ADDR="127.0.0.1", MASTER_PORT="29999")
    r = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--impl",
                        "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_config_records_how_the_plan_is_built(monkeypatch):
    """The line's config says whether layers 2.. of a step reuse the first
    layer's split plan (the default) or plan in every call (--no-plan-reuse)."""
    from invariant_paged_kv_gb300 import workload as wl
    step = wl.decode_batch(0, lanes=4)
    for argv, reused in ((["bench.py"], True), (["bench.py", "--no-plan-reuse"], False)):
        monkeypatch.setattr(sys, "argv", argv)
        args = bench.parse()
        cfg = bench.workload_config(step, 4, "decode_batch", args)
        assert ("reused" in cfg["plan"]) == reused, cfg["plan"]
        assert args.no_secondary is False
