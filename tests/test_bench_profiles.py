"""Host logic of bench.py's roofline traffic lookup, on CPU: a profile summary
under profiles/ gives the DRAM bytes per launch only while the hash of the
kernel source it names still matches, and every committed summary is well
formed (a known workload, an existing source file, the commands it was made
with, all of them committed files)."""
import glob
import hashlib
import os
import re

import bench
from exact_io_aware_14_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _fake_tree(tmp_path, src_bytes, recorded_sha, name="w1"):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "k.cu").write_bytes(src_bytes)
    (tmp_path / "profiles" / "x.md").write_text(
        "# title\n\nworkload: %s\nkernel_source: k.cu sha256:%s\ntraffic_bytes_per_launch: 12345\n\n"
        "| table | 1 |\n" % (name, recorded_sha))


def test_traffic_while_the_source_hash_matches(tmp_path, monkeypatch):
    src = b"__global__ void k() {}\n"
    _fake_tree(tmp_path, src, hashlib.sha256(src).hexdigest()[:16])
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("w1") == 12345
    assert bench.profiled_traffic("other") is None


def test_no_traffic_once_the_source_changed(tmp_path, monkeypatch):
    _fake_tree(tmp_path, b"changed\n", hashlib.sha256(b"original\n").hexdigest()[:16])
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("w1") is None


def test_committed_summaries_are_well_formed():
    names = {getattr(workloads, n).name for n in dir(workloads)
             if n.isupper() and hasattr(getattr(workloads, n), "name")}
    paths = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))
    assert paths, "no profile summaries"
    for path in paths:
        text = open(path).read()
        fields = dict(re.findall(r"^(workload|kernel_source|traffic_bytes_per_launch): (.+)$", text, re.M))
        assert fields.get("workload") in names, path
        src = fields["kernel_source"].split(" sha256:")[0]
        assert os.path.isfile(os.path.join(ROOT, src)), path
        assert int(fields["traffic_bytes_per_launch"]) > 0, path
        # the commands run committed files only, with the clocks left alone
        cmds = [ln.strip() for ln in text.splitlines() if ln.startswith("    ")]
        assert any(c.startswith("python bench.py") for c in cmds), path
        for c in cmds:
            if c.startswith("ncu"):
                assert "--clock-control none" in c, path
