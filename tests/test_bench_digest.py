"""bench.py reports a kernel's DRAM traffic from profiles/traffic.json only
while the kernel's source code is the one the record was captured from: the
record holds a digest of the source with comments and whitespace removed.
These checks need no GPU."""
import json
import os

import bench

SRC = """// header comment
__global__ void k(int *p) /* inline */ {
    p[0] = 1;  // trailing
}
"""


def _digest_of(tmp_path, text, name="k.cu"):
    f = tmp_path / name
    f.write_text(text)
    return bench.source_digest(str(f))


def test_comments_and_whitespace_do_not_change_the_digest(tmp_path):
    d0 = _digest_of(tmp_path, SRC)
    edited = SRC.replace("// header comment", "// another comment\n// two lines") \
                .replace("/* inline */", "/* a\n   longer\n   block */") \
                .replace("    p[0] = 1;", "\tp[0]   =   1;")
    assert _digest_of(tmp_path, edited) == d0


def test_code_changes_change_the_digest(tmp_path):
    d0 = _digest_of(tmp_path, SRC)
    assert _digest_of(tmp_path, SRC.replace("p[0] = 1", "p[0] = 2")) != d0
    assert _digest_of(tmp_path, SRC.replace("int *p", "int *q").replace("p[0]", "q[0]")) != d0


def test_every_record_names_a_kernel_file_and_matches_a_digest_format():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    assert rec
    for name, r in rec.items():
        assert len(r["source_sha256"]) == 64 and int(r["source_sha256"], 16) >= 0, name
        assert r["dram_bytes_per_launch"] == r["dram_read_bytes"] + r["dram_write_bytes"], name
        assert r["command"].startswith("ncu ") and "--clock-control none" in r["command"], name


def test_stale_record_reads_as_none(tmp_path, monkeypatch):
    """A record whose digest differs from the source's gives no traffic."""
    csrc = tmp_path / "persistent_kv_cache_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text(SRC)
    prof = tmp_path / "profiles"
    prof.mkdir()
    good = bench.source_digest(str(csrc / "k.cu"))
    (prof / "traffic.json").write_text(json.dumps({
        "fresh": {"source_sha256": good, "dram_bytes_per_launch": 123},
        "stale": {"source_sha256": "0" * 64, "dram_bytes_per_launch": 456}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic(("k.cu", "fresh")) == 123
    assert bench.kernel_traffic(("k.cu", "stale")) is None
    assert bench.kernel_traffic(("k.cu", "absent")) is None
