"""bench.py reports a kernel's DRAM traffic only while the kernel's source
still hashes to the one the committed ncu capture was taken on; after any
change to the source the figure is null.  A record taken on a smaller batch
gives bytes per row, scaled to the benchmark's active rows."""
import hashlib

import bench


def test_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cuh"
    src.write_bytes(b"__global__ void k() {}\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    rec = tmp_path / "traffic.txt"
    rec.write_text("# kernel=k source_sha=%s bytes_per_launch=1 (a comment is not a record)\n"
                   "kernel=other source_sha=%s bytes_per_launch=7\n"
                   "kernel=k source_sha=%s bytes_per_launch=123456 launches=2\n" % (sha, sha, sha))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(rec))
    assert bench.ncu_traffic("k", str(src)) == 123456.0
    assert bench.ncu_traffic("missing", str(src)) is None
    src.write_bytes(b"__global__ void k() { /* changed */ }\n")
    assert bench.ncu_traffic("k", str(src)) is None
    src.write_bytes(b"__global__ void k() {}\n")
    rec.write_text("kernel=k source_sha=%s rows=4096 bytes_per_row=300.5 launches=2\n" % sha)
    assert bench.ncu_traffic("k", str(src), active_rows=16384) == 300.5 * 16384
    assert bench.ncu_traffic("k", str(src)) is None  # a per-row record needs the row count
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "absent.txt"))
    assert bench.ncu_traffic("k", str(src)) is None


def test_committed_records_are_well_formed():
    for line in open(bench.TRAFFIC_FILE).read().splitlines():
        if not line.strip() or line.lstrip().startswith("#"):
            continue
        f = dict(kv.split("=", 1) for kv in line.split())
        assert set(f) >= {"kernel", "source_sha"}, line
        assert len(f["source_sha"]) == 16
        if "bytes_per_row" in f:
            assert int(f["rows"]) > 0 and float(f["bytes_per_row"]) > 0, line
        else:
            assert float(f["bytes_per_launch"]) > 0, line
