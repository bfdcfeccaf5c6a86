"""Host-side pieces of bench.py that need no GPU: the digest that ties the
committed ncu traffic figure to the decode kernel's code, and the reading of
that figure."""
import os
import shutil

import bench


def _copy_sources(dst):
    for rel in bench.KERNEL_SOURCES:
        os.makedirs(os.path.join(dst, os.path.dirname(rel)), exist_ok=True)
        shutil.copy(os.path.join(bench.ROOT, rel), os.path.join(dst, rel))


def _digest(root, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(root))
    return bench.kernel_source_hash()


def test_digest_ignores_comments_but_not_code(tmp_path, monkeypatch):
    _copy_sources(tmp_path)
    base = _digest(tmp_path, monkeypatch)
    rel = bench.KERNEL_SOURCES[0]
    path = os.path.join(tmp_path, rel)
    text = open(path, encoding="utf-8").read()
    # comment and whitespace edits keep the digest
    open(path, "w", encoding="utf-8").write(
        "// a new line comment\n/* and a block\n   comment */\n" + text.replace("\n", "\n\n", 3))
    assert _digest(tmp_path, monkeypatch) == base
    # a change to the code itself does not
    open(path, "w", encoding="utf-8").write(text + "\nstatic const int pkv_probe_value = 1;\n")
    assert _digest(tmp_path, monkeypatch) != base


def test_committed_traffic_needs_matching_digest_and_workload(tmp_path, monkeypatch):
    _copy_sources(tmp_path)
    digest = _digest(tmp_path, monkeypatch)
    f = tmp_path / "traffic.txt"
    f.write_text(f"# header\nsource_sha256: {digest}\nworkload: wl A\n"
                 "traffic_bytes_per_launch: 12345\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.committed_traffic("wl A") == 12345
    assert bench.committed_traffic("wl B") is None          # another workload
    f.write_text("source_sha256: 0000000000000000\nworkload: wl A\n"
                 "traffic_bytes_per_launch: 12345\n")
    assert bench.committed_traffic("wl A") is None          # another kernel version
