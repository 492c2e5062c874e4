"""Host-side pieces of bench.py that need no GPU: the DRAM-traffic lookup that
the roofline reports only while the kernel sources still match the capture,
and the CUDA runtime binding of the end-to-end loop."""
import hashlib
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _fake_tree(tmp_path, sources, body):
    for rel, text in sources.items():
        p = tmp_path / rel
        p.parent.mkdir(parents=True, exist_ok=True)
        p.write_text(text)
    (tmp_path / "profiles").mkdir(exist_ok=True)
    (tmp_path / "profiles" / "traffic.txt").write_text(body)


def _digest(tmp_path, rels):
    h = hashlib.sha256()
    for rel in rels:
        h.update((tmp_path / rel).read_bytes())
    return h.hexdigest()[:16]


def test_traffic_reported_only_for_the_captured_sources(tmp_path, monkeypatch):
    rels = ["k/a.cu", "k/b.cuh"]
    _fake_tree(tmp_path, {"k/a.cu": "kernel a\n", "k/b.cuh": "header b\n"}, "")
    d = _digest(tmp_path, rels)
    (tmp_path / "profiles" / "traffic.txt").write_text(
        "# comment line\n"
        f"wl stream {d} 12345 profiles/x.md\n"
        f"wl tc {d} 999 profiles/x.md\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "STAGE_SOURCES", {"stream": rels, "tc": ["k/a.cu"]})
    assert bench.measured_traffic("wl", "stream") == 12345
    assert bench.measured_traffic("other", "stream") is None     # no line for the workload
    assert bench.measured_traffic("wl", "tc") is None            # hash taken over other files
    assert bench.measured_traffic("wl", "nostage") is None
    (tmp_path / "k" / "b.cuh").write_text("header b, edited\n")  # any change to a source
    assert bench.measured_traffic("wl", "stream") is None


def test_traffic_file_lines_are_well_formed():
    """Every recorded line names a stage bench.py knows, a 16-hex-digit source
    hash, a positive byte count and an existing summary under profiles/."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    with open(path) as f:
        lines = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert lines
    for parts in lines:
        wl, stage, digest, nbytes, src = parts[:5]
        assert stage in bench.STAGE_SOURCES
        assert len(digest) == 16 and int(digest, 16) >= 0
        assert int(nbytes) > 0
        assert os.path.exists(os.path.join(ROOT, src))


def test_cuda_runtime_binding_exposes_the_loop_calls():
    try:
        rt = bench.Cudart()
    except OSError:
        pytest.skip("no CUDA runtime library on this host")
    for name in ("cudaMemcpyAsync", "cudaEventCreateWithFlags", "cudaEventRecord", "cudaStreamWaitEvent",
                 "cudaEventDestroy"):
        assert hasattr(rt.lib, name)
    assert (bench.Cudart.H2D, bench.Cudart.D2H) == (1, 2)   # cudaMemcpyHostToDevice / DeviceToHost
    with pytest.raises(RuntimeError):
        rt.check(1, "cudaEventRecord")
