"""Host-side logic of bench.py (CPU only)."""
import bench
from io_aware_exact_10_gb300 import workloads as W


def test_strip_comments():
    src = "int a; // one\n/* two\nlines */ int b;\n\n  // only a comment\nint c;   \n"
    assert bench.strip_comments(src) == "int a;\n int b;\nint c;"


def test_traffic_follows_the_backward_sources(monkeypatch):
    """The captured traffic is reported while the hash of the backward's
    sources matches the capture, and dropped (null) once it does not."""
    monkeypatch.setattr(bench, "NCU_TRAFFIC_SOURCES_SHA256", bench.kernel_sources_sha256())
    assert bench.ncu_traffic() == bench.NCU_TRAFFIC_BYTES
    monkeypatch.setattr(bench, "NCU_TRAFFIC_SOURCES_SHA256", "0" * 64)
    assert bench.ncu_traffic() is None


def test_config_names_the_shape():
    c = bench.config_of(W.PREFILL_CHUNK)
    assert (c["N"], c["N_k"], c["H"], c["H_kv"]) == (1024, 8192, 32, 8)
    c = bench.config_of(W.SPARSE_LOCAL_GLOBAL)
    assert c["block_pattern"] == "local3_global1_random0.05" and 0.10 < c["blocks_kept"] < 0.13
    c = bench.config_of(W.GPT2_MEDIUM)
    assert "N_k" not in c and "H_kv" not in c and "block_pattern" not in c
