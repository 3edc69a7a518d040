"""Host-side logic of bench.py (CPU only)."""
import bench
from io_aware_exact_10_gb300 import workloads as W


def test_strip_comments():
    src = "int a; // one\n/* two\nlines */ int b;\n\n  // only a comment\nint c;   \n"
    assert bench.strip_comments(src) == "int a;\n int b;\nint c;"


def test_traffic_follows_the_backward_sources(monkeypatch):
    """The captured traffic is reported for the workload it was captured on,
    scaled from the capture's batch to the workload's, while the hash of the
    backward's sources matches the capture, and dropped (null) once it does
    not."""
    sha = bench.kernel_sources_sha256()
    table = {W.LONG_CAUSAL.name: {"bytes": 1000.0, "capture_B": 1, "sources_sha256": sha}}
    monkeypatch.setattr(bench, "NCU_TRAFFIC", table)
    assert bench.ncu_traffic(W.LONG_CAUSAL) == 1000.0 * W.LONG_CAUSAL.B
    # the capture belongs to one workload: other lines report no traffic
    assert bench.ncu_traffic(W.GQA_CAUSAL) is None
    assert bench.ncu_traffic(W.SPARSE_LOCAL_GLOBAL) is None
    table[W.LONG_CAUSAL.name]["sources_sha256"] = "0" * 64
    assert bench.ncu_traffic(W.LONG_CAUSAL) is None


def test_default_line_is_the_long_causal_d128_workload():
    """The default bench line runs B=4, H=32, N=8192, d=128, causal, where
    the forward and backward bars are stated, and reports them."""
    w = W.WORKLOADS[bench.DEFAULT_WORKLOAD]
    assert (w.B, w.H, w.N, w.d, w.causal) == (4, 32, 8192, 128, True)
    b = bench.bars_of(w, 1200.0, 700.0, 2000.0)
    assert b["fwd_met"] and not b["bwd_met"] and abs(b["bwd_pct"] - 35.0) < 1e-9
    assert bench.bars_of(W.GPT2_MEDIUM, 1.0, 1.0, 2.0) is None
    # the oracle samples stay bounded: a few heads of the long workload
    assert 1 <= bench.oracle_heads(w, 1.0e11, 8) <= 2
    assert bench.oracle_heads(W.GPT2_MEDIUM, 4.0e11, 128) == 128


def test_config_names_the_shape():
    c = bench.config_of(W.PREFILL_CHUNK)
    assert (c["N"], c["N_k"], c["H"], c["H_kv"]) == (1024, 8192, 32, 8)
    c = bench.config_of(W.SPARSE_LOCAL_GLOBAL)
    assert c["block_pattern"] == "local3_global1_random0.05" and 0.10 < c["blocks_kept"] < 0.13
    c = bench.config_of(W.GPT2_MEDIUM)
    assert "N_k" not in c and "H_kv" not in c and "block_pattern" not in c


def test_sweep_byte_model_counts_visited_tiles():
    """The sweep's tiled byte model equals a brute-force count of the tiles
    the kernels visit (causal: key j visible to query i iff j <= i), and never
    falls below the algorithmic minimum; one pair of query tiles against two
    key tiles streams each input exactly once."""
    import bench
    for N, d, causal in ((256, 64, True), (512, 64, False), (1000, 128, True), (4096, 128, True),
                         (384, 64, True)):
        nt = -(-N // 128)
        tile = 128 * d * 2
        fwd_tiles = 0
        for p in range(-(-nt // 2)):
            last_row = min(N, (2 * p + 2) * 128) - 1
            fwd_tiles += sum(1 for j in range(nt) if not causal or j * 128 <= last_row)
        bwd_visits = sum(1 for kt in range(nt) for qt in range(nt)
                         if not causal or kt * 128 <= min(N, qt * 128 + 128) - 1)
        b = bench.sweep_bytes(N, d, 3, causal)
        assert b["fwd_model"] == 3 * (4 * N * d + 4 * N + fwd_tiles * 2 * tile)
        assert b["bwd_kernel_model"] == 3 * (nt * 4 * tile + bwd_visits * (2 * tile + 1024 + 1024 * d))
        assert b["fwd_model"] >= b["fwd_min"] - 3 * (4 * (nt * 128 - N) * d) * 2
        assert b["bwd_kernel_model"] >= b["bwd_kernel_min"]
    b = bench.sweep_bytes(256, 64, 1, True)
    assert b["fwd_model"] == b["fwd_min"]


def test_tile_sweep_layout_is_the_same_attention():
    """The tile sweep's Br = 128 layout views every 128-row query tile as its
    own query head (N_q = 128) of the original key/value head, through the
    grouped-head and cross-length rules (query head h' uses key/value head
    h' // G).  Non-causal, that is the same attention: the oracle on both
    layouts agrees to rounding."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(3)
    B, H, N, d = 1, 2, 384, 16
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    o, lse = oracle.attn_fwd(q, k, v, 0.25, False)
    nt = N // 128
    o2, lse2 = oracle.attn_fwd(q.reshape(B, H * nt, 128, d), k, v, 0.25, False)
    assert np.allclose(o2.reshape(o.shape), o, rtol=0, atol=1e-12)
    assert np.allclose(lse2.reshape(lse.shape), lse, rtol=0, atol=1e-12)
