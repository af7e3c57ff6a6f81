"""Host logic of the benchmark that needs no GPU: the key that ties the stored DRAM-traffic record to the kernel
sources (comments and layout ignored, any code change noticed)."""
import bench


def test_strip_comments():
    src = "int a; // one\n/* two\n   lines */ int b;   /* three */int c;\n"
    assert bench.strip_comments(src) == "int a; int b; int c;"


def test_source_hash_ignores_comments_not_code(monkeypatch):
    base = bench.source_hash()
    real_open = open

    def fake_open(path, *a, **k):
        f = real_open(path, *a, **k)
        if str(path).endswith("q8_device.cuh"):
            text = f.read()
            f.close()
            import io
            return io.StringIO(edit(text))
        return f

    edit = lambda t: t.replace("namespace q8 {", "// a new comment\nnamespace q8 {  /* and another */", 1)
    monkeypatch.setattr("builtins.open", fake_open)
    assert bench.source_hash() == base
    edit = lambda t: t.replace("namespace q8 {", "namespace q8 { constexpr int kUnused = 1;", 1)
    assert bench.source_hash() != base


def test_traffic_record_matches_the_committed_kernels():
    """profiles/traffic.json was captured from the stream kernels as they stand (its key is their sources' hash), so
    the bench line carries its DRAM traffic; and that traffic is the algorithmic bytes to within 2% (no weight byte is
    read twice)."""
    import json
    with open(bench.PROFILE_TRAFFIC) as f:
        rec = json.load(f)
    assert rec["source_hash"] == bench.source_hash(), "kernel sources changed since the traffic capture"
    for m in ("1", "16"):
        got = bench.traffic_record(int(m), True)
        assert got is not None
        alg = rec["by_m"][m]["algorithmic_bytes_per_call"]
        assert abs(got - alg) <= 0.02 * alg, (m, got, alg)
    assert bench.traffic_record(1, False) is None  # a variant chain is not the captured step
