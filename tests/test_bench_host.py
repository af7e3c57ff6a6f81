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
