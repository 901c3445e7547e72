"""The traffic record that bench.py attaches to its roofline line applies to
the kernel sources it was captured on: the source hash ignores comments and
spacing (an edit of the comments is no kernel change) but not code, and the
record is only returned while the hash matches."""
import json

import bench


def test_code_only_drops_comments_and_spacing_but_keeps_strings():
    a = 'int a = 1; // note\n/* block\n comment */ const char *s = "x // kept";\n'
    b = 'int a = 1;   // another note\nconst char *s = "x // kept";'
    assert bench._code_only(a) == bench._code_only(b) == 'int a = 1; const char *s = "x // kept";'
    assert bench._code_only("int a = 2;") != bench._code_only("int a = 1;")
    # an escaped quote does not end a string literal
    assert bench._code_only('const char *q = "a \\" // b"; // c') == 'const char *q = "a \\" // b";'


def test_traffic_record_is_returned_only_for_matching_sources(tmp_path, monkeypatch):
    rec = {"source_hash": bench.kernel_source_hash(),
           "dram_bytes_per_launch": {"some_kernel": 123}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic_wl.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: rec["source_hash"])
    assert bench.profiled_traffic("wl") == {"some_kernel": 123}
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.profiled_traffic("wl") == {}
    assert bench.profiled_traffic("missing") == {}
