"""Host-side logic of bench.py that needs no GPU: the comment-insensitive
code hash that links a profile summary to the kernel source it was taken
on, and the lookup of a profiled DRAM traffic figure."""
import bench


def _hash_of(tmp_path, text):
    p = tmp_path / "k.cu"
    p.write_text(text)
    return bench.code_hash(str(p))


BASE = """// header comment
__global__ void k(float* x) {  /* block comment */
    x[0] = 1.0f;  // trailing comment
    const char* s = "a // not a comment";
}
"""


def test_code_hash_ignores_comments_and_whitespace(tmp_path):
    h = _hash_of(tmp_path, BASE)
    assert len(h) == 16
    edited = BASE.replace("// header comment", "// a different header\n// over two lines")
    edited = edited.replace("/* block comment */", "/* another\n   block */")
    edited = edited.replace("x[0] = 1.0f;", "x[0]  =  1.0f ;")
    assert _hash_of(tmp_path, edited) == h


def test_code_hash_sees_code_changes(tmp_path):
    h = _hash_of(tmp_path, BASE)
    assert _hash_of(tmp_path, BASE.replace("1.0f", "2.0f")) != h
    # text inside a string literal is code, even when it looks like a comment
    assert _hash_of(tmp_path, BASE.replace("not a comment", "still code")) != h


def test_profiled_traffic_follows_the_recorded_hash(tmp_path, monkeypatch):
    csrc = tmp_path / "fp8_fine_grained_25_b300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "k.cu").write_text(BASE)
    h = bench.code_hash(str(csrc / "k.cu"))
    (tmp_path / "profiles" / "k.md").write_text(
        f"code-sha256-16 (source without comments or whitespace): k.cu {h}\n\n"
        "traffic_bytes_per_launch: 123456 (k)\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("k.md", "k.cu") == 123456
    (csrc / "k.cu").write_text(BASE.replace("// trailing comment", "// edited"))
    assert bench.profiled_traffic("k.md", "k.cu") == 123456  # comment edit: still linked
    (csrc / "k.cu").write_text(BASE.replace("1.0f", "2.0f"))
    assert bench.profiled_traffic("k.md", "k.cu") is None  # code changed: unlinked
    assert bench.profiled_traffic("missing.md", "k.cu") is None
