"""The profile digest of the attention sources ignores comments and layout, not code.

bench.py reads a committed ncu traffic figure back only while the digest it was stamped with
matches the current attention sources; a comment edit must keep it, a code edit must not.
"""
from paged_kv_attention_forward_gb300 import build


def test_code_text_drops_comments_and_layout_only():
    a = "int x = 1; // one\n/* block\n comment */ float y = x * 2;\n"
    b = "int  x = 1;\n\n\nfloat y = x * 2; // two, reworded\n"
    c = "int x = 1; float y = x * 3;\n"
    assert build.code_text(a) == build.code_text(b)
    assert build.code_text(a) != build.code_text(c)


def test_attention_digest_follows_code(tmp_path, monkeypatch):
    for name in build.ATTENTION_SOURCES:
        (tmp_path / name).write_text("// header\nint f(int a) { return a + 1; }\n")
    monkeypatch.setattr(build, "CSRC", str(tmp_path))
    d0 = build.source_digest(build.ATTENTION_SOURCES)
    (tmp_path / build.ATTENTION_SOURCES[0]).write_text("/* reworded */\nint f(int a)\n{\n    return a + 1;\n}\n")
    assert build.source_digest(build.ATTENTION_SOURCES) == d0
    (tmp_path / build.ATTENTION_SOURCES[0]).write_text("int f(int a) { return a + 2; }\n")
    assert build.source_digest(build.ATTENTION_SOURCES) != d0
