"""The kernel-source hash that keys the committed ncu traffic record: it must
ignore comments and blank lines (a comment edit leaves the compiled kernel
unchanged) and nothing else."""

import bench


def test_comments_and_blank_lines_are_ignored():
    a = "int f(int x) {\n  return x + 1;\n}\n"
    b = ("// header\n/* block\n   comment */\nint f(int x) {  // trailing\n\n"
         "  return x + /* inline */1;\n}\n")
    assert bench._code_only(a) == bench._code_only(b)


def test_code_changes_are_seen():
    a = "int f(int x) { return x + 1; }\n"
    assert bench._code_only(a) != bench._code_only(a.replace("+ 1", "+ 2"))


def test_comment_markers_inside_literals_are_code():
    src = 'const char* s = "a // b /* c */";\nchar q = \'"\';\nint k = 1;  // gone\n'
    out = bench._code_only(src)
    assert '"a // b /* c */"' in out
    assert "char q = '\"';" in out
    assert "gone" not in out and "int k = 1;" in out


def test_escaped_quote_in_string():
    src = 'const char* s = "x\\" // still string";  // comment\n'
    out = bench._code_only(src)
    assert '"x\\" // still string"' in out and "comment" not in out


def test_hash_is_stable_and_short():
    h = bench.kernel_source_hash()
    assert h == bench.kernel_source_hash() and len(h) == 16
