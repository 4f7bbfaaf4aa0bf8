"""Host checks of bench.py's bookkeeping: the kernel-code hash that keys the
stored DRAM-traffic figures ignores comments and layout but not code."""
import bench


def test_strip_comments_keeps_code_and_literals():
    src = ('int a = 1; // trailing\n'
           '/* block\n comment */ const char *s = "x // not a comment /* nor */";\n'
           "char q = '\"'; int b = a /* inline */ + 2;\n")
    got = bench.strip_comments(src)
    assert got == ('int a = 1; const char *s = "x // not a comment /* nor */"; '
                   "char q = '\"'; int b = a + 2;")


def test_code_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    csrc = tmp_path / "paged_kv_attention_kvcache_gb300" / "csrc"
    csrc.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (csrc / "k.cu").write_text("__global__ void k(int *p) { p[0] = 1; }\n")
    h0 = bench.kernel_source_hash("k.cu")
    (csrc / "k.cu").write_text("// the kernel\n__global__ void k(int *p)\n{\n  p[0] = 1;  /* one */\n}\n")
    assert bench.kernel_source_hash("k.cu") == h0
    (csrc / "k.cu").write_text("__global__ void k(int *p) { p[0] = 2; }\n")
    assert bench.kernel_source_hash("k.cu") != h0
