"""The digest that keys bench.py's stored DRAM-traffic figures to the kernel
sources they were measured on: it follows the code, not the comments."""
import bench


def test_comments_do_not_change_the_code_tokens():
    t = bench._code_tokens
    assert t("int a; // note\nint b;") == t("int a;\nint b; /* other note */")
    assert t("a /* two\nlines */ b") == "a b"
    assert t('s = "http://x"; // y') == 's = "http://x";'   # // inside a string stays
    assert t("c = '\"'; /* q */ d") == "c = '\"'; d"
    assert t('x = "a\\"//b";') == 'x = "a\\"//b";'          # escaped quote inside a string


def test_code_changes_change_the_tokens():
    t = bench._code_tokens
    assert t("int a = 1;") != t("int a = 2;")
    assert t("f(x);") != t("g(x);")


def test_digest_is_stable():
    assert bench.kernel_sources_digest() == bench.kernel_sources_digest()
    assert len(bench.kernel_sources_digest()) == 16
