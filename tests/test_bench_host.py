"""Host-side pieces of bench.py: the code identity used for the DRAM-traffic
lookup."""
import bench


def test_code_tokens_ignore_comments_and_layout_only():
    a = 'int f(int x) {\n  // a comment\n  return x + 1; /* block\n comment */\n}\n'
    b = 'int f(int x){return x+1;}'
    assert bench.code_tokens(a) == bench.code_tokens(b)
    assert bench.code_tokens('return x + 2;') != bench.code_tokens('return x + 1;')
    # "//" inside a string literal is code, not a comment
    assert bench.code_tokens('const char* s = "a//b";') == 'constchar*s="a//b";'
    assert bench.code_tokens('x = "a\\"//";') == 'x="a\\"//";'


def test_every_kernel_has_a_code_hash():
    for k in bench.KERNEL_SOURCES:
        assert len(bench.source_hash(k)) == 16
