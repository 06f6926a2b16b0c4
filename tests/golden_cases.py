"""Reader for tests/golden/page_test_cases.txt (the shapes the pages' own
attention test runs; see the citations in that file)."""
import os

_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "page_test_cases.txt")


def load():
    prefill, decode = [], []
    for line in open(_PATH):
        line = line.split("#", 1)[0].split()
        if not line:
            continue
        kind, a, b, hq, hkv, d = line[0], *map(int, line[1:])
        (prefill if kind == "prefill" else decode).append((a, b, hq, hkv, d))
    return prefill, decode
