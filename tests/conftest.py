import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="session")
def tcd():
    """The C-ABI binding over a freshly built libtcd.so (builds if stale)."""
    from trie_constrained_decoding_gb300 import build
    build.build()
    from trie_constrained_decoding_gb300 import binding
    return binding
