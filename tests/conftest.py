"""Shared pytest configuration: the ``gpu`` marker, repo-root imports and golden-file parsing."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the built CUDA library")


def read_golden(name: str) -> dict:
    """Parse a golden fixture: '#' comments, a NAME line, then whitespace-separated rows."""
    blocks: dict = {}
    cur = None
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            toks = line.split()
            if len(toks) == 1 and not _is_num(toks[0]):
                cur = toks[0]
                blocks[cur] = []
                continue
            blocks[cur].append([None if t == "-" else (int(t) if _is_int(t) else float(t))
                                for t in toks])
    return blocks


def _is_int(t: str) -> bool:
    try:
        int(t)
        return True
    except ValueError:
        return False


def _is_num(t: str) -> bool:
    try:
        float(t)
        return True
    except ValueError:
        return t == "-"


@pytest.fixture(scope="session")
def golden():
    return read_golden
