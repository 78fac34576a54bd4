import json
import os
import struct
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def golden(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)


def golden_file(case):
    """File image of a golden case (see tests/golden/format_errors.json)."""
    if "file_hex" in case:
        return bytes.fromhex(case["file_hex"])
    hb = bytes.fromhex(case["header_hex"]) if "header_hex" in case else case["header"].encode()
    n = case.get("length", len(hb))
    return struct.pack("<Q", n) + hb + bytes(case.get("data", 0))


def small_file():
    """File image of tests/golden/format_small.json."""
    g = golden("format_small.json")
    hb = g["header"].encode() + b" " * g["pad"]
    return g, struct.pack("<Q", len(hb)) + hb + bytes.fromhex(g["data_hex"])


@pytest.fixture(scope="session")
def oracle():
    from oracle import oracle as O
    O.lib()
    return O


@pytest.fixture(scope="session")
def stmat():
    """The product binding with its library built for sm_103a (host parts run
    without a GPU)."""
    from safetensors_materialization_gb300 import build as B
    B.build()
    from safetensors_materialization_gb300 import stmat as S
    S.lib()
    return S
