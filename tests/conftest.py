import os
import re
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the built CUDA library")


def read_golden(name: str) -> dict:
    """Parse a ``key = value`` golden fixture (``#`` comments; values split on spaces)."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            parts = val.split()
            nums = []
            for p in parts:
                nums.append(int(p) if re.fullmatch(r"-?\d+", p) else p)
            out[key] = nums[0] if len(nums) == 1 else tuple(nums)
    return out


def read_shape_cases(name: str) -> dict:
    """Parse the ``[case M N K BM BN BK]`` / ``label: (..) -> (..)`` fixture."""
    cases, cur = {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            m = re.fullmatch(r"\[case ([\d ]+)\]", line)
            if m:
                cur = tuple(int(x) for x in m.group(1).split())
                cases[cur] = {}
                continue
            label, shapes = (s.strip() for s in line.split(":", 1))
            levels = []
            for part in shapes.split("->"):
                nums = [int(x) for x in re.findall(r"\d+", part)]
                levels.append(tuple(nums))
            cases[cur][label] = levels
    return cases


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle

    oracle.build()
    return oracle
