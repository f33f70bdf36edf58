import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103) and the built GPU library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """With HC_PARITY_LOG set: totals of the parity tiers over the session
    (elements compared, those within the plain bound, those accepted only at
    the condition-aware magnitude or only through the rounding-flip bound, and
    the largest ulp distance in each)."""
    import json
    path = os.environ.get("HC_PARITY_LOG")
    if not path or not os.path.exists(path):
        return
    recs = [json.loads(line) for line in open(path) if line.strip()]
    recs = [r for r in recs if "kind" not in r]
    if not recs:
        return
    n = sum(r["elements"] for r in recs)
    cond = sum(r["pre_cond_rescued"] for r in recs)
    flip = sum(r["pre_flip_rescued"] for r in recs)
    terminalreporter.write_line(
        f"parity tiers: {len(recs)} comparisons, {n} pre_output elements; condition-aware tier {cond} "
        f"(largest {max(r['pre_cond_max_ulp'] for r in recs)} ulp), rounding-flip tier {flip} "
        f"(largest {max(r['pre_flip_max_ulp'] for r in recs)} ulp); post_gate within "
        f"{max(r['post_max_ulp'] for r in recs)} ulp")
