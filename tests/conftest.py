import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def has_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


@pytest.fixture(scope="session")
def gpu_lib():
    """The CUDA library, built in-tree if needed; the tests that use it are
    marked gpu and fail (not skip) when it cannot be built or loaded."""
    import draft_token_markov_gb300.build as b
    b.build()
    from draft_token_markov_gb300 import api
    return api


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The acceptance records of the full workloads (licensed deviations,
    excused tokens and the oracle's smallest winning margin), one line each,
    and as JSON in $MARKOV_ACCEPTANCE_OUT when that is set."""
    try:
        from tests import acceptance
    except Exception:  # pragma: no cover
        return
    recs = acceptance.RECORDS
    if not recs:
        return
    tr = terminalreporter
    tr.write_sep("-", "acceptance records")
    for name, r in sorted(recs.items()):
        mm = "none" if r["min_margin"] is None else f"{r['min_margin']:.3g}"
        tr.write_line(f"{name}: ok={r['ok']} positions={r['positions']} "
                      f"cache_1ulp={r['cache_1ulp']} cache_bias_ulp={r['cache_bias_ulp']} "
                      f"cache_bias_wide={r['cache_bias_wide']} excused={r['excused']} "
                      f"min_margin={mm}")
    out = os.environ.get("MARKOV_ACCEPTANCE_OUT")
    if out:
        import json
        os.makedirs(os.path.dirname(os.path.abspath(out)), exist_ok=True)
        with open(out, "w") as f:
            json.dump(recs, f, indent=1, sort_keys=True)
