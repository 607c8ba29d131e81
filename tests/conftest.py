import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running statistical test")


# The mutation tests run the oracle's pins against a copy of the oracle with
# one planted mistake; this variable points the oracle at that build.
_ORACLE_LIB = os.environ.get("D3D_ORACLE_LIB_OVERRIDE")
if _ORACLE_LIB:
    import oracle

    oracle.build = lambda force=False: _ORACLE_LIB
