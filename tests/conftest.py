import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# The planted-mistake check of the oracle's pins (tests/test_oracle_mutants.py) runs the pin file
# against a modified copy of oracle/__init__.py, named by ORACLE_PY; normally unset.
if os.environ.get("ORACLE_PY"):
    import importlib.util

    _spec = importlib.util.spec_from_file_location("oracle", os.environ["ORACLE_PY"])
    _mod = importlib.util.module_from_spec(_spec)
    sys.modules["oracle"] = _mod
    _spec.loader.exec_module(_mod)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: vocabulary-scale case (seconds of oracle time)")
