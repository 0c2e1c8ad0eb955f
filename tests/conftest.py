import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# The library runs small prefill selections (few query tiles, few pairs) on
# its dp4a row kernel. The parity tests that target the tensor-core
# selection and the routed kernel at small shapes keep them: the tensor
# cores wherever they apply, unless a test (or the caller) says otherwise.
# test_small_prefill_default_rule runs the library's own choice.
os.environ.setdefault("ESA_ROW_SELECT", "tc")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")
