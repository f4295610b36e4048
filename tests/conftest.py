import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: larger CPU cases")


# Parity bar for floating point (bf16 inputs, fp32 accumulation on the device):
# relative Frobenius error and max abs error as a fraction of rms(y_ref).
REL_FROB = 5e-3
MAX_ABS_RMS = 2e-2
