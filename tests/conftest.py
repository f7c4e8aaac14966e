import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    # GPU tests are selected with `-m gpu` and deselected with `-m "not gpu"`.
    # They are deliberately NOT auto-skipped when no device is visible: on a
    # GPU machine a missing device or library must fail loudly.
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
