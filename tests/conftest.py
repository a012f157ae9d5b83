"""Shared pytest configuration: the ``gpu`` marker and the repository root on sys.path."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def ensure_built():
    """Build libdtt.so if it is missing or older than a source file (CPU tests need it too)."""
    import glob
    from device_triggered_transfers_gb300 import LIB_PATH
    from device_triggered_transfers_gb300.build import build
    srcs = glob.glob(os.path.join(ROOT, "device_triggered_transfers_gb300", "csrc", "*")) + \
        glob.glob(os.path.join(ROOT, "include", "*"))
    if not os.path.exists(LIB_PATH) or \
            os.path.getmtime(LIB_PATH) < max(os.path.getmtime(s) for s in srcs):
        build()
