import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU; calls the library through its C ABI")


def library():
    """Build the CUDA library if it is stale, then load it (raises if it cannot)."""
    from fully_sharded_unit_gb300 import binding
    from fully_sharded_unit_gb300.build import build
    build()
    return binding.lib()
