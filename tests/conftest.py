import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    # Build the in-tree CUDA library and the CPU oracle before any test module
    # imports them (both builds are no-ops when up to date).
    from flash_mixed_chunk_gb300 import _buildlib as _b
    _b.build()
    import oracle
    oracle.build()
