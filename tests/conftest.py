import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_sessionstart(session):
    # The CUDA library and the oracle are compiled from source (nvcc cross-compiles
    # without a GPU); both builds are no-ops when up to date.
    from mla_decode_attention_02_gb300 import build as lib_build
    import oracle

    lib_build.build()
    oracle.build()
