import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def _lib_stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    srcs = [os.path.join(ROOT, "include", "mqa_decode.h")]
    csrc = os.path.join(ROOT, "mqa_decode_attention_gb300", "csrc")
    srcs += [os.path.join(csrc, f) for f in os.listdir(csrc)]
    return any(os.path.getmtime(s) > t for s in srcs)


@pytest.fixture(scope="session")
def built_lib():
    """Path of libmqa_decode.so, (re)built with nvcc when missing or stale."""
    from mqa_decode_attention_gb300.build import build, lib_path

    lib = lib_path()
    if _lib_stale(lib):
        build()
    return lib
