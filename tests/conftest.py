import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")

# A run of the parity suites against another build of the library (the
# bounds-checked one): DCN_TEST_LIBRARY names its path.  Test plumbing only;
# the library itself reads no environment variable.
if os.environ.get("DCN_TEST_LIBRARY"):
    from deformable_convolution_vision_gb300 import binding as _binding
    _binding.LIBRARY = os.environ["DCN_TEST_LIBRARY"]
    _binding._lib = None


def pytest_report_header(config):
    if os.environ.get("DCN_TEST_LIBRARY"):
        from deformable_convolution_vision_gb300 import binding
        return [f"dcn library under test: {binding.LIBRARY}"]
    return []
