"""The ragged-vocabulary parity tests (rows off 16-byte boundaries, head and
tail elements, vocabularies shorter than a vector, a tile or k) against the
library built with device-side index checks: every index a kernel computes
or reads is tested before use, and the results still match the oracle."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_ragged_vocab_under_device_checks():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_66_gb300 import _build
    _build.build(debug=True)
    env = dict(os.environ, SV_LIBRARY="debug")
    tests = ["tests/test_debug_build.py::test_loaded_variant_follows_the_environment",
             "tests/test_gpu_parity.py::test_ragged_vocab",
             "tests/test_gpu_filtered.py::test_filtered_ragged_vocab"]
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", *tests],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=1200)
    print(r.stdout[-2000:])
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and "failed" not in r.stdout
