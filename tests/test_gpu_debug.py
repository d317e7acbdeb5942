"""The debug build of the library (device-side index checks, -DTXL_DEBUG).

Its kernels check the index arithmetic of the hot path (the work split of each
block, the shared-memory ring rows through which the Appendix B shift of
"Transformer-XL: Attentive Language Models Beyond a Fixed-Length Context" is
applied, the TMEM columns of the table chunks, output rows, decode key and table
ranges, memory ring slots and window rows) and record a failure in the device
status word instead of trapping.  Here, in child processes that load the debug
library: one check failed on purpose is reported and cleared, and the kernel
parity tests (odd shapes, ragged tails, splits, the decode kernel, windows,
memory rings) pass with every check active; each of those tests reads the
status word after its kernels."""

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu


def _env():
    return dict(os.environ, TXL_DEBUG_LIB="1")


def test_debug_build_reports_a_failed_index_check():
    code = ("import transformer_xl_relative_pos_gb300 as t\n"
            "assert t.debug_checks(), 'not the debug build'\n"
            "assert t.device_status() == 0\n"
            "assert t.debug_index_probe() == -8\n"     # TXL_ERR_INDEX
            "assert t.device_status() == 0\n"          # read and cleared
            "assert t.lib_path().endswith('libtxl_gb300_debug.so')\n"
            "print('ok')\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=_env(), capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stderr[-3000:]


def test_kernel_parity_tests_pass_with_index_checks():
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        "tests/test_gpu_kernels.py", "tests/test_gpu_window.py",
                        "tests/test_gpu_decode.py", "tests/test_gpu_project.py",
                        "tests/test_gpu_bwd.py"],
                       cwd=ROOT, env=_env(), capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, (r.stdout[-3000:] + r.stderr[-2000:])
