"""The C ABI from a plain C program on the GPU: tests/c/step_c_api.c runs a
tiny decoding step as the four separate calls and through the step executor
(stream and graph mode, pinned host inputs and results) and compares the
paths bit for bit; the Python parity tests tie the calls to the oracle."""
import subprocess

import pytest

from c_api import build_c_program

pytestmark = pytest.mark.gpu


def test_c_program_runs_the_step(tmp_path):
    exe = build_c_program(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.strip() == "ok"
