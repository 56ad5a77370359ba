"""The C ABI compiles and links from plain C (no GPU needed): the program
in tests/c/step_c_api.c builds against include/medusa.h and the library."""
import os

from c_api import build_c_program


def test_c_program_builds_and_links(tmp_path):
    exe = build_c_program(tmp_path)
    assert os.access(exe, os.X_OK)
