"""The oracle's C code has no undefined behaviour (signed overflow,
out-of-range shifts or conversions, misaligned access) on its pin inputs:
the pins run against a copy built with UBSan that aborts on the first
finding. No GPU needed."""
import os
import shutil
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_oracle_pins_pass_under_ubsan(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    lib = str(tmp_path / "liboracle_ubsan.so")
    flags = [f for f in oracle._CFLAGS]
    subprocess.run(["gcc", *flags, "-g", "-fsanitize=undefined", "-fno-sanitize-recover=all",
                    "-o", lib, oracle._SRC, "-lm"], check=True)
    code = (
        "import sys\n"
        f"sys.path[:0] = [{ROOT!r}, {os.path.join(ROOT, 'tests')!r}]\n"
        "import oracle\n"
        f"oracle._LIB_PATH = {lib!r}\n"
        "import pytest\n"
        "rc = pytest.main(['-q', '-x', '-s', '-p', 'no:cacheprovider', '-m', 'not gpu', "
        f"{os.path.join(ROOT, 'tests', 'test_oracle_pins.py')!r}])\n"
        "assert oracle._lib is not None and oracle._lib._name == " f"{lib!r}\n"
        "sys.exit(rc)\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
