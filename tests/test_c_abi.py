"""The header is a plain C99 interface: a C client compiles against it with
warnings as errors, links against the built library, and gets the documented
results from the calls that need no GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libdir():
    from decode_projection_gemms_gb300.build import build
    return os.path.dirname(build())


def test_c_client(libdir, tmp_path):
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "host_calls"
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Wpedantic", "-Werror",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_abi", "host_calls.c"),
           "-L", libdir, "-lkdaproj", f"-Wl,-rpath,{libdir}", "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi ok" in r.stdout
