"""The C ABI from C: tests/c_abi_check.c compiles against include/ks.h as C11 with gcc, links
libks.so, and checks the validation-only calls (no GPU needed)."""
import os
import subprocess

from row_wise_rmsnorm_ks_gb300 import build as ks_build

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_plain_c_caller(tmp_path):
    lib = ks_build.build()
    exe = tmp_path / "c_abi_check"
    lib_dir = os.path.dirname(lib)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror",
                    f"-I{os.path.join(ROOT, 'include')}", os.path.join(HERE, "c_abi_check.c"),
                    f"-L{lib_dir}", "-lks", f"-Wl,-rpath,{lib_dir}", "-o", str(exe)],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert "c abi ok" in r.stdout
