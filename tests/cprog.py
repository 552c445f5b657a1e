"""Builds the plain-C test program tests/c/transfer_from_c.c against libkvx.so (test helper)."""
import os
import shutil
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "transfer_from_c.c")
CUDA = "/usr/local/cuda"


def build_c_program(out_path: str) -> str:
    """Compiles the program as strict C99 (warnings are errors; the CUDA headers as system
    headers) and links it against the in-tree libkvx.so and the CUDA runtime."""
    from disaggregated_paged_kv_gb300 import kvx
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no C compiler")
    lib_dir = os.path.dirname(kvx.LIB_PATH)
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), "-isystem", os.path.join(CUDA, "include"),
           SRC, "-o", out_path, "-L", lib_dir, "-l:libkvx.so",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", f"-Wl,-rpath,{lib_dir}",
           f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out_path
