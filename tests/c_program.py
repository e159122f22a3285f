"""Build helper for tests/c_abi_program.c (a plain C caller of the library)."""
import os
import shutil
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi_program.c")
LIB_DIR = os.path.join(ROOT, "gated_delta_rule_kk_gb300", "lib")


def cuda_home():
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def compile_program(out_dir, link=True):
    """gcc the program against include/gdn.h (and, with link, the built
    library and the CUDA runtime); returns the executable's path."""
    cuda = cuda_home()
    exe = os.path.join(out_dir, "c_abi_program")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), SRC]
    if link:
        cmd += ["-o", exe, "-L", LIB_DIR, "-l:libgdn_gb300.so", f"-Wl,-rpath,{LIB_DIR}",
                "-L", os.path.join(cuda, "lib64"), "-lcudart", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    else:
        cmd += ["-c", "-o", exe + ".o"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe
