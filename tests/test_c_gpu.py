"""The C ABI from a plain C99 program on the GPU: tests/c/roundtrip_gpu.c allocates device
pools with cudaMalloc and host chunks with kvx_host_alloc, runs one kvx_roundtrip_chunks and
one kvx_transform_hbm through libkvx.so, and compares every chunk and pool byte with the C
oracle compiled into the program.  No Python or torch on the data path."""
import os
import shutil
import subprocess

import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU hosts too; every test here is gpu-marked
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from paged_kv_gather_gb300.build import build  # noqa: E402

build()
from paged_kv_gather_gb300 import kvx  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_lib_dir(cuda: str) -> str:
    for sub in ("lib64", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib", "lib"):
        d = os.path.join(cuda, sub)
        if os.path.exists(os.path.join(d, "libcudart.so")):
            return d
    pytest.skip(f"no libcudart.so under {cuda}")


def test_c_program_round_trip_transform_and_bulk_mapping(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cudalib = _cuda_lib_dir(cuda)
    lib = kvx.library_path()
    exe = str(tmp_path / "roundtrip_gpu")
    subprocess.run([cc, "-std=c99", "-O1", "-Wall", "-Wextra", "-Werror",
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "oracle"),
                    "-I", os.path.join(cuda, "include"),
                    os.path.join(ROOT, "tests", "c", "roundtrip_gpu.c"), "-o", exe,
                    "-L", os.path.dirname(lib), "-l:" + os.path.basename(lib),
                    "-Wl,-rpath," + os.path.dirname(lib),
                    "-L", cudalib, "-lcudart", "-Wl,-rpath," + cudalib], check=True)
    run = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    out = dict(line.split(" ", 1) for line in run.stdout.strip().splitlines() if " " in line)
    assert run.returncode == 0, run.stdout + run.stderr
    assert out["failures"] == "0"
    assert out["roundtrip_device_flags"] == "0" and out["transform_device_flags"] == "0"
    assert out["roundtrip_chunks_mismatches"] == "0"
    assert out["transform_chunks_mismatches"] == "0"
    assert all(out[f"roundtrip_pool{i}_mismatches"] == "0" for i in range(6))
    assert out["bulk_store_device_flags"] == "0" and out["bulk_load_device_flags"] == "0"
    assert out["bulk_store_chunks_mismatches"] == "0"
    assert all(out[f"bulk_load_pool{i}_mismatches"] == "0" for i in range(6))
