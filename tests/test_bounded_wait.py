"""The bounded pipeline wait every kernel uses: a barrier that never
completes makes the wait give up after its time limit (2 s), flag
PKV_DEVERR_WAIT_TIMEOUT and return, and the CUDA context stays usable.
The failure is made on purpose by a barrier nothing arrives on; no fault,
trap or hang is involved.  The harness kernel is built from
tests/bounded_wait_kernel.cu against the library's device header."""

import ctypes
import os
import subprocess
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "bounded_wait_kernel.cu")
WAIT_TIMEOUT = 0x8


def build(out_dir: str) -> str:
    from paged_kv_cache_304_gb300 import build as B
    lib = os.path.join(out_dir, "libbounded_wait.so")
    subprocess.run([B.nvcc(), *B.ARCH, *B.NVCC_FLAGS, "-shared", SRC, "-o", lib], check=True)
    return lib


def test_harness_compiles(tmp_path):
    """nvcc cross-compiles the harness for sm_103a and it exports its entry
    point (no GPU needed)."""
    lib = ctypes.CDLL(build(str(tmp_path)))
    assert hasattr(lib, "bounded_wait_probe")


@pytest.mark.gpu
def test_wait_that_never_completes_times_out_and_context_survives(tmp_path):
    import torch
    lib = ctypes.CDLL(build(str(tmp_path)))
    lib.bounded_wait_probe.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.bounded_wait_probe.restype = ctypes.c_int
    dev = torch.device("cuda:0")
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    # a completing barrier: no flag
    assert lib.bounded_wait_probe(0, err.data_ptr(), status.data_ptr(), stream) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 1 and int(err.item()) == 0
    # a silent barrier: the wait gives up after about 2 s
    t0 = time.monotonic()
    assert lib.bounded_wait_probe(1, err.data_ptr(), status.data_ptr(), stream) == 0
    torch.cuda.synchronize()
    dt = time.monotonic() - t0
    assert int(status.item()) == 2
    assert int(err.item()) & WAIT_TIMEOUT
    assert 1.5 < dt < 30.0
    # the context is still usable
    x = torch.arange(1024, device=dev, dtype=torch.float32)
    assert float(x.sum().item()) == 1023 * 1024 / 2
