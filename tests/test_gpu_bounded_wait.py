"""The library's bounded mbarrier waits, made to run out on purpose.

Every wait in the decode and indexer kernels polls a bounded number of times
(mla_device.cuh: mbar_wait_bounded, mbar_wait_or_abort); when the phase never
completes it sets a bit in a fault word the host reads and returns, so the
CTA can drain and leave instead of hanging the GPU.  These tests compile
tests/bounded_wait_kernels.cu against the library's own device header and
check, on a barrier that nothing ever completes, that the wait gives up with
the fault bit set and the CUDA context stays usable afterwards; that a wait
told to abort by another warp leaves without a fault bit; and that a wait
whose phase does complete returns true.  Nothing here faults, traps or hangs
the GPU: the longest wait ends by its own poll budget (seconds)."""
import ctypes as C
import os
import subprocess
import time

import numpy as np
import pytest
import torch

from gpu_helpers import lib

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "sparse_mla_decode_kv_gb300", "csrc")
TEST_FAULT = 0x40


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("bounded_wait") / "libwaitprobe.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", "-I", CSRC, os.path.join(HERE, "bounded_wait_kernels.cu"), "-o", out],
                   check=True)
    so = C.CDLL(out)
    so.wait_probe.restype = C.c_int
    so.wait_probe.argtypes = [C.c_int, C.POINTER(C.c_uint), C.POINTER(C.c_int), C.POINTER(C.c_longlong)]
    torch.cuda.init()
    return so


def run(probe, mode):
    fault, ok, cycles = C.c_uint(0), C.c_int(-1), C.c_longlong(0)
    t0 = time.monotonic()
    err = probe.wait_probe(mode, C.byref(fault), C.byref(ok), C.byref(cycles))
    return err, fault.value, ok.value, cycles.value, time.monotonic() - t0


def test_wait_whose_phase_completes_returns_true(probe):
    err, fault, ok, cycles, _ = run(probe, 2)
    assert err == 0 and ok == 1 and fault == 0


def test_wait_told_to_abort_leaves_without_fault_bit(probe):
    err, fault, ok, cycles, secs = run(probe, 1)
    assert err == 0 and ok == 0 and fault == 0
    assert secs < 10.0


def test_wait_that_never_completes_gives_up_and_reports(probe):
    err, fault, ok, cycles, secs = run(probe, 0)
    assert err == 0, f"CUDA error {err}"
    assert ok == 0, "the wait must report that its phase never completed"
    assert fault & TEST_FAULT, "the fault bit must be set"
    assert cycles > 1_000_000, "the wait must actually have polled"
    assert secs < 120.0
    print(f"bounded wait gave up after {secs:.2f} s ({cycles:,} SM cycles)")
    # the context is still usable: a library call right after gives exact results
    m = lib()
    s = torch.arange(5000, dtype=torch.float32, device="cuda").remainder(977).view(1, -1).contiguous()
    cl = torch.tensor([5000], dtype=torch.int32, device="cuda")
    got = m.mla_topk(s, cl, 64).cpu().numpy()[0]
    order = np.lexsort((np.arange(5000), -s.cpu().numpy()[0].astype(np.float64)))
    assert np.array_equal(got, np.sort(order[:64]))
    assert m.mla_device_fault(clear=False) == 0
