"""Failure detection without a fault: the kernels' on-chip waits are bounded.

A wait on an mbarrier that nothing arrives on (the library's own
fm::mbar_wait, built into a test-only kernel) must give up after its time
limit (2 s), set the timeout bit of the status word it reports to and return,
and the CTA's other waiter must leave as well; afterwards the context is still
usable (the library's kernels run and give the right answer)."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "sparse_attention_kv_c4_gb300", "csrc")
TIMEOUT_BIT = 0x2  # FM_DEVERR_TIMEOUT


@pytest.fixture(scope="module")
def torch_dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return torch, torch.device("cuda:0")


def test_bounded_wait_gives_up_and_reports(torch_dev, tmp_path):
    torch, dev = torch_dev
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    so = str(tmp_path / "wait_probe.so")
    subprocess.run([nvcc, "-gencode=arch=compute_103a,code=sm_103a", "-O2", "-shared", "-Xcompiler", "-fPIC",
                    "-I", CSRC, "-o", so, os.path.join(HERE, "wait_timeout_probe.cu")], check=True)
    lib = ctypes.CDLL(so)
    lib.launch_wait_probe.argtypes = [ctypes.c_void_p] * 4
    lib.launch_wait_probe.restype = ctypes.c_int
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    results = torch.full((2,), 7, dtype=torch.int32, device=dev)
    elapsed = torch.zeros(2, dtype=torch.int64, device=dev)
    assert lib.launch_wait_probe(status.data_ptr(), results.data_ptr(), elapsed.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert results.cpu().tolist() == [0, 0]  # both waiters gave up
    assert int(status.item()) & TIMEOUT_BIT
    ns = elapsed.cpu().numpy()
    assert ns.max() >= 2_000_000_000 and ns.max() < 10_000_000_000, ns

    # the context is still usable
    import sparse_attention_kv_c4_gb300 as fm
    rng = np.random.default_rng(9)
    s = torch.from_numpy(rng.standard_normal((3, 5000)).astype(np.float32)).to(dev)
    idx = torch.empty((3, 64), dtype=torch.int32, device=dev)
    fm.fm_topk_select(s, 64, idx)
    torch.cuda.synchronize()
    ref = torch.topk(s, 64, dim=1).indices.sort(dim=1).values.to(torch.int32)
    assert torch.equal(idx, ref)
    assert fm.fm_device_status(reset=True) == 0  # the library's own status word was not touched
