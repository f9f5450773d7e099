"""The bounded device-side wait of the tensor-core kernels runs out cleanly.

dion3_wait_probe runs the GEMM's own bounded mbarrier wait on a barrier that
nothing arrives at, with a 1 ms limit: the kernel records the timeout in the
device status word and returns (no copy or MMA is in flight, nothing hangs),
dion3_device_status reports DION3_ERR_TIMEOUT once and then DION3_OK, and the
context stays usable for a GEMM afterwards.  With the arrival the same wait
succeeds and records nothing."""
import numpy as np
import pytest
import torch

import matrix_orthogonalizing_optimizer_shape_gb300 as d3

pytestmark = pytest.mark.gpu


def test_wait_without_arrival_times_out(cuda_lib):
    d3.device_status()  # start from a clear status word
    d3.wait_probe(arrive=False, limit_ns=1_000_000)
    with pytest.raises(d3.Dion3Error) as exc:
        d3.device_status()
    assert exc.value.status == d3.ERR_TIMEOUT
    d3.device_status()  # the word was cleared by the read


def test_wait_with_arrival_succeeds(cuda_lib):
    d3.device_status()
    for _ in range(3):
        d3.wait_probe(arrive=True, limit_ns=1_000_000)
    d3.device_status()


def test_context_usable_after_timeout(cuda_lib):
    d3.wait_probe(arrive=False, limit_ns=1_000)
    with pytest.raises(d3.Dion3Error):
        d3.device_status()
    rng = np.random.default_rng(3)
    A = torch.from_numpy(rng.standard_normal((256, 128)).astype(np.float16)).cuda()
    B = torch.from_numpy(rng.standard_normal((192, 128)).astype(np.float16)).cuda()
    D = torch.empty((256, 192), dtype=torch.float16, device="cuda")
    d3.gemm_f16(A, B, D=D)
    d3.device_status()
    want = A.double().cpu().numpy() @ B.double().cpu().numpy().T
    assert np.abs(D.double().cpu().numpy() - want).max() <= 2e-3 * np.abs(want).max()
