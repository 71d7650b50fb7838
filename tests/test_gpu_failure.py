"""Failure detection on the GPU without a fault: the library's bounded mbarrier wait gives
up on a barrier nothing arrives at, reports SSM_STATUS_TIMEOUT in the caller's status word,
and the context stays usable for the next call."""
import numpy as np
import pytest
import torch

from synth import Shape, Workload, batch
from tests.helpers import oracle_verify_instance, rel_err, run_tree_step, upload_tree_batch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_mamba2_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"


def test_bounded_wait_gives_up_reports_and_leaves_the_context_usable():
    from speculative_decoding_mamba2_gb300 import SSM_STATUS_TIMEOUT, ssm_selftest_bounded_wait
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    ssm_selftest_bounded_wait(2000, status)  # 2 ms
    e1.record()
    torch.cuda.synchronize()
    assert int(status) == SSM_STATUS_TIMEOUT
    assert e0.elapsed_time(e1) >= 1.5  # the wait ran for its limit, then gave up
    # the same context runs a verify round afterwards, with a clean status
    w = Workload(60, "after timeout", Shape(H=4), n_layers=1, batch=1, trees=(("random", 10, 3, 3),))
    b = batch(w)
    out = run_tree_step(upload_tree_batch(b, w))
    assert int(out["status"]) == 0
    assert rel_err(out["y"][0].cpu().numpy(), oracle_verify_instance(b, 0, 0)) <= 1e-3
