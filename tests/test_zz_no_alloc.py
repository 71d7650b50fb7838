"""ssm_tree_verify_noalloc -- the entry point for callers that cannot allocate
device memory (its scratch is an array compiled into the library) -- gives the
same outputs as ssm_tree_verify with a caller-allocated workspace, bit for bit
(the same kernels run on the same inputs; only the scratch address differs), on
calls in a row with different batches (the shared array keeps the previous
call's contents when the next starts): two tree batches, then a long chain tree,
which takes the chain kernels and their own scratch records.  Kept in a file of
its own, collected last."""
import ctypes

import pytest
import torch

from synth import Shape, Workload, batch, workload
from tests.helpers import upload_tree_batch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_mamba2_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"


def _both(d):
    from speculative_decoding_mamba2_gb300 import ssm_tree_verify, ssm_tree_verify_noalloc, ssm_tree_verify_workspace_size
    dims, S, n = d["dims"], d["n_seq"], d["n"]
    I = S * dims.n_layers
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y_ref = torch.full((I, n, dims.d_inner), float("nan"), device="cuda")
    ws = torch.empty(ssm_tree_verify_workspace_size(dims, S, n, d["depth"]), dtype=torch.uint8, device="cuda")
    ssm_tree_verify(dims, d["params"], S, n, d["depth"], d["layout"], d["xBC"], d["dt"], d["h0"], d["ring"],
                    d["ring_head"], y_ref, ws, status)
    y = torch.full_like(y_ref, float("nan"))
    ssm_tree_verify_noalloc(dims, d["params"], S, n, d["depth"], d["layout"], d["xBC"], d["dt"], d["h0"], d["ring"],
                            d["ring_head"], y, status)
    torch.cuda.synchronize()
    assert int(status) == 0
    return y, y_ref


def test_noalloc_matches_workspace_entry_point_twice():
    # first call: the 2.7B layer shape, 8 layers x 2 sequences of 16-node random trees
    w1 = Workload(70, "noalloc a", Shape(H=80), n_layers=8, batch=2, trees=(("random", 16, 3, 4),))
    y, y_ref = _both(upload_tree_batch(batch(w1), w1))
    assert torch.isfinite(y).all()
    assert torch.equal(y, y_ref)
    # second call right after, another shape and tree: the array holds the first call's data
    w2 = workload(0)
    y, y_ref = _both(upload_tree_batch(batch(w2), w2))
    assert torch.isfinite(y).all()
    assert torch.equal(y, y_ref)
    # third call: a 40-node chain (deeper than the tree kernels take), so the chain kernels
    # read their per-chunk records from the same array, over the tree calls' contents
    w3 = Workload(71, "noalloc chain", Shape(H=6), n_layers=1, batch=2, trees=(("chain", 40),))
    d3 = upload_tree_batch(batch(w3), w3)
    assert d3["depth"] == 39
    y, y_ref = _both(d3)
    assert torch.isfinite(y).all()
    assert torch.equal(y, y_ref)


def test_noalloc_rejects_batches_beyond_its_array():
    from speculative_decoding_mamba2_gb300 import (SSM_ERR_CAPACITY, SSM_NOALLOC_WORKSPACE_BYTES, Dims, SSMError,
                                                   lib, ssm_tree_verify_workspace_size)
    from speculative_decoding_mamba2_gb300.binding import ssm_dims, ssm_params
    dims = Dims(n_heads=80, n_layers=64, ring_cap=20)
    assert ssm_tree_verify_workspace_size(dims, 16, 16, 4) > SSM_NOALLOC_WORKSPACE_BYTES
    cd, cp = dims.c(), ssm_params(16, 16, 16, 16, 16)
    fake = ctypes.c_void_p(16)  # rejected before any pointer is used
    rc = lib().ssm_tree_verify_noalloc(ctypes.byref(cd), ctypes.byref(cp), 16, 16, 4, fake, fake, fake, fake, fake,
                                       fake, fake, None, None)
    assert rc == SSM_ERR_CAPACITY
    assert "bytes of scratch" in lib().ssm_last_error().decode()
