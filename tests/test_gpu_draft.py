"""Draft side on the GPU: chained ssm_draft_step calls against the oracle, and
ssm_replay against the stepped states (bit for bit) and the oracle."""
import numpy as np
import pytest
import torch

import oracle
from synth import Shape, Workload, draft_batch, workload
from tests.helpers import bf16_dev, dev, f64, params_at, params_dev, rel_err, ring_window

pytestmark = pytest.mark.gpu
TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_mamba2_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"


def run_draft(b, w, steps):
    from speculative_decoding_mamba2_gb300 import Dims, ssm_draft_step
    S, L = len(b["seqs"]), len(b["layers"])
    I = S * L
    dims = Dims(n_heads=w.shape.H, n_layers=L, ring_cap=w.ring_cap)
    prm = params_dev(b["params"])
    h_ckpt = dev(b["h0"]).view(I, dims.n_heads, dims.head_dim, dims.d_state)
    h_work = torch.empty_like(h_ckpt)
    ring = bf16_dev(b["ring"]).view(I, w.ring_cap, dims.conv_dim)
    head = dev(b["ring_head"]).view(I)
    cap = steps
    logs = dict(delta=torch.zeros(I, cap, dims.n_heads, device="cuda"),
                B=torch.zeros(I, cap, dims.d_state, device="cuda"),
                x=torch.zeros(I, cap, dims.d_inner, device="cuda"), len=torch.zeros(I, dtype=torch.int32,
                                                                                     device="cuda"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    xs = bf16_dev(b["xBC"]).view(steps, I, dims.conv_dim)
    dts = bf16_dev(b["dt"]).view(steps, I, dims.n_heads)
    states, ys = [], []
    for t in range(steps):
        y = torch.empty(I, dims.d_inner, device="cuda")
        ssm_draft_step(dims, prm, S, t, cap, xs[t], dts[t], h_ckpt if t == 0 else h_work, h_work, ring, head,
                       logs["delta"], logs["B"], logs["x"], logs["len"], y, status)
        states.append(h_work.clone())
        ys.append(y)
    torch.cuda.synchronize()
    return dict(dims=dims, prm=prm, h_ckpt=h_ckpt, ring=ring, head=head, logs=logs, status=status, states=states,
                ys=ys, cap=cap)


def replay(r, n_seq, k_list, h=None):
    from speculative_decoding_mamba2_gb300 import ssm_replay
    h = r["h_ckpt"].clone() if h is None else h
    head = r["head"].clone()
    ll = r["logs"]["len"].clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    k = torch.tensor(k_list, dtype=torch.int32, device="cuda")
    ssm_replay(r["dims"], r["prm"], n_seq, r["cap"], k, r["logs"]["delta"], r["logs"]["B"], r["logs"]["x"], ll, h,
               head, status)
    torch.cuda.synchronize()
    return h, head, ll, int(status)


def oracle_draft(b, i, j, steps):
    prm = params_at(b["params"], j)
    h = b["h0"][i, j].astype(np.float64)
    ring = f64(b["ring"][i, j])
    head = int(b["ring_head"][i, j])
    states, ys, log = [h], [], []
    for t in range(steps):
        h, y, ring, row = oracle.draft_step(prm, f64(b["xBC"][t, i, j]), f64(b["dt"][t, i, j]), h, ring, head, t)
        states.append(h)
        ys.append(y)
        log.append(row)
    return states, ys, log, ring


def test_370m_draft_chain16_and_replay():
    w = workload(1)
    b = draft_batch(w)
    r = run_draft(b, w, 16)
    assert int(r["status"]) == 0
    L = len(b["layers"])
    for j in [0, 23, 47]:
        states, ys, log, ring_ref = oracle_draft(b, 0, j, 16)
        for t in range(16):
            assert rel_err(r["ys"][t][j].double().cpu().numpy(), ys[t]) <= TOL, (j, t)
            assert rel_err(r["states"][t][j].double().cpu().numpy(), states[t + 1]) <= TOL, (j, t)
        # log rows are the post-conv intermediates the oracle logs
        for t in range(16):
            d, Bv, x = log[t]
            assert rel_err(r["logs"]["delta"][j, t].double().cpu().numpy(), d) <= TOL
            assert rel_err(r["logs"]["B"][j, t].double().cpu().numpy(), Bv) <= TOL
            assert rel_err(r["logs"]["x"][j, t].double().cpu().numpy(), x) <= TOL
        # ring rows written by the draft (bytes)
        ring_gpu = r["ring"][j].view(torch.int16).cpu().numpy().view(np.uint16)
        for t in range(16):
            np.testing.assert_array_equal(ring_gpu[(3 + t) % w.ring_cap], b["xBC"][t, 0, j])
    assert r["logs"]["len"].cpu().tolist() == [16] * L
    # replay to the sampled accepted position and to every k: bit-exact with the stepped state
    for k in sorted({int(b["k"][0]), 0, 1, 7, 15, 16}):
        h, head, ll, st = replay(r, 1, [k])
        assert st == 0
        ref = r["h_ckpt"] if k == 0 else r["states"][k - 1]
        assert torch.equal(h, ref), k
        assert head.cpu().tolist() == [3 + k] * L and ll.cpu().tolist() == [0] * L
        for j in [0, 47]:
            h_or, head_or = oracle.replay(b["params"]["A_log"][j].astype(np.float64),
                                          oracle_draft(b, 0, j, 16)[2], k, b["h0"][0, j].astype(np.float64), 3)
            assert rel_err(h[j].double().cpu().numpy(), h_or) <= TOL
            assert head_or == 3 + k
        # the conv window after replay is the three positions before the new head
        ring_gpu = r["ring"][0].view(torch.int16).cpu().numpy().view(np.uint16)
        seq = np.concatenate([b["ring"][0, 0, :3], b["xBC"][:, 0, 0]])
        np.testing.assert_array_equal(ring_window(ring_gpu, 3 + k), seq[k:k + 3])


def test_replay_k_out_of_range_is_clamped_and_flagged():
    from speculative_decoding_mamba2_gb300 import SSM_STATUS_K_RANGE
    w = Workload(60, "draft small", Shape(H=4), n_layers=2, batch=2, trees=(), draft_steps=6)
    b = draft_batch(w)
    r = run_draft(b, w, 6)
    h, head, ll, st = replay(r, 2, [9, -2])
    assert st & SSM_STATUS_K_RANGE
    assert torch.equal(h[0:2], r["states"][5][0:2])  # clamped to log_len = 6
    assert torch.equal(h[2:4], r["h_ckpt"][2:4])  # clamped to 0
    assert head.cpu().tolist() == [9, 9, 3, 3]


def test_780m_batch64_draft_replay_16():
    w = workload(4)
    b = draft_batch(w, seqs=[0, 63], layers=[0, 1, 47])
    r = run_draft(b, w, 16)
    ks = [int(x) for x in b["k"]]
    h, head, ll, st = replay(r, 2, ks)
    assert st == 0
    for i in range(2):
        for j in range(3):
            inst = i * 3 + j
            ref = r["h_ckpt"][inst] if ks[i] == 0 else r["states"][ks[i] - 1][inst]
            assert torch.equal(h[inst], ref)
            _, _, log, _ = oracle_draft(b, i, j, 16)
            h_or, _ = oracle.replay(b["params"]["A_log"][j].astype(np.float64), log, ks[i],
                                    b["h0"][i, j].astype(np.float64), 3)
            assert rel_err(h[inst].double().cpu().numpy(), h_or) <= TOL


def test_replay_longer_than_one_pass_and_ragged_heads():
    # 40 logged steps (several passes of the replay's register-held B rows) and H = 5 (the
    # last head group of the replay is ragged): replay(k) equals the stepped state bit for bit
    w = Workload(62, "draft long", Shape(H=5), n_layers=2, batch=2, trees=(), draft_steps=40, ring_cap=48)
    b = draft_batch(w)
    r = run_draft(b, w, 40)
    ks = [40, 23]
    h, head, ll, st = replay(r, 2, ks)
    assert st == 0
    for i in range(2):
        for j in range(2):
            inst = i * 2 + j
            assert torch.equal(h[inst], r["states"][ks[i] - 1][inst])
    assert head.cpu().tolist() == [3 + 40, 3 + 40, 3 + 23, 3 + 23]
    assert ll.cpu().tolist() == [0, 0, 0, 0]
