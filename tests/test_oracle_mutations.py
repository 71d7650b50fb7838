"""The pins bite: plant a plausible mistake in the oracle (in memory, on the CPU)
and check that at least one pin fails.  Nothing here touches a GPU or a file."""
import numpy as np
import pytest

import oracle
import oracle.ssm_oracle as so
import tests.test_oracle_pins as pins


def _decay_sign(h, delta, A, x, B):
    return np.exp(-delta * A)[:, None, None] * h + (delta[:, None] * x)[:, :, None] * B[None, None, :]


def _outer_transposed(h, delta, A, x, B):
    H, P = x.shape
    u = (delta[:, None] * x).sum(1) / P
    return np.exp(delta * A)[:, None, None] * h + u[:, None, None] * B[None, None, :]


def _drop_D(h, C, D, x):
    return np.einsum("hpn,n->hp", h, C)


def _swap_BC(post, H, P, N):
    x, B, C = _orig_split(post, H, P, N)
    return x, C, B


def _head_map_transposed(post, H, P, N):
    x, B, C = _orig_split(post, H, P, N)
    x = np.swapaxes(post[..., :H * P].reshape(post.shape[:-1] + (P, H)), -1, -2)
    return x, B, C


def _taps_reversed(window, conv_w, conv_b):
    return so.silu(conv_b + np.einsum("ck,kc->c", conv_w[:, ::-1], window))


def _no_bias(window, conv_w, conv_b):
    return so.silu(np.einsum("ck,kc->c", conv_w, window))


def _ring_off_by_one(lay, v, xBC, ring, head):
    rows = []
    for d in range(3, 0, -1):
        src = lay["taps"][v][d - 1]
        rows.append(xBC[src] if src >= 0 else ring[(head + src + 1) % ring.shape[0]])
    rows.append(xBC[v])
    return np.stack(rows)


def _softplus_exp(v):
    return np.exp(v)


def _accept_last_match(parent, tok, tgt):
    lay = so.tree_layout(parent)
    cur, path = 0, [0]
    while True:
        m = [c for c in lay["children"][cur] if tok[c] == tgt[cur]]
        if not m:
            return path, int(tgt[cur])
        cur = m[-1]
        path.append(cur)


def _replay_short(A_log, log_rows, k, h_ckpt, head):
    return _orig_replay(A_log, log_rows, max(0, int(k) - 1), h_ckpt, head)


_orig_split = so.split_xbc
_orig_replay = so.replay

MUTATIONS = {
    "decay sign": ("ssm_step", _decay_sign),
    "x/B outer product collapsed": ("ssm_step", _outer_transposed),
    "D·x dropped": ("ssm_out", _drop_D),
    "B and C swapped": ("split_xbc", _swap_BC),
    "head→channel map transposed": ("split_xbc", _head_map_transposed),
    "conv taps newest-first": ("conv_silu", _taps_reversed),
    "conv bias dropped": ("conv_silu", _no_bias),
    "ring row off by one": ("node_window", _ring_off_by_one),
    "softplus replaced by exp": ("softplus", _softplus_exp),
    "accept takes the last matching child": ("accept", _accept_last_match),
    "replay stops one step short": ("replay", _replay_short),
}

PIN_TESTS = [
    lambda: pins.test_softplus_matches_logaddexp(),
    lambda: [pins.test_chain_conv_matches_numpy_convolve(h) for h in (3, 9, 13)],
    lambda: pins.test_closed_form_scalar_chain(),
    lambda: pins.test_closed_form_scalar_branching(),
    lambda: pins.test_closed_form_pure_decay(),
    lambda: [pins.test_tree_matches_dual_form(s) for s in (1, 2, 3)],
    lambda: pins.test_delta_to_zero_keeps_state(),
    lambda: pins.test_accept_tie_break_lowest_index(),
    lambda: [pins.test_accept_matches_brute_force(s) for s in range(10)],
    lambda: pins.test_replay_reproduces_draft_states(),
]


def _any_pin_fails():
    for t in PIN_TESTS:
        try:
            t()
        except (AssertionError, ValueError, FloatingPointError):
            return True
    return False


def test_unmutated_oracle_passes_every_pin():
    assert not _any_pin_fails()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(so, attr, fn)
    if hasattr(oracle, attr):
        monkeypatch.setattr(oracle, attr, fn)
    with np.errstate(all="ignore"):
        assert _any_pin_fails(), f"no pin caught: {name}"
