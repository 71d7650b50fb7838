"""Test-side glue: widen generator outputs for the oracle and run it per instance."""
from __future__ import annotations

import numpy as np

import oracle
from synth import bf16_bits_to_f32


def f64(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)


def params_at(params: dict, j: int) -> dict:
    """Layer j's parameters, widened to fp64."""
    return {k: np.asarray(v[j], np.float64) for k, v in params.items()}


def oracle_verify_instance(b: dict, i: int, j: int, return_states=False):
    """Run the oracle on instance (sequence index i, layer index j) of a synth batch."""
    return oracle.verify(params_at(b["params"], j), b["parent"][i], f64(b["xBC"][i, j]), f64(b["dt"][i, j]),
                         b["h0"][i, j].astype(np.float64), f64(b["ring"][i, j]), int(b["ring_head"][i, j]),
                         return_states=return_states)


def rel_err(got, ref):
    """max |got - ref| / (1 + |ref|)  (the parity bound's left side)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if got.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref) / (1.0 + np.abs(ref))))
