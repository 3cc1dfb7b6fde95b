"""The stage-wise parity check used by the GPU tests, exercised on the CPU:
the oracle's own results pass it, and planted errors in the output, the gates
or kv fail it."""
import dataclasses

import numpy as np
import pytest

from engram_hashed_gram_gb300 import synth
import parity as P


@pytest.fixture(scope="module")
def case():
    w = dataclasses.replace(synth.workload("tiny_1x16"), B=1, T=12, mask="span10")
    inp = synth.make_inputs(w)
    inp.mask[0, 3] = 0
    tok = np.arange(w.M)
    out, g, kv = P.oracle_tokens(w, inp, tok)
    return w, inp, tok, out, g, kv


def test_oracle_passes_its_own_check(case):
    w, inp, tok, out, g, kv = case
    s = P.check_layer(w, inp, tok, out, g, kv, "self")
    assert s["end_to_end"]["max_err"] == 0.0


def test_planted_output_error_fails(case):
    w, inp, tok, out, g, kv = case
    bad = out.copy()
    bad[5, 1, 100] ^= 0x0040      # a few bf16 steps
    with pytest.raises(AssertionError):
        P.check_layer(w, inp, tok, bad, g, kv, "planted out")


def test_planted_gate_error_fails(case):
    w, inp, tok, out, g, kv = case
    bad = g.copy()
    bad[2, 3] += 0.01
    with pytest.raises(AssertionError):
        P.check_layer(w, inp, tok, out, bad, kv, "planted gate")


def test_planted_kv_error_fails(case):
    w, inp, tok, out, g, kv = case
    bad = kv.copy()
    bad[1, 7] ^= 0x0010
    with pytest.raises(AssertionError):
        P.check_layer(w, inp, tok, out, g, bad, "planted kv")
