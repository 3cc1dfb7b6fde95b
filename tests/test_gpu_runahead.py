"""The run-ahead schedule (EngramRunAhead): two Engram layers whose lookup and
projection are queued on a side stream at step start while the caller's
stream is busy (a sleeping kernel stands for the backbone), and whose gates run
at each layer's entry.  The outputs must equal engram_forward bit for bit, over
two consecutive steps that reuse the kv buffers."""
import numpy as np
import pytest
import torch

from engram_hashed_gram_gb300 import synth
from engram_hashed_gram_gb300 import synth_device as SD

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def two_layers():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from engram_hashed_gram_gb300 import build as B
    B.build()
    from engram_hashed_gram_gb300.layer import EngramLayer
    w = synth.workload("tiny_1x16")
    table, scale = SD.make_table(w)
    inp = synth.make_inputs(w)
    d = SD.upload_inputs(inp)
    w2 = synth.Workload("second", 1, 16, 4096, seed=9)
    wkv2 = SD.bits_to_device(synth.make_wkv(w2))
    q2, k2 = (SD.bits_to_device(a) for a in synth.make_qk(w2))
    layers = [EngramLayer(table, scale, d["wkv"], d["q"], d["k"], max_tokens=512),
              EngramLayer(table, scale, wkv2, q2, k2, max_tokens=512)]
    yield w, layers, (table, scale, d, wkv2, q2, k2)
    for lay in layers:
        lay.close()


def _step_inputs(w, B, T, seed):
    rng = np.random.default_rng([seed, 21])
    wb = synth.Workload(w.name, B, T, w.prime_base, seed=w.seed)
    lengths, offsets = wb.layout()
    ids = [torch.from_numpy(synth.make_hash_ids(wb, lengths, offsets, rng)).cuda() for _ in range(2)]
    x = SD.bits_to_device(synth.make_x(wb, rng))
    mask = torch.from_numpy((rng.random((B, T)) > 0.1).astype(np.uint8)).cuda()
    return ids, x, mask


@pytest.mark.parametrize("B,T", [(64, 1), (2, 150)])
def test_run_ahead_equals_forward(two_layers, B, T):
    from engram_hashed_gram_gb300.layer import EngramRunAhead
    w, layers, _ = two_layers
    ra = EngramRunAhead(layers, max_tokens=512)
    for step in range(2):
        ids, x, mask = _step_inputs(w, B, T, seed=10 * step + B)
        # reference: the two layers in sequence, each by engram_forward
        ref1 = layers[0].forward(ids[0], x, mask)
        ref2 = layers[1].forward(ids[1], ref1, mask)
        torch.cuda.synchronize()
        # run ahead: projections on the side stream while the main stream sleeps
        ra.issue(ids)
        torch.cuda._sleep(int(2e6))                 # backbone stand-in before layer 1
        out1 = ra.apply(0, x, mask)
        torch.cuda._sleep(int(2e6))                 # layers between the two Engram layers
        out2 = ra.apply(1, out1, mask)
        torch.cuda.synchronize()
        assert torch.equal(out1.view(torch.int16), ref1.view(torch.int16)), f"step {step}: layer 1"
        assert torch.equal(out2.view(torch.int16), ref2.view(torch.int16)), f"step {step}: layer 2"
        for lay in layers:
            assert lay.sync_status()[0] == 0


def test_run_ahead_with_sm_budget(two_layers):
    """With the projections capped at 24 SMs the split-K plan changes (and with
    it kv's summation order); the run-ahead result equals forward under the
    same budget bit for bit, and the budget is restored afterwards."""
    from engram_hashed_gram_gb300.layer import EngramRunAhead
    w, layers, _ = two_layers
    full_plan = layers[0].plan(64)
    ra = EngramRunAhead(layers, max_tokens=512, sm_budget=24)
    assert layers[0].plan(64)[1] <= 24 and layers[0].plan(64) != full_plan
    try:
        ids, x, mask = _step_inputs(w, 64, 1, seed=5)
        ref1 = layers[0].forward(ids[0], x, mask)
        ref2 = layers[1].forward(ids[1], ref1, mask)
        ra.issue(ids)
        torch.cuda._sleep(int(2e6))
        out1 = ra.apply(0, x, mask)
        out2 = ra.apply(1, out1, mask)
        torch.cuda.synchronize()
        assert torch.equal(out1.view(torch.int16), ref1.view(torch.int16))
        assert torch.equal(out2.view(torch.int16), ref2.view(torch.int16))
    finally:
        for lay in layers:
            lay.set_sm_budget(0)
    assert layers[0].plan(64) == full_plan


def test_run_ahead_argument_errors(two_layers):
    from engram_hashed_gram_gb300.layer import EngramRunAhead
    w, layers, _ = two_layers
    ra = EngramRunAhead(layers, max_tokens=32)
    ids, x, _ = _step_inputs(w, 64, 1, seed=3)
    with pytest.raises(ValueError):
        ra.issue(ids)                               # 64 tokens > max_tokens
    with pytest.raises(ValueError):
        ra.issue(ids[:1])                           # one id tensor per layer
    with pytest.raises(RuntimeError):
        EngramRunAhead(layers, max_tokens=32).apply(0, x)   # apply before issue
