"""engram_forward_noalloc, the entry point for callers that cannot allocate
device memory (an engine that owns all of HBM through its own allocator, a
plugin inside a process that owns the GPU's memory budget): it must give the
result of engram_forward within the parity tolerance on two calls in a row,
while its scratch stays in the library's static device array -- no device
memory is taken after its first call on the device.

This file is collected last on purpose, and it sets up everything it needs,
so it passes alone in a fresh process as well as after the other tests."""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from engram_hashed_gram_gb300 import build as B
    B.build()
    from engram_hashed_gram_gb300 import _lib, synth
    from engram_hashed_gram_gb300 import synth_device as SD
    from engram_hashed_gram_gb300.layer import EngramLayer
    w = synth.workload("tiny_1x16")
    table, scale = SD.make_table(w)
    inp = synth.make_inputs(w)
    d = SD.upload_inputs(inp)
    layer = EngramLayer(table, scale, d["wkv"], d["q"], d["k"], max_tokens=_lib.NOALLOC_MAX_TOKENS)
    weights = _lib.EngramWeights(table=table.data_ptr(), scale=scale.data_ptr(), wkv=d["wkv"].data_ptr(),
                                 q_weight=d["q"].data_ptr(), k_weight=d["k"].data_ptr())
    yield dict(w=w, lib=_lib, synth=synth, SD=SD, layer=layer, weights=weights, keep=(table, scale, d))
    layer.close()


def _batch(env, B, T, seed, mask_frac):
    synth = env["synth"]
    w = dataclasses.replace(env["w"], B=B, T=T)
    rng = np.random.default_rng([seed, 7])
    ids = torch.from_numpy(synth.make_hash_ids(w, rng=rng)).cuda()
    x = env["SD"].bits_to_device(synth.make_x(w, rng))
    mask = None
    if mask_frac:
        mask = torch.from_numpy((rng.random((B, T)) >= mask_frac).astype(np.uint8)).cuda()
    return ids, x, mask


def _noalloc(env, ids, x, mask, out):
    B, T = ids.shape[0], ids.shape[1]
    return env["lib"].engram().engram_forward_noalloc(
        ctypes.byref(env["layer"].cfg), ctypes.byref(env["weights"]), ids.data_ptr(), x.data_ptr(),
        None if mask is None else mask.data_ptr(), out.data_ptr(), B, T, torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_forward_on_two_calls_in_a_row(env):
    import parity as P
    SD = env["SD"]
    # a full 64-token batch (the split-K plan), then a smaller masked batch over
    # the scratch the first call left behind
    calls = [_batch(env, 64, 1, 1, 0.0), _batch(env, 2, 9, 2, 0.3)]
    outs = []
    for i, (ids, x, mask) in enumerate(calls):
        out = torch.empty_like(x)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        assert _noalloc(env, ids, x, mask, out) == 0
        torch.cuda.synchronize()
        if i > 0:   # after its first call on the device the entry point takes no device memory
            assert torch.cuda.mem_get_info()[0] == free_before
        outs.append(out)
    for (ids, x, mask), out in zip(calls, outs):
        ref = env["layer"].forward(ids, x, mask)
        torch.cuda.synchronize()
        s = P.compare_out(SD.device_bits(out), SD.device_bits(ref))
        assert s["ok"], s
        if mask is not None:
            off = mask == 0
            assert torch.equal(out[off].view(torch.int16), x[off].view(torch.int16))
    assert env["layer"].sync_status()[0] == 0


def test_noalloc_rejects_batches_beyond_its_scratch(env):
    lib = env["lib"]
    ids, x, _ = _batch(env, 1, lib.NOALLOC_MAX_TOKENS + 1, 3, 0.0)
    out = torch.zeros_like(x)
    assert _noalloc(env, ids, x, None, out) == lib.ENGRAM_EINVAL
    torch.cuda.synchronize()
    assert int(out.view(torch.int16).abs().sum()) == 0     # nothing was queued
