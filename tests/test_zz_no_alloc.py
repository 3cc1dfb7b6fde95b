"""engram_forward_noalloc, the entry point for callers that cannot allocate
device memory (an engine that owns all of HBM through its own allocator, a
plugin inside a process that owns the GPU's memory budget).

It must give the layer's result on two calls in a row while its scratch stays
in the library's static device array -- no device memory is taken after its
first call on the device.  Each call is checked three ways:
  * bit for bit against engram_forward on a context (the two entry points run
    the same kernels with the same plan);
  * against the oracle, stage by stage (tests/parity.py check_layer), with the
    context's kv and gates -- the same bits the allocation-free call formed
    internally -- explaining the kv-induced part of the difference;
  * masked tokens pass through bit for bit.
Two shapes: the V4.1 shape (dim 5120: 100 N tiles, whole-K tiles, bf16 kv in
the scratch) and dim 512 (10 N tiles: the split-K plan, fp32 partial sums in
the scratch, the gate summing them).

This file is collected last on purpose, and it sets up everything it needs,
so it passes alone in a fresh process as well as after the other tests."""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _setup(w):
    from engram_hashed_gram_gb300 import _lib, synth
    from engram_hashed_gram_gb300 import synth_device as SD
    from engram_hashed_gram_gb300.layer import EngramLayer
    table, scale = SD.make_table(w)
    inp = synth.make_inputs(w)
    d = SD.upload_inputs(inp)
    layer = EngramLayer(table, scale, d["wkv"], d["q"], d["k"], dim=w.dim, max_tokens=_lib.NOALLOC_MAX_TOKENS)
    weights = _lib.EngramWeights(table=table.data_ptr(), scale=scale.data_ptr(), wkv=d["wkv"].data_ptr(),
                                 q_weight=d["q"].data_ptr(), k_weight=d["k"].data_ptr())
    return dict(w=w, inp=inp, layer=layer, weights=weights, keep=(table, scale, d))


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from engram_hashed_gram_gb300 import build as B
    B.build()
    from engram_hashed_gram_gb300 import _lib, synth
    from engram_hashed_gram_gb300 import synth_device as SD
    tiny = synth.workload("tiny_1x16")
    shapes = {"v41": _setup(tiny), "dim512": _setup(dataclasses.replace(tiny, dim=512))}
    yield dict(lib=_lib, synth=synth, SD=SD, shapes=shapes)
    for s in shapes.values():
        s["layer"].close()


def _batch(env, shape, B, T, seed, mask_frac):
    """Device ids, x, mask of a fresh batch, and its host inputs for the oracle."""
    synth, SD = env["synth"], env["SD"]
    sh = env["shapes"][shape]
    w = dataclasses.replace(sh["w"], B=B, T=T)
    rng = np.random.default_rng([seed, 7])
    ids_h = synth.make_hash_ids(w, rng=rng)
    x_h = synth.make_x(w, rng)
    mask_h = (rng.random((B, T)) >= mask_frac).astype(np.uint8) if mask_frac else None
    inp = dataclasses.replace(sh["inp"], w=w, hash_ids=ids_h, x=x_h, mask=mask_h)
    ids = torch.from_numpy(ids_h).cuda()
    x = SD.bits_to_device(x_h)
    mask = None if mask_h is None else torch.from_numpy(mask_h).cuda()
    return ids, x, mask, inp


def _noalloc(env, shape, ids, x, mask, out, weights=None):
    sh = env["shapes"][shape]
    B, T = ids.shape[0], ids.shape[1]
    return env["lib"].engram().engram_forward_noalloc(
        ctypes.byref(sh["layer"].cfg), ctypes.byref(sh["weights"] if weights is None else weights), ids.data_ptr(),
        x.data_ptr(), None if mask is None else mask.data_ptr(), out.data_ptr(), B, T,
        torch.cuda.current_stream().cuda_stream)


def _two_calls_in_a_row(env, shape, batches, expect_plan):
    import parity as P
    SD = env["SD"]
    layer = env["shapes"][shape]["layer"]
    calls = [_batch(env, shape, *b) for b in batches]
    outs = []
    for i, (ids, x, mask, _) in enumerate(calls):
        assert layer.plan(ids.shape[0] * ids.shape[1]) == expect_plan
        out = torch.empty_like(x)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        assert _noalloc(env, shape, ids, x, mask, out) == 0
        torch.cuda.synchronize()
        if i > 0:   # after its first call on the device the entry point takes no device memory
            assert torch.cuda.mem_get_info()[0] == free_before
        outs.append(out)
    for (ids, x, mask, inp), out in zip(calls, outs):
        M = ids.shape[0] * ids.shape[1]
        ref = layer.forward(ids, x, mask)
        kv = layer.lookup_project(ids)
        gates = torch.empty((ids.shape[0], ids.shape[1], inp.w.hc_mult), dtype=torch.float32, device="cuda")
        layer.gate_apply(kv, x, mask, gates=gates)
        torch.cuda.synchronize()
        # the same kernels and plan as the context's forward: the same bits
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"{shape}: noalloc vs engram_forward"
        if mask is not None:
            off = mask == 0
            assert int(off.sum()) > 0
            assert torch.equal(out[off].view(torch.int16), x[off].view(torch.int16))
        summary = P.check_layer(inp.w, inp, np.arange(M), SD.device_bits(out), gates.cpu().numpy(),
                                SD.device_bits(kv), f"noalloc {shape}")
        print(f"noalloc {shape} {M} tokens: {summary['end_to_end']}")
    assert layer.sync_status()[0] == 0


def test_noalloc_matches_forward_and_oracle_v41_shape(env):
    # a full 64-token batch, then a smaller masked batch over the scratch the
    # first call left behind; at dim 5120 both take whole-K tiles on 100 CTAs
    _two_calls_in_a_row(env, "v41", [(64, 1, 1, 0.0), (2, 9, 2, 0.3)], (1, 100))


def test_noalloc_matches_forward_and_oracle_split_k(env):
    # dim 512: 10 N tiles fill too little of the grid, so both entry points cut
    # K into 8 ranges and the gate kernel sums the fp32 partials in the scratch
    _two_calls_in_a_row(env, "dim512", [(48, 1, 3, 0.0), (37, 1, 4, 0.25)], (8, 80))


def test_noalloc_rejects_batches_beyond_its_scratch(env):
    lib = env["lib"]
    ids, x, _, _ = _batch(env, "v41", 1, lib.NOALLOC_MAX_TOKENS + 1, 3, 0.0)
    out = torch.zeros_like(x)
    assert _noalloc(env, "v41", ids, x, None, out) == lib.ENGRAM_EINVAL
    torch.cuda.synchronize()
    assert int(out.view(torch.int16).abs().sum()) == 0     # nothing was queued


def test_noalloc_rejects_a_table_the_device_cannot_read(env):
    """A pageable host table (plain numpy memory) is refused before anything
    is queued: no kernel ever dereferences it."""
    lib = env["lib"]
    sh = env["shapes"]["v41"]
    host_table = np.zeros((sh["w"].num_rows(), sh["w"].head_dim), dtype=np.uint8)
    bad = lib.EngramWeights(table=host_table.ctypes.data, scale=sh["weights"].scale, wkv=sh["weights"].wkv,
                            q_weight=sh["weights"].q_weight, k_weight=sh["weights"].k_weight)
    ids, x, _, _ = _batch(env, "v41", 4, 1, 5, 0.0)
    out = torch.zeros_like(x)
    assert _noalloc(env, "v41", ids, x, None, out, weights=bad) == lib.ENGRAM_EINVAL
    torch.cuda.synchronize()
    assert int(out.view(torch.int16).abs().sum()) == 0
