"""GPU parity of layer shapes other than V4.1's (dim 5120, 4 streams): the
kernels take dim as any multiple of 256 up to 5120 and 1 to 4 residual
streams.  For each shape, a batch through every plan the library picks --
one CTA with the 4-CTA cluster gate kernel (100 tokens), CTA pairs with the
streaming gate kernel (300), CTA pairs with the gate in the epilogue
(1,200) -- against the oracle on every token, and forward equal to
lookup_project + gate_apply bit for bit."""
import dataclasses

import numpy as np
import pytest
import torch

import parity as P
from engram_hashed_gram_gb300 import synth

pytestmark = pytest.mark.gpu

SHAPES = [(2048, 2), (1280, 3), (512, 1)]


@pytest.fixture(scope="module", params=SHAPES, ids=[f"dim{d}_hc{h}" for d, h in SHAPES])
def shape(request):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from engram_hashed_gram_gb300 import build as B
    B.build()
    from engram_hashed_gram_gb300 import synth_device as SD
    from engram_hashed_gram_gb300.layer import EngramLayer
    dim, hc = request.param
    w = dataclasses.replace(synth.workload("tiny_1x16"), dim=dim, hc_mult=hc, B=1, T=1200, mask="span10")
    table, scale = SD.make_table(w)
    inp = synth.make_inputs(w)
    d = SD.upload_inputs(inp)
    layer = EngramLayer(table, scale, d["wkv"], d["q"], d["k"], dim=dim, hc_mult=hc, max_tokens=w.M, eps=w.eps,
                        scale_block=w.scale_block)
    yield dict(w=w, inp=inp, d=d, SD=SD, layer=layer, keep=(table, scale))
    layer.close()


@pytest.mark.parametrize("T,pairs,fused", [(100, 0, 0), (300, 1, 0), (1200, 1, 1)])
def test_shape_every_plan(shape, T, pairs, fused):
    w, inp, d, SD, layer = shape["w"], shape["inp"], shape["d"], shape["SD"], shape["layer"]
    info = layer.describe_plan(T)
    assert (info["cta_pairs"], info["fused_gate"]) == (pairs, fused)
    ids = d["hash_ids"][:, :T].contiguous()
    x = d["x"][:, :T].contiguous()
    mask = d["mask"][:, :T].contiguous()
    sub = dataclasses.replace(inp, w=dataclasses.replace(w, T=T), hash_ids=inp.hash_ids[:, :T],
                              x=inp.x[:, :T], mask=inp.mask[:, :T])
    out = layer.forward(ids, x, mask)
    kv = layer.lookup_project(ids)
    gates = torch.empty((1, T, w.hc_mult), dtype=torch.float32, device="cuda")
    split = layer.gate_apply(kv, x, mask, gates=gates)
    inplace = x.clone()
    layer.forward(ids, inplace, mask, out=inplace)
    st, _ = layer.sync_status()
    assert st == 0
    assert torch.equal(out.view(torch.int16), split.view(torch.int16))
    assert torch.equal(out.view(torch.int16), inplace.view(torch.int16))
    off = mask == 0
    assert torch.equal(out[off].view(torch.int16), x[off].view(torch.int16))
    summary = P.check_layer(sub.w, sub, np.arange(T), SD.device_bits(out), gates.cpu().numpy(), SD.device_bits(kv),
                            f"dim {w.dim} hc {w.hc_mult} T {T}")
    print(summary)
