"""GPU parity of the V4.1-native formats through the C ABI, on a small table
(24 prime ranges above 4096): an MXFP8 table (e4m3 codes, one E8M0 scale per
32 channels) with the bf16 weight, and with the MXFP8 weight on the
block-scaled FP8 tensor-core path.  kv is compared element by element with the
oracle within the fp32 dot-product bound, gates and outputs through the
stage-wise check of parity.py; rows and scales bit for bit."""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

from engram_hashed_gram_gb300 import synth
from engram_hashed_gram_gb300 import synth_device as SD
from oracle import engram_oracle as O
import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from engram_hashed_gram_gb300 import build as B
    B.build()
    from engram_hashed_gram_gb300 import _lib
    from engram_hashed_gram_gb300.layer import EngramLayer
    w = synth.workload("tiny_1x16_mxfp8")
    table, scale = SD.make_table(w)
    inp = synth.make_inputs(w)
    dev = SD.upload_inputs(inp)
    kw = dict(scale_block=32, scale_fmt=_lib.SCALE_E8M0, max_tokens=512)
    layer = EngramLayer(table, scale, dev["wkv"], dev["q"], dev["k"], wkv_scale=dev["wkv_scale"], **kw)
    wkv_bf16 = synth.make_wkv(w)
    layer_bf16 = EngramLayer(table, scale, SD.bits_to_device(wkv_bf16), dev["q"], dev["k"], **kw)
    yield dict(w=w, table=table, scale=scale, inp=inp, dev=dev, layer=layer, layer_bf16=layer_bf16,
               wkv_bf16=wkv_bf16, lib=_lib, kw=kw)
    layer.close()
    layer_bf16.close()


def _inputs(mx, B, T, mask_frac=0.0, seed=0, bad_ids=0, bf16_weight=False):
    w = dataclasses.replace(mx["w"], B=B, T=T)
    rng = np.random.default_rng([seed, B, T, 8])
    lengths, offsets = w.layout()
    ids = synth.make_hash_ids(w, lengths, offsets, rng)
    if bad_ids:
        flat = ids.reshape(-1)
        pos = rng.choice(flat.size, size=bad_ids, replace=False)
        flat[pos[0::2]] = -1 - rng.integers(0, 1000, size=pos[0::2].size)
        flat[pos[1::2]] = w.num_rows() + rng.integers(0, 1000, size=pos[1::2].size)
    x = synth.make_x(w, rng)
    mask = None
    if mask_frac > 0:
        mask = (rng.random((B, T)) >= mask_frac).astype(np.uint8)
    base = mx["inp"]
    if bf16_weight:
        inp = synth.HostInputs(w=w, hash_ids=ids, x=x, mask=mask, wkv=mx["wkv_bf16"], q=base.q, k=base.k)
    else:
        inp = synth.HostInputs(w=w, hash_ids=ids, x=x, mask=mask, wkv=base.wkv, q=base.q, k=base.k,
                               wkv_scale=base.wkv_scale)
    return w, inp


def _dev(inp):
    return (torch.from_numpy(inp.hash_ids).cuda(), SD.bits_to_device(inp.x),
            None if inp.mask is None else torch.from_numpy(inp.mask).cuda())


def test_device_e8m0_scales_match_host_twin(mx):
    w = mx["w"]
    R = w.num_rows()
    rows = np.array([0, 1, 17, 4096, R // 2, R - 1])
    codes, scales = synth.table_rows(w.seed, rows, w.head_dim, w.scale_block, scale_fmt=1)
    sel = torch.from_numpy(rows).cuda()
    assert np.array_equal(mx["table"][sel].cpu().numpy(), codes)
    assert np.array_equal(mx["scale"][sel].cpu().numpy(), scales)
    _, s2 = synth.table_rows(w.seed, np.arange(3000, 7000), w.head_dim, w.scale_block, scale_fmt=1)
    assert np.array_equal(mx["scale"][3000:7000].cpu().numpy(), s2)


@pytest.mark.parametrize("B,T", [(1, 16), (3, 61)])
def test_lookup_rows_e8m0_bit_exact(mx, B, T):
    w, inp = _inputs(mx, B, T, bad_ids=4)
    ids, _, _ = _dev(inp)
    rows = mx["layer"].lookup(ids)
    M = B * T
    cids, codes, scales = P.compact_rows(w, inp.hash_ids.reshape(M, -1))
    want = O.lookup(cids, codes, scales, w.scale_block, w.scale_fmt)
    P.assert_bits_equal_nan_aware(SD.device_bits(rows).reshape(M, -1), want, "gathered rows")


def _kv_report(err, bound):
    """Where kv falls outside its bound: counts by 32-row group of the M tile
    and by 128-column group of the N tile (a scale placed in the wrong tensor
    memory lane or column shows up as whole groups)."""
    bad = err > bound
    rows = np.flatnonzero(bad.any(1))
    cols = np.flatnonzero(bad.any(0))
    by_rq = np.bincount((np.arange(bad.shape[0]) % 128) // 32, weights=bad.sum(1), minlength=4)
    by_cq = np.bincount((np.arange(bad.shape[1]) % 256) // 128, weights=bad.sum(0), minlength=2)
    return (f"{int(bad.sum())} of {bad.size} kv outside the bound; rows {rows[:8].tolist()}, cols "
            f"{cols[:8].tolist()}; by row quarter {by_rq.tolist()}, by column half {by_cq.tolist()}")


@pytest.mark.parametrize("budget", [0, 64])
@pytest.mark.parametrize("B,T", [(1, 16), (64, 1), (2, 100), (1, 300), (1, 512)])
def test_fp8_projection_kv(mx, B, T, budget):
    """lookup_project with the MXFP8 weight against the oracle's
    project_mxfp8, element by element (whole-K plans; split-K plans with the
    projection capped at 64 SMs; several M tiles and a ragged tail)."""
    w, inp = _inputs(mx, B, T, bad_ids=2)
    ids, _, _ = _dev(inp)
    layer = mx["layer"]
    layer.set_sm_budget(budget)
    try:
        kv = layer.lookup_project(ids)
        plan = layer.plan(B * T)
        st, _ = layer.sync_status()
    finally:
        layer.set_sm_budget(0)
    assert st == 0
    if budget and B * T <= 128:
        assert plan[0] > 1
    M = B * T
    e = P.oracle_rows(w, inp, np.arange(M))
    ref = O.project_mxfp8(e, inp.wkv, inp.wkv_scale)
    got = O.bf16_value(SD.device_bits(kv).reshape(M, -1))
    bound = P.kv_bound(e, P.weight_values(inp), ref, w.K, splits=8)
    err = np.abs(got - O.bf16_value(ref))
    assert np.all(err <= bound), _kv_report(err, bound)
    print(f"B={B} T={T} plan={plan} kv differing from the oracle: {float((err > 0).mean()):.4f}")


@pytest.mark.parametrize("B,T,mask_frac", [(1, 16, 0.0), (64, 1, 0.2), (3, 70, 0.1), (200, 1, 0.0), (1, 300, 0.1),
                                           (2, 256, 0.05)])
def test_fp8_forward_matches_oracle(mx, B, T, mask_frac):
    w, inp = _inputs(mx, B, T, mask_frac, seed=1)
    ids, x, mask = _dev(inp)
    layer = mx["layer"]
    out = layer.forward(ids, x, mask)
    out_again = layer.forward(ids, x, mask)
    kv = layer.lookup_project(ids)
    gates = torch.empty((B, T, 4), dtype=torch.float32, device="cuda")
    out2 = layer.gate_apply(kv, x, mask, gates=gates)
    st, _ = layer.sync_status()
    assert st == 0
    M = B * T
    summary = P.check_layer(w, inp, np.arange(M), SD.device_bits(out), gates.cpu().numpy(), SD.device_bits(kv),
                            f"fp8 B={B} T={T}")
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16)), "forward vs lookup_project + gate_apply"
    assert torch.equal(out.view(torch.int16), out_again.view(torch.int16)), "run to run"
    if mask is not None:
        off = mask == 0
        assert torch.equal(out[off].view(torch.int16), x[off].view(torch.int16))
    print(f"fp8 B={B} T={T} plan={layer.plan(M)} {summary}")


@pytest.mark.parametrize("B,T,mask_frac", [(1, 16, 0.0), (64, 1, 0.1), (2, 90, 0.0)])
def test_mxfp8_table_with_bf16_weight(mx, B, T, mask_frac):
    """The MXFP8 table through the bf16 path (dequantised rows, bf16 MMA)."""
    w, inp = _inputs(mx, B, T, mask_frac, seed=2, bf16_weight=True)
    ids, x, mask = _dev(inp)
    layer = mx["layer_bf16"]
    out = layer.forward(ids, x, mask)
    kv = layer.lookup_project(ids)
    gates = torch.empty((B, T, 4), dtype=torch.float32, device="cuda")
    layer.gate_apply(kv, x, mask, gates=gates)
    st, _ = layer.sync_status()
    assert st == 0
    M = B * T
    P.check_layer(w, inp, np.arange(M), SD.device_bits(out), gates.cpu().numpy(), SD.device_bits(kv),
                  f"e8m0 table, bf16 weight B={B} T={T}")


def test_fp8_configuration_errors(mx):
    lib = mx["lib"]
    dev = mx["dev"]
    w = mx["w"]
    eng = lib.engram()

    def create(**over):
        cfg = lib.EngramConfig(dim=w.dim, hc_mult=w.hc_mult, n_cols=w.n_cols, head_dim=w.head_dim, scale_block=32,
                               scale_fmt=lib.SCALE_E8M0, num_rows=w.num_rows(), eps=1e-6, clamp=1e-6,
                               max_tokens=16, wkv_fmt=lib.WKV_MXFP8)
        ws = lib.EngramWeights(table=mx["table"].data_ptr(), scale=mx["scale"].data_ptr(),
                               wkv=dev["wkv"].data_ptr(), q_weight=dev["q"].data_ptr(), k_weight=dev["k"].data_ptr(),
                               wkv_scale=dev["wkv_scale"].data_ptr())
        cfg_fields = {f for f, _ in lib.EngramConfig._fields_}
        for k, v in over.items():
            setattr(cfg if k in cfg_fields else ws, k, v)
        h = ctypes.c_void_p()
        rc = eng.engram_create(ctypes.byref(h), ctypes.byref(cfg), ctypes.byref(ws))
        if rc == 0:
            eng.engram_destroy(h)
        return rc, cfg, ws

    assert create()[0] == 0
    assert create(scale_block=128)[0] == lib.ENGRAM_EUNSUPPORTED       # MXFP8 weight needs E8M0 per 32
    assert create(scale_fmt=lib.SCALE_F32)[0] == lib.ENGRAM_EUNSUPPORTED
    assert create(wkv_fmt=7)[0] == lib.ENGRAM_EUNSUPPORTED
    assert create(wkv_scale=None)[0] == lib.ENGRAM_EINVAL
    # the allocation-free entry point keeps to the bf16 weight
    _, cfg, ws = create()
    ids = torch.zeros((1, 1, w.n_cols), dtype=torch.int64, device="cuda")
    x = torch.zeros((1, 1, w.hc_mult, w.dim), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(x)
    rc = eng.engram_forward_noalloc(ctypes.byref(cfg), ctypes.byref(ws), ids.data_ptr(), x.data_ptr(), None,
                                    out.data_ptr(), 1, 1, torch.cuda.current_stream().cuda_stream)
    assert rc == lib.ENGRAM_EUNSUPPORTED


def test_fp8_remainder_split(mx):
    """2,500 tokens with the MXFP8 weight: 20 M tiles x 100 N tiles = 2,000
    tiles on 152 SMs, 24 more than 13 waves, which the plan cuts into K
    ranges (fp32 sums to the workspace, reduced in range order).  Every token
    against the oracle (kv within the dot-product bound, gates and outputs by
    the stage-wise check), and forward equal to lookup_project + gate_apply
    bit for bit."""
    from engram_hashed_gram_gb300.layer import EngramLayer
    dev = mx["dev"]
    B, T = 1, 2500
    layer = EngramLayer(mx["table"], mx["scale"], dev["wkv"], dev["q"], dev["k"], wkv_scale=dev["wkv_scale"],
                        **dict(mx["kw"], max_tokens=2560))
    try:
        info = layer.describe_plan(B * T)
        assert info["cta_pairs"] == 0 and info["rem_tiles"] == 24 and info["rem_splits"] >= 2 and info["fused_gate"] == 0
        w, inp = _inputs(mx, B, T, mask_frac=0.05, seed=3, bad_ids=4)
        ids, x, mask = _dev(inp)
        out = layer.forward(ids, x, mask)
        kv = layer.lookup_project(ids)
        gates = torch.empty((B, T, 4), dtype=torch.float32, device="cuda")
        split = layer.gate_apply(kv, x, mask, gates=gates)
        st, _ = layer.sync_status()
        assert st == 0
        assert torch.equal(out.view(torch.int16), split.view(torch.int16))
        M = B * T
        summary = P.check_layer(w, inp, np.arange(M), SD.device_bits(out), gates.cpu().numpy(), SD.device_bits(kv),
                                "fp8 2500 tokens")
        e = P.oracle_rows(w, inp, np.arange(M))
        ref = O.project_mxfp8(e, inp.wkv, inp.wkv_scale)
        bound = P.kv_bound(e, P.weight_values(inp), ref, w.K, splits=8)
        err = np.abs(O.bf16_value(SD.device_bits(kv).reshape(M, -1)) - O.bf16_value(ref))
        assert np.all(err <= bound), _kv_report(err, bound)
        print(summary)
    finally:
        layer.close()
