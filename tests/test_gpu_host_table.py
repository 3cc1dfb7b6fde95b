"""The host-resident table tier: the table and its scales in pinned host memory,
read in place by the gather kernel over the host link.  On the tiny table
(24 prime ranges above 4096) the rows are checked bit for bit against the
oracle and the whole layer bit for bit against the same layer with the table
in device memory (the same kernels on the same values), for the bf16 and the
MXFP8 formats; host memory the device cannot read is refused at create time,
before any kernel runs."""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

from engram_hashed_gram_gb300 import synth
from engram_hashed_gram_gb300 import synth_device as SD
import parity as P

pytestmark = pytest.mark.gpu


def _setup(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from engram_hashed_gram_gb300 import build as B
    B.build()
    from engram_hashed_gram_gb300.layer import EngramLayer
    w = synth.workload(name)
    inp = synth.make_inputs(w)
    dev = SD.upload_inputs(inp)
    d_table, d_scale = SD.make_table(w)
    h_table, h_scale = SD.make_table(w, host=True)
    kw = dict(scale_block=w.scale_block, scale_fmt=w.scale_fmt, wkv_scale=dev["wkv_scale"], max_tokens=512)
    on_dev = EngramLayer(d_table, d_scale, dev["wkv"], dev["q"], dev["k"], **kw)
    on_host = EngramLayer(h_table, h_scale, dev["wkv"], dev["q"], dev["k"], **kw)
    return dict(w=w, inp=inp, dev=dev, d=(d_table, d_scale), h=(h_table, h_scale), on_dev=on_dev,
                on_host=on_host)


@pytest.fixture(scope="module", params=["tiny_1x16", "tiny_1x16_mxfp8"])
def tier(request):
    s = _setup(request.param)
    yield s
    s["on_dev"].close()
    s["on_host"].close()


def _ids_x_mask(w, B, T, seed, bad_ids=0, mask_frac=0.0):
    w = dataclasses.replace(w, B=B, T=T)
    rng = np.random.default_rng([seed, B, T, 5])
    lengths, offsets = w.layout()
    ids = synth.make_hash_ids(w, lengths, offsets, rng)
    if bad_ids:
        flat = ids.reshape(-1)
        pos = rng.choice(flat.size, size=bad_ids, replace=False)
        flat[pos[0::2]] = -1 - rng.integers(0, 1000, size=pos[0::2].size)
        flat[pos[1::2]] = w.num_rows() + rng.integers(0, 1000, size=pos[1::2].size)
    x = synth.make_x(w, rng)
    mask = (rng.random((B, T)) >= mask_frac).astype(np.uint8) if mask_frac > 0 else None
    return w, ids, x, mask


def test_host_table_holds_the_generator_rows(tier):
    w = tier["w"]
    h_table, h_scale = tier["h"]
    assert not h_table.is_cuda and h_table.is_pinned()
    R = w.num_rows()
    rows = np.array([0, 1, 17, 4096, R // 2, R - 1])
    codes, scales = synth.table_rows(w.seed, rows, w.head_dim, w.scale_block, scale_fmt=w.scale_fmt)
    assert np.array_equal(h_table.numpy()[rows], codes)
    assert np.array_equal(h_scale.numpy()[rows], scales)
    d_table, d_scale = tier["d"]
    assert torch.equal(h_table, d_table.cpu()) and torch.equal(h_scale, d_scale.cpu())


@pytest.mark.parametrize("B,T", [(1, 16), (64, 1), (3, 70)])
def test_rows_from_host_bit_exact(tier, B, T):
    w, ids, x, mask = _ids_x_mask(tier["w"], B, T, seed=1, bad_ids=4)
    rows = tier["on_host"].lookup(torch.from_numpy(ids).cuda())
    M = B * T
    base = tier["inp"]
    inp = synth.HostInputs(w=w, hash_ids=ids, x=x, mask=mask, wkv=base.wkv, q=base.q, k=base.k,
                           wkv_scale=base.wkv_scale)
    P.assert_bits_equal_nan_aware(SD.device_bits(rows).reshape(M, -1), P.oracle_rows(w, inp, np.arange(M)),
                                  "rows from the host table")


@pytest.mark.parametrize("B,T,mask_frac", [(64, 1, 0.0), (1, 16, 0.2), (2, 150, 0.1)])
def test_layer_with_host_table_equals_device_table(tier, B, T, mask_frac):
    w, ids, x, mask = _ids_x_mask(tier["w"], B, T, seed=2, mask_frac=mask_frac)
    ids_d = torch.from_numpy(ids).cuda()
    x_d = SD.bits_to_device(x)
    m_d = None if mask is None else torch.from_numpy(mask).cuda()
    out_h = tier["on_host"].forward(ids_d, x_d, m_d)
    out_d = tier["on_dev"].forward(ids_d, x_d, m_d)
    kv_h = tier["on_host"].lookup_project(ids_d)
    kv_d = tier["on_dev"].lookup_project(ids_d)
    for layer in (tier["on_host"], tier["on_dev"]):
        st, _ = layer.sync_status()
        assert st == 0
    assert torch.equal(kv_h.view(torch.int16), kv_d.view(torch.int16)), "kv"
    assert torch.equal(out_h.view(torch.int16), out_d.view(torch.int16)), "out"


def test_unreadable_host_memory_is_refused():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from engram_hashed_gram_gb300 import build as B
    B.build()
    from engram_hashed_gram_gb300 import _lib
    w = synth.workload("tiny_1x16")
    inp = synth.make_inputs(w)
    dev = SD.upload_inputs(inp)
    d_table, d_scale = SD.make_table(w)
    R = w.num_rows()
    pageable = np.zeros((1024, w.head_dim), dtype=np.uint8)       # ordinary host memory, not registered
    eng = _lib.engram()

    def create(table_ptr, scale_ptr):
        cfg = _lib.EngramConfig(dim=w.dim, hc_mult=w.hc_mult, n_cols=w.n_cols, head_dim=w.head_dim,
                                scale_block=w.scale_block, scale_fmt=_lib.SCALE_F32, num_rows=R, eps=1e-6,
                                clamp=1e-6, max_tokens=16, wkv_fmt=_lib.WKV_BF16)
        ws = _lib.EngramWeights(table=table_ptr, scale=scale_ptr, wkv=dev["wkv"].data_ptr(),
                                q_weight=dev["q"].data_ptr(), k_weight=dev["k"].data_ptr(), wkv_scale=None)
        h = ctypes.c_void_p()
        rc = eng.engram_create(ctypes.byref(h), ctypes.byref(cfg), ctypes.byref(ws))
        if rc == 0:
            eng.engram_destroy(h)
        return rc

    assert create(d_table.data_ptr(), d_scale.data_ptr()) == 0
    assert create(pageable.ctypes.data, d_scale.data_ptr()) == _lib.ENGRAM_EINVAL
    scale_pageable = np.zeros((1024, 2), dtype=np.float32)
    assert create(d_table.data_ptr(), scale_pageable.ctypes.data) == _lib.ENGRAM_EINVAL
