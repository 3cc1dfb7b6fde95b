"""Parity at the benchmark workloads' full sizes, in the launch configuration
the benchmark times (one engram_forward over the whole batch):

  decode_64x1          B=64,   T=1,    25,169,534 rows (6.4 GB)
  prefill_1x4096_zipf  B=1,    T=4096, 402,659,764 rows (103 GB), Zipf ids, 10% masked span
  decode_512x1_skew    B=512,  T=1,    100,667,472 rows (25.8 GB), hot-set ids, near-zero streams
  full_2x8192          B=2,    T=8192, 384,016,682 rows (98.3 GB), 5% masked
  decode_64x1_mxfp8, prefill_1x4096_mxfp8: the decode and prefill shapes with
                       the MXFP8 table (E8M0 per 32) and the MXFP8 weight

The table is filled on the device by the generator's twin; the oracle
regenerates only the rows the batch references.  Every token of every
workload is compared with the oracle element by element, in chunks of
CHUNK tokens: the gathered rows bit for bit, kv within the dot-product bound,
gates and outputs stage by stage (tests/parity.py check_layer).  Properties
checked on the whole batch besides: masked tokens pass through bit for bit,
the fused call equals lookup_project + gate_apply bit for bit, and a second
run is bit-identical."""
import numpy as np
import pytest
import torch

from engram_hashed_gram_gb300 import synth
from engram_hashed_gram_gb300 import synth_device as SD
from oracle import engram_oracle as O
import parity as P

pytestmark = pytest.mark.gpu

CHUNK = 2048   # tokens per oracle pass (bounds the oracle's float64 buffers to a few GB)

WORKLOADS = ["decode_64x1", "prefill_1x4096_zipf", "decode_512x1_skew", "full_2x8192", "decode_64x1_mxfp8",
             "prefill_1x4096_mxfp8"]


@pytest.mark.parametrize("name", WORKLOADS)
def test_workload_parity(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from engram_hashed_gram_gb300 import build as B
    B.build()
    from engram_hashed_gram_gb300.layer import EngramLayer
    w = synth.workload(name)
    M = w.M
    inp = synth.make_inputs(w)
    table, scale = SD.make_table(w)
    d = SD.upload_inputs(inp)
    layer = EngramLayer(table, scale, d["wkv"], d["q"], d["k"], max_tokens=M, eps=w.eps, scale_block=w.scale_block,
                        scale_fmt=w.scale_fmt, wkv_scale=d["wkv_scale"])
    try:
        ids, x, mask = d["hash_ids"], d["x"], d["mask"]
        out = layer.forward(ids, x, mask)
        out_again = layer.forward(ids, x, mask)
        kv = layer.lookup_project(ids)
        gates = torch.empty((w.B, w.T, w.hc_mult), dtype=torch.float32, device="cuda")
        out_split = layer.gate_apply(kv, x, mask, gates=gates)
        st, _ = layer.sync_status()
        assert st == 0
        assert torch.equal(out.view(torch.int16), out_again.view(torch.int16)), "run-to-run"
        assert torch.equal(out.view(torch.int16), out_split.view(torch.int16)), "fused vs split"
        if mask is not None:
            off = mask == 0
            assert int(off.sum()) > 0
            assert torch.equal(out[off].view(torch.int16), x[off].view(torch.int16)), "masked pass-through"
            assert torch.all(gates[off] == 0)

        # every token against the oracle, CHUNK tokens at a time
        out_h = SD.device_bits(out.reshape(M, w.hc_mult, w.dim))
        gates_h = gates.reshape(M, w.hc_mult).cpu().numpy()
        kv_h = SD.device_bits(kv.reshape(M, -1))
        del kv
        rows_h = SD.device_bits(layer.lookup(ids).reshape(M, -1))
        worst = {"max_err": 0.0, "rel_l2": 0.0, "pairs_gate_over_tol": 0, "pairs": 0}
        for c0 in range(0, M, CHUNK):
            tok = np.arange(c0, min(M, c0 + CHUNK))
            P.assert_bits_equal_nan_aware(rows_h[tok], P.oracle_rows(w, inp, tok), f"{name} rows {c0}")
            summary = P.check_layer(w, inp, tok, out_h[tok], gates_h[tok], kv_h[tok], f"{name} tokens {c0}..")
            e2e = summary["end_to_end"]
            worst["max_err"] = max(worst["max_err"], e2e["max_err"])
            worst["rel_l2"] = max(worst["rel_l2"], e2e["rel_l2"])
            worst["pairs_gate_over_tol"] += summary["pairs_gate_over_tol"]
            worst["pairs"] += summary["pairs"]
        print(f"{name}: all {M} tokens, plan={layer.plan(M)}, {worst}")
    finally:
        layer.close()
        del table, scale, d
        torch.cuda.empty_cache()
