"""GPU parity of the CUDA path against the oracle, through the C ABI, on the
tiny table (24 prime ranges above 4096, 100,776 rows): shapes that span one
and several 128-token tiles with ragged tails, the whole-K decode plan, the
split-K plan (under an SM budget), the single-pass plans on one CTA and on
CTA pairs, masks, in-place calls, out-of-range ids and argument errors."""
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
def tiny():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from engram_hashed_gram_gb300 import build as B
    B.build()
    from engram_hashed_gram_gb300.layer import EngramLayer
    w = synth.workload("tiny_1x16")
    table, scale = SD.make_table(w)
    inp = synth.make_inputs(w)
    dev = SD.upload_inputs(inp)
    layer = EngramLayer(table, scale, dev["wkv"], dev["q"], dev["k"], max_tokens=1024)
    yield dict(w=w, table=table, scale=scale, inp=inp, dev=dev, layer=layer)
    layer.close()


def _inputs(tiny, B, T, mask_frac=0.0, seed=0, bad_ids=0):
    w = dataclasses.replace(tiny["w"], B=B, T=T)
    rng = np.random.default_rng([seed, B, T])
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
    inp = synth.HostInputs(w=w, hash_ids=ids, x=x, mask=mask, wkv=tiny["inp"].wkv, q=tiny["inp"].q,
                           k=tiny["inp"].k)
    return w, inp


def _dev(inp):
    return (torch.from_numpy(inp.hash_ids).cuda(), SD.bits_to_device(inp.x),
            None if inp.mask is None else torch.from_numpy(inp.mask).cuda())


def test_device_table_matches_host_twin(tiny):
    w = tiny["w"]
    R = w.num_rows()
    rows = np.array([0, 1, 2, 17, 4095, 4096, R // 2, R - 2, R - 1])
    codes, scales = synth.table_rows(w.seed, rows)
    got_c = tiny["table"][torch.from_numpy(rows).cuda()].cpu().numpy()
    got_s = tiny["scale"][torch.from_numpy(rows).cuda()].cpu().numpy()
    assert np.array_equal(got_c, codes)
    assert np.array_equal(got_s.view(np.uint32), scales.view(np.uint32))
    # a whole chunk, bit for bit
    c2, s2 = synth.table_rows(w.seed, np.arange(5000, 9000))
    assert np.array_equal(tiny["table"][5000:9000].cpu().numpy(), c2)
    assert np.array_equal(tiny["scale"][5000:9000].cpu().numpy().view(np.uint32), s2.view(np.uint32))


@pytest.mark.parametrize("B,T", [(1, 16), (3, 61), (1, 1), (200, 1)])
def test_lookup_rows_bit_exact(tiny, B, T):
    w, inp = _inputs(tiny, B, T, bad_ids=6)
    ids, _, _ = _dev(inp)
    rows = tiny["layer"].lookup(ids)
    st, bad = tiny["layer"].sync_status()
    assert st == 0 and bad == 0          # check_ids is off: no error, zero rows
    M = B * T
    cids, codes, scales = P.compact_rows(w, inp.hash_ids.reshape(M, -1))
    want = O.lookup(cids, codes, scales, w.scale_block)
    P.assert_bits_equal_nan_aware(SD.device_bits(rows).reshape(M, -1), want, "gathered rows")


@pytest.mark.parametrize("B,T,mask_frac", [(1, 16, 0.0), (1, 1, 0.0), (64, 1, 0.0), (2, 100, 0.1),
                                           (3, 61, 0.3), (300, 1, 0.05)])
def test_forward_matches_oracle(tiny, B, T, mask_frac):
    w, inp = _inputs(tiny, B, T, mask_frac)
    ids, x, mask = _dev(inp)
    layer = tiny["layer"]
    out = layer.forward(ids, x, mask)
    kv = layer.lookup_project(ids)
    gates = torch.empty((B, T, 4), dtype=torch.float32, device="cuda")
    out2 = layer.gate_apply(kv, x, mask, gates=gates)
    st, _ = layer.sync_status()
    assert st == 0
    M = B * T
    summary = P.check_layer(w, inp, np.arange(M), SD.device_bits(out), gates.cpu().numpy(),
                            SD.device_bits(kv), f"B={B} T={T}")
    # fused == lookup_project + gate_apply, bit for bit
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    print(f"B={B} T={T} plan={layer.plan(M)} {summary}")


def test_masked_tokens_pass_through_bitwise_in_place(tiny):
    w, inp = _inputs(tiny, 4, 50, mask_frac=0.5, seed=3)
    inp.mask[0, 0] = 0
    ids, x, mask = _dev(inp)
    x0 = x.clone()
    x[0, 0, 1, :7] = -0.0
    x0[0, 0, 1, :7] = -0.0
    out = tiny["layer"].forward(ids, x, mask, out=x)      # in place
    torch.cuda.synchronize()
    off = mask == 0
    assert int(off.sum()) > 0
    assert torch.equal(out[off].view(torch.int16), x0[off].view(torch.int16))
    assert not torch.equal(out[~off].view(torch.int16), x0[~off].view(torch.int16))


def test_deterministic_bitwise(tiny):
    w, inp = _inputs(tiny, 2, 130, mask_frac=0.1, seed=4)
    ids, x, mask = _dev(inp)
    a = tiny["layer"].forward(ids, x, mask)
    b = tiny["layer"].forward(ids, x, mask)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    w2, inp2 = _inputs(tiny, 64, 1, seed=5)
    ids2, x2, _ = _dev(inp2)
    c = tiny["layer"].forward(ids2, x2)
    d = tiny["layer"].forward(ids2, x2)
    assert torch.equal(c.view(torch.int16), d.view(torch.int16))


def test_check_ids_reports_range_errors(tiny):
    from engram_hashed_gram_gb300.layer import EngramLayer
    dev = tiny["dev"]
    layer = EngramLayer(tiny["table"], tiny["scale"], dev["wkv"], dev["q"], dev["k"], max_tokens=64,
                        check_ids=True)
    w, inp = _inputs(tiny, 2, 8, bad_ids=5, seed=6)
    ids, x, _ = _dev(inp)
    rows = layer.lookup(ids)
    st, bad = layer.sync_status()
    assert st == -4 and bad == 5
    st, bad = layer.sync_status()
    assert st == 0 and bad == 0           # cleared
    flat = inp.hash_ids.reshape(-1)
    zero = (flat < 0) | (flat >= w.num_rows())
    r = SD.device_bits(rows).reshape(-1, 256)
    assert np.all(r[zero] == 0) and np.any(r[~zero] != 0)
    layer.forward(ids, x)
    st, bad = layer.sync_status()
    assert st == -4 and bad == 5
    layer.close()


def test_argument_errors_queue_nothing(tiny):
    import ctypes
    from engram_hashed_gram_gb300 import _lib
    lib = _lib.engram()
    ctx = tiny["layer"]._ctx
    w, inp = _inputs(tiny, 1, 4)
    ids, x, _ = _dev(inp)
    out = torch.empty_like(x)
    s = torch.cuda.current_stream().cuda_stream
    assert lib.engram_forward(None, ids.data_ptr(), x.data_ptr(), None, out.data_ptr(), 1, 4, s) == -1
    assert lib.engram_forward(ctx, None, x.data_ptr(), None, out.data_ptr(), 1, 4, s) == -1
    assert lib.engram_forward(ctx, ids.data_ptr(), x.data_ptr() + 2, None, out.data_ptr(), 1, 4, s) == -1
    assert lib.engram_forward(ctx, ids.data_ptr(), x.data_ptr(), None, out.data_ptr(), 1, 1025, s) == -1
    assert lib.engram_forward(ctx, ids.data_ptr(), x.data_ptr(), None, out.data_ptr(), -1, 4, s) == -1
    assert lib.engram_forward(ctx, ids.data_ptr(), x.data_ptr(), None, out.data_ptr(), 0, 4, s) == 0
    # an unsupported shape is refused at create
    cfg = _lib.EngramConfig(dim=5000, hc_mult=4, n_cols=24, head_dim=256, scale_block=128, scale_fmt=0,
                            num_rows=10, eps=1e-6, clamp=1e-6, max_tokens=8, check_ids=0)
    wt = _lib.EngramWeights(table=tiny["table"].data_ptr(), scale=tiny["scale"].data_ptr(),
                            wkv=tiny["dev"]["wkv"].data_ptr(), q_weight=tiny["dev"]["q"].data_ptr(),
                            k_weight=tiny["dev"]["k"].data_ptr())
    h = ctypes.c_void_p()
    assert lib.engram_create(ctypes.byref(h), ctypes.byref(cfg), ctypes.byref(wt)) == -6
    assert tiny["layer"].sync_status()[0] == 0


def test_empty_batch_is_a_no_op(tiny):
    layer = tiny["layer"]
    ids = torch.empty((0, 5, 24), dtype=torch.int64, device="cuda")
    x = torch.empty((0, 5, 4, 5120), dtype=torch.bfloat16, device="cuda")
    out = layer.forward(ids, x)
    assert out.shape == x.shape
    assert layer.sync_status()[0] == 0


@pytest.mark.parametrize("B,T,mask_frac", [(1, 150, 0.1), (300, 1, 0.0), (7, 100, 0.3), (64, 1, 0.2), (1, 16, 0.0),
                                           (1, 2300, 0.1), (3, 1400, 0.05)])
def test_fused_epilogue_matches_split_path(tiny, B, T, mask_frac):
    """fuse_gate: the gate and residual add run in the projection's epilogue
    (plans without split-K); the result must equal lookup_project + gate_apply
    bit for bit, and match the oracle.  Below 256 tokens the one-CTA kernel
    runs it, from 256 on the CTA-pair kernel (300 and 4,200 tokens: an odd
    number of M tiles, so the last pair's second CTA holds no rows).  2,300
    and 4,200 tokens span 18 and 33 M tiles: several groups of 16 M tiles (8
    pairs) in the fused unit order (key tiles of a group, then the value
    tiles of the group before), the last one partial."""
    from engram_hashed_gram_gb300.layer import EngramLayer
    dev = tiny["dev"]
    fused = EngramLayer(tiny["table"], tiny["scale"], dev["wkv"], dev["q"], dev["k"], max_tokens=4200,
                        fuse_gate=True)
    w, inp = _inputs(tiny, B, T, mask_frac, seed=21)
    ids, x, mask = _dev(inp)
    out = fused.forward(ids, x, mask)
    again = fused.forward(ids, x, mask)
    kv = fused.lookup_project(ids)
    gates = torch.empty((B, T, 4), dtype=torch.float32, device="cuda")
    split = fused.gate_apply(kv, x, mask, gates=gates)
    inplace = x.clone()
    fused.forward(ids, inplace, mask, out=inplace)
    assert fused.sync_status()[0] == 0
    assert fused.plan(B * T)[0] == 1                      # the fused epilogue needs a plan without split-K
    info = fused.describe_plan(B * T)
    assert info["fused_gate"] == 1 and info["rem_splits"] == 0
    assert info["cta_pairs"] == (1 if B * T >= 256 else 0)
    assert torch.equal(out.view(torch.int16), split.view(torch.int16))
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))
    assert torch.equal(out.view(torch.int16), inplace.view(torch.int16))
    M = B * T
    P.check_layer(w, inp, np.arange(M), SD.device_bits(out), gates.cpu().numpy(), SD.device_bits(kv), "fused")
    fused.close()


def test_stream_gate_kernel_matches_cluster_kernel(tiny):
    """Batches of 256 tokens and more take the persistent streaming gate
    kernel (one CTA per SM, several tokens each), smaller ones the 4-CTA
    cluster kernel; both form the sums in the same order, so the same tokens
    give the same bits either way."""
    w, inp = _inputs(tiny, 2, 512, mask_frac=0.1, seed=4)
    ids, x, mask = _dev(inp)
    layer = tiny["layer"]
    kv = layer.lookup_project(ids)
    g_stream = torch.empty((2, 512, 4), dtype=torch.float32, device="cuda")
    out_stream = layer.gate_apply(kv, x, mask, gates=g_stream)              # 1024 tokens
    outs, gs = [], []
    for b in range(2):
        for t0 in range(0, 512, 128):                                      # 128 tokens per call
            sl = (slice(b, b + 1), slice(t0, t0 + 128))
            g = torch.empty((1, 128, 4), dtype=torch.float32, device="cuda")
            outs.append(layer.gate_apply(kv[sl].contiguous(), x[sl].contiguous(), mask[sl].contiguous(), gates=g))
            gs.append(g)
    st, _ = layer.sync_status()
    assert st == 0
    assert torch.equal(out_stream.view(torch.int16),
                       torch.cat(outs, dim=1).reshape(2, 512, 4, -1).view(torch.int16))
    assert torch.equal(g_stream.view(torch.int32), torch.cat(gs, dim=1).reshape(2, 512, 4).view(torch.int32))
    # in place: out may be x
    x2 = x.clone()
    layer.gate_apply(kv, x2, mask, out=x2)
    st, _ = layer.sync_status()
    assert st == 0
    assert torch.equal(x2.view(torch.int16), out_stream.view(torch.int16))
    summary = P.check_layer(w, inp, np.arange(1024), SD.device_bits(out_stream), g_stream.cpu().numpy(),
                            SD.device_bits(kv), "streaming gate 1024 tokens")
    print(summary)


@pytest.mark.parametrize("T", [200, 600])
def test_bounded_wait_runs_out_and_the_context_recovers(tiny, T):
    """Failure detection without a fault: with the test hook, the fused
    epilogue never raises its gates-ready flags, the value tiles' bounded wait
    (two seconds) runs out, every role of the projection leaves its loop, and
    engram_sync_status() reports ENGRAM_ETIMEOUT.  The next call on the same
    context is correct again (equal to its lookup_project + gate_apply).
    200 tokens run the one-CTA kernel, 600 the CTA-pair kernel."""
    import time
    from engram_hashed_gram_gb300 import _lib
    from engram_hashed_gram_gb300.layer import EngramLayer
    w, inp = _inputs(tiny, 1, T, seed=6)
    ids, x, _ = _dev(inp)
    dev = tiny["dev"]
    fused = EngramLayer(tiny["table"], tiny["scale"], dev["wkv"], dev["q"], dev["k"], max_tokens=T, fuse_gate=True)
    try:
        assert fused.plan(T)[0] == 1                         # single pass: the fused epilogue runs
        assert fused.describe_plan(T)["cta_pairs"] == (1 if T >= 256 else 0)
        assert _lib.engram().engram_test_hook(fused._ctx, _lib.TEST_HOLD_GATE_FLAGS) == 0
        t0 = time.perf_counter()
        fused.forward(ids, x)
        st, _ = fused.sync_status()
        elapsed = time.perf_counter() - t0
        assert st == _lib.ENGRAM_ETIMEOUT, st
        assert elapsed < 20.0
        assert _lib.engram().engram_test_hook(fused._ctx, 0) == 0
        out = fused.forward(ids, x)
        st, _ = fused.sync_status()
        assert st == 0
        ref = fused.gate_apply(fused.lookup_project(ids), x)     # the same plan through the separate kernels
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    finally:
        fused.close()


@pytest.mark.parametrize("budget", [48, 96])
def test_split_k_plans(tiny, budget):
    """Decode batches on all SMs take whole-K tiles; with the projection capped
    at fewer SMs than tiles the plan cuts K (fp32 partial sums, summed by the
    gate kernel and by lookup_project's reduction).  Those plans against the
    oracle, and forward against lookup_project + gate_apply bit for bit."""
    layer = tiny["layer"]
    assert layer.plan(64)[0] == 1
    layer.set_sm_budget(budget)
    try:
        for B, T in [(64, 1), (1, 16), (3, 37)]:
            M = B * T
            splits, ctas = layer.plan(M)
            assert splits > 1 and ctas <= budget
            w, inp = _inputs(tiny, B, T, mask_frac=0.1, seed=9)
            ids, x, mask = _dev(inp)
            out = layer.forward(ids, x, mask)
            kv = layer.lookup_project(ids)
            gates = torch.empty((B, T, 4), dtype=torch.float32, device="cuda")
            split = layer.gate_apply(kv, x, mask, gates=gates)
            assert layer.sync_status()[0] == 0
            assert torch.equal(out.view(torch.int16), split.view(torch.int16))
            summary = P.check_layer(w, inp, np.arange(M), SD.device_bits(out), gates.cpu().numpy(),
                                    SD.device_bits(kv), f"split-K {splits} B={B} T={T}")
            print(f"budget {budget}: B={B} T={T} plan={(splits, ctas)} {summary}")
    finally:
        layer.set_sm_budget(0)
    assert layer.plan(64)[0] == 1


def test_remainder_split_tiles(tiny):
    """1,300 tokens make 11 x 100 = 1,100 output tiles: with the projection
    held to 137 SMs (so that the one-CTA kernel runs), eight full waves and 4
    tiles left over, which the plan cuts into four K ranges each (their fp32
    sums reduced in range order by a separate kernel).  Those tiles hold
    the value columns of every token; every token is checked against the
    oracle, and forward equals lookup_project + gate_apply bit for bit."""
    from engram_hashed_gram_gb300.layer import EngramLayer
    dev = tiny["dev"]
    layer = EngramLayer(tiny["table"], tiny["scale"], dev["wkv"], dev["q"], dev["k"], max_tokens=1408)
    try:
        w, inp = _inputs(tiny, 2, 650, mask_frac=0.05, seed=8)
        ids, x, mask = _dev(inp)
        out = layer.forward(ids, x, mask)
        kv = layer.lookup_project(ids)
        gates = torch.empty((2, 650, 4), dtype=torch.float32, device="cuda")
        split = layer.gate_apply(kv, x, mask, gates=gates)
        assert layer.sync_status()[0] == 0
        # on all SMs this batch takes CTA pairs (whole 256 x 256 tiles) with the
        # gate in their epilogue; on 137 SMs the one-CTA plan with the separate
        # gate kernel cuts the 4 tiles of its last wave into K ranges
        assert layer.plan(1300) == (1, 152)
        assert layer.forward_kernels(1300) == 2
        assert torch.equal(out.view(torch.int16), split.view(torch.int16))
        layer.set_sm_budget(137)
        assert layer.plan(1300) == (1, 137)
        # gather, projection, the remainder's sums, gate; no remainder at 1,233 tokens (9 full waves)
        assert layer.forward_kernels(1300) == 4
        assert layer.forward_kernels(1233) == 3
        assert layer.forward_kernels(64) == 3 and layer.forward_kernels(0) == 0
        out = layer.forward(ids, x, mask)
        kv = layer.lookup_project(ids)
        split = layer.gate_apply(kv, x, mask, gates=gates)
        assert layer.sync_status()[0] == 0
        assert torch.equal(out.view(torch.int16), split.view(torch.int16))
        M = 1300
        summary = P.check_layer(w, inp, np.arange(M), SD.device_bits(out.reshape(M, 4, -1)),
                                gates.reshape(M, 4).cpu().numpy(), SD.device_bits(kv.reshape(M, -1)),
                                "remainder split")
        print(summary)
    finally:
        layer.close()


@pytest.mark.parametrize("B,T", [(1, 256), (3, 100), (1, 1000), (1, 1750)])
def test_cta_pair_projection(tiny, B, T):
    """From 256 tokens on, the projection runs on CTA pairs (tcgen05
    cta_group::2, 256 x 256 tiles; 300 tokens leave the odd CTA of the last
    pair without a row of the batch; 1,750 tokens make 700 pair tiles, 16 more
    than 9 waves of 76 pairs, which the plan cuts into K ranges).  Held to 150
    SMs the same batch takes the one-CTA kernel: both are checked against the
    oracle on every token, and their kv agree within the dot-product bound.
    (The separate gate kernel throughout: the fused epilogue has its own tests.)"""
    from engram_hashed_gram_gb300.layer import EngramLayer
    w, inp = _inputs(tiny, B, T, mask_frac=0.1, seed=12)
    ids, x, mask = _dev(inp)
    dev = tiny["dev"]
    layer = EngramLayer(tiny["table"], tiny["scale"], dev["wkv"], dev["q"], dev["k"], max_tokens=2048,
                        fuse_gate=False)
    M = B * T
    if M == 1750:
        assert layer.forward_kernels(M) == 4           # gather, pairs, the remainder's sums, gate
    res = {}
    try:
        for budget in (0, 150):
            layer.set_sm_budget(budget)
            out = layer.forward(ids, x, mask)
            kv = layer.lookup_project(ids)
            gates = torch.empty((B, T, 4), dtype=torch.float32, device="cuda")
            split = layer.gate_apply(kv, x, mask, gates=gates)
            assert layer.sync_status()[0] == 0
            assert torch.equal(out.view(torch.int16), split.view(torch.int16))
            P.check_layer(w, inp, np.arange(M), SD.device_bits(out), gates.cpu().numpy(), SD.device_bits(kv),
                          f"budget {budget}")
            res[budget] = SD.device_bits(kv).reshape(M, -1)
        layer.set_sm_budget(0)
        assert layer.plan(M) == (1, 152)
    finally:
        layer.close()
    rows = P.oracle_rows(w, inp, np.arange(M))
    bound = P.kv_bound(rows, P.weight_values(inp), res[150], w.K)
    diff = np.abs(O.bf16_value(res[0]) - O.bf16_value(res[150]))
    assert np.all(diff <= 2 * bound)
    print(f"{M} tokens: pair vs one-CTA kv identical in {float((diff == 0).mean()):.6f} of the elements")


def test_library_choice_fuses_large_batches_on_pairs(tiny):
    """fuse_gate left to the library: from 1,024 tokens on, with all SMs, the
    gate and the residual add run in the CTA-pair projection's epilogue (two
    kernels per forward); below that, or held to fewer SMs, the separate gate
    kernel.  The fused forward equals lookup_project + gate_apply bit for bit
    and matches the oracle on every token."""
    from engram_hashed_gram_gb300.layer import EngramLayer
    dev = tiny["dev"]
    layer = EngramLayer(tiny["table"], tiny["scale"], dev["wkv"], dev["q"], dev["k"], max_tokens=2048)
    try:
        assert layer.describe_plan(512)["fused_gate"] == 0 and layer.describe_plan(512)["cta_pairs"] == 1
        info = layer.describe_plan(1200)
        assert info["fused_gate"] == 1 and info["cta_pairs"] == 1 and info["rem_splits"] == 0
        assert layer.forward_kernels(1200) == 2
        layer.set_sm_budget(150)
        assert layer.describe_plan(1200)["fused_gate"] == 0 and layer.describe_plan(1200)["cta_pairs"] == 0
        layer.set_sm_budget(0)
        B, T = 2, 600
        w, inp = _inputs(tiny, B, T, mask_frac=0.1, seed=31)
        ids, x, mask = _dev(inp)
        out = layer.forward(ids, x, mask)
        kv = layer.lookup_project(ids)
        gates = torch.empty((B, T, 4), dtype=torch.float32, device="cuda")
        split = layer.gate_apply(kv, x, mask, gates=gates)
        assert layer.sync_status()[0] == 0
        assert torch.equal(out.view(torch.int16), split.view(torch.int16))
        P.check_layer(w, inp, np.arange(B * T), SD.device_bits(out), gates.cpu().numpy(), SD.device_bits(kv),
                      "library choice, 1200 tokens")
    finally:
        layer.close()


def test_stage_timing_over_a_run_of_calls(tiny):
    """engram_enable_stage_timing(ctx, n) keeps the stage events of the last n
    calls: after five forwards with n = 3, stage_times_n(3) gives three
    (gather, projection, gate) triples of positive durations, the last equal
    to stage_times(); asking for more calls than remembered is refused."""
    from engram_hashed_gram_gb300._lib import EngramError
    layer = tiny["layer"]
    w, inp = _inputs(tiny, 1, 300, seed=14)
    ids, x, mask = _dev(inp)
    layer.enable_stage_timing(True, calls=3)
    try:
        with pytest.raises(EngramError):
            layer.stage_times_n(1)                       # nothing timed yet
        for _ in range(5):
            layer.forward(ids, x, mask)
        runs = layer.stage_times_n(3)
        last = layer.stage_times()
        assert len(runs) == 3 and runs[-1] == last
        assert all(g > 0 and p > 0 and t > 0 for g, p, t in runs)
        with pytest.raises(EngramError):
            layer.stage_times_n(4)
    finally:
        layer.enable_stage_timing(False)
    assert layer.sync_status()[0] == 0


@pytest.mark.parametrize("T", [600, 2300])
def test_fused_epilogue_beside_other_work(tiny, T):
    """The fused epilogue takes its tiles from a work counter, so its value
    tiles' waits never depend on a CTA that has not started: run while bf16
    matmuls on another stream hold SMs (600 and 2,300 tokens, both on CTA
    pairs), it still finishes with status 0 and equals lookup_project +
    gate_apply bit for bit."""
    from engram_hashed_gram_gb300.layer import EngramLayer
    dev = tiny["dev"]
    fused = EngramLayer(tiny["table"], tiny["scale"], dev["wkv"], dev["q"], dev["k"], max_tokens=2300,
                        fuse_gate=True)
    try:
        w, inp = _inputs(tiny, 1, T, mask_frac=0.1, seed=23)
        ids, x, mask = _dev(inp)
        ref = fused.gate_apply(fused.lookup_project(ids), x, mask)
        a = torch.randn(8192, 8192, dtype=torch.bfloat16, device="cuda")
        b = torch.randn(8192, 8192, dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        side = torch.cuda.Stream()
        with torch.cuda.stream(side):
            for _ in range(8):
                torch.mm(a, b)
        outs = [fused.forward(ids, x, mask) for _ in range(4)]
        torch.cuda.synchronize()
        assert fused.sync_status()[0] == 0
        for out in outs:
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    finally:
        fused.close()


def test_plan_invariants_over_batch_sizes(tiny):
    """The projection's plan over 1 to 20,000 tokens (queries only, nothing
    runs): CTA pairs exactly from 256 tokens, the gate in the epilogue
    exactly from 1,024 (on pairs, whole tiles), split-K only up to 128 tokens,
    a remainder split only for a last wave of at most a quarter of the grid,
    an even CTA count on pairs, and forward's kernel count to match; under an
    SM budget, neither pairs nor the fused epilogue."""
    from engram_hashed_gram_gb300.layer import EngramLayer
    dev = tiny["dev"]
    layer = EngramLayer(tiny["table"], tiny["scale"], dev["wkv"], dev["q"], dev["k"], max_tokens=20000)
    try:
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        for budget in (0, 120):
            layer.set_sm_budget(budget)
            cap = sms if budget == 0 else budget
            for M in list(range(1, 300, 7)) + list(range(300, 20001, 173)) + [128, 129, 255, 256, 1023, 1024]:
                p = layer.describe_plan(M)
                k = layer.forward_kernels(M)
                pairs = budget == 0 and M >= 256
                fused = budget == 0 and M >= 1024
                assert p["cta_pairs"] == int(pairs), (M, budget, p)
                assert p["fused_gate"] == int(fused), (M, budget, p)
                assert p["splits"] == 1 or M <= 128, (M, p)
                assert p["ctas"] <= cap, (M, p)
                if pairs:
                    assert p["ctas"] % 2 == 0, (M, p)
                if fused:
                    assert p["rem_tiles"] == 0 and p["splits"] == 1 and k == 2, (M, p, k)
                else:
                    assert k == 3 + (1 if p["rem_tiles"] else 0), (M, p, k)
                if p["rem_tiles"]:
                    slots = p["ctas"] // 2 if pairs else p["ctas"]
                    assert 0 < p["rem_tiles"] <= slots // 4 and 2 <= p["rem_splits"] <= 4, (M, p)
    finally:
        layer.close()
