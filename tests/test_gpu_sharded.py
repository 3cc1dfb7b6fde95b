"""The row-split table on one GPU: two shard contexts (table rows [0, P) and
[P, R), P = ceil(R/2), as `ParallelEngramEmbedding` splits them) over the same
device table stand in for two ranks; their gathered rows, summed the way
exchange_rows sums them, equal the whole table's rows bit for bit, and
engram_forward_rows on the sum equals engram_forward bit for bit.  Each shard's
rows also match the oracle's shard lookup bit for bit.  The multi-rank NCCL
exchange itself needs more than one GPU; its gloo form is tested on CPU
(tests/test_sharded.py)."""
import dataclasses
import os
import socket

import numpy as np
import pytest
import torch

from engram_hashed_gram_gb300 import synth
from oracle import engram_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from engram_hashed_gram_gb300 import build as B
    B.build()
    from engram_hashed_gram_gb300 import synth_device as SD
    from engram_hashed_gram_gb300.layer import EngramLayer, shard_rows
    w = dataclasses.replace(synth.workload("tiny_1x16"), B=1, T=1200, mask="span10")
    table, scale = SD.make_table(w)
    inp = synth.make_inputs(w)
    d = SD.upload_inputs(inp)
    R = table.shape[0]
    kw = dict(max_tokens=w.M, eps=w.eps, scale_block=w.scale_block)
    whole = EngramLayer(table, scale, d["wkv"], d["q"], d["k"], **kw)
    shards = []
    for r in range(2):
        s, e = shard_rows(R, r, 2)
        shards.append((s, e, EngramLayer(table[s:e], scale[s:e], d["wkv"], d["q"], d["k"], row_offset=s,
                                         check_ids=True, **kw)))
    ids = d["hash_ids"].clone()
    ids[0, 0, :4] = torch.tensor([-1, R, R + 5, -(1 << 40)])     # outside every shard
    yield dict(w=w, inp=inp, d=d, SD=SD, table=table, scale=scale, whole=whole, shards=shards, ids=ids, R=R)
    whole.close()
    for _, _, lay in shards:
        lay.close()


def test_shard_rows_sum_to_the_whole_lookup(env):
    SD, ids = env["SD"], env["ids"]
    whole = env["whole"].lookup(ids)
    parts = [lay.lookup(ids) for _, _, lay in env["shards"]]
    summed = parts[0].view(torch.int32) + parts[1].view(torch.int32)     # exchange_rows' integer sum
    torch.cuda.synchronize()
    assert torch.equal(summed.view(torch.int16), whole.view(torch.int16))
    # each shard against the oracle's `ParallelEngramEmbedding` step on its rows
    ids_h = ids.cpu().numpy().reshape(-1, env["w"].n_cols)
    codes, scales = synth.host_table(env["w"].seed, env["R"], env["w"].head_dim, env["w"].scale_block)
    for (s, e, _), p in zip(env["shards"], parts):
        ref = O.lookup_shard(ids_h, codes[s:e], scales[s:e], s, env["w"].scale_block)
        assert np.array_equal(SD.device_bits(p).reshape(ref.shape), ref)


@pytest.mark.parametrize("T", [1200, 300])
def test_forward_rows_on_the_exchanged_rows_equals_forward(env, T):
    """1,200 tokens run the CTA-pair projection with the gate in its epilogue,
    300 tokens the CTA-pair projection and the separate gate kernel."""
    ids, d = env["ids"][:, :T].contiguous(), env["d"]
    x, mask = d["x"][:, :T].contiguous(), d["mask"][:, :T].contiguous()
    assert env["whole"].describe_plan(T)["fused_gate"] == (1 if T >= 1024 else 0)
    parts = [lay.lookup(ids) for _, _, lay in env["shards"]]
    rows = (parts[0].view(torch.int32) + parts[1].view(torch.int32)).view(torch.bfloat16)
    for s, e, lay in env["shards"]:           # every rank gets the whole output from the exchanged rows
        out_rows = lay.forward_rows(rows, x, mask)
        ref = env["whole"].forward(ids, x, mask)
        torch.cuda.synchronize()
        assert torch.equal(out_rows.view(torch.int16), ref.view(torch.int16))
    # in place as well
    y = x.clone()
    env["shards"][0][2].forward_rows(rows, y, mask, out=y)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), ref.view(torch.int16))


def test_shard_counts_ids_outside_it(env):
    ids = env["ids"]
    ids_h = ids.cpu().numpy().reshape(-1)
    for s, e, lay in env["shards"]:
        lay.sync_status()
        lay.lookup(ids)
        st, bad = lay.sync_status()
        outside = int(((ids_h < s) | (ids_h >= e)).sum())
        assert (st, bad) == (-4, outside)


def _free_port():
    sock = socket.socket()
    sock.bind(("127.0.0.1", 0))
    port = sock.getsockname()[1]
    sock.close()
    return port


def test_engram_shard_on_a_one_rank_nccl_group(env):
    """EngramShard with a one-rank NCCL process group holds the whole table
    and equals engram_forward bit for bit; NCCL's integer all-reduce of the
    rows (the exchange's collective) is the identity on one rank."""
    import torch.distributed as dist
    from engram_hashed_gram_gb300.layer import EngramShard
    if dist.is_initialized():
        pytest.skip("a process group already exists")
    if not dist.is_nccl_available():
        pytest.skip("torch.distributed has no NCCL backend here")
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(_free_port())
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
    try:
        d, w = env["d"], env["w"]
        sh = EngramShard(env["table"], env["scale"], d["wkv"], d["q"], d["k"], num_rows=env["R"], max_tokens=w.M,
                         eps=w.eps, scale_block=w.scale_block)
        out = sh.forward(env["ids"], d["x"], d["mask"])
        ref = env["whole"].forward(env["ids"], d["x"], d["mask"])
        rows = env["whole"].lookup(env["ids"])
        before = rows.clone()
        dist.all_reduce(rows.view(torch.int32), op=dist.ReduceOp.SUM)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        assert torch.equal(rows.view(torch.int16), before.view(torch.int16))
        sh.close()
    finally:
        dist.destroy_process_group()
