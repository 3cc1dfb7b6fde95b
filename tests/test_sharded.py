"""The row-split table on CPU (no GPU): the oracle's shard lookup
(`ParallelEngramEmbedding.forward` of atlas.klimoza.dev "deepseek-v4.1 /
engram-second") pinned against the whole-table lookup, the product's shard
bounds against the excerpt's rule, and the product's exchange (exchange_rows,
one all-reduce) run by world_size-2 and -3 gloo ranks: the shards' rows, once
exchanged, are the whole table's rows bit for bit."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from engram_hashed_gram_gb300 import synth
from engram_hashed_gram_gb300.layer import exchange_rows, shard_rows
from oracle import engram_oracle as O

R, HD, BS = 29, 32, 16


def _tiny_table(seed=3, scale_fmt=O.SCALE_F32):
    codes, scales = synth.table_rows(seed, np.arange(R), HD, BS, scale_fmt)
    # every code at least once, including +-0 and the NaN codes, in rows 0..7
    codes[:8] = np.arange(256, dtype=np.uint8).reshape(8, HD)
    return codes, scales


def _ids(rng, M=40, C=5):
    ids = rng.integers(0, R, size=(M, C), dtype=np.int64)
    ids[0, :] = [-1, R, R + 7, -(1 << 62), (1 << 62)]        # outside the table
    ids[1, :] = [0, R - 1, 3, 4, 5]
    return ids


def test_shard_bounds_follow_the_excerpt_rule():
    # part = ceil(R / world) rows per rank, rank r from r * part; the last ends at R
    assert [O.shard_bounds(10, r, 3) for r in range(3)] == [(0, 4), (4, 8), (8, 10)]
    assert [O.shard_bounds(3, r, 4) for r in range(4)] == [(0, 1), (1, 2), (2, 3), (3, 3)]
    for rows in (0, 1, 7, 29, 384_016_682):
        for world in (1, 2, 3, 5, 8):
            b = [O.shard_bounds(rows, r, world) for r in range(world)]
            assert b[0][0] == 0 and b[-1][1] == rows
            assert all(b[i][1] == b[i + 1][0] for i in range(world - 1))        # no gap, no overlap
            assert [shard_rows(rows, r, world) for r in range(world)] == b       # the product's helper agrees
    with pytest.raises(ValueError):
        shard_rows(10, 3, 3)


@pytest.mark.parametrize("scale_fmt", [O.SCALE_F32, O.SCALE_E8M0])
@pytest.mark.parametrize("world", [1, 2, 3, 5])
def test_shard_lookups_sum_to_the_whole_table(world, scale_fmt):
    """Every row is held by exactly one rank: the ranks' rows summed as integers
    are the whole lookup's bits, and summed as floats (the excerpt's all-reduce)
    its values, except that -0.0 becomes +0.0 there."""
    codes, scales = _tiny_table(scale_fmt=scale_fmt)
    ids = _ids(np.random.default_rng(world))
    whole = O.lookup(ids, codes, scales, BS, scale_fmt)
    parts = []
    for r in range(world):
        s, e = O.shard_bounds(R, r, world)
        parts.append(O.lookup_shard(ids, codes[s:e], scales[s:e], s, BS, scale_fmt))
    # bits: one non-zero contribution per element
    nonzero = sum((p != 0).astype(np.int64) for p in parts)
    assert nonzero.max() <= 1
    assert np.array_equal(sum(p.astype(np.int64) for p in parts).astype(np.uint16), whole)
    # values: as the excerpt's floating-point all-reduce sums them
    fsum = sum(O.bf16_value(p) for p in parts)
    wv = O.bf16_value(whole)
    both_nan = np.isnan(fsum) & np.isnan(wv)
    assert np.array_equal(fsum[~both_nan], wv[~both_nan])
    if world == 1:
        assert np.array_equal(parts[0], whole)


def test_shard_lookup_zeroes_rows_outside_its_shard():
    codes, scales = _tiny_table()
    ids = np.array([[9, 10, 19, 20, -1]], dtype=np.int64)
    part = O.lookup_shard(ids, codes[10:20], scales[10:20], 10, BS).reshape(5, HD)
    whole = O.lookup(ids, codes, scales, BS).reshape(5, HD)
    assert not part[0].any() and not part[3].any() and not part[4].any()
    assert np.array_equal(part[1], whole[1]) and np.array_equal(part[2], whole[2])


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        codes, scales = _tiny_table()
        ids = _ids(np.random.default_rng(11))
        s, e = shard_rows(R, rank, world)
        mine = O.lookup_shard(ids, codes[s:e], scales[s:e], s, BS)
        rows = torch.from_numpy(mine.view(np.int16).copy()).view(torch.bfloat16).reshape(ids.shape[0], 1, -1)
        out = exchange_rows(rows)                                  # the product's exchange, in place
        got = out.view(torch.int16).numpy().view(np.uint16).reshape(ids.shape[0], -1)
        q.put((rank, bool(np.array_equal(got, O.lookup(ids, codes, scales, BS))), int((mine != 0).sum())))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_exchange_over_gloo_ranks_gives_the_whole_table(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert [r for r, _, _ in res] == list(range(world))
    assert all(ok for _, ok, _ in res), res
    assert all(nz > 0 for _, _, nz in res)          # every rank held some of the rows


def test_exchange_without_a_process_group_is_a_no_op():
    rows = torch.arange(12, dtype=torch.int16).view(torch.bfloat16).reshape(1, 2, 6)
    before = rows.clone()
    assert exchange_rows(rows) is rows
    assert torch.equal(rows.view(torch.int16), before.view(torch.int16))
