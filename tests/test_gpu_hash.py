"""GPU parity of engram_hash against the hash oracle, bit for bit: random
configurations with masks, out-of-vocabulary ids and chunked calls; the V4.1
layout (two layers, the 48 primes above 16,000,000); and the whole pipeline
token ids -> hash -> layer on the small table."""
import dataclasses

import numpy as np
import pytest
import torch

from engram_hashed_gram_gb300 import synth
from engram_hashed_gram_gb300 import synth_device as SD
from oracle import engram_oracle as O
from oracle import hash_oracle as H
import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from engram_hashed_gram_gb300 import build as B
    B.build()


def _params(rng, n_layers, n, heads, vocab, primes=None):
    token_map = rng.integers(0, 99_092, size=vocab).astype(np.int32)
    mult = (rng.integers(1, 1 << 62, size=(n_layers, n)) * 2 + 1).astype(np.int64)
    if primes is None:
        primes = rng.integers(1_000_003, 16_000_057, size=(n_layers, n - 1, heads)).astype(np.int64)
    offsets = np.zeros((n_layers, (n - 1) * heads), dtype=np.int64)
    for g in range(n_layers):
        offsets[g] = np.concatenate([[0], np.cumsum(primes[g].reshape(-1))[:-1]])
    return token_map, mult, primes, offsets


def _dev(*arrays):
    return [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in arrays]


@pytest.mark.parametrize("n_layers,n,heads", [(2, 4, 8), (1, 3, 5), (3, 5, 2)])
def test_hash_matches_oracle_over_chunked_calls(built, n_layers, n, heads):
    from engram_hashed_gram_gb300.layer import EngramHasher
    rng = np.random.default_rng([n_layers, n, heads])
    vocab = 4000
    token_map, mult, primes, offsets = _params(rng, n_layers, n, heads, vocab)
    B, Ltot = 3, 300
    ids = rng.integers(0, vocab, size=(B, Ltot))
    ids[0, 7] = vocab + 5                                  # outside the map
    ids[2, 100] = -3
    mask = (rng.random((B, Ltot)) > 0.1).astype(np.uint8)
    hasher = EngramHasher(*_dev(token_map, mult, primes, offsets), max_batch=4, max_len=512)
    cache = np.zeros((4, 512), np.int64)
    for s, e in ((0, 1), (1, 130), (130, 131), (131, 300)):
        got = hasher(torch.from_numpy(ids[:, s:e]).cuda(), s, torch.from_numpy(mask[:, s:e]).cuda())
        want = H.ngram_hash(ids[:, s:e], s, cache, token_map, mult, primes, offsets, 2, -1, mask[:, s:e])
        assert np.array_equal(got.cpu().numpy(), np.transpose(want, (2, 0, 1, 3)))
    assert np.array_equal(hasher.cache[:B, :Ltot].cpu().numpy(), cache[:B, :Ltot])


def test_extreme_divisors(built):
    """The remainder for divisors from 1 to 2^63-1 (powers of two, 2^32 +- 1,
    the largest int64) on hashes that cover the whole int64 range, including
    its most negative value (multiplier 2^63 with an odd id)."""
    from engram_hashed_gram_gb300.layer import EngramHasher
    rng = np.random.default_rng(63)
    divisors = np.array([1, 2, 3, 7, 1 << 20, (1 << 31) - 1, (1 << 32) - 1, 1 << 32, (1 << 32) + 1,
                         (1 << 40) + 7, (1 << 62) - 57, 1 << 62, (1 << 62) + 135, (1 << 63) - 25,
                         (1 << 63) - 1, 16_000_057], dtype=np.int64).reshape(2, 1, 8)
    token_map, mult, primes, offsets = _params(rng, 2, 2, 8, 500, primes=divisors)
    mult[0, 1] = np.int64(-(1 << 63))                       # products 0 or INT64_MIN
    offsets[:] = 0                                          # the divisors' sums overflow int64
    ids = rng.integers(0, 500, size=(4, 64))
    hasher = EngramHasher(*_dev(token_map, mult, primes, offsets), max_batch=4, max_len=64)
    got = hasher(torch.from_numpy(ids).cuda()).cpu().numpy()
    want = H.ngram_hash(ids, 0, np.zeros((4, 64), np.int64), token_map, mult, primes, offsets, 2, -1)
    assert np.array_equal(got, np.transpose(want, (2, 0, 1, 3)))


def test_v41_layout(built):
    """Two layers, 3 orders x 8 heads, the 48 primes above 16,000,000 (first 24
    for the first module, next 24 for the second); every id lies in its
    layer's table and matches the oracle."""
    from engram_hashed_gram_gb300.layer import EngramHasher
    rng = np.random.default_rng(41)
    pr = np.array(synth.consecutive_primes_above(16_000_000, 48), dtype=np.int64).reshape(2, 3, 8)
    token_map, mult, primes, offsets = _params(rng, 2, 4, 8, 129_280, primes=pr)
    ids = rng.integers(0, 129_280, size=(2, 257))
    hasher = EngramHasher(*_dev(token_map, mult, primes, offsets), max_batch=2, max_len=257)
    got = hasher(torch.from_numpy(ids).cuda()).cpu().numpy()
    want = H.ngram_hash(ids, 0, np.zeros((2, 257), np.int64), token_map, mult, primes, offsets, 2, -1)
    assert np.array_equal(got, np.transpose(want, (2, 0, 1, 3)))
    assert got[0].min() >= 0 and got[0].max() < 384_006_168
    assert got[1].min() >= 0 and got[1].max() < 384_016_682


def test_argument_errors(built):
    from engram_hashed_gram_gb300 import _lib
    from engram_hashed_gram_gb300.layer import EngramHasher
    rng = np.random.default_rng(3)
    hasher = EngramHasher(*_dev(*_params(rng, 1, 4, 8, 100)), max_batch=2, max_len=16)
    ids = torch.zeros((2, 8), dtype=torch.int64, device="cuda")
    with pytest.raises(_lib.EngramError):
        hasher(ids, start_pos=9)                           # 9 + 8 > max_len
    with pytest.raises(_lib.EngramError):
        hasher(torch.zeros((3, 4), dtype=torch.int64, device="cuda"))   # B > max_batch
    assert hasher(torch.zeros((2, 0), dtype=torch.int64, device="cuda")).numel() == 0


def test_pipeline_token_ids_to_layer_output(built):
    """hash (one layer, the small table's 24 prime ranges) -> engram_forward,
    against the oracle chain."""
    from engram_hashed_gram_gb300.layer import EngramHasher, EngramLayer
    w = dataclasses.replace(synth.workload("tiny_1x16"), B=2, T=40)
    lengths, offsets0 = w.layout()
    rng = np.random.default_rng(5)
    pr = lengths.reshape(1, 3, 8).astype(np.int64)
    token_map, mult, primes, offsets = _params(rng, 1, 4, 8, 5000, primes=pr)
    assert np.array_equal(offsets[0], offsets0)
    ids = rng.integers(0, 5000, size=(w.B, w.T))
    mask = np.ones((w.B, w.T), np.uint8)
    mask[1, 10:15] = 0                                     # an image span
    hasher = EngramHasher(*_dev(token_map, mult, primes, offsets), max_batch=w.B, max_len=w.T)
    hid = hasher(torch.from_numpy(ids).cuda(), 0, torch.from_numpy(mask).cuda())[0]   # [B, T, 24]
    table, scale = SD.make_table(w)
    inp = synth.make_inputs(w)
    d = SD.upload_inputs(inp)
    layer = EngramLayer(table, scale, d["wkv"], d["q"], d["k"], max_tokens=w.M)
    m = torch.from_numpy(mask).cuda()
    out = layer.forward(hid.contiguous(), d["x"], m)
    assert layer.sync_status()[0] == 0
    want_ids = H.ngram_hash(ids, 0, np.zeros((w.B, w.T), np.int64), token_map, mult, primes, offsets, 2, -1, mask)
    assert np.array_equal(hid.cpu().numpy(), want_ids[:, :, 0, :])
    inp2 = dataclasses.replace(inp, hash_ids=want_ids[:, :, 0, :].astype(np.int64), mask=mask)
    ref_out, ref_g, ref_kv = P.oracle_tokens(w, inp2, np.arange(w.M))
    s = P.compare_out(SD.device_bits(out).reshape(w.M, w.hc_mult, w.dim), ref_out)
    assert s["rel_l2"] <= P.REL_L2_TOL
    off = mask.reshape(-1) == 0
    assert np.array_equal(SD.device_bits(out).reshape(w.M, -1)[off], inp.x.reshape(w.M, -1)[off])
    layer.close()


def test_full_size_chunked_v41(built):
    """The full-size workload's shape: B = 2 sessions of 8,192 tokens in four
    chunks of 2,048, V4.1 layout, with DEAD positions (mask) and ids outside
    the map; every output id against the oracle."""
    from engram_hashed_gram_gb300.layer import EngramHasher
    rng = np.random.default_rng(8192)
    vocab = 129_280
    pr = np.array(synth.consecutive_primes_above(16_000_000, 48), dtype=np.int64).reshape(2, 3, 8)
    token_map, mult, primes, offsets = _params(rng, 2, 4, 8, vocab, primes=pr)
    B, L = 2, 8192
    ids = rng.integers(0, vocab, size=(B, L))
    ids[0, ::997] = vocab + 11
    mask = (rng.random((B, L)) > 0.02).astype(np.uint8)
    hasher = EngramHasher(*_dev(token_map, mult, primes, offsets), max_batch=B, max_len=L)
    cache = np.zeros((B, L), np.int64)
    for s in range(0, L, 2048):
        got = hasher(torch.from_numpy(ids[:, s:s + 2048]).cuda(), s, torch.from_numpy(mask[:, s:s + 2048]).cuda())
        want = H.ngram_hash(ids[:, s:s + 2048], s, cache, token_map, mult, primes, offsets, 2, -1, mask[:, s:s + 2048])
        assert np.array_equal(got.cpu().numpy(), np.transpose(want, (2, 0, 1, 3))), f"chunk at {s}"
