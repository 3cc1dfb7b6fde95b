"""Pins of the n-gram hash oracle: the page's demo vector, torch's int64
semantics, the blocking rules by hand, chunked calls and the column layout."""
import os

import numpy as np
import pytest
import torch

from oracle import hash_oracle as H

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _golden():
    out = {}
    for line in open(os.path.join(ROOT, "tests", "golden", "hash_demo.txt")):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = (s.strip() for s in line.split("=", 1))
            out[k] = [int(t, 0) for t in v.split()]
    return out


def test_demo_vector_exact_integers():
    g = _golden()
    ids = np.array([g["ids"]], dtype=np.int64)
    n = len(g["multipliers"])                                   # 3: orders 2 and 3
    primes = np.array([[[17, 19, 23], g["primes"]]], dtype=object)
    offsets = np.zeros((1, (n - 1) * 3), dtype=object)
    cache = np.zeros((1, 8), dtype=np.int64)
    out = H.ngram_hash(ids, 0, cache, np.arange(8), [g["multipliers"]], primes, offsets, pad_id=0, dead_id=-1,
                       arith="bigint")
    assert [int(v) for v in out[0, -1, 0, 3:6]] == g["rows_3gram_at_last"]


def test_int64_semantics_match_torch():
    """Steps 4-5 in torch int64 (wrapping products, XOR, remainder with the
    divisor's sign) on the oracle's look-back tokens."""
    rng = np.random.default_rng(0)
    B, L, n, heads, nl = 3, 17, 4, 8, 2
    vocab = 500
    token_map = rng.integers(0, 99_092, size=vocab)
    ids = rng.integers(0, vocab, size=(B, L))
    mult = rng.integers(1, 1 << 62, size=(nl, n)) * 2 + 1                    # odd, large: products overflow
    primes = rng.integers(1_000_003, 16_000_057, size=(nl, n - 1, heads))
    offsets = rng.integers(0, 1 << 30, size=(nl, (n - 1) * heads))
    mask = rng.random((B, L)) > 0.1
    cache = np.zeros((4, 64), dtype=np.int64)
    got = H.ngram_hash(ids, 5, cache.copy(), token_map, mult, primes, offsets, 2, -1, mask, arith="int64")
    toks = torch.tensor(H.ngram_tokens(ids, 5, cache.copy(), token_map, 2, -1, n, mask), dtype=torch.int64)
    prods = toks.unsqueeze(2) * torch.from_numpy(mult)                        # [B, L, nl, n]
    rolling, cols = prods[..., 0], []
    for i in range(1, n):
        rolling = torch.bitwise_xor(rolling, prods[..., i])
        cols.append(rolling.unsqueeze(-1) % torch.from_numpy(primes[:, i - 1]))
    want = (torch.cat(cols, dim=-1) + torch.from_numpy(offsets)).numpy()
    assert np.array_equal(got, want)
    # and the exact-integer mode differs once products overflow
    big = H.ngram_hash(ids, 5, cache.copy(), token_map, mult, primes, offsets, 2, -1, mask, arith="bigint")
    assert any(int(a) != int(b) for a, b in zip(got.ravel(), big.ravel()))


def test_blocking_rules_by_hand():
    DEAD, PAD = -7, 2
    token_map = np.arange(100) + 10                                         # id t -> 10 + t
    ids = np.array([[5, 6, 7, 8, 9, 1]])
    mask = np.array([[1, 0, 1, 1, 1, 1]], dtype=bool)                        # position 1 is an image token
    cache = np.zeros((1, 16), dtype=np.int64)
    toks = H.ngram_tokens(ids, 0, cache, token_map, PAD, DEAD, 4, mask)[0]
    assert toks[0] == [15, PAD, PAD, PAD]                                   # nothing before position 0
    assert toks[1] == [PAD, PAD, PAD, PAD]                                  # a DEAD token blocks itself
    assert toks[2] == [17, PAD, PAD, PAD]                                   # ... and every n-gram reaching it
    assert toks[3] == [18, 17, PAD, PAD]
    assert toks[4] == [19, 18, 17, PAD]
    assert toks[5] == [11, 19, 18, 17]
    assert list(cache[0, :6]) == [15, DEAD, 17, 18, 19, 11]


def test_chunked_calls_equal_one_call():
    rng = np.random.default_rng(1)
    n, heads, nl = 4, 8, 2
    token_map = rng.integers(0, 99_092, size=300)
    ids = rng.integers(0, 300, size=(2, 23))
    ids[1, 4] = 1000                                                         # outside the map: DEAD
    mask = rng.random((2, 23)) > 0.15
    mult = rng.integers(1, 1 << 62, size=(nl, n)) * 2 + 1
    primes = rng.integers(1_000_003, 16_000_057, size=(nl, n - 1, heads))
    offsets = rng.integers(0, 1 << 30, size=(nl, (n - 1) * heads))
    whole = H.ngram_hash(ids, 0, np.zeros((2, 32), np.int64), token_map, mult, primes, offsets, 2, -1, mask)
    cache = np.zeros((2, 32), np.int64)
    parts = []
    for s, e in ((0, 1), (1, 9), (9, 10), (10, 23)):
        parts.append(H.ngram_hash(ids[:, s:e], s, cache, token_map, mult, primes, offsets, 2, -1, mask[:, s:e]))
    assert np.array_equal(np.concatenate(parts, axis=1), whole)


def test_column_layout_and_offsets():
    """With multipliers [1, 0, 0, 0] every order's hash is the current token:
    column (order - 2) * heads + head holds token % prime[order, head] + offset."""
    rng = np.random.default_rng(2)
    n, heads = 4, 8
    primes = rng.integers(50, 1000, size=(1, n - 1, heads))
    offsets = rng.integers(0, 10_000, size=(1, (n - 1) * heads))
    ids = np.array([[3, 141, 59, 265]])
    out = H.ngram_hash(ids, 0, np.zeros((1, 8), np.int64), np.arange(1000), [[1, 0, 0, 0]], primes, offsets, 2, -1)
    for l in range(4):
        for i in range(n - 1):
            for h in range(heads):
                c = i * heads + h
                assert out[0, l, 0, c] == ids[0, l] % primes[0, i, h] + offsets[0, c]
