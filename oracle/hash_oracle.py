"""CPU oracle of the Engram n-gram hash -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline may import this module; the product path never does.

It follows the hash ``forward`` excerpt of atlas.klimoza.dev "deepseek-v4.1 /
engram-second" step by step, in plain Python integers:

  1. compressed = token_map[input_ids]; positions where token_mask is False
     become DEAD (they take part in no n-gram);
  2. the session cache row of each sequence receives the compressed ids at
     positions start_pos .. start_pos + L - 1;
  3. for shift = 0 .. max_ngram_size-1: the token `shift` positions back (from
     the cache), and a `blocked` flag that accumulates over the shifts (the
     position is < shift, or that token is DEAD); a blocked look-back is pad_id;
  4. products = token[shift] * multiplier[layer, shift]; the running XOR of the
     products after shift i is the hash of the (i+1)-gram;
  5. each (i+1)-gram hash modulo each head's prime (the remainder takes the
     divisor's sign, as ``%`` does on torch integer tensors), plus the column's
     row offset; columns are ordered (order, head).

Arithmetic: ``arith="int64"`` wraps the products to signed 64 bits, as int64
tensors do (the excerpt's semantics); ``arith="bigint"`` keeps exact integers,
as the demo on monishver11.github.io "DeepSeek's Other Modules" (section "Check
it in Python") does.  Readings: an input id outside [0, len(token_map)) is
treated as DEAD (the excerpt would raise on such an index).
"""
from __future__ import annotations

import numpy as np

MASK64 = (1 << 64) - 1


def _signed64(v: int) -> int:
    v &= MASK64
    return v - (1 << 64) if v >> 63 else v


def ngram_tokens(input_ids, start_pos: int, cache, token_map, pad_id: int, dead_id: int, max_ngram_size: int,
                 token_mask=None):
    """Steps 1-3: the look-back tokens, [B, L, max_ngram_size] Python ints.
    `cache` (a [B_max, L_max] integer array) is updated in place."""
    ids = np.asarray(input_ids, dtype=np.int64)
    B, L = ids.shape
    vocab = len(token_map)
    for b in range(B):
        for l in range(L):
            t = int(ids[b, l])
            c = int(token_map[t]) if 0 <= t < vocab else dead_id
            if token_mask is not None and not bool(np.asarray(token_mask)[b, l]):
                c = dead_id
            cache[b, start_pos + l] = c
    out = [[[0] * max_ngram_size for _ in range(L)] for _ in range(B)]
    for b in range(B):
        for l in range(L):
            pos = start_pos + l
            blocked = False
            for shift in range(max_ngram_size):
                src = int(cache[b, max(pos - shift, 0)])
                blocked = blocked or pos < shift or src == dead_id
                out[b][l][shift] = pad_id if blocked else src
    return out


def ngram_hash(input_ids, start_pos: int, cache, token_map, multipliers, primes, offsets, pad_id: int,
               dead_id: int, token_mask=None, arith: str = "int64") -> np.ndarray:
    """Hash ids [B, L, n_layers, (max_ngram_size-1) * n_heads] (int64 numpy;
    object dtype in "bigint" mode).

    multipliers: [n_layers, max_ngram_size]; primes: [n_layers,
    max_ngram_size-1, n_heads]; offsets: [n_layers, (max_ngram_size-1)*n_heads]."""
    mult = [[int(v) for v in row] for row in np.asarray(multipliers, dtype=object)]
    pr = np.asarray(primes, dtype=object)
    off = np.asarray(offsets, dtype=object)
    n_layers, n = len(mult), len(mult[0])
    heads = pr.shape[2]
    toks = ngram_tokens(input_ids, start_pos, cache, token_map, pad_id, dead_id, n, token_mask)
    B, L = len(toks), len(toks[0]) if toks else 0
    out = np.empty((B, L, n_layers, (n - 1) * heads), dtype=object)
    for b in range(B):
        for l in range(L):
            for g in range(n_layers):
                prods = []
                for s in range(n):
                    p = toks[b][l][s] * mult[g][s]
                    prods.append(_signed64(p) if arith == "int64" else p)
                rolling = prods[0]
                for i in range(1, n):
                    rolling = rolling ^ prods[i]      # two's complement XOR of in-range ints
                    for h in range(heads):
                        c = (i - 1) * heads + h
                        out[b, l, g, c] = rolling % int(pr[g, i - 1, h]) + int(off[g, c])
    return out.astype(np.int64) if arith == "int64" else out
