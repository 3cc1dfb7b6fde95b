"""Python binding of the Engram layer's C ABI (include/engram.h).

Argument marshalling only: shapes, dtypes and device pointers of torch tensors
are checked and handed to libengram.so; every step of the layer runs in the
library's CUDA kernels on the tensors' device, on the current torch stream
unless another is given.  PyTorch is used for device memory and streams.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import EngramConfig, EngramHashConfig, EngramWeights, check

_U16 = (torch.bfloat16, torch.int16, torch.uint16)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtypes, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the layer on {device}")


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


class EngramLayer:
    """One Engram instance bound to caller-owned device tensors.

    table: uint8 [R, head_dim] e4m3 codes; scale: float32 [R, head_dim/scale_block]
    (or uint8 E8M0 codes with scale_fmt=SCALE_E8M0); wkv: bf16 [dim*(hc+1),
    n_cols*head_dim], or its uint8 e4m3 codes together with wkv_scale (uint8
    E8M0 [dim*(hc+1), n_cols*head_dim/32]) for the MXFP8 weight; q_weight,
    k_weight: bf16 [hc, dim].  The tensors are referenced, not copied, and are
    kept alive by this object.  table and scale may instead be pinned host
    tensors (``pin_memory()``): the gather then reads them in place over the
    host link, the layer runs on ``device`` (default: the current CUDA
    device).  With ``row_offset`` the table is one shard of a row-split table:
    it holds global rows [row_offset, row_offset + R), and every other id
    gives a zero row (see EngramShard).  fuse_gate: None lets the library
    choose where the gate is formed (in the projection's epilogue or in a
    kernel of its own) by batch size, True / False force one or the other;
    the result is the same either way."""

    def __init__(self, table, scale, wkv, q_weight, k_weight, *, dim=5120, hc_mult=4, n_cols=24, head_dim=256,
                 scale_block=128, scale_fmt=_lib.SCALE_F32, eps=1e-6, clamp=1e-6, max_tokens=4096,
                 check_ids=False, fuse_gate=None, wkv_scale=None, device=None, row_offset=0):
        if table.device.type == "cuda":
            dev = table.device
        elif table.is_pinned():
            dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        else:
            raise ValueError("table must be a CUDA tensor or a pinned host tensor")
        if dev.type != "cuda":
            raise ValueError("the Engram layer runs on a CUDA device only")
        R = table.shape[0]
        tdev = table.device
        if tdev.type != "cuda" and not (scale.device.type == "cpu" and scale.is_pinned()):
            raise ValueError("with a pinned host table, scale must be pinned host memory too")
        _need(table, "table", (torch.uint8,), (R, head_dim), tdev)
        _need(scale, "scale", (torch.float32,) if scale_fmt == _lib.SCALE_F32 else (torch.uint8,),
              (R, head_dim // scale_block), tdev)
        wkv_fmt = _lib.WKV_BF16 if wkv_scale is None else _lib.WKV_MXFP8
        if wkv_fmt == _lib.WKV_BF16:
            _need(wkv, "wkv", _U16, (dim * (hc_mult + 1), n_cols * head_dim), dev)
        else:
            _need(wkv, "wkv", (torch.uint8,), (dim * (hc_mult + 1), n_cols * head_dim), dev)
            _need(wkv_scale, "wkv_scale", (torch.uint8,), (dim * (hc_mult + 1), n_cols * head_dim // 32), dev)
        _need(q_weight, "q_weight", _U16, (hc_mult, dim), dev)
        _need(k_weight, "k_weight", _U16, (hc_mult, dim), dev)
        self.device = dev
        self.dim, self.hc_mult, self.n_cols, self.head_dim = dim, hc_mult, n_cols, head_dim
        self.N = dim * (hc_mult + 1)
        self.K = n_cols * head_dim
        self.max_tokens = max_tokens
        self._keep = (table, scale, wkv, q_weight, k_weight, wkv_scale)
        self.cfg = EngramConfig(dim=dim, hc_mult=hc_mult, n_cols=n_cols, head_dim=head_dim,
                                scale_block=scale_block, scale_fmt=scale_fmt, num_rows=R, eps=eps, clamp=clamp,
                                max_tokens=max_tokens, check_ids=1 if check_ids else 0,
                                fuse_gate=0 if fuse_gate is None else (1 if fuse_gate else -1), wkv_fmt=wkv_fmt,
                                row_offset=row_offset)
        w = EngramWeights(table=_ptr(table), scale=_ptr(scale), wkv=_ptr(wkv), q_weight=_ptr(q_weight),
                          k_weight=_ptr(k_weight), wkv_scale=_ptr(wkv_scale))
        self._ctx = ctypes.c_void_p()
        self._lib = _lib.engram()
        with torch.cuda.device(dev):
            check(self._lib.engram_create(ctypes.byref(self._ctx), ctypes.byref(self.cfg), ctypes.byref(w)),
                  "engram_create")

    # ------------------------------------------------------------------ calls
    def _tokens(self, hash_ids):
        _need(hash_ids, "hash_ids", (torch.int64,), None, self.device)
        if hash_ids.dim() != 3 or hash_ids.shape[2] != self.n_cols:
            raise ValueError(f"hash_ids must be [B, T, {self.n_cols}]")
        return hash_ids.shape[0], hash_ids.shape[1]

    def _mask(self, token_mask, B, T):
        if token_mask is None:
            return None
        if token_mask.dtype == torch.bool:
            token_mask = token_mask.view(torch.uint8)
        _need(token_mask, "token_mask", (torch.uint8,), (B, T), self.device)
        return token_mask

    def forward(self, hash_ids, x, token_mask=None, out=None, stream=None):
        """out = Engram(x); out may be x (in place)."""
        B, T = self._tokens(hash_ids)
        _need(x, "x", _U16, (B, T, self.hc_mult, self.dim), self.device)
        m = self._mask(token_mask, B, T)
        if out is None:
            out = torch.empty_like(x)
        _need(out, "out", _U16, tuple(x.shape), self.device)
        check(self._lib.engram_forward(self._ctx, _ptr(hash_ids), _ptr(x), _ptr(m), _ptr(out), B, T,
                                       _stream(stream)), "engram_forward")
        return out

    __call__ = forward

    def lookup_project(self, hash_ids, kv=None, stream=None):
        B, T = self._tokens(hash_ids)
        if kv is None:
            kv = torch.empty((B, T, self.N), dtype=torch.bfloat16, device=self.device)
        _need(kv, "kv", _U16, (B, T, self.N), self.device)
        check(self._lib.engram_lookup_project(self._ctx, _ptr(hash_ids), _ptr(kv), B, T, _stream(stream)),
              "engram_lookup_project")
        return kv

    def gate_apply(self, kv, x, token_mask=None, out=None, gates=None, stream=None):
        B, T = x.shape[0], x.shape[1]
        _need(kv, "kv", _U16, (B, T, self.N), self.device)
        _need(x, "x", _U16, (B, T, self.hc_mult, self.dim), self.device)
        m = self._mask(token_mask, B, T)
        if out is None:
            out = torch.empty_like(x)
        _need(out, "out", _U16, tuple(x.shape), self.device)
        if gates is not None:
            _need(gates, "gates", (torch.float32,), (B, T, self.hc_mult), self.device)
        check(self._lib.engram_gate_apply(self._ctx, _ptr(kv), _ptr(x), _ptr(m), _ptr(out), _ptr(gates), B, T,
                                          _stream(stream)), "engram_gate_apply")
        return out

    def lookup(self, hash_ids, rows=None, stream=None):
        B, T = self._tokens(hash_ids)
        if rows is None:
            rows = torch.empty((B, T, self.K), dtype=torch.bfloat16, device=self.device)
        _need(rows, "rows", _U16, (B, T, self.K), self.device)
        check(self._lib.engram_lookup(self._ctx, _ptr(hash_ids), _ptr(rows), B, T, _stream(stream)),
              "engram_lookup")
        return rows

    def forward_rows(self, rows, x, token_mask=None, out=None, stream=None):
        """out = Engram(x) from gathered rows [B, T, n_cols*head_dim] bf16 (as
        lookup() writes them, or their sum over the shards of a row-split
        table); out may be x."""
        B, T = x.shape[0], x.shape[1]
        _need(rows, "rows", _U16, (B, T, self.K), self.device)
        _need(x, "x", _U16, (B, T, self.hc_mult, self.dim), self.device)
        m = self._mask(token_mask, B, T)
        if out is None:
            out = torch.empty_like(x)
        _need(out, "out", _U16, tuple(x.shape), self.device)
        check(self._lib.engram_forward_rows(self._ctx, _ptr(rows), _ptr(x), _ptr(m), _ptr(out), B, T,
                                            _stream(stream)), "engram_forward_rows")
        return out

    def sync_status(self, stream=None):
        """(status, bad_ids): waits for the stream, returns and clears the
        device-detected error."""
        bad = ctypes.c_int64(0)
        st = self._lib.engram_sync_status(self._ctx, _stream(stream), ctypes.byref(bad))
        return st, bad.value

    def plan(self, m_tokens):
        s, c = ctypes.c_int32(0), ctypes.c_int32(0)
        check(self._lib.engram_plan(self._ctx, m_tokens, ctypes.byref(s), ctypes.byref(c)), "engram_plan")
        return s.value, c.value

    def describe_plan(self, m_tokens):
        """The projection's plan for m_tokens tokens as a dict (engram_describe_plan)."""
        info = _lib.EngramPlanInfo()
        check(self._lib.engram_describe_plan(self._ctx, m_tokens, ctypes.byref(info)), "engram_describe_plan")
        return {f: getattr(info, f) for f, _ in info._fields_}

    def forward_kernels(self, m_tokens):
        """How many kernels one forward over m_tokens tokens launches."""
        k = ctypes.c_int32(0)
        check(self._lib.engram_forward_kernels(self._ctx, m_tokens, ctypes.byref(k)), "engram_forward_kernels")
        return k.value

    def set_sm_budget(self, sms: int):
        """At most `sms` SMs for the projection's grid (0 = all of them)."""
        check(self._lib.engram_set_sm_budget(self._ctx, sms), "engram_set_sm_budget")

    def enable_stage_timing(self, enable=True, calls=1):
        """Records stage events for the last `calls` forward / lookup_project
        calls (engram_enable_stage_timing); enable=False drops them."""
        n = int(calls) if enable else 0
        check(self._lib.engram_enable_stage_timing(self._ctx, n), "engram_enable_stage_timing")

    def stage_times(self):
        """(gather, projection, gate) milliseconds of the last forward /
        lookup_project call, from CUDA events on its stream."""
        ms = (ctypes.c_float * 3)()
        check(self._lib.engram_stage_times(self._ctx, ms), "engram_stage_times")
        return tuple(ms)

    def stage_times_n(self, n):
        """[(gather, projection, gate)] milliseconds of the last n calls, oldest first."""
        ms = (ctypes.c_float * (3 * n))()
        check(self._lib.engram_stage_times_n(self._ctx, n, ms), "engram_stage_times_n")
        return [tuple(ms[3 * i:3 * i + 3]) for i in range(n)]

    def close(self):
        if getattr(self, "_ctx", None) is not None and self._ctx.value:
            self._lib.engram_destroy(self._ctx)
            self._ctx = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def shard_rows(num_rows: int, rank: int, world_size: int) -> tuple[int, int]:
    """Rows [start, end) of the table that `rank` of `world_size` holds when
    the table is split by rows the way `ParallelEngramEmbedding` splits it
    (atlas.klimoza.dev "deepseek-v4.1 / engram-second"): P = ceil(R /
    world_size) rows per rank, rank r from r*P.  The last shard ends at R
    (the excerpt's last part is padded to P rows that no id reaches)."""
    if world_size < 1 or not 0 <= rank < world_size or num_rows < 0:
        raise ValueError("need 0 <= rank < world_size and num_rows >= 0")
    part = -(-num_rows // world_size)
    start = min(rank * part, num_rows)
    return start, min(start + part, num_rows)


def exchange_rows(rows: torch.Tensor, group=None) -> torch.Tensor:
    """The one exchange of the row-split layer, in place: every rank's
    gathered rows (zero for ids outside its shard) summed over the ranks of
    `group`, the `dist.all_reduce` of `ParallelEngramEmbedding.forward`.  The
    sum runs on the rows' bit patterns as 32-bit integers: exactly one rank
    holds each row and the others hold zero bits, so the sum is that rank's
    bits exactly -- including -0.0, which a floating-point sum would turn into
    +0.0.  A no-op without an initialised process group of more than one
    rank.  Collective: every rank of the group must call it."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size(group) == 1:
        return rows
    if rows.element_size() * rows.numel() % 4 != 0 or not rows.is_contiguous():
        raise ValueError("rows must be contiguous and a whole number of 32-bit words")
    dist.all_reduce(rows.view(torch.int32), op=dist.ReduceOp.SUM, group=group)
    return rows


class EngramShard:
    """One rank's part of an Engram layer whose table is split by rows over
    the ranks of a process group (one GPU per rank), as `ParallelEngramEmbedding`
    splits it: this rank holds rows shard_rows(R, rank, world_size) of the
    table (table and scale are that shard), wkv and q/k weights whole.

    forward(): engram_lookup on the shard (zero rows for ids outside it) ->
    exchange_rows (one all-reduce of [B*T, n_cols*head_dim] bf16 over the
    group) -> engram_forward_rows.  Every rank passes the same hash ids and x
    and gets the whole layer's output; with one rank it equals
    EngramLayer.forward bit for bit.  Keyword arguments are EngramLayer's
    (bf16 weight only)."""

    def __init__(self, table, scale, wkv, q_weight, k_weight, *, num_rows, group=None, **kw):
        import torch.distributed as dist
        dist_on = dist.is_available() and dist.is_initialized()
        self.group = group
        self.rank = dist.get_rank(group) if dist_on else 0
        self.world_size = dist.get_world_size(group) if dist_on else 1
        start, end = shard_rows(num_rows, self.rank, self.world_size)
        if table.shape[0] != end - start:
            raise ValueError(f"rank {self.rank} holds rows [{start}, {end}): table has {table.shape[0]} rows")
        if kw.get("wkv_scale") is not None:
            raise ValueError("the row-split layer takes the bf16 weight")
        self.layer = EngramLayer(table, scale, wkv, q_weight, k_weight, row_offset=start, **kw)
        self.rows_range = (start, end)

    def forward(self, hash_ids, x, token_mask=None, out=None, rows=None):
        """out = Engram(x), on the current torch stream; rows: optional
        [B, T, K] bf16 buffer for the exchanged rows."""
        rows = self.layer.lookup(hash_ids, rows=rows)
        exchange_rows(rows, self.group)
        return self.layer.forward_rows(rows, x, token_mask, out=out)

    __call__ = forward

    def close(self):
        self.layer.close()


class EngramHasher:
    """The n-gram hash of every Engram layer of a model (include/engram.h,
    engram_hash), with its session cache.

    token_map: int32 [vocab]; multipliers: int64 [n_layers, max_ngram_size];
    primes: int64 [n_layers, max_ngram_size-1, n_heads]; offsets: int64
    [n_layers, (max_ngram_size-1)*n_heads]; all on one CUDA device.  The cache
    ([max_batch, max_len] int32) is allocated here and holds each sequence's
    compressed history between calls."""

    def __init__(self, token_map, multipliers, primes, offsets, *, max_batch, max_len, pad_id=2, dead_id=-1):
        dev = token_map.device
        n_layers, n = multipliers.shape
        heads = primes.shape[2]
        _need(token_map, "token_map", (torch.int32,), None, dev)
        _need(multipliers, "multipliers", (torch.int64,), (n_layers, n), dev)
        _need(primes, "primes", (torch.int64,), (n_layers, n - 1, heads), dev)
        _need(offsets, "offsets", (torch.int64,), (n_layers, (n - 1) * heads), dev)
        self.device = dev
        self.n_layers, self.cols = n_layers, (n - 1) * heads
        self.cfg = EngramHashConfig(n_layers=n_layers, max_ngram_size=n, n_heads=heads, max_batch=max_batch,
                                    max_len=max_len, vocab_size=token_map.numel(), pad_id=pad_id, dead_id=dead_id)
        self.cache = torch.zeros((max_batch, max_len), dtype=torch.int32, device=dev)
        self._keep = (token_map, multipliers, primes, offsets)
        self._lib = _lib.engram()

    def __call__(self, input_ids, start_pos=0, token_mask=None, out=None, stream=None):
        """hash ids [n_layers, B, L, cols] for positions [start_pos, start_pos + L)."""
        _need(input_ids, "input_ids", (torch.int64,), None, self.device)
        B, L = input_ids.shape
        if token_mask is not None:
            if token_mask.dtype == torch.bool:
                token_mask = token_mask.view(torch.uint8)
            _need(token_mask, "token_mask", (torch.uint8,), (B, L), self.device)
        if out is None:
            out = torch.empty((self.n_layers, B, L, self.cols), dtype=torch.int64, device=self.device)
        _need(out, "out", (torch.int64,), (self.n_layers, B, L, self.cols), self.device)
        tm, mu, pr, of = self._keep
        check(self._lib.engram_hash(ctypes.byref(self.cfg), _ptr(tm), _ptr(mu), _ptr(pr), _ptr(of), _ptr(self.cache),
                                    _ptr(input_ids), _ptr(token_mask), start_pos, _ptr(out), B, L, _stream(stream)),
              "engram_hash")
        return out


class EngramRunAhead:
    """Run-ahead schedule of the Engram layers of one model step.

    The lookup and the projection depend only on the token ids, so they can
    run ahead of the backbone; only the gate needs the hidden state at the
    layer's entry (zhuai.tech "Engram in DeepSeek V4.1 Flash", section "Run
    projection early: overlap CPU work with the GPU"; monishver11.github.io
    "DeepSeek's Other Modules", section "Serving cost: gathers, not FLOPs": the
    addresses are known early, so the fetch overlaps the first block).

    issue(hash_ids_per_layer) queues every layer's engram_lookup_project on a
    side stream as soon as the ids are ready on the caller's stream;
    apply(i, x, ...) makes the caller's stream wait for layer i's kv and runs
    engram_gate_apply there.  The result equals each layer's engram_forward
    bit for bit.  One kv buffer per layer ([max_tokens, N] bf16) is owned
    here; the next issue() waits for the caller's stream, so it never
    overwrites a kv an earlier apply() still reads."""

    def __init__(self, layers, max_tokens: int, sm_budget=None):
        """sm_budget: if given (one count for every layer, or one per layer),
        the layers' projections are capped at that many SMs
        (engram_set_sm_budget; 0 = all), leaving the rest to the caller's
        stream.  A layer far from the step's start can trickle on a few SMs
        while the backbone runs; the first one is needed soon and takes all."""
        if not layers:
            raise ValueError("at least one layer")
        self.layers = list(layers)
        self.device = self.layers[0].device
        for lay in self.layers:
            if lay.device != self.device:
                raise ValueError("all layers must be on one device")
        self.max_tokens = max_tokens
        self.side = torch.cuda.Stream(self.device)
        self._kv = [torch.empty((max_tokens, lay.N), dtype=torch.bfloat16, device=self.device) for lay in self.layers]
        self._ready = [torch.cuda.Event() for _ in self.layers]
        self._shape = None
        if sm_budget is not None:
            budgets = list(sm_budget) if isinstance(sm_budget, (list, tuple)) else [sm_budget] * len(self.layers)
            if len(budgets) != len(self.layers):
                raise ValueError("one SM budget per layer")
            for lay, b in zip(self.layers, budgets):
                lay.set_sm_budget(int(b))

    def issue(self, hash_ids_per_layer, stream=None):
        """Queues lookup_project of every layer on the side stream, after the
        work already queued on `stream` (the current stream by default)."""
        if len(hash_ids_per_layer) != len(self.layers):
            raise ValueError("one hash-id tensor per layer")
        main = torch.cuda.current_stream(self.device) if stream is None else stream
        B, T = hash_ids_per_layer[0].shape[0], hash_ids_per_layer[0].shape[1]
        if B * T > self.max_tokens:
            raise ValueError(f"{B * T} tokens exceed max_tokens {self.max_tokens}")
        self.side.wait_stream(main)
        for i, (lay, ids) in enumerate(zip(self.layers, hash_ids_per_layer)):
            if ids.shape[0] != B or ids.shape[1] != T:
                raise ValueError("every layer's hash ids must cover the same [B, T]")
            kv = self._kv[i][: B * T].view(B, T, lay.N)
            lay.lookup_project(ids, kv=kv, stream=self.side)
            self._ready[i].record(self.side)
        self._shape = (B, T)

    def apply(self, i, x, token_mask=None, out=None, gates=None, stream=None):
        """Layer i at its entry: waits (on `stream`) for its kv, then gates."""
        if self._shape is None:
            raise RuntimeError("issue() first")
        B, T = self._shape
        main = torch.cuda.current_stream(self.device) if stream is None else stream
        main.wait_event(self._ready[i])
        kv = self._kv[i][: B * T].view(B, T, self.layers[i].N)
        return self.layers[i].gate_apply(kv, x, token_mask, out=out, gates=gates, stream=main)
