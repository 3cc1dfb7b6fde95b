"""Device side of the seeded input generators: fills a synthetic table on the
GPU with the device twin (include/engram_synth.h) of synth.table_rows(), and
uploads the host-made small inputs of a workload.  Input generation only."""
from __future__ import annotations

import numpy as np
import torch

from . import _lib, synth


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise RuntimeError(f"{where} failed with {rc}")


def _cuda_device(t: torch.Tensor) -> torch.device:
    """The device whose kernels fill t: its own, or the current CUDA device for
    a pinned host tensor (written in place over the host link)."""
    if t.is_cuda:
        return t.device
    if not t.is_pinned():
        raise ValueError("a host tensor filled by the device generator must be pinned")
    return torch.device("cuda", torch.cuda.current_device())


def fill_table(table: torch.Tensor, scale: torch.Tensor | None, seed: int, scale_block: int = 128,
               row_begin: int = 0, row_end: int | None = None, stream=None) -> None:
    """Writes rows [row_begin, row_end) of a uint8 [R, head_dim] table and its
    fp32 [R, head_dim/scale_block] scales exactly as synth.table_rows(seed, ...)."""
    lib = _lib.synth()
    R, head_dim = table.shape
    row_end = R if row_end is None else row_end
    dev = _cuda_device(table)
    cq = torch.from_numpy(synth.code_quantile_table().copy()).to(dev)
    sq = torch.from_numpy(synth.scale_quantile_table().copy()).to(dev)
    st = torch.cuda.current_stream(dev).cuda_stream if stream is None else int(stream)
    chunk = 1 << 26   # rows per launch
    for b in range(row_begin, row_end, chunk):
        e = min(row_end, b + chunk)
        _check(lib.engram_synth_fill_table(table.data_ptr(), None if scale is None else scale.data_ptr(), b, e,
                                           head_dim, scale_block, synth.stream_key(seed, synth.TAG_CODES),
                                           synth.stream_key(seed, synth.TAG_SCALES), cq.data_ptr(), sq.data_ptr(),
                                           st), "engram_synth_fill_table")
    torch.cuda.current_stream(dev).synchronize()


def fill_scales_e8m0(scale: torch.Tensor, seed: int, head_dim: int, scale_block: int, stream=None) -> None:
    """Writes the E8M0 scales (uint8 [R, head_dim/scale_block]) exactly as
    synth.table_rows(seed, ..., scale_fmt=1)."""
    lib = _lib.synth()
    R = scale.shape[0]
    dev = _cuda_device(scale)
    eq = torch.from_numpy(synth.e8m0_quantile_table().copy()).to(dev)
    st = torch.cuda.current_stream(dev).cuda_stream if stream is None else int(stream)
    _check(lib.engram_synth_fill_scales_e8m0(scale.data_ptr(), 0, R, head_dim, scale_block,
                                             synth.stream_key(seed, synth.TAG_SCALES), eq.data_ptr(), st),
           "engram_synth_fill_scales_e8m0")
    torch.cuda.current_stream(dev).synchronize()


def make_table(w: synth.Workload, device="cuda", num_rows: int | None = None, host: bool = False):
    """(table uint8 [R, head_dim], scales [R, head_dim/scale_block]) on the
    device, or in pinned host memory with host=True (filled in place by the
    device generator): fp32 scales, or E8M0 bytes for the mxfp8 format."""
    R = w.num_rows() if num_rows is None else num_rows
    nb = w.head_dim // w.scale_block
    sdt = torch.uint8 if w.scale_fmt == 1 else torch.float32
    if host:
        table = torch.empty((R, w.head_dim), dtype=torch.uint8, pin_memory=True)
        scale = torch.empty((R, nb), dtype=sdt, pin_memory=True)
    else:
        table = torch.empty((R, w.head_dim), dtype=torch.uint8, device=device)
        scale = torch.empty((R, nb), dtype=sdt, device=device)
    if w.scale_fmt == 1:
        fill_table(table, None, w.seed, w.scale_block)
        fill_scales_e8m0(scale, w.seed, w.head_dim, w.scale_block)
    else:
        fill_table(table, scale, w.seed, w.scale_block)
    return table, scale


def bits_to_device(a: np.ndarray, device="cuda", dtype=torch.bfloat16) -> torch.Tensor:
    """uint16 bit patterns -> a device tensor of the given 16-bit dtype."""
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.to(device).view(dtype)


def device_bits(t: torch.Tensor) -> np.ndarray:
    """A 16-bit device tensor -> uint16 bit patterns on the host."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def upload_inputs(inp: synth.HostInputs, device="cuda"):
    """dict of device tensors: hash_ids, x, mask, wkv, q, k, wkv_scale (None
    for a bf16 weight; for the mxfp8 format wkv holds the uint8 codes)."""
    fp8 = inp.wkv_scale is not None
    return dict(
        hash_ids=torch.from_numpy(inp.hash_ids).to(device),
        x=bits_to_device(inp.x, device),
        mask=None if inp.mask is None else torch.from_numpy(inp.mask).to(device),
        wkv=torch.from_numpy(inp.wkv).to(device) if fp8 else bits_to_device(inp.wkv, device),
        q=bits_to_device(inp.q, device),
        k=bits_to_device(inp.k, device),
        wkv_scale=torch.from_numpy(inp.wkv_scale).to(device) if fp8 else None,
    )
