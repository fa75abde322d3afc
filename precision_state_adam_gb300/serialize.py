"""Save and restore optimizer state (moments, codes, scales, step) in one file.

AiDotNet PR #814 ("add 8-bit Adam optimizer for memory efficiency") serializes the 8-bit
optimizer as its options, a flag telling whether both moments are compressed, the first
moment (codes + scales, or full precision), a marker telling whether a quantized second
moment follows, and that moment's codes and scales. This module writes the same facts for
every moment mode of this library, host side (the state is a handful of caller-owned
tensors; nothing here is on the update's hot path).

File layout, little-endian:
    8 bytes   magic b"PSADAMST"
    u32       format version (1)
    u32       n = length of the JSON header that follows
    n bytes   UTF-8 JSON: {"mode", "step", "block_size", "compress_both_moments",
              "has_v_quantized", "hparams", "q8", "numel": [...], "arrays": [[name, dtype,
              count], ...]}
    ...       the arrays in the order listed, raw bytes (bf16 as its 16-bit patterns)
    u32       CRC-32 (zlib) of every byte before it
"""
from __future__ import annotations

import json
import struct
import zlib
from typing import BinaryIO

import torch

MAGIC = b"PSADAMST"
VERSION = 1
BLOCK = 2048       # default 8-bit block size
MAX_BLOCK = 16384  # largest block size the library accepts

# per mode: the state tensors of one parameter tensor, as (name, dtype, count kind)
_LAYOUT = {
    "fp32": (("m", torch.float32, "n"), ("v", torch.float32, "n")),
    "bf16m": (("m", torch.bfloat16, "n"), ("v", torch.bfloat16, "n")),
    "q8": (("m_code", torch.int8, "n"), ("v_code", torch.uint8, "n"),
           ("m_scale", torch.float32, "b"), ("v_scale", torch.float32, "b")),
    "q8v": (("m", torch.float32, "n"), ("v_code", torch.uint8, "n"), ("v_scale", torch.float32, "b")),
}
_DTYPE_NAME = {torch.float32: "f32", torch.bfloat16: "bf16", torch.int8: "i8", torch.uint8: "u8"}
_NAME_DTYPE = {v: k for k, v in _DTYPE_NAME.items()}


class StateFormatError(ValueError):
    pass


def _count(kind: str, n: int, bs: int) -> int:
    return n if kind == "n" else (n + bs - 1) // bs


def _raw(t: torch.Tensor) -> bytes:
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.numpy().tobytes()


def save_state(f: str | BinaryIO, mode: str, state, step: int, hparams: dict | None = None,
               q8: dict | None = None, block_size: int = BLOCK) -> None:
    """Write ``state`` (as returned by ``zeros_state(params, mode, block_size)``), the number
    of steps taken, and optionally the hyper-parameters and 8-bit options."""
    if mode not in _LAYOUT:
        raise ValueError(f"unknown moment mode {mode!r}")
    if not 1 <= block_size <= MAX_BLOCK:
        raise ValueError(f"block size {block_size} outside 1..{MAX_BLOCK}")
    layout = _LAYOUT[mode]
    if len(state) != len(layout):
        raise ValueError(f"{mode} state has {len(layout)} parts, got {len(state)}")
    numel = [int(t.numel()) for t in state[0]]
    arrays, blobs = [], []
    for i, n in enumerate(numel):
        for (name, dtype, kind), part in zip(layout, state):
            t = part[i]
            if t.dtype != dtype or t.numel() != _count(kind, n, block_size):
                raise ValueError(f"tensor {i} {name}: expected {_count(kind, n, block_size)} x {dtype}, "
                                 f"got {t.numel()} x {t.dtype}")
            arrays.append([f"{i}.{name}", _DTYPE_NAME[dtype], t.numel()])
            blobs.append(_raw(t))
    header = {
        "mode": mode, "step": int(step), "block_size": int(block_size),
        "compress_both_moments": mode == "q8", "has_v_quantized": mode in ("q8", "q8v"),
        "hparams": hparams or {}, "q8": q8 or {}, "numel": numel, "arrays": arrays,
    }
    hb = json.dumps(header, sort_keys=True).encode()
    body = MAGIC + struct.pack("<II", VERSION, len(hb)) + hb + b"".join(blobs)
    data = body + struct.pack("<I", zlib.crc32(body) & 0xFFFFFFFF)
    if isinstance(f, str):
        with open(f, "wb") as fh:
            fh.write(data)
    else:
        f.write(data)


def load_state(f: str | BinaryIO, device=None):
    """Read a state file. Returns (mode, state, step, header); ``state`` has the layout of
    ``zeros_state(..., mode)`` with tensors on ``device`` (default CPU)."""
    data = open(f, "rb").read() if isinstance(f, str) else f.read()
    if len(data) < 20 or data[:8] != MAGIC:
        raise StateFormatError("not a psadam state file")
    (crc,) = struct.unpack("<I", data[-4:])
    if zlib.crc32(data[:-4]) & 0xFFFFFFFF != crc:
        raise StateFormatError("checksum mismatch: the file is damaged")
    version, hlen = struct.unpack("<II", data[8:16])
    if version != VERSION:
        raise StateFormatError(f"unsupported format version {version}")
    if 16 + hlen > len(data) - 4:
        raise StateFormatError("header runs past the end of the file")
    try:
        header = json.loads(data[16:16 + hlen].decode())
        mode = header["mode"]
        bs = header.get("block_size")
        flags = (header["compress_both_moments"], header["has_v_quantized"])
        numel, arrays = header["numel"], header["arrays"]
        int(header["step"])
    except (ValueError, UnicodeDecodeError, KeyError, TypeError, AttributeError) as e:
        raise StateFormatError(f"unreadable header: {e}") from None
    if mode not in _LAYOUT or not isinstance(bs, int) or not 1 <= bs <= MAX_BLOCK:
        raise StateFormatError(f"unsupported mode / block size: {mode}, {bs}")
    if flags != (mode == "q8", mode in ("q8", "q8v")):
        raise StateFormatError("flags disagree with the moment mode")
    if not isinstance(numel, list) or not all(isinstance(n, int) and n >= 0 for n in numel):
        raise StateFormatError("numel must be a list of non-negative integers")
    layout = _LAYOUT[mode]
    if not isinstance(arrays, list) or len(arrays) != len(numel) * len(layout) or \
            not all(isinstance(a, list) and len(a) == 3 for a in arrays):
        raise StateFormatError(f"array list does not match {len(numel)} tensors of the {mode} layout")
    parts = [[] for _ in layout]
    off = 16 + hlen
    it = iter(arrays)
    for i, n in enumerate(numel):
        for j, (name, dtype, kind) in enumerate(layout):
            aname, dname, count = next(it)
            if aname != f"{i}.{name}" or _NAME_DTYPE.get(dname) != dtype or count != _count(kind, n, bs):
                raise StateFormatError(f"array {aname} does not match the {mode} layout")
            size = count * (2 if dtype == torch.bfloat16 else torch.empty(0, dtype=dtype).element_size())
            raw = bytearray(data[off:min(off + size, len(data) - 4)])  # never into the checksum
            if len(raw) != size:
                raise StateFormatError("file is truncated")
            off += size
            if dtype == torch.bfloat16:
                t = torch.frombuffer(raw, dtype=torch.int16).view(torch.bfloat16) if count else torch.empty(0, dtype=dtype)
            else:
                t = torch.frombuffer(raw, dtype=dtype) if count else torch.empty(0, dtype=dtype)
            parts[j].append(t.clone().to(device) if device is not None else t.clone())
    if off != len(data) - 4:
        raise StateFormatError("trailing bytes after the last array")
    return mode, tuple(parts), int(header["step"]), header
