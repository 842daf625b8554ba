"""Loader for the hand-derived golden streams under tests/golden/."""
from __future__ import annotations

import glob
import os
import struct

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def distinct_u32(n: int) -> np.ndarray:
    # (i + 1) * odd constant mod 2^32 is a bijection, so the words are distinct
    i = np.arange(1, n + 1, dtype=np.uint64)
    return ((i * np.uint64(2654435761)) & np.uint64(0xFFFFFFFF)).astype(np.uint32)


def _make_input(spec: str) -> np.ndarray:
    kind, *args = spec.split()
    if kind == "repeat_u32":
        return np.full(int(args[1]), int(args[0], 0), np.uint32).view(np.uint8)
    if kind == "bytes":
        return np.frombuffer(bytes.fromhex(args[0]), np.uint8).copy()
    if kind == "period_distinct_u32":
        p, n = int(args[0]), int(args[1])
        return np.tile(distinct_u32(p), n // p + 1)[:n].view(np.uint8).copy()
    if kind == "zero_then_distinct_u32":
        n = int(args[0])
        return np.concatenate([np.zeros(n, np.uint32), distinct_u32(n)]).view(np.uint8)
    if kind == "distinct_u32_with":
        # n distinct words, then edits in order:
        #   copy:dst:src:len  w[dst + k] = w[src + k] for k < len
        #   set:i:value       w[i] = value
        #   pairs:start:count w[start + 2j + 1] = w[start + 2j] for j < count
        w = distinct_u32(int(args[0]))
        for op in args[1:]:
            name, *v = op.split(":")
            v = [int(t, 0) for t in v]
            if name == "copy":
                for k in range(v[2]):
                    w[v[0] + k] = w[v[1] + k]
            elif name == "set":
                w[v[0]] = v[1]
            elif name == "pairs":
                for j in range(v[1]):
                    w[v[0] + 2 * j + 1] = w[v[0] + 2 * j]
            else:
                raise ValueError(op)
        return w.view(np.uint8).copy()
    raise ValueError(spec)


def _layout_stream(layout: str, x: np.ndarray, ws: int, cs: int) -> np.ndarray:
    out = bytearray()
    n_chunks = (x.size + cs - 1) // cs
    for part in layout.split("|"):
        kind, *args = part.split()
        if kind == "header":
            out += struct.pack("<IHBBIIQQ", 0x5A4C5047, 1, ws, 0, cs, n_chunks, x.size,
                               int(args[0], 0))
        elif kind == "entry":
            out += struct.pack("<II", int(args[0], 0), int(args[1], 0))
        elif kind == "raw_copy_of_input":
            out += bytes(x[int(args[0]):int(args[1])])
        elif kind == "hex":
            out += bytes.fromhex("".join(args))
        else:
            raise ValueError(part)
    return np.frombuffer(bytes(out), np.uint8).copy()


def load_all():
    cases = []
    for path in sorted(glob.glob(os.path.join(GOLDEN_DIR, "*.txt"))):
        meta = {}
        hexlines = []
        in_stream = False
        with open(path) as f:
            for line in f:
                line = line.strip()
                if not line or line.startswith("#"):
                    continue
                if in_stream:
                    hexlines.append(line.replace(" ", ""))
                    continue
                key, _, val = line.partition(":")
                val = val.strip()
                if key == "stream":
                    in_stream = True
                    continue
                meta[key] = val
        ws = int(meta["word_size"])
        cs = int(meta["chunk_size"])
        levels = [int(v) for v in meta["match_level"].split()]
        windows = [int(v) for v in meta.get("window", "32").split()]
        x = _make_input(meta["input"])
        assert x.size == int(meta["n_bytes"])
        if hexlines:
            stream = np.frombuffer(bytes.fromhex("".join(hexlines)), np.uint8).copy()
        else:
            stream = _layout_stream(meta["stream_layout"], x, ws, cs)
        cases.append(dict(name=os.path.basename(path), ws=ws, cs=cs, levels=levels,
                          windows=windows, x=x, stream=stream))
    return cases
