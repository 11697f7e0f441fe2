"""Calibration cache ("FlashRT docs/architecture.md", 6 Calibration
Framework): the activation scales of a plan, saved as JSON under a key made
of a hash of the checkpoint and the token count, "{hash}_Se{M}.json", so a
later process with the same weights and M loads them instead of measuring.

A record holds the known fields (shape, activation, per-layer s_x, s_h and the
weight scales s_gu, s_down they were measured against) and a free-form
`extra` map.  A record whose shape or weight scales differ from the plan's is
stale and is not used.  Scales are fp32; JSON keeps them exactly (the decimal
repr of a float32 widened to a Python float parses back to the same float32).
Host code: no CUDA kernels (weights_digest reads tensors back to the host).
"""
from __future__ import annotations

import hashlib
import json
import math
import os
import struct

import torch

FORMAT = "frt_ffn_calibration/1"


def default_dir() -> str:
    """FRT_FFN_CALIB_DIR, else ~/.cache/frt_ffn/calibration."""
    return os.environ.get("FRT_FFN_CALIB_DIR") or os.path.join(os.path.expanduser("~"), ".cache", "frt_ffn",
                                                                "calibration")


def weights_digest(tag: bytes, tensors, chunk_elems: int = 1 << 26) -> str:
    """SHA-256 over every element of each tensor in order (its raw bytes,
    read in chunks so that host memory stays bounded), after a tag naming
    how the tensors are used (e.g. whether the norm weight is folded).  Two
    weight sets that differ in any element get different digests."""
    h = hashlib.sha256(tag)
    for t in tensors:
        flat = t.detach().reshape(-1)
        h.update(("%s:%d;" % (str(flat.dtype), flat.numel())).encode())
        raw = flat.view(torch.uint8) if flat.element_size() == 1 else flat.view(torch.int16) \
            if flat.element_size() == 2 else flat.view(torch.int32)
        for part in raw.split(chunk_elems):
            h.update(part.contiguous().cpu().numpy())
    return h.hexdigest()


def checkpoint_hash(shape: dict, layer_digests) -> str:
    """16 hex digits of SHA-256 over the plan shape and each layer's weight
    digest (None for a layer without weights)."""
    h = hashlib.sha256()
    h.update(json.dumps(shape, sort_keys=True).encode())
    for dg in layer_digests:
        h.update((dg or "-").encode())
        h.update(b"\0")
    return h.hexdigest()[:16]


def cache_key(ckpt_hash: str, M: int) -> str:
    if M < 1:
        raise ValueError("M must be >= 1")
    return "%s_Se%d" % (ckpt_hash, M)


def _f32(x) -> float:
    return struct.unpack("<f", struct.pack("<f", float(x)))[0]


def make_record(shape: dict, M: int, scales: dict, extra: dict | None = None) -> dict:
    rec = {"format": FORMAT, "M": int(M)}
    rec.update({k: shape[k] for k in ("d", "ff", "act", "n_layers")})
    for k in ("s_x", "s_h", "s_gu", "s_down"):
        v = [_f32(x) for x in scales[k]]
        if len(v) != shape["n_layers"]:
            raise ValueError("%s has %d entries for %d layers" % (k, len(v), shape["n_layers"]))
        rec[k] = v
    rec["extra"] = dict(extra or {})
    return rec


def save(directory: str, key: str, record: dict) -> str:
    """Write record to directory/key.json atomically; returns the path."""
    os.makedirs(directory, exist_ok=True)
    path = os.path.join(directory, key + ".json")
    tmp = "%s.tmp%d" % (path, os.getpid())
    with open(tmp, "w") as f:
        json.dump(record, f, indent=1)
    os.replace(tmp, path)
    return path


def load(directory: str, key: str, shape: dict, M: int, weight_scales: dict) -> dict | None:
    """The record under key if it exists and matches the plan (shape, M and
    weight scales, compared as fp32); None otherwise."""
    path = os.path.join(directory, key + ".json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if not isinstance(rec, dict) or rec.get("format") != FORMAT or rec.get("M") != M:
        return None
    if any(rec.get(k) != shape[k] for k in ("d", "ff", "act", "n_layers")):
        return None
    L = shape["n_layers"]
    for k in ("s_x", "s_h", "s_gu", "s_down"):
        v = rec.get(k)
        if not isinstance(v, list) or len(v) != L:
            return None
    for k in ("s_gu", "s_down"):
        if [_f32(x) for x in rec[k]] != [_f32(x) for x in weight_scales[k]]:
            return None
    if any(not (math.isfinite(_f32(x)) and _f32(x) > 0.0) for k in ("s_x", "s_h") for x in rec[k]):
        return None
    rec["s_x"] = [_f32(x) for x in rec["s_x"]]
    rec["s_h"] = [_f32(x) for x in rec["s_h"]]
    return rec
