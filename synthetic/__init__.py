"""Seeded synthetic inputs for the FP8 FFN sublayer workloads.

This module is shared by the oracle tests, the GPU tests and the benchmark.
It holds no arithmetic of the method itself: it only draws seeded normal
numbers, scales them, marks outlier channels and rounds them to BF16 (torch's
round-to-nearest-even cast).

Workload shapes stand in for the pages' own workloads, which used real
checkpoints and robot observations that are not available here:
  * VLA action expert (action chunk of 50 tokens, Gemma-expert width) and VLA
    prefix (2 camera views x 256 SigLIP tokens + 456 text tokens), from the
    itsolotime FlashRT article, 6.2 (SigLIP 256 tokens per view) and 3.1
    (num_views=2);
  * batch-1 LLM decode and long prefill at Qwen3.6-27B-like width, from the
    itsolotime article, 8.1 and 2.2 (Qwen3.6-27B NVFP4 decode).

Recipe (seeded per workload):
  * residual and hidden ~ N(0, 1), fp32 -> BF16;
  * outlier workloads: ceil(0.001 d) channels, chosen by a seeded permutation,
    multiplied by 20 in the residual, hidden and calibration batches alike;
  * RMSNorm weight = 1 + N(0, 0.1); W_gate, W_up, W_down ~ N(0, 0.02);
  * calibration: 4 batches of M rows for the tiny workload, 1 batch otherwise.
Each tensor has its own seed derived from (workload seed, stream, layer), so
any layer can be generated alone.  Generation runs on a chosen torch device;
the CPU and CUDA generators give different numbers for the same seed, so a
test draws once and hands the same tensors to both sides.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

GEGLU_TANH = "geglu_tanh"
SWIGLU = "swiglu"


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    d: int
    ff: int
    act: str
    L: int
    seed: int
    outliers: bool
    n_calib: int

    @property
    def act_id(self) -> int:
        return 0 if self.act == GEGLU_TANH else 1

    @property
    def weight_bytes_per_layer(self) -> int:
        return 3 * self.d * self.ff

    def with_(self, **kw) -> "Workload":
        fields = dict(self.__dict__)
        fields.update(kw)
        return Workload(**fields)


WORKLOADS = {
    "tiny": Workload("tiny", M=8, d=256, ff=1024, act=GEGLU_TANH, L=1, seed=0, outliers=False, n_calib=4),
    "vla_action_expert": Workload("vla_action_expert", M=50, d=1024, ff=4096, act=GEGLU_TANH, L=18, seed=1,
                                  outliers=True, n_calib=1),
    "vla_prefix": Workload("vla_prefix", M=968, d=2048, ff=16384, act=GEGLU_TANH, L=18, seed=2,
                           outliers=True, n_calib=1),
    "llm_decode": Workload("llm_decode", M=1, d=5120, ff=17408, act=SWIGLU, L=64, seed=3,
                           outliers=False, n_calib=1),
    "long_prefill": Workload("long_prefill", M=8192, d=5120, ff=17408, act=SWIGLU, L=4, seed=4,
                             outliers=True, n_calib=1),
}

# Attention-input projections of each workload's model family (readings: the
# pages name the models, not their heads): (query heads, key/value heads,
# head dim, RoPE base) -- Gemma-style 8 query heads sharing one 256-wide
# key/value head for the VLA shapes (base 10^4), a Qwen-style 40 / 8 heads of
# 128 at width 5120 (base 10^6) for the LLM shapes.
ATTENTION = {
    "tiny": (4, 1, 64, 1.0e4),
    "vla_action_expert": (8, 1, 256, 1.0e4),
    "vla_prefix": (8, 1, 256, 1.0e4),
    "llm_decode": (40, 8, 128, 1.0e6),
    "long_prefill": (40, 8, 128, 1.0e6),
}
DECODE_CONTEXT = 4096  # the decoded token's position in the LLM decode workload

# sub-stream identifiers
_S_WNORM, _S_WGATE, _S_WUP, _S_WDOWN, _S_RES, _S_HID, _S_OUTL = range(7)
_S_WQ, _S_WK, _S_WV, _S_WNORM_ATTN = range(7, 11)
_S_MOD = 11
_S_CALIB_BASE = 1000


def _seed(*parts: int) -> int:
    return int(np.random.SeedSequence([int(p) for p in parts]).generate_state(1, dtype=np.uint64)[0] >> 1)


def _normal(shape, seed: int, device) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def outlier_channels(wl: Workload) -> list[int]:
    if not wl.outliers:
        return []
    k = math.ceil(0.001 * wl.d)
    g = torch.Generator(device="cpu")
    g.manual_seed(_seed(wl.seed, _S_OUTL))
    return sorted(torch.randperm(wl.d, generator=g)[:k].tolist())


def layer_weights(wl: Workload, layer: int, device="cpu") -> dict[str, torch.Tensor]:
    """BF16 master weights of one layer: w_norm [d], w_gate [ff,d], w_up [ff,d], w_down [d,ff]."""
    s = wl.seed
    w_norm = 1.0 + 0.1 * _normal((wl.d,), _seed(s, _S_WNORM, layer), device)
    w_gate = 0.02 * _normal((wl.ff, wl.d), _seed(s, _S_WGATE, layer), device)
    w_up = 0.02 * _normal((wl.ff, wl.d), _seed(s, _S_WUP, layer), device)
    w_down = 0.02 * _normal((wl.d, wl.ff), _seed(s, _S_WDOWN, layer), device)
    return {k: v.to(torch.bfloat16) for k, v in
            dict(w_norm=w_norm, w_gate=w_gate, w_up=w_up, w_down=w_down).items()}


def modulation(wl: Workload, layer: int, rows: int, device="cpu") -> torch.Tensor:
    """AdaRMSNorm modulation of one layer, BF16 [rows, 3d] = [scale | shift | gate]
    (the outputs of the conditioning Dense layers): scale, shift ~ N(0, 0.1),
    gate ~ 1 + N(0, 0.1); rows = 1 (one conditioning for all tokens) or M."""
    z = _normal((rows, 3 * wl.d), _seed(wl.seed, _S_MOD, layer), device)
    z = 0.1 * z
    z[:, 2 * wl.d:] += 1.0
    return z.to(torch.bfloat16)


def qkv_weights(wl: Workload, layer: int, device="cpu") -> dict[str, torch.Tensor]:
    """BF16 attention-input weights of one layer: w_norm [d], w_q [Hq hd, d],
    w_k [Hkv hd, d], w_v [Hkv hd, d]; same distributions as the FFN's."""
    nq, nkv, hd, _ = ATTENTION.get(wl.name, ATTENTION["tiny"])
    s = wl.seed
    w = dict(w_norm=1.0 + 0.1 * _normal((wl.d,), _seed(s, _S_WNORM_ATTN, layer), device),
             w_q=0.02 * _normal((nq * hd, wl.d), _seed(s, _S_WQ, layer), device),
             w_k=0.02 * _normal((nkv * hd, wl.d), _seed(s, _S_WK, layer), device),
             w_v=0.02 * _normal((nkv * hd, wl.d), _seed(s, _S_WV, layer), device))
    return {k: v.to(torch.bfloat16) for k, v in w.items()}


def positions(wl: Workload, M: int | None = None) -> np.ndarray:
    """Token positions (int32): the decode workload's token sits after a
    DECODE_CONTEXT-token context; the other workloads start at 0."""
    M = wl.M if M is None else M
    p0 = DECODE_CONTEXT if wl.name == "llm_decode" else 0
    return (p0 + np.arange(M)).astype(np.int32)


def _activation(wl: Workload, M: int, seed: int, device) -> torch.Tensor:
    x = _normal((M, wl.d), seed, device)
    ch = outlier_channels(wl)
    if ch:
        idx = torch.tensor(ch, device=device, dtype=torch.long)
        x[:, idx] *= 20.0
    return x.to(torch.bfloat16)


def inputs(wl: Workload, device="cpu", M: int | None = None) -> tuple[torch.Tensor, torch.Tensor]:
    """(residual, hidden) BF16 [M,d] for the timed / compared forward."""
    M = wl.M if M is None else M
    return (_activation(wl, M, _seed(wl.seed, _S_RES), device),
            _activation(wl, M, _seed(wl.seed, _S_HID), device))


def calibration_batches(wl: Workload, device="cpu", M: int | None = None):
    """[(residual_b, hidden_b)] for b < n_calib, each BF16 [M,d]."""
    M = wl.M if M is None else M
    out = []
    for b in range(wl.n_calib):
        out.append((_activation(wl, M, _seed(wl.seed + _S_CALIB_BASE + b, _S_RES), device),
                    _activation(wl, M, _seed(wl.seed + _S_CALIB_BASE + b, _S_HID), device)))
    return out


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """BF16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bf16_bits(a: np.ndarray, device="cpu") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).to(device)
