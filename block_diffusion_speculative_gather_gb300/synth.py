"""Seeded synthetic inputs: weights, prompts, tap rows, hc streams, KV.

This module holds no arithmetic of the method: it only draws numbers.  It is
the one module that both the CUDA path's callers and the CPU oracle's callers
use, so that both see the same inputs.

Every tensor is drawn from its own counter-keyed Philox stream (key = base
seed, a stable id of the tensor's name, chunk index), so a tensor's values do
not depend on which other tensors were drawn or in which order, and large
tensors are drawn in parallel chunks.  Weights are N(0, std) in fp32, rounded
to bf16 for bf16 models; norm weights are ones, or N(1, norm_std) when a
caller asks for it (so that a kernel which drops or swaps a norm weight
changes the result); prompts are uniform ids.
"""

from __future__ import annotations

import os
import zlib
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, List, Sequence

import numpy as np
import torch

_CHUNK = 1 << 22
_THREADS = max(1, min(16, os.cpu_count() or 1))

WEIGHT_SEED = 0
PROMPT_SEED = 1
TAP_SEED = 2
KV_SEED = 3


def _key(seed: int, name: str, chunk: int) -> int:
    return (int(seed) << 64) | (zlib.crc32(name.encode()) << 32) | int(chunk)


def _draw_chunk(args):
    seed, name, chunk, count = args
    rng = np.random.Generator(np.random.Philox(key=_key(seed, name, chunk)))
    return rng.standard_normal(count, dtype=np.float32)


def normal(shape: Sequence[int], std: float, seed: int, name: str) -> np.ndarray:
    """N(0, std^2) fp32 array of `shape`, keyed by (seed, name)."""
    total = int(np.prod(shape))
    jobs = [(seed, name, c, min(_CHUNK, total - c * _CHUNK))
            for c in range((total + _CHUNK - 1) // _CHUNK)]
    if len(jobs) > 1:
        with ThreadPoolExecutor(_THREADS) as ex:
            parts = list(ex.map(_draw_chunk, jobs))
    else:
        parts = [_draw_chunk(j) for j in jobs] or [np.zeros(0, np.float32)]
    out = np.concatenate(parts) if len(parts) > 1 else parts[0]
    if std != 1.0:
        out *= np.float32(std)
    return out.reshape(shape)


def as_torch(a: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    return torch.from_numpy(a).to(dtype)


def uniform_ids(n: int, vocab: int, seed: int = PROMPT_SEED, name: str = "prompt") -> np.ndarray:
    rng = np.random.Generator(np.random.Philox(key=_key(seed, name, 0)))
    return rng.integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


LAYER_KEYS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")
NORM_KEYS = ("ln_attn", "ln_mlp", "q_norm", "k_norm")


def layer_shapes(hidden: int, n_q: int, n_kv: int, head_dim: int, ffn: int) -> Dict[str, tuple]:
    """nn.Linear layouts [out, in] of one Qwen3-shaped decoder layer."""
    return {
        "wq": (n_q * head_dim, hidden),
        "wk": (n_kv * head_dim, hidden),
        "wv": (n_kv * head_dim, hidden),
        "wo": (hidden, n_q * head_dim),
        "w_gate": (ffn, hidden),
        "w_up": (ffn, hidden),
        "w_down": (hidden, ffn),
    }


def norm_weight(n: int, norm_std: float, seed: int, name: str) -> torch.Tensor:
    """fp32 RMSNorm weight of width n: ones, or N(1, norm_std) keyed by name."""
    if norm_std <= 0.0:
        return torch.ones(n, dtype=torch.float32)
    return torch.from_numpy(normal((n,), norm_std, seed, name) + np.float32(1.0))


def decoder_layers(prefix: str, n_layers: int, hidden: int, n_q: int, n_kv: int,
                   head_dim: int, ffn: int, dtype: torch.dtype, std: float = 0.02,
                   seed: int = WEIGHT_SEED, norm_std: float = 0.0) -> List[Dict[str, torch.Tensor]]:
    """Weights of n_layers decoder layers as CPU tensors.

    Projections are N(0, std) drawn in fp32 and cast to `dtype` (fp32 or
    bf16); norm weights (attention/MLP input norms, q/k head norms) are fp32,
    ones or N(1, norm_std) (each its own stream).
    """
    shapes = layer_shapes(hidden, n_q, n_kv, head_dim, ffn)
    widths = {"ln_attn": hidden, "ln_mlp": hidden, "q_norm": head_dim, "k_norm": head_dim}
    layers = []
    for l in range(n_layers):
        lw = {}
        for k in LAYER_KEYS:
            lw[k] = as_torch(normal(shapes[k], std, seed, f"{prefix}.{l}.{k}"), dtype)
        for k in NORM_KEYS:
            lw[k] = norm_weight(widths[k], norm_std, seed, f"{prefix}.{l}.{k}")
        layers.append(lw)
    return layers


def matrix(name: str, rows: int, cols: int, dtype: torch.dtype, std: float = 0.02,
           seed: int = WEIGHT_SEED) -> torch.Tensor:
    return as_torch(normal((rows, cols), std, seed, name), dtype)


def tap_rows(n_rows: int, width: int, dtype: torch.dtype = torch.bfloat16,
             seed: int = TAP_SEED, name: str = "taps") -> torch.Tensor:
    """N(0, 1) hidden rows standing in for target taps, [n_rows, width]."""
    return as_torch(normal((n_rows, width), 1.0, seed, name), dtype)


def hc_streams(n_layers: int, n_rows: int, hc: int, hidden: int,
               dtype: torch.dtype = torch.bfloat16, seed: int = TAP_SEED) -> torch.Tensor:
    """[n_layers, n_rows, hc * hidden] N(0, 1) hyper-connection streams."""
    return as_torch(normal((n_layers, n_rows, hc * hidden), 1.0, seed, "hc"), dtype)


def kv_rows(n_layers: int, n_kv: int, n_pos: int, head_dim: int,
            dtype: torch.dtype = torch.bfloat16, seed: int = KV_SEED) -> torch.Tensor:
    """[n_layers, 2, n_kv, n_pos, head_dim] N(0, 1) synthetic K/V."""
    return as_torch(normal((n_layers, 2, n_kv, n_pos, head_dim), 1.0, seed, "kv"), dtype)


class ModelTensors:
    """Every synthetic tensor of a workload (CPU tensors).

    embed [vocab, H] (also the tied LM head), per-layer weights of the target
    ("tgt") and the drafter ("drf"), fc [H, n_taps*H] and fp32 weights of the
    final norms and the drafter's context norm (ones, or N(1, norm_std) when
    norm_std > 0).  Layers stored as INT4 (the drafter's or the target's) are
    drawn in fp32; the quantiser of each side turns them into INT4.
    """

    def __init__(self, w, std: float = 0.02, seed: int = WEIGHT_SEED, norm_std: float = 0.0):
        dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
        self.w = w
        self.norm_std = norm_std
        self.embed = matrix("embed", w.vocab, w.hidden, dt, std, seed)
        self.final_norm_t = norm_weight(w.hidden, norm_std, seed, "final_norm_tgt")
        self.final_norm_d = norm_weight(w.hidden, norm_std, seed, "final_norm_drf")
        self.ctx_norm = norm_weight(w.hidden, norm_std, seed, "ctx_norm")
        tdt = torch.float32 if getattr(w, "tgt_int4", False) else dt
        self.tgt = decoder_layers("tgt", w.tgt_layers, w.hidden, w.n_q, w.n_kv, w.head_dim,
                                  w.ffn, tdt, std, seed, norm_std)
        ddt = torch.float32 if w.drf_int4 else dt
        self.drf = decoder_layers("drf", w.drf_layers, w.hidden, w.n_q, w.n_kv, w.head_dim,
                                  w.ffn, ddt, std, seed, norm_std)
        self.fc = matrix("fc", w.hidden, w.n_taps * w.hidden, dt, std, seed) \
            if w.drf_layers else None
