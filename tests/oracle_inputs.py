"""Builds the oracle's inputs from the seeded synthetic generators.

Tensors drawn by ``synth`` (bf16 or fp32 CPU tensors) are handed to the oracle
as float32 numpy arrays; bf16 and fp32 values convert exactly.
"""

from __future__ import annotations

from typing import Dict, List

import numpy as np
import torch

from block_diffusion_speculative_gather_gb300 import synth
from block_diffusion_speculative_gather_gb300.synth import ModelTensors  # noqa: F401
from block_diffusion_speculative_gather_gb300.configs import Workload
from oracle import dflash_oracle as O


def np32(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float32).cpu().numpy()


def oracle_config(w: Workload, **kw) -> O.OracleConfig:
    cfg = O.OracleConfig(
        hidden=w.hidden, n_q=w.n_q, n_kv=w.n_kv, head_dim=w.head_dim, ffn=w.ffn,
        vocab=w.vocab, tgt_layers=w.tgt_layers, drf_layers=w.drf_layers,
        tap_layers=list(w.tap_layers), block=w.block, window=w.window,
        max_seq=w.max_seq, eos_id=w.eos_id, rms_eps=w.rms_eps,
        rope_theta=w.rope_theta, ctx_norm=w.ctx_norm,
        adaptive_block=getattr(w, "adaptive_block", False))
    for k, v in kw.items():
        setattr(cfg, k, v)
    return cfg


def torch_dtype(w: Workload) -> torch.dtype:
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def oracle_layers(layers: List[Dict[str, torch.Tensor]], int4: bool = False):
    out = []
    for lw in layers:
        d = {}
        for k, t in lw.items():
            a = np32(t)
            if int4 and k in synth.LAYER_KEYS:
                packed, s = O.quantize_int4_g64(a)
                a = O.dequant_int4_g64(packed, s)
            d[k] = a
        out.append(d)
    return out


def int4_roundtrip(w: np.ndarray) -> np.ndarray:
    """The values an INT4 group-64 copy of w holds (the oracle's quantiser)."""
    packed, s = O.quantize_int4_g64(w)
    return O.dequant_int4_g64(packed, s)


def oracle_target(m: ModelTensors) -> O.TargetWeights:
    w = m.w
    embed = np32(m.embed)
    return O.TargetWeights(embed=embed, layers=oracle_layers(m.tgt, getattr(w, "tgt_int4", False)),
                           final_norm=np32(m.final_norm_t),
                           lm_head=int4_roundtrip(embed) if getattr(w, "lm_int4", False) else None)


def oracle_draft(m: ModelTensors) -> O.DraftWeights:
    return O.DraftWeights(layers=oracle_layers(m.drf, m.w.drf_int4), fc=np32(m.fc),
                          ctx_norm=np32(m.ctx_norm), final_norm=np32(m.final_norm_d))
