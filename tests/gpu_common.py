"""Helpers shared by the GPU parity tests (built library + oracle inputs)."""

from __future__ import annotations

import numpy as np
import torch


def build_lib():
    from block_diffusion_speculative_gather_gb300 import build
    build.build()


def rel_err_rows(gpu: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Per row: max_v |g_v - o_v| / max_v |o_v| (the logit tolerance measure)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return np.max(np.abs(gpu - ref), axis=-1) / np.max(np.abs(ref), axis=-1)


def decidable(ref_row: np.ndarray, tol: float) -> bool:
    """The top-2 margin of the oracle row exceeds 2 * tol * max|o| (then an
    implementation within tol of the oracle must pick the same argmax)."""
    top = np.sort(np.asarray(ref_row, dtype=np.float64))[-2:]
    return (top[1] - top[0]) > 2 * tol * np.max(np.abs(ref_row))


def check_ids(gpu_ids, ref_logits: np.ndarray, tol: float):
    """GPU ids equal the oracle argmax on every decidable row."""
    n_dec = 0
    for i, g in enumerate(gpu_ids):
        if decidable(ref_logits[i], tol):
            assert int(g) == int(np.argmax(ref_logits[i])), f"row {i}"
            n_dec += 1
    return n_dec


def compared_prefix(gpu_tokens, ref_tokens, ref_logits_rows, tol: float) -> int:
    """Length of the token-stream prefix that must agree: up to and including
    the first undecidable row (sequences may legitimately split there)."""
    n = 0
    for g, r, lg in zip(gpu_tokens, ref_tokens, ref_logits_rows):
        if not decidable(lg, tol):
            break
        assert g == r, f"token {n}: gpu {g} oracle {r}"
        n += 1
    return n


def logits_buf(vocab: int) -> torch.Tensor:
    return torch.zeros((16, vocab), dtype=torch.float32, device="cuda")
