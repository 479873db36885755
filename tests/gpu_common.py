"""Helpers shared by the GPU parity tests (built library + oracle inputs).

Decidable rows.  A logits row is decidable when the oracle's top-2 margin
exceeds twice the GPU row's distance from it: with
e_r = max_v |g_v - o_v| / max_v |o_v| measured on the GPU's own logits row
(the values its argmax epilogue reduced), a margin
o_top1 - o_top2 > 2 e_r max_v |o_v| leaves the GPU no other argmax, so its
id must equal the oracle's.  Every such check also asserts e_r below the
workload's tolerance (rel 1e-4 fp32, 2e-2 bf16/INT4), and a floor on how many
rows were decidable: the rows whose margin exceeds 2 * dec_tol * max|o| for
the accuracy the kernels are expected to reach (dec_tol, stated per test), so
a precision loss shows up as a failed floor, not as a silently shorter check.
"""

from __future__ import annotations

import json
import os

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


def margin_ratio(ref_row: np.ndarray) -> float:
    """(o_top1 - o_top2) / max_v |o_v| of an oracle row."""
    r = np.asarray(ref_row, dtype=np.float64)
    top = np.sort(r)[-2:]
    return float((top[1] - top[0]) / np.max(np.abs(r)))


def decidable(ref_row: np.ndarray, tol: float) -> bool:
    """The top-2 margin of the oracle row exceeds 2 * tol * max|o| (then an
    implementation within tol of the oracle must pick the same argmax)."""
    return margin_ratio(ref_row) > 2 * tol


def report(name: str, **values):
    """Appends measured parity figures to the JSON-lines file named by
    DFLASH_PARITY_REPORT (nothing when it is unset)."""
    path = os.environ.get("DFLASH_PARITY_REPORT")
    if not path:
        return
    rec = {"test": name}
    for k, v in values.items():
        rec[k] = v.tolist() if isinstance(v, np.ndarray) else v
    with open(path, "a") as f:
        f.write(json.dumps(rec) + "\n")


def check_rows(name: str, gpu_logits, gpu_ids, ref_logits, tol: float, dec_tol: float,
               min_decidable: int = -1):
    """Logits of every row within tol of the oracle; on every row decidable at
    the row's measured error, the GPU id equals the oracle's argmax.  Asserts
    at least min_decidable decidable rows (default: every row decidable at
    dec_tol).  Returns the boolean decidable mask."""
    g = np.asarray(gpu_logits, dtype=np.float64)
    o = np.asarray(ref_logits, dtype=np.float64)
    err = rel_err_rows(g, o)
    assert err.max() < tol, (name, err)
    ratios = np.array([margin_ratio(r) for r in o])
    dec = ratios > 2 * err
    if min_decidable < 0:
        min_decidable = int(np.sum(ratios > 2 * dec_tol))
    report(name, err=err, margin=ratios, decidable=dec.astype(int),
           floor=min_decidable)
    if gpu_ids is not None:
        for i, gid in enumerate(gpu_ids):
            if dec[i]:
                assert int(gid) == int(np.argmax(o[i])), f"{name}: row {i}"
    assert int(dec.sum()) >= min_decidable, (name, int(dec.sum()), min_decidable, err)
    assert int(dec.sum()) > 0, (name, err, ratios)
    return dec


def check_ids(gpu_ids, ref_logits: np.ndarray, tol: float):
    """GPU ids equal the oracle argmax on every row decidable at tol."""
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


def stream_prefix(name: str, gpu_tokens, gpu_step_logits, ref_tokens, ref_logits_rows,
                  tol: float):
    """Greedy streams: token k of both streams must agree while every earlier
    token agreed and row k is decidable at the GPU step's measured error
    (the GPU step's logits are for the same prefix as the oracle's row k
    only while the streams agree).  Returns the compared length."""
    n = 0
    errs = []
    for g, gl, r, ol in zip(gpu_tokens, gpu_step_logits, ref_tokens, ref_logits_rows):
        e = float(rel_err_rows(np.asarray(gl)[None], np.asarray(ol)[None])[0])
        errs.append(e)
        assert e < tol, (name, n, e)
        if not margin_ratio(ol) > 2 * e:
            break
        assert g == r, f"{name}: token {n}: gpu {g} oracle {r}"
        n += 1
    report(name, compared=n, err=errs)
    return n


def logits_buf(vocab: int) -> torch.Tensor:
    return torch.zeros((16, vocab), dtype=torch.float32, device="cuda")


def accept_check(name: str, toks, n_emitted: int, st, ref_logits, drafts, gpu_logits,
                 tol: float, pos0: int):
    """Acceptance of a verify against the oracle's: on rows 0..a (a the
    oracle's accepted drafts) every row must be decidable at the GPU's
    measured error (asserted: the check never passes vacuously), then the
    emitted tokens, their count and the rolled-back KV length are exact."""
    from oracle import dflash_oracle as O
    o = np.asarray(ref_logits, dtype=np.float64)
    y = [int(np.argmax(r)) for r in o]
    a, emitted, _ = O.accept(drafts, y, -1)
    err = rel_err_rows(np.asarray(gpu_logits, np.float64)[: len(o)], o)
    dec = [margin_ratio(o[i]) > 2 * err[i] for i in range(a + 1)]
    report(name, a=a, emitted=len(emitted), err=err, decidable=[int(d) for d in dec])
    assert all(dec), (name, "rows 0..a not all decidable", err[: a + 1],
                      [margin_ratio(o[i]) for i in range(a + 1)])
    assert toks[:n_emitted] == emitted, (name, toks[:n_emitted], emitted)
    assert n_emitted == len(emitted)
    assert st.n == pos0 + len(emitted) and st.last_accept == a
    return a


def accept_prefix_check(name: str, toks, n_emitted: int, st, ref_logits, drafts, gpu_logits,
                        tol: float, dec_tol: float, pos0: int):
    """Acceptance against the oracle's where some rows may be undecidable:
    k = the first row not decidable at the GPU's measured error.  The GPU's
    emitted tokens equal the oracle's argmaxes on rows < k; when k covers the
    oracle's accepted rows 0..a, acceptance, emitted tokens and the
    rolled-back length are exact; otherwise both accepted at least k drafts.
    A floor: k >= the first row whose margin is below 2 * dec_tol."""
    from oracle import dflash_oracle as O
    o = np.asarray(ref_logits, dtype=np.float64)
    y = [int(np.argmax(r)) for r in o]
    a, emitted, _ = O.accept(drafts, y, -1)
    err = rel_err_rows(np.asarray(gpu_logits, np.float64)[: len(o)], o)
    assert err.max() < tol, (name, err)
    ratios = [margin_ratio(r) for r in o]
    k = next((i for i in range(len(o)) if not ratios[i] > 2 * err[i]), len(o))
    floor = next((i for i in range(len(o)) if not ratios[i] > 2 * dec_tol), len(o))
    a_gpu = n_emitted - 1
    report(name, a=a, a_gpu=a_gpu, k=k, floor=floor, err=err, margin=ratios)
    for i in range(min(k, n_emitted)):
        assert toks[i] == y[i], (name, i, toks[i], y[i])
    if k > a:
        assert toks[:n_emitted] == emitted, (name, toks[:n_emitted], emitted)
        assert n_emitted == len(emitted) and st.last_accept == a
        assert st.n == pos0 + len(emitted)
    else:
        assert a_gpu >= k and a >= k, (name, a_gpu, a, k)
    assert k >= floor, (name, k, floor, err)
    return a, k
