"""Plain CPU oracle for the DFlash block-diffusion speculative round.

TEST INFRASTRUCTURE ONLY.  This module is the slow, obviously-correct
definition that the CUDA path is checked against.  Only the test suite,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import it.  It shares no code with the CUDA library
and never imports the product package; the only thing both sides share are
the seeded input generators, which hold none of the method's arithmetic.

Precision: float64 throughout (weights given as bf16/fp32 values are upcast
exactly).  Where floating point decides an integer code (the INT4 quantiser),
the decision is taken in fp32, the precision the CUDA kernel takes it in.

Sources (three pull-request pages on one subject):
  * "[RFC] DFlash" -- ExecuTorch PR #20840 (sections "DFlash Overview",
    "Key Implementation Details", the review "Requested changes" 1-6 and the
    author's reply "1. Dynamic block_len" / "3. Draft KV cache").
  * "feat: DFlash2 block-diffusion drafter for Qwen 3.8" -- Mference PR #22
    (commit messages, "What's here").
  * "dflash: the chain verify builds pipelined and defers the qwen4 PLE
    gather" -- mlx-serve PR #937 (first commit message: hcStreamMean).

Readings where the pages are silent:
  * decoder layer = Qwen3: pre-norm RMSNorm (eps 1e-6), per-head q/k RMSNorm
    before rotate-half RoPE (theta 1e6), GQA, SwiGLU MLP, no biases, final
    RMSNorm, LM head tied to the embedding;
  * a tap at layer l is the residual stream after decoder layer l
    (0-indexed); taps are concatenated in increasing layer order;
  * drafter context c = RMSNorm_ctx(fc(taps)); per draft layer the context
    keys are RoPE(k_norm(W_k c)) at the tap rows' absolute positions and the
    values W_v c; they are concatenated with the block's keys/values along
    the key axis ("[sliding ctx | bidirectional block]");
  * the sliding window is anchored at the block start: every block row sees
    context positions [max(0, n - W), n) (W = 0: all) and every block row;
  * the mask token is vocab - 1; argmax ties go to the lowest index;
  * INT4: symmetric, group 64 along K, bf16 scale = bf16(absmax / 7),
    code = clamp(rint(w / s), -8, 7) stored as u4 = code + 8, low nibble =
    even k.

Parity status: every function below is pinned by the ``-m "not gpu"`` tests
(library routines, closed forms, brute force, hand examples and the
speculative == greedy invariant).  The drafter's architecture choices listed
above are readings of the pages, not facts the pages fix; the functions that
implement them are pinned, the choices themselves are not (no trained
checkpoint is available to pin them against).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Callable, Dict, List, Optional, Sequence

import numpy as np

F64 = np.float64


# --------------------------------------------------------------------------
# configuration
# --------------------------------------------------------------------------

@dataclass
class OracleConfig:
    """Shapes of the target and the drafter (both Qwen3-shaped)."""

    hidden: int
    n_q: int
    n_kv: int
    head_dim: int
    ffn: int
    vocab: int
    tgt_layers: int
    drf_layers: int
    tap_layers: Sequence[int]
    block: int
    window: int = 0           # 0 = the whole context is visible
    max_seq: int = 1 << 30
    eos_id: int = -1          # -1 = no EOS
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    ctx_norm: bool = True
    adaptive_block: bool = False   # per-round block cap from recent acceptance

    @property
    def mask_id(self) -> int:
        return self.vocab - 1

    @property
    def n_taps(self) -> int:
        return len(self.tap_layers)


# --------------------------------------------------------------------------
# primitives (Qwen3 decoder conventions)
# --------------------------------------------------------------------------

def f64(a) -> np.ndarray:
    return np.asarray(a, dtype=F64)


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * w."""
    x = f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * f64(w)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y = x W^T with W stored [out, in] (the nn.Linear layout)."""
    return f64(x) @ f64(w).T


def rope_angles(positions: Sequence[int], head_dim: int, theta: float) -> np.ndarray:
    """angle[p, i] = pos_p * theta^(-2i/d), i < d/2, in float64."""
    half = head_dim // 2
    inv = theta ** (-(2.0 * np.arange(half, dtype=F64)) / head_dim)
    return np.asarray(positions, dtype=F64)[:, None] * inv[None, :]


def rope_rotate_half(x: np.ndarray, positions: Sequence[int], theta: float) -> np.ndarray:
    """Rotate-half RoPE on x[..rows.., heads, d]; element i pairs with i + d/2."""
    x = f64(x)
    d = x.shape[-1]
    half = d // 2
    ang = rope_angles(positions, d, theta)            # [rows, half]
    cos = np.cos(ang)[:, None, :]
    sin = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, visible: np.ndarray,
              scale: float) -> np.ndarray:
    """Grouped-query attention.

    q [Tq, n_q, d], k/v [Tk, n_kv, d], visible [Tq, Tk] bool.  Query head h
    reads key/value head h // (n_q // n_kv).  Softmax over the visible keys
    only; every query row must see at least one key.
    """
    q, k, v = f64(q), f64(k), f64(v)
    n_q, n_kv = q.shape[1], k.shape[1]
    group = n_q // n_kv
    out = np.zeros_like(q)
    for h in range(n_q):
        kh = h // group
        s = (q[:, h, :] @ k[:, kh, :].T) * scale        # [Tq, Tk]
        s = np.where(visible, s, -np.inf)
        m = np.max(s, axis=1, keepdims=True)
        p = np.exp(s - m)
        p = p / np.sum(p, axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, kh, :]
    return out


def argmax_lowest(logits_row: np.ndarray) -> int:
    """argmax with ties resolved to the lowest index."""
    return int(np.argmax(logits_row))


# --------------------------------------------------------------------------
# masks
# --------------------------------------------------------------------------

def causal_visible(q_pos: Sequence[int], k_pos: Sequence[int]) -> np.ndarray:
    """Target verify/prefill rows: key position <= query position."""
    return np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None]


def block_context_range(n: int, window: int) -> range:
    """Context positions every block row sees: [max(0, n - W), n), W=0 = all.

    [RFC] DFlash, "Requested changes" 2 (the Qwen draft is non-causal), and
    DFlash2 drafter, first commit ("block attention over [sliding ctx |
    bidirectional block]"); the window is anchored at the block start.
    """
    lo = 0 if window <= 0 else max(0, n - window)
    return range(lo, n)


def block_visible(ctx_pos: Sequence[int], n: int, bl: int, window: int) -> np.ndarray:
    """Visibility of keys [ctx rows | block rows] for the bl block rows."""
    rng = block_context_range(n, window)
    ctx_ok = np.array([rng.start <= p < rng.stop for p in ctx_pos], dtype=bool)
    vis = np.ones((bl, len(ctx_pos) + bl), dtype=bool)
    vis[:, :len(ctx_pos)] = ctx_ok[None, :]
    return vis


# --------------------------------------------------------------------------
# decoder layer
# --------------------------------------------------------------------------

def qkv_project(h: np.ndarray, lw: Dict[str, np.ndarray], cfg: OracleConfig,
                positions: Sequence[int]):
    """q, k, v of normed rows h: per-head RMSNorm on q and k, then RoPE."""
    T = h.shape[0]
    d = cfg.head_dim
    q = linear(h, lw["wq"]).reshape(T, cfg.n_q, d)
    k = linear(h, lw["wk"]).reshape(T, cfg.n_kv, d)
    v = linear(h, lw["wv"]).reshape(T, cfg.n_kv, d)
    q = rms_norm(q, lw["q_norm"], cfg.rms_eps)
    k = rms_norm(k, lw["k_norm"], cfg.rms_eps)
    q = rope_rotate_half(q, positions, cfg.rope_theta)
    k = rope_rotate_half(k, positions, cfg.rope_theta)
    return q, k, v


def mlp(x: np.ndarray, lw: Dict[str, np.ndarray], cfg: OracleConfig) -> np.ndarray:
    h = rms_norm(x, lw["ln_mlp"], cfg.rms_eps)
    return linear(silu(linear(h, lw["w_gate"])) * linear(h, lw["w_up"]), lw["w_down"])


class KVCache:
    """Per-layer K (post-norm, post-RoPE) and V, indexed by absolute position."""

    def __init__(self, n_layers: int, n_kv: int, head_dim: int):
        self.k: List[Dict[int, np.ndarray]] = [dict() for _ in range(n_layers)]
        self.v: List[Dict[int, np.ndarray]] = [dict() for _ in range(n_layers)]

    def write(self, layer: int, positions: Sequence[int], k: np.ndarray, v: np.ndarray):
        for i, p in enumerate(positions):
            self.k[layer][p] = k[i].copy()
            self.v[layer][p] = v[i].copy()

    def read(self, layer: int, length: int):
        k = np.stack([self.k[layer][p] for p in range(length)])
        v = np.stack([self.v[layer][p] for p in range(length)])
        return k, v

    def truncate(self, length: int):
        """KV-position rollback: forget every position >= length."""
        for layer in range(len(self.k)):
            for p in [p for p in self.k[layer] if p >= length]:
                del self.k[layer][p]
                del self.v[layer][p]


def target_layer(x: np.ndarray, lw, cfg: OracleConfig, positions: Sequence[int],
                 cache: KVCache, layer: int) -> np.ndarray:
    """One target decoder layer over rows x at `positions` (contiguous).

    Writes this layer's K/V at those positions, then attends causally over
    the cache [0, last position].
    """
    h = rms_norm(x, lw["ln_attn"], cfg.rms_eps)
    q, k, v = qkv_project(h, lw, cfg, positions)
    cache.write(layer, positions, k, v)
    kv_len = positions[-1] + 1
    K, V = cache.read(layer, kv_len)
    vis = causal_visible(positions, range(kv_len))
    a = attention(q, K, V, vis, 1.0 / math.sqrt(cfg.head_dim))
    x = x + linear(a.reshape(x.shape[0], -1), lw["wo"])
    return x + mlp(x, lw, cfg)


# --------------------------------------------------------------------------
# target forward: logits + taps
# --------------------------------------------------------------------------

@dataclass
class TargetWeights:
    embed: np.ndarray                      # [vocab, H] (also the LM head when tied)
    layers: List[Dict[str, np.ndarray]]
    final_norm: np.ndarray
    # LM head [vocab, H] when it is not the embedding itself: the 4-bit
    # models of "[RFC] DFlash" ("Test Plan": target and draft both 4-bit)
    # read the logits from an INT4 group-64 copy (dequantised values here)
    lm_head: Optional[np.ndarray] = None

    def head(self) -> np.ndarray:
        return self.embed if self.lm_head is None else self.lm_head


def target_forward(tw: TargetWeights, cfg: OracleConfig, tokens: Sequence[int],
                   pos0: int, cache: KVCache):
    """Target forward over rows `tokens` at positions pos0..pos0+T-1.

    Returns (logits [T, vocab], taps [T, n_taps * H]).  The taps are the
    residual stream after each tap layer, concatenated in increasing layer
    order ([RFC] DFlash, "Key Implementation Details", Phase 1: the target
    returns logits plus concatenated hidden states of the selected layers).
    """
    positions = list(range(pos0, pos0 + len(tokens)))
    x = f64(tw.embed[np.asarray(tokens)])
    taps = {}
    for l, lw in enumerate(tw.layers):
        x = target_layer(x, lw, cfg, positions, cache, l)
        if l in cfg.tap_layers:
            taps[l] = x.copy()
    h = rms_norm(x, tw.final_norm, cfg.rms_eps)
    logits = linear(h, tw.head())
    tap = np.concatenate([taps[l] for l in sorted(cfg.tap_layers)], axis=-1) \
        if cfg.tap_layers else np.zeros((len(tokens), 0))
    return logits, tap


def greedy(tw: TargetWeights, cfg: OracleConfig, prompt: Sequence[int], n_new: int):
    """Plain greedy decoding: tok_{k+1} = argmax target(tok_0..tok_k).

    The first generated token comes from the prompt's last row; each later
    token from a one-row forward of the previous one.
    """
    cache = KVCache(len(tw.layers), cfg.n_kv, cfg.head_dim)
    logits, _ = target_forward(tw, cfg, prompt, 0, cache)
    out = [argmax_lowest(logits[-1])]
    pos = len(prompt)
    while len(out) < n_new:
        if cfg.eos_id >= 0 and out[-1] == cfg.eos_id:
            break
        logits, _ = target_forward(tw, cfg, [out[-1]], pos, cache)
        out.append(argmax_lowest(logits[0]))
        pos += 1
    return out


# --------------------------------------------------------------------------
# hc-stream mean tap and INT4 group-64 format
# --------------------------------------------------------------------------

def hc_mean(x: np.ndarray, hc: int) -> np.ndarray:
    """Per-token mean over hyper-connection streams.

    x [L, hc * H] laid out stream-major (stream s owns columns s*H..s*H+H-1)
    -> [L, H]; the unflatten(-1, (hc, hidden)).mean(-2) of mlx-serve PR #937,
    first commit (hcStreamMean).  Summed in stream order, then scaled by 1/hc.
    """
    x = f64(x)
    L, width = x.shape
    H = width // hc
    acc = np.zeros((L, H), dtype=F64)
    for s in range(hc):
        acc = acc + x[:, s * H:(s + 1) * H]
    return acc * (1.0 / hc)


def tap_concat(per_layer_streams: Sequence[np.ndarray], hc: int) -> np.ndarray:
    """hc-mean each tap layer's streams, concatenate in tap-layer order."""
    return np.concatenate([hc_mean(s, hc) for s in per_layer_streams], axis=-1)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest, ties to even); returns uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> 16) & 1
    b = (b + 0x7FFF + lsb) >> 16
    return b.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(F64)


def quantize_int4_g64(w: np.ndarray):
    """Symmetric INT4 with group 64 along K and a bf16 scale per group.

    w [N, K] fp32 -> (packed uint8 [N, K/2], scale bits uint16 [N, K/64]).
    s = bf16(absmax(group) / 7); code = clamp(rint(w / s), -8, 7), 0 where
    s == 0; stored u4 = code + 8, low nibble = even k.  The scale and the
    division are computed in fp32 (the precision the kernel decides in).
    DFlash2 drafter, third commit (projections quantised at load into an
    INT4 format); group size and bf16 scales as the long-context config.
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    g = w.reshape(N, K // 64, 64)
    absmax = np.max(np.abs(g), axis=-1)
    s_bits = f32_to_bf16_bits(absmax / np.float32(7.0))
    s = bf16_bits_to_f64(s_bits).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        qf = np.where(s[..., None] > 0, g / s[..., None], np.float32(0.0))
    q = np.clip(np.rint(qf), -8, 7).astype(np.int32).reshape(N, K)
    u = (q + 8).astype(np.uint8)
    packed = (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)
    return packed, s_bits


def dequant_int4_g64(packed: np.ndarray, s_bits: np.ndarray) -> np.ndarray:
    """w = (u4 - 8) * s, exact in float64."""
    N, half = packed.shape
    K = half * 2
    u = np.empty((N, K), dtype=np.int32)
    u[:, 0::2] = packed & 0xF
    u[:, 1::2] = packed >> 4
    s = bf16_bits_to_f64(s_bits)
    return (u - 8).astype(F64) * np.repeat(s, 64, axis=1)


# --------------------------------------------------------------------------
# drafter (uncached: re-projects the context window on every call)
# --------------------------------------------------------------------------

@dataclass
class DraftWeights:
    layers: List[Dict[str, np.ndarray]]    # wq..w_down may be INT4 via dequant
    fc: np.ndarray                         # [H, n_taps * H]
    ctx_norm: np.ndarray                   # [H]
    final_norm: np.ndarray                 # [H]


def draft_context(dw: DraftWeights, cfg: OracleConfig, taps: np.ndarray) -> np.ndarray:
    """c = RMSNorm_ctx(fc(taps)) ([RFC] DFlash, review #3: self.fc(target_hidden))."""
    c = linear(taps, dw.fc)
    return rms_norm(c, dw.ctx_norm, cfg.rms_eps) if cfg.ctx_norm else c


def draft_forward(dw: DraftWeights, embed: np.ndarray, cfg: OracleConfig,
                  taps_by_pos: np.ndarray, t_n: int, n: int, bl: int,
                  lm_head: Optional[np.ndarray] = None):
    """One drafter forward over the masked block at positions n..n+bl-1.

    taps_by_pos[p] is the concatenated tap row of absolute position p (p < n).
    The block is [t_n, MASK x (bl-1)] ([RFC] DFlash, "DFlash Overview": one
    forward predicts a whole masked block).  Target hidden states enter the
    K/V of every draft layer ("added into the Key/Value projections of every
    draft"), as context keys/values for the window
    [max(0, n-W), n) concatenated with the block's own.  The block attends
    bidirectionally.  Returns (logits [bl, vocab], draft ids [bl - 1]) where
    draft id j-1 = argmax of block row j, j = 1..bl-1 (row 0 is discarded).
    The drafter shares the target's embedding and LM head (lm_head None: the
    embedding itself).
    """
    ctx_pos = list(block_context_range(n, cfg.window))
    c = draft_context(dw, cfg, taps_by_pos[ctx_pos]) if ctx_pos else \
        np.zeros((0, cfg.hidden))
    blk_pos = list(range(n, n + bl))
    x = f64(embed[np.asarray([t_n] + [cfg.mask_id] * (bl - 1))])
    vis = block_visible(ctx_pos, n, bl, cfg.window)
    d = cfg.head_dim
    for lw in dw.layers:
        h = rms_norm(x, lw["ln_attn"], cfg.rms_eps)
        q, kb, vb = qkv_project(h, lw, cfg, blk_pos)
        kc = linear(c, lw["wk"]).reshape(len(ctx_pos), cfg.n_kv, d)
        kc = rope_rotate_half(rms_norm(kc, lw["k_norm"], cfg.rms_eps), ctx_pos,
                              cfg.rope_theta) if ctx_pos else kc
        vc = linear(c, lw["wv"]).reshape(len(ctx_pos), cfg.n_kv, d)
        K = np.concatenate([kc, kb], axis=0)
        V = np.concatenate([vc, vb], axis=0)
        a = attention(q, K, V, vis, 1.0 / math.sqrt(d))
        x = x + linear(a.reshape(bl, -1), lw["wo"])
        x = x + mlp(x, lw, cfg)
    logits = linear(rms_norm(x, dw.final_norm, cfg.rms_eps),
                    embed if lm_head is None else lm_head)
    ids = [argmax_lowest(logits[j]) for j in range(1, bl)]
    return logits, ids


# --------------------------------------------------------------------------
# acceptance, block length, the speculative loop
# --------------------------------------------------------------------------

def first_mismatch(draft_ids: Sequence[int], target_ids: Sequence[int]) -> int:
    """Number a of accepted drafts: the longest prefix with d[j] == y[j-1].

    draft_ids has T-1 entries (block rows 1..T-1) and target_ids T entries
    (one per verify row), so target_ids[a] is always in range: the bonus
    token ([RFC] DFlash, first code review, the first_mismatch note).
    """
    a = 0
    while a < len(draft_ids) and draft_ids[a] == target_ids[a]:
        a += 1
    return a


def accept(draft_ids: Sequence[int], target_ids: Sequence[int], eos_id: int):
    """Emit y[0..a]; if an EOS lands at e <= a emit y[0..e] and finish.

    Returns (a, emitted tokens, finished).  Accepted length = a + 1.
    [RFC] DFlash, "Key Implementation Details" Phase 3 (first-mismatch
    acceptance) and the second review's note on EOS truncation keeping the
    first EOS.
    """
    a = first_mismatch(draft_ids, target_ids)
    emitted = list(target_ids[: a + 1])
    finished = False
    if eos_id >= 0 and eos_id in emitted:
        emitted = emitted[: emitted.index(eos_id) + 1]
        finished = True
    return a, emitted, finished


def block_len(block: int, max_new: int, generated: int, max_seq: int, pos: int) -> int:
    """min(block, max_new - generated, max_seq - pos) ([RFC] DFlash,
    "Requested changes" 1, Make block_len dynamic)."""
    return min(block, max_new - generated, max_seq - pos)


# Adaptive block length.  The mlx-serve page's round policy picks the block
# size per round ("dflash: the chain verify builds pipelined ...", first
# commit: the DFlash round policy drives the targets) without giving its
# rule; reading taken: an exponential average of the accepted drafts a,
# ema <- ema / 2 + a / 2 in fp32 (the precision the kernel decides in),
# starting from block - 1, caps the next block at 4 rows (ema < 1.5),
# 8 rows (ema < 4.5) or 16 rows: m in {3, 7, 15} drafts.

def adaptive_block_cap(ema: float, block: int) -> int:
    e = np.float32(ema)
    cap = 4 if e < np.float32(1.5) else (8 if e < np.float32(4.5) else 16)
    return min(block, cap)


def adaptive_ema_update(ema: float, accepted: int) -> float:
    half = np.float32(0.5)
    return float(half * np.float32(ema) + half * np.float32(accepted))


@dataclass
class SpecTrace:
    tokens: List[int] = field(default_factory=list)
    rounds: int = 0
    accept_hist: List[int] = field(default_factory=list)   # per draft position
    per_round: List[dict] = field(default_factory=list)
    ctx_taps: List[np.ndarray] = field(default_factory=list)  # draft context, by position


DraftFn = Callable[[int, int, int, List[int]], List[int]]


def spec_rounds(tw: TargetWeights, dw: Optional[DraftWeights], cfg: OracleConfig,
                prompt: Sequence[int], n_new: int,
                draft_override: Optional[DraftFn] = None):
    """The speculative loop: draft -> verify -> accept -> roll back, as a
    generator: yields (trace, 0) after the prompt's forward and (trace, bl)
    after every round, bl = the rows that round's verify ran.

    Per round ([RFC] DFlash, "Key Implementation Details" Phase 3, and
    "Requested changes" 1 and 3):
      bl = min(B, n_new - generated, max_seq - n); bl == 1 -> plain step;
      draft bl-1 ids from [t_n, MASK...] over the tap context;
      verify [t_n, d_1..d_{bl-1}] at positions n..n+bl-1 in one forward;
      accept a = first mismatch, emit y_0..y_a (EOS-truncated);
      roll the target KV back to n + #emitted and append the taps of verify
      rows 0..#emitted-1 to the draft context.
    draft_override(t_n, n, bl, history) replaces the drafter's ids (used to
    pin the loop with adversarial drafts); the drafter is then not run.
    """
    B = cfg.block
    cache = KVCache(len(tw.layers), cfg.n_kv, cfg.head_dim)
    logits, taps = target_forward(tw, cfg, prompt, 0, cache)
    ctx_taps = [row for row in taps]                  # position p -> tap row
    tr = SpecTrace(tokens=[argmax_lowest(logits[-1])], accept_hist=[0] * (B - 1),
                   ctx_taps=ctx_taps)
    n = len(prompt)
    finished = cfg.eos_id >= 0 and tr.tokens[0] == cfg.eos_id
    ema = float(np.float32(B - 1))
    yield tr, 0
    while len(tr.tokens) < n_new and not finished:
        t_n = tr.tokens[-1]
        cap = adaptive_block_cap(ema, B) if cfg.adaptive_block else B
        bl = block_len(cap, n_new, len(tr.tokens), cfg.max_seq, n)
        if bl <= 1:
            d = []
        elif draft_override is not None:
            d = list(draft_override(t_n, n, bl, list(prompt) + tr.tokens))
        else:
            _, d = draft_forward(dw, tw.embed, cfg, np.stack(ctx_taps), t_n, n, bl,
                                 lm_head=tw.lm_head)
        logits, vtaps = target_forward(tw, cfg, [t_n] + d, n, cache)
        y = [argmax_lowest(logits[i]) for i in range(len(d) + 1)]
        a, emitted, finished = accept(d, y, cfg.eos_id)
        ema = adaptive_ema_update(ema, a)
        for j in range(min(a, len(tr.accept_hist))):
            tr.accept_hist[j] += 1
        # rollback: positions n..n+#emitted-1 hold the confirmed inputs
        n_new_len = n + len(emitted)
        cache.truncate(n_new_len)
        ctx_taps.extend(vtaps[i] for i in range(len(emitted)))
        tr.per_round.append(dict(n=n, bl=bl, a=a, emitted=len(emitted),
                                 kv_len=n_new_len, ctx_len=len(ctx_taps)))
        tr.tokens.extend(emitted)
        tr.rounds += 1
        n = n_new_len
        yield tr, bl


def spec_decode(tw: TargetWeights, dw: Optional[DraftWeights], cfg: OracleConfig,
                prompt: Sequence[int], n_new: int,
                draft_override: Optional[DraftFn] = None) -> SpecTrace:
    """The whole speculative loop of one sequence (spec_rounds run out)."""
    tr = None
    for tr, _ in spec_rounds(tw, dw, cfg, prompt, n_new, draft_override):
        pass
    return tr


@dataclass
class BatchTrace:
    traces: List[SpecTrace]
    rounds: int = 0                                            # batched rounds
    rows_per_round: List[int] = field(default_factory=list)   # verify rows, all sequences


def spec_decode_batch(tw: TargetWeights, dw: Optional[DraftWeights], cfg: OracleConfig,
                      prompts: Sequence[Sequence[int]], n_new,
                      draft_overrides: Optional[Sequence[Optional[DraftFn]]] = None) -> BatchTrace:
    """Several independent sequences decoded in lockstep rounds.

    The pages verify one sequence's 1+m rows per forward ([RFC] DFlash,
    "Key Implementation Details" Phase 3: a [1, 1+m] batch).  Batching
    sequences is this library's extension (a reading): in each batched
    round every unfinished sequence takes its own round (its own block
    length, drafts, acceptance and rollback), and the batched verify runs
    the sum of their rows.  Sequences share only the weights, so each
    sequence's result is its single-sequence speculative decode.  n_new is
    one budget for all sequences or one per sequence; draft_overrides, one
    per sequence, as spec_decode's draft_override.
    """
    budgets = list(n_new) if isinstance(n_new, (list, tuple)) else [n_new] * len(prompts)
    fns = list(draft_overrides) if draft_overrides is not None else [None] * len(prompts)
    gens = [spec_rounds(tw, dw, cfg, p, b, f) for p, b, f in zip(prompts, budgets, fns)]
    bt = BatchTrace(traces=[next(g)[0] for g in gens])
    active = list(range(len(gens)))
    while active:
        rows, still = 0, []
        for i in active:
            step = next(gens[i], None)
            if step is None:
                continue
            bt.traces[i], bl = step
            rows += bl
            still.append(i)
        if still:
            bt.rounds += 1
            bt.rows_per_round.append(rows)
        active = still
    return bt
