"""The five workloads the library is built and measured on.

tiny          2-layer fp32 target (hidden 256, 4 q / 2 kv heads, head_dim 64,
              SwiGLU 1024, vocab 4096) tapped at layers 0 and 1; 1-layer
              drafter; fc 512 -> 256; block 8; window 64; 32-token prompt,
              64 greedy tokens.
draft_bf16    Qwen3-4B-shaped 5-layer bf16 drafter alone: hidden 2560,
              32 q / 8 kv heads, head_dim 128, SwiGLU 9728, vocab 151936;
              1024 N(0,1) tap rows of 5 x 2560; block 16.
draft_int4    the same drafter with q/k/v/o/gate/up/down in INT4 group-64
              with bf16 scales; 16384 prefilled tap rows, window 2048, block 8.
e2e_bf16      36-layer Qwen3-4B-shaped bf16 target, taps at 5 evenly spaced
              layers, the draft_bf16 drafter; 1024-token prompt, 512 tokens;
              verify batches of 1+m rows, m in {3, 7, 15}.
hc_sweep      hyper-connection taps: [L, 4 x 4096] bf16 streams at 4 layers,
              mean over the 4 streams; verify forward of the e2e target at
              T = 1, 2, 4, 8, 16 rows over a 16384-token KV cache.
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Tuple


@dataclass(frozen=True)
class Workload:
    name: str
    hidden: int
    n_q: int
    n_kv: int
    head_dim: int
    ffn: int
    vocab: int
    tgt_layers: int          # 0 = drafter alone (taps supplied externally)
    drf_layers: int
    tap_layers: Tuple[int, ...]
    block: int
    window: int              # 0 = whole context
    dtype: str               # "f32" | "bf16": embedding, fc, caches, activations
    drf_int4: bool = False
    tgt_int4: bool = False   # target q/k/v/o/gate/up/down in INT4 group-64
    lm_int4: bool = False    # LM head: INT4 group-64 copy of the embedding
    adaptive_block: bool = False   # per-round block cap from recent acceptance
    prompt_len: int = 0
    n_new: int = 0
    n_ctx: int = 0           # externally supplied tap rows (drafter alone)
    max_seq: int = 0
    hc: int = 1
    eos_id: int = -1
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    ctx_norm: bool = True

    @property
    def n_taps(self) -> int:
        return len(self.tap_layers)

    @property
    def mask_id(self) -> int:
        return self.vocab - 1

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def evenly_spaced_taps(n_layers: int, n_taps: int) -> Tuple[int, ...]:
    """floor(i * (L - 1) / (n - 1)), i = 0..n-1: {0, 8, 17, 26, 35} for 36/5."""
    return tuple((i * (n_layers - 1)) // (n_taps - 1) for i in range(n_taps))


TINY = Workload(
    name="tiny", hidden=256, n_q=4, n_kv=2, head_dim=64, ffn=1024, vocab=4096,
    tgt_layers=2, drf_layers=1, tap_layers=(0, 1), block=8, window=64, dtype="f32",
    prompt_len=32, n_new=64, max_seq=256)

QWEN3_4B = dict(hidden=2560, n_q=32, n_kv=8, head_dim=128, ffn=9728, vocab=151936)

DRAFT_BF16 = Workload(
    name="draft_bf16", **QWEN3_4B, tgt_layers=0, drf_layers=5,
    tap_layers=evenly_spaced_taps(36, 5), block=16, window=0, dtype="bf16",
    n_ctx=1024, max_seq=1024 + 64)

DRAFT_INT4 = Workload(
    name="draft_int4", **QWEN3_4B, tgt_layers=0, drf_layers=5,
    tap_layers=evenly_spaced_taps(36, 5), block=8, window=2048, dtype="bf16",
    drf_int4=True, n_ctx=16384, max_seq=16384 + 64)

E2E_BF16 = Workload(
    name="e2e_bf16", **QWEN3_4B, tgt_layers=36, drf_layers=5,
    tap_layers=evenly_spaced_taps(36, 5), block=16, window=0, dtype="bf16",
    prompt_len=1024, n_new=512, max_seq=1024 + 512 + 64)

HC_SWEEP = Workload(
    name="hc_sweep", **QWEN3_4B, tgt_layers=36, drf_layers=0,
    tap_layers=evenly_spaced_taps(36, 5), block=16, window=0, dtype="bf16",
    prompt_len=16384, max_seq=16384 + 64, hc=4)

HC_TAP = dict(hc=4, hidden=4096, n_layers=4, rows=(16, 2048, 16384))

ALL = {w.name: w for w in (TINY, DRAFT_BF16, DRAFT_INT4, E2E_BF16, HC_SWEEP)}
