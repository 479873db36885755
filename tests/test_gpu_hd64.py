"""GPU parity of a bf16 model with head_dim 64 (hidden 512, 8 q / 4 kv heads,
SwiGLU 1536, vocab 4096, a 2-layer target tapped at layers 0 and 1, a
1-layer drafter): the 64-wide instantiations of the fused split-KV attention,
the dense prefill's attention and its row kernels (two elements per lane and
RoPE pair), the dense window ingest, against the CPU oracle.

Tolerance as in the Qwen3-4B-shaped tests: logits within rel 2e-2 of the
oracle, ids bit-exact where the oracle's top-2 margin is decidable;
speculative == greedy bit-exactly on the GPU.
"""

import numpy as np
import pytest
import torch

from block_diffusion_speculative_gather_gb300 import synth
from block_diffusion_speculative_gather_gb300.configs import Workload
from oracle import dflash_oracle as O
from tests import gpu_common as G
from tests.oracle_inputs import ModelTensors, oracle_config, oracle_draft, oracle_target

pytestmark = pytest.mark.gpu
TOL = 2e-2
W = Workload(name="hd64", hidden=512, n_q=8, n_kv=4, head_dim=64, ffn=1536, vocab=4096, tgt_layers=2,
             drf_layers=1, tap_layers=(0, 1), block=16, window=0, dtype="bf16", prompt_len=200, n_new=40,
             max_seq=512)


@pytest.fixture(scope="module")
def hd64():
    G.build_lib()
    m = ModelTensors(W, std=0.05, norm_std=0.1)
    prompt = synth.uniform_ids(W.prompt_len, W.vocab, seed=21)
    tw, dw, cfg = oracle_target(m), oracle_draft(m), oracle_config(W)
    ref, _ = O.target_forward(tw, cfg, prompt.tolist(), 0, O.KVCache(2, W.n_kv, W.head_dim))
    return dict(m=m, prompt=torch.from_numpy(prompt), tw=tw, dw=dw, cfg=cfg, ref=ref)


def _prefill(hd64, env, monkeypatch):
    from block_diffusion_speculative_gather_gb300.runtime import DFlash
    if env is not None:
        monkeypatch.setenv("DFLASH_DENSE_PREFILL", env)
    dec = DFlash(W, hd64["m"])
    monkeypatch.delenv("DFLASH_DENSE_PREFILL", raising=False)
    vl = G.logits_buf(W.vocab)
    dec.set_logits_out(vl, None)
    dec.prefill(hd64["prompt"], W.n_new)
    dec.check()
    dec.set_logits_out(None, None)
    return dec, vl


@pytest.mark.parametrize("env", [None, "0"], ids=["dense", "chunked"])
def test_hd64_prefill_logits(hd64, monkeypatch, env):
    dec, vl = _prefill(hd64, env, monkeypatch)
    P = W.prompt_len
    last = (P - 1) // 16 * 16
    rows = G.check_rows(f"hd64_prefill_{env}", vl[:P - last].cpu().numpy(), None,
                        hd64["ref"][last:P], TOL, 1e-3)
    if rows[-1]:
        assert dec.stats().t_n == int(np.argmax(hd64["ref"][P - 1]))
    dec.close()


def test_hd64_dense_matches_chunked_caches(hd64, monkeypatch):
    caps = (W.max_seq + 63) // 64 * 64
    kv = []
    for env in (None, "0"):
        dec, _ = _prefill(hd64, env, monkeypatch)
        kt = dec.kv_target.view(torch.float16).view(W.tgt_layers, 2, W.n_kv, caps, W.head_dim)
        kd = dec.kv_draft.view(torch.float16).view(W.drf_layers, 2, W.n_kv, caps, W.head_dim)
        kv.append((kt[:, :, :, :W.prompt_len].float().clone(), kd[:, :, :, :W.prompt_len].float().clone()))
        dec.close()
    for a, b in zip(kv[0], kv[1]):
        scale = b.abs().amax(dim=-1, keepdim=True).clamp_min(1e-6)
        assert ((a - b).abs() / scale).max().item() < 2.0 ** -8


def test_hd64_spec_equals_greedy_and_oracle(hd64, monkeypatch):
    dec, _ = _prefill(hd64, None, monkeypatch)
    gg = dec.greedy(hd64["prompt"], W.n_new)
    sp = dec.generate(hd64["prompt"], W.n_new)
    dec.check()
    assert sp == gg
    # the GPU greedy steps again with each step's logits, against the
    # oracle's greedy decoding (each step's logits kept for the margin test)
    P = W.prompt_len
    vl = G.logits_buf(W.vocab)
    dec.set_logits_out(vl, None)
    dec.prefill(hd64["prompt"], W.n_new)
    gl = [vl[(P - 1) % 16].clone()]
    st = dec.stats()
    while not st.finished and len(gl) < W.n_new:
        dec.verify(None)
        gl.append(vl[0].clone())
        st = dec.stats()
    dec.check()
    dec.close()
    cache = O.KVCache(W.tgt_layers, W.n_kv, W.head_dim)
    lg, _ = O.target_forward(hd64["tw"], hd64["cfg"], hd64["prompt"].tolist(), 0, cache)
    rows, toks, pos = [lg[-1]], [O.argmax_lowest(lg[-1])], P
    while len(toks) < W.n_new:
        lg, _ = O.target_forward(hd64["tw"], hd64["cfg"], [toks[-1]], pos, cache)
        rows.append(lg[0])
        toks.append(O.argmax_lowest(lg[0]))
        pos += 1
    floor = next((i for i, r in enumerate(rows) if not G.decidable(r, 1e-3)), len(rows))
    n = G.stream_prefix("hd64_greedy_stream", gg, [r.cpu().numpy() for r in gl], toks, rows, TOL)
    assert n >= floor and n > 0, (n, floor)
