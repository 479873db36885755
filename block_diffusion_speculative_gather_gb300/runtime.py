"""Python harness over the C ABI: PyTorch owns the device memory and the
stream, the library runs every step of the round in its own kernels.

    dec = DFlash(workload, ModelTensors(workload))
    dec.prefill(prompt)              # target prefill, or dec.prefill_taps(...)
    d = dec.draft()                  # draft ids on the device
    toks, n = dec.verify(d)          # accept + rollback + tap commit

`DFlash.generate` is the speculative loop; `DFlash.greedy` runs the same
verify kernels one row at a time (plain greedy decoding).
"""

from __future__ import annotations

import ctypes as C
from typing import List, Optional

import torch

from . import capi
from .configs import Workload


def _dtype_code(w: Workload) -> int:
    return capi.DFLASH_F32 if w.dtype == "f32" else capi.DFLASH_BF16


def make_config(w: Workload, **over) -> capi.dflash_config:
    cfg = capi.dflash_config()
    cfg.hidden, cfg.n_q, cfg.n_kv, cfg.head_dim = w.hidden, w.n_q, w.n_kv, w.head_dim
    cfg.ffn, cfg.vocab = w.ffn, w.vocab
    cfg.tgt_layers, cfg.drf_layers = w.tgt_layers, w.drf_layers
    cfg.n_taps = w.n_taps if w.drf_layers else 0
    for i, l in enumerate(w.tap_layers[: capi.MAX_TAPS]):
        cfg.tap_layer[i] = l
    cfg.block_max, cfg.window, cfg.max_seq, cfg.eos_id = w.block, w.window, w.max_seq, w.eos_id
    cfg.dtype = _dtype_code(w)
    cfg.tgt_wfmt = _dtype_code(w)
    cfg.drf_wfmt = capi.DFLASH_INT4G64 if w.drf_int4 else _dtype_code(w)
    if w.tgt_int4:
        cfg.tgt_wfmt = capi.DFLASH_INT4G64
    cfg.lm_wfmt = capi.DFLASH_INT4G64 if w.lm_int4 else 0
    cfg.adaptive_block = 1 if w.adaptive_block else 0
    cfg.ctx_norm = 1 if w.ctx_norm else 0
    cfg.rms_eps, cfg.rope_theta = w.rms_eps, w.rope_theta
    for k, v in over.items():
        setattr(cfg, k, v)
    return cfg


class DFlash:
    """One generation context on one GPU."""

    def __init__(self, w: Workload, model, device: str = "cuda", stream=None, **cfg_over):
        self._load(w, model, device, stream, **cfg_over)
        kvt = capi.dflash_kv_target_bytes(self.cfg)
        kvd = capi.dflash_kv_draft_bytes(self.cfg)
        wsb = capi.dflash_workspace_bytes(self.cfg)
        if wsb == 0:
            capi.check(-1)
        self.kv_target = torch.zeros(max(kvt, 16), dtype=torch.uint8, device=self.device)
        self.kv_draft = torch.zeros(max(kvd, 16), dtype=torch.uint8, device=self.device)
        self.workspace = torch.zeros(wsb, dtype=torch.uint8, device=self.device)
        torch.cuda.synchronize(self.device)
        self.ctx = capi.dflash_init(self.cfg, self._weights, self.kv_target, self.kv_draft,
                                    self.workspace)
        B = w.block
        self.draft_ids = torch.full((max(1, B - 1),), -1, dtype=torch.int32, device=self.device)
        self.tokens_out = torch.full((B,), -1, dtype=torch.int32, device=self.device)
        self.n_emitted = torch.zeros(1, dtype=torch.int32, device=self.device)

    def _load(self, w: Workload, model, device, stream, **cfg_over):
        """Weights on the device (INT4 copies made by the library's
        quantiser) and the C structs that point at them."""
        self.w = w
        self.device = torch.device(device)
        self._stream = stream      # None: the current stream at each call
        self.cfg = make_config(w, **cfg_over)
        dev = lambda t: None if t is None else t.to(self.device).contiguous()
        self.embed = dev(model.embed)
        self.final_norm_t = dev(model.final_norm_t)
        self.final_norm_d = dev(model.final_norm_d)
        self.ctx_norm = dev(model.ctx_norm)
        self.fc = dev(model.fc)
        self.tgt = [{k: dev(v) for k, v in lw.items()} for lw in model.tgt]
        self.drf = [{k: dev(v) for k, v in lw.items()} for lw in model.drf]
        if w.drf_int4:
            self._quantize_layers(self.drf)
        if w.tgt_int4:
            self._quantize_layers(self.tgt)
        self.lm_head = self.lm_scales = None
        if w.lm_int4:
            self.lm_head, self.lm_scales = self._quantize(self.embed)
        self._layers_t = (capi.dflash_layer * max(1, len(self.tgt)))(
            *[self._layer(lw) for lw in self.tgt])
        self._layers_d = (capi.dflash_layer * max(1, len(self.drf)))(
            *[self._layer(lw) for lw in self.drf])
        wts = capi.dflash_weights()
        wts.embed = self.embed.data_ptr()
        wts.final_norm_tgt = self.final_norm_t.data_ptr()
        wts.final_norm_drf = self.final_norm_d.data_ptr()
        wts.fc = self.fc.data_ptr() if self.fc is not None else None
        wts.ctx_norm = self.ctx_norm.data_ptr()
        wts.tgt = C.cast(self._layers_t, C.POINTER(capi.dflash_layer))
        wts.drf = C.cast(self._layers_d, C.POINTER(capi.dflash_layer))
        if self.lm_head is not None:
            wts.lm_head = self.lm_head.data_ptr()
            wts.lm_scales = self.lm_scales.data_ptr()
        self._weights = wts

    def _quantize(self, w: torch.Tensor):
        """INT4 group-64 (packed [n][k/2], bf16 scales [k/64][n]) of w [n][k]."""
        wf = w.float().contiguous()
        n, kk = wf.shape
        packed = torch.empty((n, kk // 2), dtype=torch.uint8, device=self.device)
        scales = torch.empty((kk // 64, n), dtype=torch.int16, device=self.device)
        capi.dflash_quantize_int4g64(wf, packed, scales, self.stream)
        return packed, scales

    def _quantize_layers(self, layers):
        for lw in layers:
            for k in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down"):
                lw[k], lw["s" + k[1:]] = self._quantize(lw[k])   # wq -> sq, w_gate -> s_gate

    @staticmethod
    def _layer(lw) -> capi.dflash_layer:
        l = capi.dflash_layer()
        for k in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "ln_attn", "ln_mlp",
                  "q_norm", "k_norm"):
            setattr(l, k, lw[k].data_ptr())
        for k in ("sq", "sk", "sv", "so", "s_gate", "s_up", "s_down"):
            if k in lw:
                setattr(l, k, lw[k].data_ptr())
        return l

    @property
    def stream(self):
        return self._stream if self._stream is not None else torch.cuda.current_stream(self.device)

    # ------------------------------------------------------------ the calls

    def prefill(self, prompt: torch.Tensor, max_new: int):
        self._prompt = prompt.to(self.device, torch.int32).contiguous()
        capi.dflash_prefill_taps(self.ctx, self._prompt, None, 0, 1, 0, max_new, self.stream)

    def prefill_taps(self, taps: torch.Tensor, hc: int, first_token: int, max_new: int):
        """taps: [n_taps, n_ext, hc * hidden] in the workload dtype."""
        self._taps = taps.to(self.device).contiguous()
        capi.dflash_prefill_taps(self.ctx, None, self._taps, self._taps.shape[1], hc,
                                 first_token, max_new, self.stream)

    def adopt_kv(self, n: int, pending_token: int, max_new: int):
        """Continue from caches filled by the caller (positions [0, n))."""
        capi.dflash_adopt_kv(self.ctx, n, pending_token, max_new, self.stream)

    def draft(self, out: Optional[torch.Tensor] = None) -> torch.Tensor:
        out = self.draft_ids if out is None else out
        capi.dflash_draft_block(self.ctx, out, self.stream)
        return out

    def verify(self, draft_ids: Optional[torch.Tensor]):
        capi.dflash_verify_accept(self.ctx, draft_ids, self.tokens_out, self.n_emitted,
                                  self.stream)
        return self.tokens_out, self.n_emitted

    def rollback(self, new_len: int, token: int):
        capi.dflash_rollback(self.ctx, new_len, token, self.stream)

    def stats(self) -> capi.dflash_stats_t:
        return capi.dflash_stats(self.ctx, self.stream)

    def check(self):
        capi.dflash_check(self.ctx, self.stream)

    def set_logits_out(self, verify_logits=None, draft_logits=None):
        capi.dflash_set_logits_out(self.ctx, verify_logits, draft_logits)

    # ------------------------------------------------------------ loops

    def _collect(self, out: List[int]):
        n = int(self.n_emitted.item())
        out.extend(self.tokens_out[:n].tolist())
        return n

    def generate(self, prompt: torch.Tensor, max_new: int, draft_fn=None) -> List[int]:
        """Speculative decoding; draft_fn(dec) may replace the drafter's ids."""
        self.prefill(prompt, max_new)
        st = self.stats()
        out = [st.t_n]
        while not st.finished and len(out) < max_new:
            d = draft_fn(self) if draft_fn is not None else self.draft()
            self.verify(d)
            self._collect(out)
            st = self.stats()
        return out

    def generate_graphed(self, prompt: torch.Tensor, max_new: int,
                         rounds_per_replay: int = 16) -> List[int]:
        """Speculative decoding with the rounds replayed from one CUDA graph of
        `rounds_per_replay` rounds.  Each replay ends by copying its rounds'
        emitted tokens and the progress words to pinned host memory; the
        host waits once per replay, collects the tokens and stops when the
        state says finished (rounds after that are empty on the device)."""
        B, K = self.w.block, rounds_per_replay
        self.prefill(prompt, max_new)
        graph = getattr(self, "_round_graph", None)
        if graph is None or graph[0] != K:
            self._round_graph = None
            stage = torch.zeros((K, B + 1), dtype=torch.int32, device=self.device)
            prog = torch.zeros(4, dtype=torch.int32, device=self.device)
            host_stage = torch.zeros((K, B + 1), dtype=torch.int32).pin_memory()
            host_prog = torch.zeros(4, dtype=torch.int32).pin_memory()
            s = torch.cuda.Stream(self.device)
            s.wait_stream(torch.cuda.current_stream(self.device))
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for r in range(K):
                    self.verify(self.draft())
                    stage[r, :B].copy_(self.tokens_out)
                    stage[r, B:].copy_(self.n_emitted)
                capi.dflash_progress(self.ctx, prog, s)
                host_stage.copy_(stage, non_blocking=True)
                host_prog.copy_(prog, non_blocking=True)
            self._round_graph = (K, g, stage, prog, host_stage, host_prog)
            # the capture ran nothing; the prefill above still holds
        _, g, stage, prog, host_stage, host_prog = self._round_graph
        st = self.stats()
        out = [st.t_n]
        done = bool(st.finished)
        ev = torch.cuda.Event()
        while not done and len(out) < max_new:
            g.replay()
            ev.record()
            ev.synchronize()
            rows = host_stage.tolist()
            for r in range(K):
                n = rows[r][B]
                out.extend(rows[r][:n])
            done = bool(host_prog[0].item())
        return out[:max_new]

    def greedy(self, prompt: torch.Tensor, max_new: int) -> List[int]:
        """Plain greedy decoding through the same verify kernels, one row a step."""
        self.prefill(prompt, max_new)
        st = self.stats()
        out = [st.t_n]
        while not st.finished and len(out) < max_new:
            self.verify(None)
            self._collect(out)
            st = self.stats()
        return out

    def close(self):
        self._round_graph = None
        if getattr(self, "ctx", None):
            capi.dflash_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class DFlashBatch(DFlash):
    """S independent sequences of one model decoded in lockstep rounds: one
    drafter forward and one target forward over all sequences' rows per
    round (dflash_batch_*).  Each sequence is a context of its own."""

    def __init__(self, w: Workload, model, S: int, device: str = "cuda", stream=None, **cfg_over):
        self._load(w, model, device, stream, **cfg_over)
        self.S = S
        kvt = capi.dflash_kv_target_bytes(self.cfg)
        kvd = capi.dflash_kv_draft_bytes(self.cfg)
        wsb = capi.dflash_batch_workspace_bytes(self.cfg, S)
        if wsb == 0:
            capi.check(-1)
        self.kv_target = torch.zeros(max(S * kvt, 16), dtype=torch.uint8, device=self.device)
        self.kv_draft = torch.zeros(max(S * kvd, 16), dtype=torch.uint8, device=self.device)
        self.workspace = torch.zeros(wsb, dtype=torch.uint8, device=self.device)
        torch.cuda.synchronize(self.device)
        self.batch = capi.dflash_batch_init(self.cfg, self._weights, S, self.kv_target,
                                            self.kv_draft, self.workspace)
        self.ctxs = [capi.dflash_batch_context(self.batch, s) for s in range(S)]
        self.ctx = None
        B = w.block
        self.draft_ids = torch.full((S, max(1, B - 1)), -1, dtype=torch.int32, device=self.device)
        self.tokens_out = torch.full((S, B), -1, dtype=torch.int32, device=self.device)
        self.n_emitted = torch.zeros(S, dtype=torch.int32, device=self.device)
        self._prompts = [None] * S

    def prefill(self, prompts, max_new):
        """prompts: S token tensors (lengths may differ); max_new: one budget
        or one per sequence."""
        budgets = list(max_new) if isinstance(max_new, (list, tuple)) else [max_new] * self.S
        for s, (p, b) in enumerate(zip(prompts, budgets)):
            self._prompts[s] = p.to(self.device, torch.int32).contiguous()
            capi.dflash_prefill_taps(self.ctxs[s], self._prompts[s], None, 0, 1, 0, b, self.stream)

    def draft(self, out: Optional[torch.Tensor] = None) -> torch.Tensor:
        out = self.draft_ids if out is None else out
        capi.dflash_batch_draft(self.batch, out, self.stream)
        return out

    def verify(self, draft_ids: Optional[torch.Tensor]):
        capi.dflash_batch_verify_accept(self.batch, draft_ids, self.tokens_out, self.n_emitted,
                                        self.stream)
        return self.tokens_out, self.n_emitted

    def stats(self, s: int = 0) -> capi.dflash_stats_t:
        return capi.dflash_stats(self.ctxs[s], self.stream)

    def check(self):
        capi.dflash_batch_check(self.batch, self.stream)

    def set_logits_out(self, verify_logits=None, draft_logits=None):
        capi.dflash_batch_set_logits_out(self.batch, verify_logits, draft_logits)

    def rollback(self, new_len: int, token: int, s: int = 0):
        capi.dflash_rollback(self.ctxs[s], new_len, token, self.stream)

    def _loop(self, prompts, max_new, speculative: bool, draft_fn=None) -> List[List[int]]:
        self.prefill(prompts, max_new)
        outs = [[self.stats(s).t_n] for s in range(self.S)]
        while True:
            sts = [self.stats(s) for s in range(self.S)]
            if all(st.finished for st in sts):
                break
            if speculative:
                d = draft_fn(self) if draft_fn is not None else self.draft()
            else:
                d = None
            toks, n = self.verify(d)
            toks, n = toks.cpu().tolist(), n.cpu().tolist()
            for s in range(self.S):
                outs[s].extend(toks[s][: n[s]])
        return outs

    def generate(self, prompts, max_new, draft_fn=None) -> List[List[int]]:
        """Speculative decoding of every sequence in lockstep rounds."""
        return self._loop(prompts, max_new, True, draft_fn)

    def greedy(self, prompts, max_new) -> List[List[int]]:
        """Plain greedy decoding of every sequence, one batched row each step."""
        return self._loop(prompts, max_new, False)

    def close(self):
        if getattr(self, "batch", None):
            capi.dflash_batch_destroy(self.batch)
            self.batch = None
            self.ctxs = []
