"""ctypes binding of libdflash.so (include/dflash.h), names as in the header.

Argument marshalling only: every step of the round runs in the library's
CUDA kernels.  Importing this module loads the library and raises if it is
missing; there is no other implementation to fall back to.
"""

from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdflash.so")

DFLASH_OK = 0
ERRORS = {-1: "CONFIG", -2: "CAPACITY", -3: "ARG", -4: "CUDA", -5: "DEVICE", -6: "TIMEOUT",
          -7: "STATE"}
DFLASH_F32, DFLASH_BF16, DFLASH_INT4G64 = 0, 1, 2
MAX_TAPS = 8
MAX_BLOCK = 16


class DFlashError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"DFLASH_ERR_{ERRORS.get(code, code)}: {msg}")
        self.code = code


class dflash_config(C.Structure):
    _fields_ = [
        ("hidden", C.c_int32), ("n_q", C.c_int32), ("n_kv", C.c_int32), ("head_dim", C.c_int32),
        ("ffn", C.c_int32), ("vocab", C.c_int32), ("tgt_layers", C.c_int32),
        ("drf_layers", C.c_int32), ("n_taps", C.c_int32), ("tap_layer", C.c_int32 * MAX_TAPS),
        ("block_max", C.c_int32), ("window", C.c_int32), ("max_seq", C.c_int32),
        ("eos_id", C.c_int32), ("dtype", C.c_int32), ("tgt_wfmt", C.c_int32),
        ("drf_wfmt", C.c_int32), ("ctx_norm", C.c_int32), ("rms_eps", C.c_float),
        ("rope_theta", C.c_float), ("lm_wfmt", C.c_int32), ("adaptive_block", C.c_int32),
    ]


class dflash_layer(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in (
        "wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down",
        "sq", "sk", "sv", "so", "s_gate", "s_up", "s_down",
        "ln_attn", "ln_mlp", "q_norm", "k_norm")]


class dflash_weights(C.Structure):
    _fields_ = [
        ("embed", C.c_void_p), ("final_norm_tgt", C.c_void_p), ("final_norm_drf", C.c_void_p),
        ("fc", C.c_void_p), ("ctx_norm", C.c_void_p),
        ("tgt", C.POINTER(dflash_layer)), ("drf", C.POINTER(dflash_layer)),
        ("lm_head", C.c_void_p), ("lm_scales", C.c_void_p),
    ]


class dflash_stats_t(C.Structure):
    _fields_ = [
        ("rounds", C.c_int64), ("emitted", C.c_int64), ("accept_hist", C.c_int64 * MAX_BLOCK),
        ("n", C.c_int32), ("t_n", C.c_int32), ("block_len", C.c_int32), ("generated", C.c_int32),
        ("max_new", C.c_int32), ("ctx_len", C.c_int32), ("finished", C.c_int32),
        ("last_accept", C.c_int32), ("device_error", C.c_int32), ("pad_", C.c_int32),
    ]


class dflash_profile_t(C.Structure):
    _fields_ = [("gemm_launches", C.c_int64), ("gemm_ms", C.c_double), ("gemm_bytes", C.c_double),
                ("gemm_weight_bytes", C.c_double)]


def _load() -> C.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with "
            "`python -m block_diffusion_speculative_gather_gb300.build` (no fallback exists)")
    lib = C.CDLL(LIB_PATH)
    vp, i32, i64, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
    sig = {
        "dflash_workspace_bytes": (sz, [C.POINTER(dflash_config)]),
        "dflash_kv_target_bytes": (sz, [C.POINTER(dflash_config)]),
        "dflash_kv_draft_bytes": (sz, [C.POINTER(dflash_config)]),
        "dflash_init": (C.c_int, [C.POINTER(dflash_config), C.POINTER(dflash_weights), vp, vp,
                                  vp, sz, C.POINTER(vp)]),
        "dflash_prefill_taps": (C.c_int, [vp, vp, i32, vp, i32, i32, i32, i32, vp]),
        "dflash_draft_block": (C.c_int, [vp, vp, vp]),
        "dflash_verify_accept": (C.c_int, [vp, vp, vp, vp, vp]),
        "dflash_rollback": (C.c_int, [vp, i64, i32, vp]),
        "dflash_stats": (C.c_int, [vp, C.POINTER(dflash_stats_t), vp]),
        "dflash_check": (C.c_int, [vp, vp]),
        "dflash_set_logits_out": (C.c_int, [vp, vp, vp]),
        "dflash_destroy": (None, [vp]),
        "dflash_last_error": (C.c_char_p, []),
        "dflash_tap_reduce": (C.c_int, [C.POINTER(vp), i32, i32, i32, i32, vp, vp]),
        "dflash_quantize_int4g64": (C.c_int, [vp, i32, i32, vp, vp, vp]),
        "dflash_profile": (C.c_int, [vp, i32, C.POINTER(dflash_profile_t)]),
        "dflash_launch_count": (i64, []),
        "dflash_selftest_timeout": (C.c_int, [vp, i64, vp]),
        "dflash_adopt_kv": (C.c_int, [vp, i32, i32, i32, vp]),
        "dflash_linear_workspace_bytes": (sz, [i32, i32]),
        "dflash_linear": (C.c_int, [vp, vp, i32, i32, vp, vp, sz, vp, vp]),
        "dflash_linear_noalloc": (C.c_int, [vp, vp, i32, i32, vp, vp, vp]),
        "dflash_progress": (C.c_int, [vp, vp, vp]),
        "dflash_attention_form": (C.c_int, [vp, i32]),
        "dflash_linear_dense": (C.c_int, [vp, vp, vp, i32, i32, i32, vp, vp, vp]),
        "dflash_batch_workspace_bytes": (sz, [C.POINTER(dflash_config), i32]),
        "dflash_batch_init": (C.c_int, [C.POINTER(dflash_config), C.POINTER(dflash_weights), i32, vp,
                                        vp, vp, sz, C.POINTER(vp)]),
        "dflash_batch_context": (vp, [vp, i32]),
        "dflash_batch_draft": (C.c_int, [vp, vp, vp]),
        "dflash_batch_verify_accept": (C.c_int, [vp, vp, vp, vp, vp]),
        "dflash_batch_set_logits_out": (C.c_int, [vp, vp, vp]),
        "dflash_batch_check": (C.c_int, [vp, vp]),
        "dflash_batch_destroy": (None, [vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


lib = _load()

EXPORTED = ("dflash_workspace_bytes", "dflash_kv_target_bytes", "dflash_kv_draft_bytes",
            "dflash_init", "dflash_prefill_taps", "dflash_draft_block", "dflash_verify_accept",
            "dflash_rollback", "dflash_stats", "dflash_check", "dflash_set_logits_out",
            "dflash_destroy", "dflash_last_error", "dflash_tap_reduce",
            "dflash_quantize_int4g64", "dflash_profile", "dflash_launch_count",
            "dflash_selftest_timeout", "dflash_adopt_kv", "dflash_linear_workspace_bytes",
            "dflash_linear", "dflash_linear_noalloc",
            "dflash_progress", "dflash_attention_form", "dflash_linear_dense",
            "dflash_batch_workspace_bytes", "dflash_batch_init", "dflash_batch_context",
            "dflash_batch_draft", "dflash_batch_verify_accept", "dflash_batch_set_logits_out",
            "dflash_batch_check", "dflash_batch_destroy")


def check(rc: int) -> None:
    if rc != DFLASH_OK:
        raise DFlashError(rc, lib.dflash_last_error().decode())


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


DFLASH_ERR_ARG = -3


def _need(t, name: str, dtypes, shape) -> None:
    """Binding-side argument check of a standalone operation's tensor (the C
    ABI sees only pointers and sizes): dtype, shape (None = any extent) and
    row-major contiguity.  Raises DFlashError(ARG) before any device work."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise DFlashError(DFLASH_ERR_ARG, f"{name}: a torch tensor is required")
    if dtypes is not None and t.dtype not in dtypes:
        raise DFlashError(DFLASH_ERR_ARG, f"{name}: dtype {t.dtype}, expected one of {dtypes}")
    if shape is not None and (t.dim() != len(shape) or
                              any(e is not None and e != d for e, d in zip(shape, t.shape))):
        raise DFlashError(DFLASH_ERR_ARG, f"{name}: shape {tuple(t.shape)}, expected {shape}")
    if not t.is_contiguous():
        raise DFlashError(DFLASH_ERR_ARG, f"{name}: must be contiguous (row-major)")


def _on_gpu(**tensors) -> None:
    """Every tensor on one CUDA device: the library reads device pointers and
    has no CPU path."""
    devs = set()
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise DFlashError(DFLASH_ERR_ARG, f"{name}: a CUDA tensor is required (no CPU path)")
        devs.add(t.device)
    if len(devs) > 1:
        raise DFlashError(DFLASH_ERR_ARG, f"tensors on several devices: {sorted(map(str, devs))}")


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def dflash_workspace_bytes(cfg: dflash_config) -> int:
    return lib.dflash_workspace_bytes(C.byref(cfg))


def dflash_kv_target_bytes(cfg: dflash_config) -> int:
    return lib.dflash_kv_target_bytes(C.byref(cfg))


def dflash_kv_draft_bytes(cfg: dflash_config) -> int:
    return lib.dflash_kv_draft_bytes(C.byref(cfg))


def dflash_init(cfg, weights, kv_target, kv_draft, workspace) -> int:
    out = C.c_void_p()
    check(lib.dflash_init(C.byref(cfg), C.byref(weights), _ptr(kv_target), _ptr(kv_draft),
                          _ptr(workspace), workspace.numel() * workspace.element_size(),
                          C.byref(out)))
    return out.value


def dflash_prefill_taps(ctx, prompt_ids, ext_taps, n_ext, hc, first_token, max_new, stream=None):
    n_prompt = 0 if prompt_ids is None else prompt_ids.numel()
    check(lib.dflash_prefill_taps(ctx, _ptr(prompt_ids), n_prompt, _ptr(ext_taps), n_ext, hc,
                                  first_token, max_new, _stream(stream)))


def dflash_draft_block(ctx, draft_ids, stream=None):
    check(lib.dflash_draft_block(ctx, _ptr(draft_ids), _stream(stream)))


def dflash_verify_accept(ctx, draft_ids, tokens_out, n_emitted, stream=None):
    check(lib.dflash_verify_accept(ctx, _ptr(draft_ids), _ptr(tokens_out), _ptr(n_emitted),
                                   _stream(stream)))


def dflash_rollback(ctx, new_len: int, token: int, stream=None):
    check(lib.dflash_rollback(ctx, new_len, token, _stream(stream)))


def dflash_stats(ctx, stream=None) -> dflash_stats_t:
    out = dflash_stats_t()
    check(lib.dflash_stats(ctx, C.byref(out), _stream(stream)))
    return out


def dflash_check(ctx, stream=None):
    check(lib.dflash_check(ctx, _stream(stream)))


def dflash_set_logits_out(ctx, verify_logits, draft_logits):
    check(lib.dflash_set_logits_out(ctx, _ptr(verify_logits), _ptr(draft_logits)))


def dflash_destroy(ctx):
    lib.dflash_destroy(ctx)


def dflash_tap_reduce(layer_streams, rows: int, hc: int, hidden: int, out, stream=None):
    import torch
    for i, t in enumerate(layer_streams):
        _need(t, f"layer_streams[{i}]", (torch.bfloat16,), (rows, hc * hidden))
    _need(out, "out", (torch.float32,), (rows, len(layer_streams) * hidden))
    _on_gpu(out=out, **{f"layer_streams[{i}]": t for i, t in enumerate(layer_streams)})
    arr = (C.c_void_p * len(layer_streams))(*[t.data_ptr() for t in layer_streams])
    check(lib.dflash_tap_reduce(arr, len(layer_streams), rows, hc, hidden, _ptr(out),
                                _stream(stream)))


def dflash_quantize_int4g64(w, packed, scales, stream=None):
    import torch
    _need(w, "w", (torch.float32,), (None, None))
    n, k = w.shape
    _need(packed, "packed", (torch.uint8,), (n, k // 2))
    two_byte = tuple(d for d in (torch.int16, getattr(torch, "uint16", None)) if d is not None)
    _need(scales, "scales", two_byte, (k // 64, n))
    _on_gpu(w=w, packed=packed, scales=scales)
    check(lib.dflash_quantize_int4g64(_ptr(w), n, k, _ptr(packed), _ptr(scales), _stream(stream)))


def dflash_profile(ctx, mode: int) -> dflash_profile_t:
    """mode 1 start, 2 read, 0 read and stop (see include/dflash.h)."""
    out = dflash_profile_t()
    check(lib.dflash_profile(ctx, mode, C.byref(out)))
    return out


def dflash_launch_count() -> int:
    return lib.dflash_launch_count()


def dflash_selftest_timeout(ctx, limit_ns: int, stream=None):
    check(lib.dflash_selftest_timeout(ctx, limit_ns, _stream(stream)))


def dflash_adopt_kv(ctx, n: int, pending_token: int, max_new: int, stream=None):
    check(lib.dflash_adopt_kv(ctx, n, pending_token, max_new, _stream(stream)))


def dflash_linear_workspace_bytes(n: int, k: int) -> int:
    return lib.dflash_linear_workspace_bytes(n, k)


def _linear_operands(w, x, y):
    import torch
    _need(w, "w", (torch.bfloat16,), (None, None))
    n, k = w.shape
    _need(x, "x", (torch.bfloat16,), (MAX_BLOCK, k))
    _need(y, "y", (torch.float32,), (MAX_BLOCK, n))
    return n, k


def dflash_linear(w, x, y, workspace, err, stream=None):
    """y = x w^T (16 rows); err (int32[2] on the device) receives the GEMM's
    error words after it: {0, 0}, or {1, site} when a bounded wait ran out."""
    import torch
    n, k = _linear_operands(w, x, y)
    _need(workspace, "workspace", None, None)
    _need(err, "err", (torch.int32,), (2,))
    _on_gpu(w=w, x=x, y=y, workspace=workspace, err=err)
    check(lib.dflash_linear(_ptr(w), _ptr(x), n, k, _ptr(y), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _ptr(err),
                            _stream(stream)))


def dflash_linear_noalloc(w, x, y, err, stream=None):
    """y = x w^T like dflash_linear, with the library's fixed scratch instead
    of a caller workspace (for callers that cannot allocate device memory);
    err as in dflash_linear."""
    import torch
    n, k = _linear_operands(w, x, y)
    _need(err, "err", (torch.int32,), (2,))
    _on_gpu(w=w, x=x, y=y, err=err)
    check(lib.dflash_linear_noalloc(_ptr(w), _ptr(x), n, k, _ptr(y), _ptr(err), _stream(stream)))


def dflash_progress(ctx, out, stream=None):
    """Enqueue the progress words (finished, generated, n, emitted) into the
    int32[4] device tensor `out`."""
    check(lib.dflash_progress(ctx, _ptr(out), _stream(stream)))


def dflash_attention_form(ctx, model: int) -> int:
    """Attention form of the target (model 0) or drafter (model 1):
    2 tcgen05, 1 mma.sync split-KV, 0 separate partial/combine kernels."""
    r = lib.dflash_attention_form(ctx, model)
    check(min(r, 0))
    return r


def dflash_linear_dense(w, x, y, err, x_lo=None, stream=None):
    """y[m][n] = x[m] . w[n] (+ x_lo[m] . w[n]) on the tcgen05 dense GEMM:
    x, x_lo bf16 [M][K], w bf16 [N][K], y fp32 [M][N], err int32[2] zeros."""
    import torch
    _need(x, "x", (torch.bfloat16,), (None, None))
    m, k = x.shape
    _need(w, "w", (torch.bfloat16,), (None, k))
    n = w.shape[0]
    _need(y, "y", (torch.float32,), (m, n))
    if x_lo is not None:
        _need(x_lo, "x_lo", (torch.bfloat16,), (m, k))
    _need(err, "err", (torch.int32,), (None,))
    if err.numel() < 2:
        raise DFlashError(DFLASH_ERR_ARG, "err: int32[2] required")
    _on_gpu(w=w, x=x, x_lo=x_lo, y=y, err=err)
    check(lib.dflash_linear_dense(_ptr(w), _ptr(x), _ptr(x_lo), m, n, k, _ptr(y), _ptr(err),
                                  _stream(stream)))


# ---- several sequences in lockstep rounds

def dflash_batch_workspace_bytes(cfg, S: int) -> int:
    return lib.dflash_batch_workspace_bytes(C.byref(cfg), S)


def dflash_batch_init(cfg, weights, S: int, kv_target, kv_draft, workspace):
    out = C.c_void_p()
    check(lib.dflash_batch_init(C.byref(cfg), C.byref(weights), S, _ptr(kv_target), _ptr(kv_draft),
                                _ptr(workspace), workspace.numel() * workspace.element_size(),
                                C.byref(out)))
    return out.value


def dflash_batch_context(b, s: int):
    c = lib.dflash_batch_context(b, s)
    if not c:
        check(DFLASH_ERR_ARG)
    return c


def dflash_batch_draft(b, draft_ids, stream=None):
    check(lib.dflash_batch_draft(b, _ptr(draft_ids), _stream(stream)))


def dflash_batch_verify_accept(b, draft_ids, tokens_out, n_emitted, stream=None):
    check(lib.dflash_batch_verify_accept(b, _ptr(draft_ids), _ptr(tokens_out), _ptr(n_emitted),
                                         _stream(stream)))


def dflash_batch_set_logits_out(b, verify_logits=None, draft_logits=None):
    check(lib.dflash_batch_set_logits_out(b, _ptr(verify_logits), _ptr(draft_logits)))


def dflash_batch_check(b, stream=None):
    check(lib.dflash_batch_check(b, _stream(stream)))


def dflash_batch_destroy(b) -> None:
    lib.dflash_batch_destroy(b)
