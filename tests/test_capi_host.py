"""Host-side checks of the C ABI (no GPU): the library loads, exports every
entry point include/dflash.h declares, and its configuration guards reject
bad shapes before any buffer is touched."""

import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def capi():
    from block_diffusion_speculative_gather_gb300 import build
    build.build()
    from block_diffusion_speculative_gather_gb300 import capi as m
    return m


def _declared():
    src = open(os.path.join(ROOT, "include", "dflash.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash_[a-z0-9_]+)\s*\(", src)))


def test_header_symbols_exported(capi):
    names = _declared()
    assert len(names) >= 15
    for n in names:
        assert hasattr(capi.lib, n), n
    assert set(names) == set(capi.EXPORTED)


def test_struct_sizes_match_header(capi):
    # 19 int32 fields, the int32 tap array and 2 floats
    assert C.sizeof(capi.dflash_config) == 4 * (19 + capi.MAX_TAPS + 2)
    assert C.sizeof(capi.dflash_weights) == 9 * 8
    assert C.sizeof(capi.dflash_layer) == 18 * 8
    assert C.sizeof(capi.dflash_stats_t) == 8 * (2 + capi.MAX_BLOCK) + 4 * 10


def _cfg(capi, **kw):
    from block_diffusion_speculative_gather_gb300.configs import TINY
    from block_diffusion_speculative_gather_gb300.runtime import make_config
    return make_config(TINY, **kw)


def test_sizes_for_valid_config(capi):
    cfg = _cfg(capi)
    assert capi.dflash_workspace_bytes(cfg) > 0
    assert capi.dflash_kv_target_bytes(cfg) == 2 * 2 * 2 * 256 * 64 * 4
    assert capi.dflash_kv_draft_bytes(cfg) == 1 * 2 * 2 * 256 * 64 * 4


@pytest.mark.parametrize("field,value", [
    ("hidden", 200), ("head_dim", 96), ("n_kv", 3), ("vocab", 4000), ("block_max", 17),
    ("block_max", 0), ("ffn", 1000), ("dtype", 7), ("drf_wfmt", 1), ("n_taps", 0),
    ("eos_id", 4096), ("max_seq", 1),
])
def test_config_guard_rejects_before_buffers(capi, field, value):
    cfg = _cfg(capi, **{field: value})
    assert capi.dflash_workspace_bytes(cfg) == 0
    out = C.c_void_p()
    w = capi.dflash_weights()
    rc = capi.lib.dflash_init(C.byref(cfg), C.byref(w), None, None, None, 0, C.byref(out))
    assert rc == -1, capi.lib.dflash_last_error()
    assert out.value is None


def test_bf16_query_group_guard(capi):
    # the tensor-core attention gives one warp to each q head of a kv head's group
    from block_diffusion_speculative_gather_gb300.configs import E2E_BF16
    from block_diffusion_speculative_gather_gb300.runtime import make_config
    assert capi.dflash_workspace_bytes(make_config(E2E_BF16)) > 0          # 32 / 8
    assert capi.dflash_workspace_bytes(make_config(E2E_BF16, n_kv=4)) == 0  # 32 / 4
    assert capi.dflash_workspace_bytes(_cfg(capi, n_q=16, n_kv=2)) > 0     # fp32: 8 per kv head


def test_tap_layer_guard(capi):
    cfg = _cfg(capi)
    cfg.tap_layer[1] = 5            # beyond the 2-layer target
    assert capi.dflash_workspace_bytes(cfg) == 0
    cfg = _cfg(capi)
    cfg.tap_layer[0], cfg.tap_layer[1] = 1, 0   # not increasing
    assert capi.dflash_workspace_bytes(cfg) == 0


def test_missing_weights_rejected(capi):
    cfg = _cfg(capi)
    out = C.c_void_p()
    w = capi.dflash_weights()       # all NULL
    rc = capi.lib.dflash_init(C.byref(cfg), C.byref(w), None, None, None, 0, C.byref(out))
    assert rc == -3 and "embed" in capi.lib.dflash_last_error().decode()


def test_null_context_calls_fail_cleanly(capi):
    assert capi.lib.dflash_draft_block(None, None, None) == -3
    assert capi.lib.dflash_verify_accept(None, None, None, None, None) == -3
    assert capi.lib.dflash_rollback(None, 5, 0, None) == -3
    assert capi.lib.dflash_attention_form(None, 0) == -3
    assert capi.lib.dflash_linear_dense(None, None, None, 1, 4, 64, None, None, None) == -3


def test_dense_linear_argument_guards(capi):
    # rejected before anything touches the device: the pointers are never read
    p = C.c_void_p(1 << 20)                       # 16-byte aligned, never dereferenced
    bad = [(1, 4, 96),     # k not a multiple of 64
           (1, 6, 64),     # n not a multiple of 4 (rows of y stay 16-byte aligned)
           (0, 4, 64),     # no rows
           (1, 4, 0)]      # no k
    for m, n, k in bad:
        assert capi.lib.dflash_linear_dense(p, p, None, m, n, k, p, p, None) == -3, (m, n, k)
    q = C.c_void_p((1 << 20) + 8)                 # misaligned
    assert capi.lib.dflash_linear_dense(q, p, None, 1, 4, 64, p, p, None) == -3
    assert capi.lib.dflash_prefill_taps(None, None, 0, None, 0, 1, 0, 1, None) == -3
    assert capi.lib.dflash_quantize_int4g64(None, 1, 256, None, None, None) == -3
    assert capi.lib.dflash_tap_reduce(None, 1, 1, 1, 8, None, None) == -3


def test_binding_checks_standalone_operands_before_the_library(capi):
    """The bindings of the standalone operations check dtype, shape,
    contiguity and device before calling the library (which sees only
    pointers): mismatches raise DFlashError(ARG) on the host, and host tensors
    are refused (the library has no CPU path)."""
    import torch
    bf, f32 = torch.bfloat16, torch.float32
    e = lambda: torch.zeros(2, dtype=torch.int32)
    cases = [
        ("w", lambda: capi.dflash_linear_dense(torch.zeros(8, 128, dtype=bf), torch.zeros(4, 64, dtype=bf),
                                               torch.zeros(4, 8), e())),
        ("y", lambda: capi.dflash_linear_dense(torch.zeros(8, 64, dtype=bf), torch.zeros(4, 64, dtype=bf),
                                               torch.zeros(8, 4), e())),
        ("x_lo", lambda: capi.dflash_linear_dense(torch.zeros(8, 64, dtype=bf), torch.zeros(4, 64, dtype=bf),
                                                  torch.zeros(4, 8), e(),
                                                  x_lo=torch.zeros(4, 64, dtype=f32))),
        ("err", lambda: capi.dflash_linear_dense(torch.zeros(8, 64, dtype=bf), torch.zeros(4, 64, dtype=bf),
                                                 torch.zeros(4, 8), torch.zeros(1, dtype=torch.int32))),
        ("x", lambda: capi.dflash_linear(torch.zeros(128, 64, dtype=bf), torch.zeros(8, 64, dtype=bf),
                                         torch.zeros(16, 128), torch.zeros(64, dtype=torch.uint8), e())),
        ("x", lambda: capi.dflash_linear_noalloc(torch.zeros(128, 64, dtype=bf),
                                                 torch.zeros(128, 16, dtype=bf).t(), torch.zeros(16, 128),
                                                 e())),
        ("err", lambda: capi.dflash_linear_noalloc(torch.zeros(128, 64, dtype=bf),
                                                   torch.zeros(16, 64, dtype=bf), torch.zeros(16, 128),
                                                   torch.zeros(2, dtype=torch.int64))),
        ("scales", lambda: capi.dflash_quantize_int4g64(torch.zeros(4, 256), torch.zeros(4, 128, dtype=torch.uint8),
                                                        torch.zeros(2, 4, dtype=torch.int16))),
        ("out", lambda: capi.dflash_tap_reduce([torch.zeros(3, 4 * 64, dtype=bf)] * 2, 3, 4, 64,
                                               torch.zeros(3, 64))),
        ("CUDA", lambda: capi.dflash_linear_dense(torch.zeros(8, 64, dtype=bf), torch.zeros(4, 64, dtype=bf),
                                                  torch.zeros(4, 8), e())),
        ("CUDA", lambda: capi.dflash_tap_reduce([torch.zeros(3, 4 * 64, dtype=bf)] * 2, 3, 4, 64,
                                                torch.zeros(3, 128))),
    ]
    for word, call in cases:
        with pytest.raises(capi.DFlashError) as exc:
            call()
        assert exc.value.code == -3 and word in str(exc.value), (word, str(exc.value))


def test_batch_workspace_guard(capi):
    # many-sequence rounds: 1 <= S <= 32 sequences of a bf16 model
    from block_diffusion_speculative_gather_gb300.configs import E2E_BF16
    from block_diffusion_speculative_gather_gb300.runtime import make_config
    cfg = make_config(E2E_BF16)
    sizes = [capi.dflash_batch_workspace_bytes(cfg, S) for S in (1, 8, 9, 16, 32)]
    assert all(b > 0 for b in sizes)
    assert sizes == sorted(sizes) and len(set(sizes)) == len(sizes)   # grows with S
    assert capi.dflash_batch_workspace_bytes(cfg, 0) == 0
    assert capi.dflash_batch_workspace_bytes(cfg, 33) == 0
    assert capi.dflash_batch_workspace_bytes(make_config(E2E_BF16.with_(tgt_int4=True)), 8) == 0
    assert capi.dflash_batch_workspace_bytes(make_config(E2E_BF16.with_(drf_int4=True)), 8) == 0
    assert capi.dflash_batch_workspace_bytes(_cfg(capi), 8) == 0      # fp32 model
