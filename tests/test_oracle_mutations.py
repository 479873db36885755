"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in one oracle function, on the CPU: the
function's source with one edit, compiled in the oracle module's namespace
and patched in for the duration of the case.  The mistakes are the kind a
restatement of the pages could make: a wrong GQA head mapping, RoPE pairing,
sign or frequency, a dropped norm weight or k-norm, swapped SwiGLU operands,
a causal mask off by one, the sliding window's anchor off by one, argmax ties
to the highest index, acceptance or rollback off by one, the bonus token
dropped, taps committed from the wrong rows or taken before the layer, the
hc layout interleaved, INT4 nibbles or scale wrong, drafts read from block
row 0, a causal draft block, the drafter's context keys and values built
wrong, the mask token replaced, the attention scale or residual wrong, the
untied LM head ignored, EOS truncation or the hc scale wrong, the adaptive
average or the batched row count wrong.  Every case must make at least one pin of the
oracle test modules fail an assertion; the unmutated oracle passes them all.
"""

import inspect
import itertools
import signal
import textwrap

import pytest

from block_diffusion_speculative_gather_gb300 import synth
from block_diffusion_speculative_gather_gb300.configs import TINY
from oracle import dflash_oracle as O
from tests import test_formats as TF
from tests import test_oracle_model as TM
from tests import test_oracle_pins as TN
from tests import test_oracle_primitives as TP
from tests.oracle_inputs import ModelTensors, oracle_config, oracle_draft, oracle_target

MUTATIONS = [
    ("gqa_head_mapping", "attention", "kh = h // group", "kh = h % n_kv"),
    ("rope_sign", "rope_rotate_half", "x1 * cos - x2 * sin, x2 * cos + x1 * sin",
     "x1 * cos + x2 * sin, x2 * cos - x1 * sin"),
    ("rope_adjacent_pairs", "rope_rotate_half", "x1, x2 = x[..., :half], x[..., half:]",
     "x1, x2 = x[..., 0::2], x[..., 1::2]"),
    ("rope_frequency", "rope_angles", "(-(2.0 * np.arange(half, dtype=F64)) / head_dim)",
     "(-(np.arange(half, dtype=F64)) / head_dim)"),
    ("rms_norm_weight_dropped", "rms_norm", "np.sqrt(ms + eps) * f64(w)", "np.sqrt(ms + eps)"),
    ("silu_sign", "silu", "np.exp(-x)", "np.exp(x)"),
    ("swiglu_operands_swapped", "mlp",
     'silu(linear(h, lw["w_gate"])) * linear(h, lw["w_up"])',
     'silu(linear(h, lw["w_up"])) * linear(h, lw["w_gate"])'),
    ("k_norm_dropped", "qkv_project", 'k = rms_norm(k, lw["k_norm"], cfg.rms_eps)', "k = k"),
    ("causal_off_by_one", "causal_visible", "<= np.asarray(q_pos)[:, None]",
     "<= np.asarray(q_pos)[:, None] + 1"),
    ("window_anchor_off_by_one", "block_context_range", "max(0, n - window)",
     "max(0, n - window + 1)"),
    ("argmax_ties_highest", "argmax_lowest", "int(np.argmax(logits_row))",
     "int(len(logits_row) - 1 - np.argmax(np.asarray(logits_row)[::-1]))"),
    ("acceptance_index_shift", "first_mismatch", "draft_ids[a] == target_ids[a]",
     "draft_ids[a] == target_ids[min(a + 1, len(target_ids) - 1)]"),
    ("bonus_token_dropped", "accept", "emitted = list(target_ids[: a + 1])",
     "emitted = list(target_ids[: max(a, 1)])"),
    ("block_len_budget_off_by_one", "block_len", "return min(block, max_new - generated,",
     "return min(block, max_new - generated + 1,"),
    ("rollback_off_by_one", "spec_rounds", "n_new_len = n + len(emitted)",
     "n_new_len = n + len(emitted) - (1 if len(emitted) > 1 else 0)"),
    ("tap_commit_from_row_0", "spec_rounds", "ctx_taps.extend(vtaps[i] for i in range(len(emitted)))",
     "ctx_taps.extend(vtaps[0] for i in range(len(emitted)))"),
    ("tap_before_layer", "target_forward",
     "x = target_layer(x, lw, cfg, positions, cache, l)\n        if l in cfg.tap_layers:\n"
     "            taps[l] = x.copy()",
     "if l in cfg.tap_layers:\n            taps[l] = x.copy()\n"
     "        x = target_layer(x, lw, cfg, positions, cache, l)"),
    ("hc_layout_interleaved", "hc_mean", "x[:, s * H:(s + 1) * H]", "x[:, s::hc]"),
    ("int4_nibble_order", "quantize_int4_g64", "(u[:, 0::2] | (u[:, 1::2] << 4))",
     "((u[:, 0::2] << 4) | u[:, 1::2])"),
    ("int4_scale_divisor", "quantize_int4_g64", "absmax / np.float32(7.0)", "absmax / np.float32(8.0)"),
    ("int4_dequant_offset", "dequant_int4_g64", "(u - 8)", "(u - 7)"),
    ("drafts_from_row_0", "draft_forward", "for j in range(1, bl)]", "for j in range(0, bl - 1)]"),
    ("draft_block_causal", "block_visible", "vis[:, :len(ctx_pos)] = ctx_ok[None, :]",
     "vis[:, :len(ctx_pos)] = ctx_ok[None, :]\n"
     "    vis[:, len(ctx_pos):] = np.tril(np.ones((bl, bl), dtype=bool))"),
    ("adaptive_threshold_inclusive", "adaptive_block_cap", "e < np.float32(1.5)", "e <= np.float32(1.5)"),
    ("adaptive_average_weights", "adaptive_ema_update",
     "half * np.float32(ema) + half * np.float32(accepted)",
     "np.float32(0.75) * np.float32(ema) + np.float32(0.25) * np.float32(accepted)"),
    ("ctx_rope_positions_shifted", "draft_forward", "ctx_pos,\n                              cfg.rope_theta",
     "[p + 1 for p in ctx_pos],\n                              cfg.rope_theta"),
    ("ctx_k_norm_dropped", "draft_forward", 'rope_rotate_half(rms_norm(kc, lw["k_norm"], cfg.rms_eps), ctx_pos,',
     "rope_rotate_half(kc, ctx_pos,"),
    ("ctx_values_from_w_k", "draft_forward", 'vc = linear(c, lw["wv"])', 'vc = linear(c, lw["wk"])'),
    ("mask_token_replaced", "draft_forward", "[t_n] + [cfg.mask_id] * (bl - 1)", "[t_n] * bl"),
    ("attention_scale", "target_layer", "1.0 / math.sqrt(cfg.head_dim)", "1.0 / cfg.head_dim"),
    ("attention_residual_dropped", "target_layer", 'x = x + linear(a.reshape(x.shape[0], -1), lw["wo"])',
     'x = linear(a.reshape(x.shape[0], -1), lw["wo"])'),
    ("untied_lm_head_ignored", "target_forward", "logits = linear(h, tw.head())",
     "logits = linear(h, tw.embed)"),
    ("eos_dropped_from_output", "accept", "emitted = emitted[: emitted.index(eos_id) + 1]",
     "emitted = emitted[: max(emitted.index(eos_id), 1)]"),
    ("hc_mean_scale", "hc_mean", "acc * (1.0 / hc)", "acc * (1.0 / max(hc - 1, 1))"),
    ("batch_rows_counted_per_sequence", "spec_decode_batch", "rows += bl", "rows += 1"),
]


def _mutant(fn_name, old, new):
    src = textwrap.dedent(inspect.getsource(getattr(O, fn_name)))
    assert src.count(old) == 1, (fn_name, old)
    ns = {}
    exec(compile(src.replace(old, new), O.__file__, "exec"), O.__dict__, ns)
    return ns[fn_name]


def _checks(tiny):
    """Every test function of the oracle test modules, parametrisations
    expanded, with the `tiny` model fixture supplied; cheap modules first."""
    out = []
    for mod in (TP, TN, TF, TM):
        for name, fn in vars(mod).items():
            if not name.startswith("test_") or not inspect.isfunction(fn):
                continue
            params = list(inspect.signature(fn).parameters)
            grids = []
            for m in getattr(fn, "pytestmark", []):
                if m.name != "parametrize":
                    continue
                names = m.args[0].split(",") if isinstance(m.args[0], str) else list(m.args[0])
                vals = [v.values if hasattr(v, "values") else v for v in m.args[1]]
                vals = [v if isinstance(v, tuple) and len(names) > 1 else (v,) for v in vals]
                grids.append([dict(zip([n.strip() for n in names], v)) for v in vals])
            if set(params) - {"tiny"} - {k for g in grids for d in g for k in d}:
                continue                      # needs a fixture this runner does not supply
            for combo in itertools.product(*grids) if grids else [()]:
                kw = {k: v for d in combo for k, v in d.items()}
                if "tiny" in params:
                    kw["tiny"] = tiny
                out.append((f"{mod.__name__}.{name}", fn, kw))
    return out


@pytest.fixture(scope="module")
def tiny():
    m = ModelTensors(TINY, std=0.1)
    return dict(tw=oracle_target(m), dw=oracle_draft(m), cfg=oracle_config(TINY),
                prompt=synth.uniform_ids(TINY.prompt_len, TINY.vocab).tolist())


def _first_failure(checks, limit_s=120):
    def on_alarm(signum, frame):
        raise TimeoutError("pin run exceeded its time limit")
    old = signal.signal(signal.SIGALRM, on_alarm)
    signal.alarm(limit_s)
    # the primitives' module-level generator is restored afterwards, so the
    # pin modules draw the same inputs whether or not this runner ran first
    rng_state = TP.RNG.bit_generator.state
    try:
        for label, fn, kw in checks:
            try:
                fn(**kw)
            except Exception as e:   # AssertionError or an error the mistake provokes
                return label, e
        return None
    finally:
        signal.alarm(0)
        signal.signal(signal.SIGALRM, old)
        TP.RNG.bit_generator.state = rng_state


def test_unmutated_oracle_passes_every_pin(tiny):
    checks = _checks(tiny)
    assert len(checks) > 60
    assert _first_failure(checks) is None


@pytest.mark.parametrize("case", MUTATIONS, ids=[c[0] for c in MUTATIONS])
def test_planted_mistake_fails_a_pin(tiny, monkeypatch, case):
    label, fn_name, old, new = case
    monkeypatch.setattr(O, fn_name, _mutant(fn_name, old, new))
    hit = _first_failure(_checks(tiny))
    assert hit is not None, f"no pin caught the planted mistake {label}"
    # a pin's own check, not an incidental error of the edited source
    assert isinstance(hit[1], AssertionError), (label, hit[0], repr(hit[1]))
