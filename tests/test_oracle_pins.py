"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test names what fixes the expected value: a value the pages print, a closed form, an
invariant of the op, a library routine, or an independent float64 restatement (tests/torch_ref.py).
These run on the CPU only.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle
import synth
from tests import torch_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def facts():
    with open(os.path.join(GOLDEN, "archdef_facts.json")) as f:
        return json.load(f)


# ---------------------------------------------------------------- dequantisation (GGUF formats)

def test_half_to_float_all_bit_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float32)
    got = oracle.dequant(synth.GGML_F16, bits.view(np.uint8), 65536)
    same = (got.view(np.uint32) == want.view(np.uint32)) | (np.isnan(got) & np.isnan(want))
    assert same.all()


def test_q8_0_hand_built_block():
    # d = 0.5, codes -16..15: weights are exactly -8.0 .. 7.5 in steps of 0.5
    blk = np.zeros(34, np.uint8)
    blk[0:2] = np.array([0.5], np.float16).view(np.uint8)
    blk[2:] = np.arange(-16, 16, dtype=np.int8).view(np.uint8)
    got = oracle.dequant(synth.GGML_Q8_0, blk, 32)
    assert np.array_equal(got, np.arange(-16, 16, dtype=np.float32) * 0.5)


def test_q8_0_two_blocks_use_their_own_scale():
    blk = np.zeros(68, np.uint8)
    blk[0:2] = np.array([0.25], np.float16).view(np.uint8)
    blk[2:34] = np.full(32, 4, np.int8).view(np.uint8)
    blk[34:36] = np.array([-2.0], np.float16).view(np.uint8)
    blk[36:68] = np.full(32, -3, np.int8).view(np.uint8)
    got = oracle.dequant(synth.GGML_Q8_0, blk, 64)
    assert np.array_equal(got[:32], np.full(32, 1.0, np.float32))
    assert np.array_equal(got[32:], np.full(32, 6.0, np.float32))


def test_q4_0_hand_built_block_nibble_order():
    # byte j holds element j in its low nibble and element j+16 in its high nibble (GGUF Q4_0);
    # with low = j and high = 15 - j the weights are d*(j-8) and d*(7-j).
    blk = np.zeros(18, np.uint8)
    blk[0:2] = np.array([0.125], np.float16).view(np.uint8)
    j = np.arange(16, dtype=np.uint8)
    blk[2:] = j | ((15 - j) << 4)
    got = oracle.dequant(synth.GGML_Q4_0, blk, 32)
    want = np.concatenate([(j.astype(np.float32) - 8), (7 - j.astype(np.float32))]) * 0.125
    assert np.array_equal(got, want)


def test_dequant_f32_is_identity():
    x = np.random.default_rng(0).standard_normal(37).astype(np.float32)
    assert np.array_equal(oracle.dequant(synth.GGML_F32, x.view(np.uint8), 37), x)


# ---------------------------------------------------------------- rms_norm

def test_rms_norm_unit_weights_give_unit_rms():
    x = np.random.default_rng(1).standard_normal(4096).astype(np.float32) * 37.0
    y = oracle.rms_norm(x, np.ones_like(x), 0.0)
    assert abs(np.sqrt(np.mean(y.astype(np.float64) ** 2)) - 1.0) < 1e-6


def test_rms_norm_scale_invariance_and_weight_is_elementwise():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(256).astype(np.float32)
    w = (1 + 0.1 * rng.standard_normal(256)).astype(np.float32)
    y1 = oracle.rms_norm(x, w, 0.0)
    y2 = oracle.rms_norm(x * np.float32(8.0), w, 0.0)  # exact power-of-two scale
    assert np.array_equal(y1, y2)
    y_unit = oracle.rms_norm(x, np.ones_like(w), 0.0).astype(np.float64)
    assert np.allclose(y1, y_unit * w, rtol=2e-7, atol=0)


def test_rms_norm_eps_matters_for_small_inputs():
    x = np.full(16, 1e-4, np.float32)
    y = oracle.rms_norm(x, np.ones_like(x), 1e-6)
    # closed form: 1e-4 / sqrt(1e-8 + 1e-6)
    assert np.allclose(y, 1e-4 / math.sqrt(1e-8 + 1e-6), rtol=1e-6)


# ---------------------------------------------------------------- rope

@pytest.mark.parametrize("adjacent", [False, True])
def test_rope_identity_at_position_zero(adjacent):
    v = np.random.default_rng(3).standard_normal(4 * 64).astype(np.float32)
    assert np.array_equal(oracle.rope(v, 4, 0, 1e6, adjacent), v)


@pytest.mark.parametrize("adjacent", [False, True])
def test_rope_preserves_each_pair_norm(adjacent):
    hd = 128
    v = np.random.default_rng(4).standard_normal(hd).astype(np.float32)
    r = oracle.rope(v, 1, 777, 5e5, adjacent).astype(np.float64)
    v = v.astype(np.float64)
    if adjacent:
        a, b = v.reshape(-1, 2).T, r.reshape(-1, 2).T
    else:
        a, b = (v[: hd // 2], v[hd // 2:]), (r[: hd // 2], r[hd // 2:])
    assert np.allclose(np.hypot(*a), np.hypot(*b), rtol=1e-6)


@pytest.mark.parametrize("adjacent", [False, True])
def test_rope_relative_position_property(adjacent):
    # <R(p+s) q, R(s) k> does not depend on s
    rng = np.random.default_rng(5)
    q = rng.standard_normal(64).astype(np.float32)
    k = rng.standard_normal(64).astype(np.float32)
    dots = [float(np.dot(oracle.rope(q, 1, 5 + s, 1e4, adjacent).astype(np.float64),
                         oracle.rope(k, 1, s, 1e4, adjacent).astype(np.float64)))
            for s in (0, 1, 17, 300)]
    assert np.allclose(dots, dots[0], rtol=1e-5)


@pytest.mark.parametrize("adjacent", [False, True])
def test_rope_pairing_and_frequencies(adjacent):
    # Pair 0 has frequency base^0 = 1, so at position p it turns by exactly p radians; pair j turns
    # by p * base^(-2j/hd). A unit vector in pair j's first slot lands on (cos, sin) of that angle.
    hd, base, p = 16, 100.0, 3
    for j in range(hd // 2):
        i0, i1 = (2 * j, 2 * j + 1) if adjacent else (j, j + hd // 2)
        e = np.zeros(hd, np.float32)
        e[i0] = 1.0
        r = oracle.rope(e, 1, p, base, adjacent)
        ang = p * base ** (-2.0 * j / hd)
        assert abs(r[i0] - math.cos(ang)) < 1e-7 and abs(r[i1] - math.sin(ang)) < 1e-7
        others = np.delete(r, [i0, i1])
        assert not others.any()


def test_norm_heads_then_rope_differs_from_rope_then_norm_heads():
    # The order matters with a non-uniform head weight, and not with unit weights (rope keeps the
    # head's norm), so a test with unit weights would prove nothing.
    rng = np.random.default_rng(6)
    hd, nh = 64, 2
    v = rng.standard_normal(nh * hd).astype(np.float32)
    w = (1 + 0.1 * rng.standard_normal(hd)).astype(np.float32)

    def norm_heads(x, w):
        return np.concatenate([oracle.rms_norm(x[h * hd:(h + 1) * hd], w, 1e-6) for h in range(nh)])
    a = oracle.rope(norm_heads(v, w), nh, 9, 1e6, False)
    b = norm_heads(oracle.rope(v, nh, 9, 1e6, False), w)
    assert np.abs(a - b).max() > 1e-3
    one = np.ones(hd, np.float32)
    a1 = oracle.rope(norm_heads(v, one), nh, 9, 1e6, False)
    b1 = norm_heads(oracle.rope(v, nh, 9, 1e6, False), one)
    assert np.allclose(a1, b1, atol=1e-6)


# ---------------------------------------------------------------- attention

def test_attention_single_key_returns_its_value():
    rng = np.random.default_rng(7)
    q, K, V = (rng.standard_normal((1, 64)).astype(np.float32) for _ in range(3))
    assert np.array_equal(oracle.attend(q[0], K, V, 0, 0), V[0])


def test_attention_identical_keys_average_the_values():
    rng = np.random.default_rng(8)
    q = rng.standard_normal(32).astype(np.float32)
    K = np.tile(rng.standard_normal(32).astype(np.float32), (5, 1))
    V = rng.standard_normal((5, 32)).astype(np.float32)
    assert np.allclose(oracle.attend(q, K, V, 0, 4), V.astype(np.float64).mean(0), atol=1e-6)


def test_attention_weights_are_the_softmax_and_sum_to_one():
    # With V = identity rows the output is the weight vector itself.
    rng = np.random.default_rng(9)
    hd, n = 32, 20
    q = rng.standard_normal(hd).astype(np.float32)
    K = rng.standard_normal((n, hd)).astype(np.float32)
    V = np.eye(n, hd, dtype=np.float32)
    p = oracle.attend(q, K, V, 0, n - 1)[:n].astype(np.float64)
    want = scipy.special.softmax(K.astype(np.float64) @ q.astype(np.float64) / math.sqrt(hd))
    assert abs(p.sum() - 1.0) < 1e-6
    assert np.allclose(p, want, rtol=1e-6, atol=1e-9)


def test_attention_range_excludes_keys_outside_it():
    rng = np.random.default_rng(10)
    q = rng.standard_normal(16).astype(np.float32)
    K = rng.standard_normal((10, 16)).astype(np.float32)
    V = rng.standard_normal((10, 16)).astype(np.float32)
    full = oracle.attend(q, K[4:8], V[4:8], 0, 3)
    ranged = oracle.attend(q, K, V, 4, 7)
    assert np.array_equal(full, ranged)


# ---------------------------------------------------------------- activations

def test_gelu_is_x_times_normal_cdf():
    x = np.linspace(-8, 8, 4001).astype(np.float32)
    want = x.astype(np.float64) * scipy.stats.norm.cdf(x.astype(np.float64))
    assert np.allclose(oracle.act("gelu", x), want, rtol=1e-6, atol=1e-7)


def test_gelu_and_gelu_tanh_differ_by_about_1e_3():
    # The pages say the two gates differ by about 1e-3 and that gemma3 needs the tanh one. The
    # largest gap over [-8, 8] is 4.7e-4, at |x| = 2.7 (the gap is even in x, since both gates
    # satisfy f(x) - f(-x) = x): the same order, and far above f32 noise.
    x = np.linspace(-8, 8, 160001).astype(np.float32)
    d = np.abs(oracle.act("gelu", x).astype(np.float64) - oracle.act("gelu_tanh", x))
    assert 4.5e-4 < d.max() < 5.0e-4
    assert 2.5 < abs(x[d.argmax()]) < 2.9


@pytest.mark.parametrize("kind", ["silu", "gelu", "gelu_tanh", "relu"])
def test_gates_satisfy_f_x_minus_f_minus_x_equals_x(kind):
    # x*s(x) - (-x)*s(-x) = x*(s(x) + s(-x)) = x for s = sigmoid, Phi, the tanh form and the step.
    x = np.linspace(-6, 6, 1201).astype(np.float32)
    f = oracle.act(kind, x).astype(np.float64)
    g = oracle.act(kind, -x).astype(np.float64)
    assert np.allclose(f - g, x, atol=2e-6)


def test_silu_is_x_times_logistic():
    x = np.linspace(-20, 20, 2001).astype(np.float32)
    want = x.astype(np.float64) * scipy.special.expit(x.astype(np.float64))
    assert np.allclose(oracle.act("silu", x), want, rtol=1e-6, atol=1e-12)


# ---------------------------------------------------------------- matmul

@pytest.mark.parametrize("wtype", ["f32", "f16", "q8_0", "q4_0"])
def test_matvec_matches_numpy_float64(wtype):
    t = synth.make_weight(11, "w", wtype, (96, 40))
    x = np.random.default_rng(12).standard_normal(96).astype(np.float32)
    got = oracle.matvec(t.dtype, t.data, 96, 40, x)
    want = torch_ref.dequant(t) @ x.astype(np.float64)
    assert np.allclose(got, want, rtol=1e-6, atol=1e-7 * np.abs(want).max())


# ---------------------------------------------------------------- archdef facts

@pytest.mark.parametrize("arch", ["gemma3", "llama", "qwen2", "qwen3"])
def test_shipped_archdefs_have_the_published_step_counts(arch):
    cfg = {"qwen3": "tiny", "llama": "llama3_8b", "qwen2": "qwen2_7b", "gemma3": "gemma3_1b"}[arch]
    m = oracle.Model(arch, oracle.load_archdef(arch), synth.metadata(synth.CONFIGS[cfg]), 8)
    assert m.steps(1) == facts()["steps_per_layer"][arch]


def test_oracle_rejects_unknown_ops_and_wrong_arch_name():
    text = oracle.load_archdef("qwen3")
    with pytest.raises(oracle.OracleError, match="line 28"):
        oracle.Model("qwen3", text.replace("silu(g)", "siluu(g)"), synth.metadata(synth.CONFIGS["tiny"]), 8)
    with pytest.raises(oracle.OracleError, match="declares"):
        oracle.Model("llama", text, synth.metadata(synth.CONFIGS["tiny"]), 8)


# ---------------------------------------------------------------- whole forward

def _tiny_like(arch, **over):
    base = {"qwen3": "tiny", "llama": "llama3_8b", "qwen2": "qwen2_7b", "gemma3": "gemma3_1b"}[arch]
    small = dict(n_layer=3, n_embd=128, n_head=4, n_head_kv=2, head_dim=32, n_ff=192, n_vocab=300,
                 context_length=64)
    if arch == "gemma3":
        small.update(n_layer=7, n_head_kv=1, head_dim=64, sliding_window=5)
    small.update(over)
    return synth.scaled(synth.CONFIGS[base], name=f"{arch}_small", **small)


ARCH_OPTS = {
    "qwen3": dict(rope_adjacent=False),
    "llama": dict(rope_adjacent=True),
    "qwen2": dict(rope_adjacent=False),
    "gemma3": dict(rope_adjacent=False, window_pattern=6, embed_scale=33.941125, act="gelu_tanh"),
}


@pytest.mark.parametrize("arch", ["qwen3", "llama", "qwen2", "gemma3"])
@pytest.mark.parametrize("wtype", ["f32", "f16", "q8_0", "q4_0"])
def test_forward_matches_independent_float64_restatement(arch, wtype):
    cfg = _tiny_like(arch, wtype=wtype)
    W = synth.make_model(cfg, seed=0)
    toks = synth.tokens(cfg, 12)
    m = oracle.model_from_synth(cfg, W, 32)
    got = [m.forward(toks[i:i + 1], i) for i in range(len(toks))]
    want, _ = torch_ref.forward(cfg, W, toks, **ARCH_OPTS[arch])
    for i in range(len(toks)):
        err = np.abs(got[i] - want[i]).max() / np.abs(want[i]).max()
        assert err < 2e-5, (i, err)


def test_bulk_prefill_equals_token_by_token_exactly():
    cfg = _tiny_like("qwen2")
    W = synth.make_model(cfg)
    toks = synth.tokens(cfg, 9)
    a = oracle.model_from_synth(cfg, W, 32)
    b = oracle.model_from_synth(cfg, W, 32)
    for i in range(8):
        la = a.forward(toks[i:i + 1], i)
    lb = b.forward(toks[:8], 0)
    assert np.array_equal(la, lb)
    assert np.array_equal(a.forward(toks[8:9], 8), b.forward(toks[8:9], 8))


@pytest.mark.parametrize("arch", ["qwen2", "gemma3"])
def test_chunked_prefill_equals_one_bulk_forward_exactly(arch):
    """Bulk forwards at positions > 0 attend to the cache the earlier forwards left: three chunks
    (4 + 3 + 5 rows at positions 0, 4, 7) give the same last logits and the same cache as one
    12-row forward (gemma3: through its sliding-window layers too)."""
    cfg = _tiny_like(arch)                       # gemma3: window of 5 keys on its local layers
    W = synth.make_model(cfg)
    toks = synth.tokens(cfg, 13)
    a = oracle.model_from_synth(cfg, W, 32)
    b = oracle.model_from_synth(cfg, W, 32)
    for p0, p1 in ((0, 4), (4, 7), (7, 12)):
        la = a.forward(toks[p0:p1], p0)
    lb = b.forward(toks[:12], 0)
    assert np.array_equal(la, lb)
    for layer in range(cfg.n_layer):
        ka, va = a.read_kv(layer, 0, 12, cfg.n_head_kv, cfg.head_dim)
        kb, vb = b.read_kv(layer, 0, 12, cfg.n_head_kv, cfg.head_dim)
        assert np.array_equal(ka, kb) and np.array_equal(va, vb)
    assert np.array_equal(a.forward(toks[12:13], 12), b.forward(toks[12:13], 12))


def test_scale_by_a_metadata_key_equals_scale_by_its_value():
    """`scale(x, embedding_length)` multiplies by the metadata value (256 for this model), exactly as
    the literal does."""
    cfg = _tiny_like("qwen3", n_embd=256)
    W = synth.make_model(cfg)
    toks = synth.tokens(cfg, 3)
    base = oracle.load_archdef("qwen3")
    texts = [base.replace("  x = embed(token_embd.weight)\n", f"  x = embed(token_embd.weight)\n  scale(x, {c})\n", 1)
             for c in ("embedding_length", "256")]
    assert all(t != base for t in texts)
    a = oracle.model_from_synth(cfg, W, 8, archdef_text=texts[0])
    b = oracle.model_from_synth(cfg, W, 8, archdef_text=texts[1])
    c = oracle.model_from_synth(cfg, W, 8)
    for i in range(3):
        la, lb, lc = (x.forward(toks[i:i + 1], i) for x in (a, b, c))
        assert np.array_equal(la, lb) and not np.array_equal(la, lc)


def test_copy_makes_an_independent_register():
    """`c = copy(x)` holds the value of x at that step: `add(x, c)` right after it is x + x = 2x,
    bit for bit `scale(x, 2)` (doubling is exact in f32); and with x doubled after the copy,
    `add(x, c)` is 2x + x = 3x, bit for bit `scale(x, 3)` (2x is exact, so both round 3x once). A
    copy that aliased x would give 4x there."""
    cfg = _tiny_like("llama")
    W = synth.make_model(cfg)
    toks = synth.tokens(cfg, 3)
    base = oracle.load_archdef("llama")
    embed = "  x = embed(token_embd.weight)\n"

    def with_prologue(extra):
        t = base.replace(embed, embed + extra, 1)
        assert t != base
        return t

    texts = {
        "copy_add": with_prologue("  c = copy(x)\n  add(x, c)\n"),
        "scale2": with_prologue("  scale(x, 2)\n"),
        "copy_scale_add": with_prologue("  c = copy(x)\n  scale(x, 2)\n  add(x, c)\n"),
        "scale3": with_prologue("  scale(x, 3)\n"),
    }
    ms = {k: oracle.model_from_synth(cfg, W, 8, archdef_text=t) for k, t in texts.items()}
    plain = oracle.model_from_synth(cfg, W, 8)
    for i in range(3):
        out = {k: m.forward(toks[i:i + 1], i) for k, m in ms.items()}
        assert np.array_equal(out["copy_add"], out["scale2"])
        assert np.array_equal(out["copy_scale_add"], out["scale3"])
        assert not np.array_equal(out["scale2"], out["scale3"])
        assert not np.array_equal(out["scale2"], plain.forward(toks[i:i + 1], i))


def test_tied_embedding_fallback():
    cfg = _tiny_like("qwen3", tied=True)
    W = synth.make_model(cfg)
    assert "output.weight" not in W
    W2 = dict(W)
    e = W["token_embd.weight"]
    W2["output.weight"] = synth.Tensor("output.weight", e.dtype, e.ne, e.data.copy())
    toks = synth.tokens(cfg, 4)
    a = oracle.model_from_synth(cfg, W, 16)
    b = oracle.model_from_synth(cfg, W2, 16)
    for i in range(4):
        assert np.array_equal(a.forward(toks[i:i + 1], i), b.forward(toks[i:i + 1], i))


def test_zero_blocks_leave_the_embedding_closed_form():
    # All block matrices zero: every branch adds 0, so x stays the embedding row and the logits are
    # W_out . rms_norm(E[token]) * output_norm.
    cfg = _tiny_like("llama", wtype="f32")
    W = synth.make_model(cfg)
    for name, t in W.items():
        if name.startswith("blk.") and len(t.ne) == 2:
            W[name] = synth.Tensor(name, t.dtype, t.ne, np.zeros_like(t.data))
    toks = synth.tokens(cfg, 3)
    m = oracle.model_from_synth(cfg, W, 8)
    E = torch_ref.dequant(W["token_embd.weight"])
    O = torch_ref.dequant(W["output.weight"])
    wn = W["output_norm.weight"].data.view(np.float32).astype(np.float64)
    for i, t in enumerate(toks):
        e = E[t]
        want = O @ (e / np.sqrt(np.mean(e * e) + cfg.eps) * wn)
        got = m.forward(toks[i:i + 1], i)
        assert np.allclose(got, want, rtol=1e-5, atol=1e-6 * np.abs(want).max())


def test_swapping_norm_heads_and_rope_changes_the_model():
    cfg = _tiny_like("qwen3")
    W = synth.make_model(cfg)
    text = oracle.load_archdef("qwen3")
    lines = text.split("\n")
    i_nq = next(i for i, l in enumerate(lines) if "norm_heads(q" in l)
    i_rq = next(i for i, l in enumerate(lines) if "rope(q" in l)
    i_nk = next(i for i, l in enumerate(lines) if "norm_heads(k" in l)
    i_rk = next(i for i, l in enumerate(lines) if "rope(k" in l)
    lines[i_nq], lines[i_rq] = lines[i_rq], lines[i_nq]
    lines[i_nk], lines[i_rk] = lines[i_rk], lines[i_nk]
    swapped = "\n".join(lines)
    toks = synth.tokens(cfg, 4)
    a = oracle.model_from_synth(cfg, W, 8)
    b = oracle.model_from_synth(cfg, W, 8, archdef_text=swapped)
    diffs = [np.abs(a.forward(toks[i:i + 1], i) - b.forward(toks[i:i + 1], i)).max() for i in range(4)]
    assert diffs[0] < 1e-6          # position 0: rope is the identity, order cannot matter
    assert max(diffs[1:]) > 1e-3    # later positions: a different model


def test_window_at_least_context_equals_global_attention():
    cfg = _tiny_like("gemma3")
    W = synth.make_model(cfg)
    toks = synth.tokens(cfg, 8)
    wide = synth.scaled(cfg, sliding_window=64)
    none = synth.scaled(cfg, sliding_window=0)
    a = oracle.model_from_synth(wide, W, 16)
    b = oracle.model_from_synth(none, W, 16)
    for i in range(8):
        assert np.array_equal(a.forward(toks[i:i + 1], i), b.forward(toks[i:i + 1], i))


@pytest.mark.parametrize("t,sees", [(0, "global"), (7, "global"), (8, "all")])
def test_only_every_sixth_gemma3_layer_sees_keys_outside_the_window(t, sees):
    """Five of every six gemma3 layers attend over a sliding window, the sixth over everything, and a
    window of W keys at position p allows keys p - W + 1 .. p. With W = 5, 7 layers and a step at
    position 12, change the cached key and value of position t in one layer: the logits move iff
    that layer can see t, i.e. t = 8 in every layer, t = 7 or 0 only in layer 5 (i mod 6 = 5); an
    unseen change leaves them bit for bit."""
    cfg = _tiny_like("gemma3")                  # 7 layers, window 5
    assert cfg.n_layer == 7 and cfg.sliding_window == 5
    W = synth.make_model(cfg)
    toks = synth.tokens(cfg, 13)
    base = oracle.model_from_synth(cfg, W, 16)
    base.forward(toks[:12], 0)
    ref = base.forward(toks[12:13], 12)
    for layer in range(cfg.n_layer):
        m = oracle.model_from_synth(cfg, W, 16)
        m.forward(toks[:12], 0)
        k, v = m.read_kv(layer, t, 1, cfg.n_head_kv, cfg.head_dim)
        m.write_kv(layer, t, k + 3.0, -v)
        moved = not np.array_equal(m.forward(toks[12:13], 12), ref)
        assert moved == (sees == "all" or layer % 6 == 5), (t, layer)


def test_cache_rows_past_the_current_position_are_never_read():
    """Causality: a step at position p attends over keys 0 .. p only. Huge values written into the
    cache rows p + 1 .. (left over from an earlier, longer conversation, say) leave the logits bit
    for bit."""
    cfg = _tiny_like("llama", wtype="q8_0")
    W = synth.make_model(cfg)
    toks = synth.tokens(cfg, 6)
    a = oracle.model_from_synth(cfg, W, 16)
    b = oracle.model_from_synth(cfg, W, 16)
    junk = np.full((cfg.n_head_kv, 10, cfg.head_dim), 1e6, np.float32)
    for layer in range(cfg.n_layer):
        b.write_kv(layer, 6, junk, -junk)
    a.forward(toks[:5], 0)
    b.forward(toks[:5], 0)
    assert np.array_equal(a.forward(toks[5:6], 5), b.forward(toks[5:6], 5))


def test_injected_kv_reproduces_the_prefix():
    cfg = _tiny_like("qwen3")
    W = synth.make_model(cfg)
    toks = synth.tokens(cfg, 7)
    a = oracle.model_from_synth(cfg, W, 16)
    for i in range(6):
        a.forward(toks[i:i + 1], i)
    b = oracle.model_from_synth(cfg, W, 16)
    for l in range(cfg.n_layer):
        k, v = a.read_kv(l, 0, 6, cfg.n_head_kv, cfg.head_dim)
        b.write_kv(l, 0, k, v)
    b.set_kv_len(6)
    assert np.array_equal(a.forward(toks[6:7], 6), b.forward(toks[6:7], 6))


def test_injected_random_kv_matches_restatement():
    cfg = _tiny_like("llama", wtype="q8_0")
    W = synth.make_model(cfg)
    P = 20
    pre = [synth.kv_fill(cfg, l, P) for l in range(cfg.n_layer)]
    m = oracle.model_from_synth(cfg, W, 32)
    for l, (k, v) in enumerate(pre):
        m.write_kv(l, 0, k, v)
    m.set_kv_len(P)
    toks = synth.tokens(cfg, 1)
    got = m.forward(toks, P)
    want, _ = torch_ref.forward(cfg, W, toks, rope_adjacent=True, kv_prefix=pre)
    assert np.abs(got - want[0]).max() < 2e-5 * np.abs(want[0]).max()


# ------------------------------------------------------------------------------ f16 KV configuration

def test_round_to_half_matches_numpy_float16():
    """The oracle's f32 -> f16 rounding (used only by the f16-KV configuration) against numpy's
    conversion: random magnitudes across the normal and subnormal ranges, exact ties between
    neighbouring halves (ties go to even), and the overflow boundary."""
    L = oracle.lib()
    rng = np.random.default_rng(5)
    halves = np.arange(0, 0x7c00, dtype=np.uint16).view(np.float16).astype(np.float32)
    ties = ((halves[:-1].astype(np.float64) + halves[1:]) / 2).astype(np.float32)
    vals = np.concatenate([rng.normal(0, 1, 4000), rng.normal(0, 1e-5, 2000), rng.normal(0, 3e4, 2000),
                           ties[::7], -ties[::11], [65504.0, 65519.99, 65520.0, 70000.0, 6e-8, 2.9e-8, 3.0e-8, 0.0]])
    vals = vals.astype(np.float32)
    with np.errstate(over="ignore"):            # values past 65520 round to infinity, on purpose
        want = vals.astype(np.float16).astype(np.float32)
    got = np.array([L.orc_round_to_half(float(v)) for v in vals], np.float32)
    assert np.array_equal(got, want)


def test_f16_kv_configuration_stores_the_rounded_keys_and_values():
    """With the f16-KV configuration the cache holds exactly the f16 rounding of what the f32
    configuration stores. Layer 0's keys and values depend only on the embeddings, so they are
    computed identically in both models and must match bit for bit after rounding."""
    L = oracle.lib()
    cfg = synth.CONFIGS["tiny"]
    W = synth.make_model(cfg)
    a = oracle.model_from_synth(cfg, W, 16)
    b = oracle.model_from_synth(cfg, W, 16)
    a.set_kv_f16(True)
    toks = synth.tokens(cfg, 5, seed=1)
    la = a.forward(toks[:3], 0)
    lb = b.forward(toks[:3], 0)
    ka, va = a.read_kv(0, 0, 3, cfg.n_head_kv, cfg.head_dim)
    kb, vb = b.read_kv(0, 0, 3, cfg.n_head_kv, cfg.head_dim)
    rk = np.array([L.orc_round_to_half(float(x)) for x in kb.ravel()], np.float32).reshape(kb.shape)
    rv = np.array([L.orc_round_to_half(float(x)) for x in vb.ravel()], np.float32).reshape(vb.shape)
    assert np.array_equal(ka, rk) and np.array_equal(va, rv)
    assert not np.array_equal(ka, kb)
    # the logits move by the rounding only
    assert 0 < np.abs(la - lb).max() <= 2e-3 * np.abs(lb).max()
