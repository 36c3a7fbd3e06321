"""GPU parity at the full sizes of the four named workloads (the tiny one is in test_gpu_parity.py).

For each model: the same seeded weights on both sides, a 16-token prompt run as one bulk forward,
then 16 teacher-forced decode steps; then, after a KV reset, the same N(0, 1) keys and values
injected into positions [0, L-4) on both sides and 4 teacher-forced steps ending at position L-1,
with L the context length the decode is measured at (4096 for qwen3-0.6B, 8192 for llama-3-8B and
gemma3-1B, where 22 of the 26 layers only see their last 512 keys, 2048 for qwen2-7B).

qwen2-7B (Q4_0, Q/K/V bias) also runs its 2048-token prompt as one bulk forward and token by token
on the GPU: the last row's logits and every cached key and value must agree within the tolerance;
and a 64-token bulk forward is compared with the oracle's.

Tolerances as in test_gpu_parity.py: max|dlogit| <= 2e-3 * max|logit| per step, argmax equal where
the oracle's top-2 gap exceeds twice that.
"""
import numpy as np
import pytest

import oracle
import synth
from decoder_token_step_gb300 import build as syn_build
from decoder_token_step_gb300 import syn

pytestmark = pytest.mark.gpu

TOL = 2e-3
LONG = {"qwen3_0_6b": 4096, "llama3_8b": 8192, "gemma3_1b": 8192, "qwen2_7b": 2048}


@pytest.fixture(scope="module", autouse=True)
def library():
    syn_build.build()
    syn.lib()


def rel(got, want):
    return float(np.abs(got.astype(np.float64) - want).max() / np.abs(want).max())


def argmax_ok(top, want):
    s = np.sort(want)
    if s[-1] - s[-2] > 2 * TOL * np.abs(want).max():
        return top == int(np.argmax(want))
    return True


def gpu_model(cfg, W, max_ctx):
    m = syn.Model(syn.read_archdef(cfg.arch), synth.metadata(cfg, max_ctx), max_ctx, arch=cfg.arch)
    m.load_tensors(W)
    m.finalize()
    return m


def check(m, o, toks, pos0):
    for i, t in enumerate(toks):
        got, top = m.forward([int(t)], pos0 + i)
        want = o.forward([int(t)], pos0 + i)
        e = rel(got, want)
        assert e <= TOL, f"step {pos0 + i}: relative logit error {e:.3g}"
        assert argmax_ok(top, want), f"step {pos0 + i}: argmax {top} vs {int(np.argmax(want))}"


@pytest.mark.parametrize("name", ["qwen3_0_6b", "gemma3_1b", "qwen2_7b", "llama3_8b"])
def test_full_size_prompt_decode_and_long_context(name):
    cfg = synth.CONFIGS[name]
    L = LONG[name]
    W = synth.make_model(cfg, seed=0)
    m = gpu_model(cfg, W, L)
    o = oracle.model_from_synth(cfg, W, L)
    toks = synth.tokens(cfg, 32, seed=1)

    got, top = m.forward(toks[:16], 0)
    want = o.forward(toks[:16], 0)
    assert rel(got, want) <= TOL
    assert argmax_ok(top, want)
    check(m, o, toks[16:], 16)

    m.reset_kv()
    o.reset_kv()
    P = L - 4
    for layer in range(cfg.n_layer):
        k, v = synth.kv_fill(cfg, layer, P, seed=2)
        m.write_kv(layer, 0, k, v)
        o.write_kv(layer, 0, k, v)
    o.set_kv_len(P)
    check(m, o, synth.tokens(cfg, 4, seed=3), P)
    m.close()
    o.close()


def test_qwen2_7b_bulk_prefill_2048_matches_token_by_token_and_oracle():
    cfg = synth.CONFIGS["qwen2_7b"]
    n = 2048
    W = synth.make_model(cfg, seed=0)
    m = gpu_model(cfg, W, n)
    toks = synth.tokens(cfg, n, seed=1)

    bulk, _ = m.forward(toks, 0)
    kv_bulk = [m.read_kv(layer, 0, n, cfg.n_head_kv, cfg.head_dim) for layer in range(cfg.n_layer)]
    m.reset_kv()
    for i in range(n - 1):
        m.forward([int(toks[i])], i, want_logits=False)
    step, _ = m.forward([int(toks[n - 1])], n - 1)
    assert rel(bulk, step.astype(np.float64)) <= TOL
    for layer in range(cfg.n_layer):
        kt, vt = m.read_kv(layer, 0, n, cfg.n_head_kv, cfg.head_dim)
        kb, vb = kv_bulk[layer]
        assert np.abs(kb - kt).max() <= 1e-3 * np.abs(kt).max(), f"layer {layer}: keys"
        assert np.abs(vb - vt).max() <= 1e-3 * np.abs(vt).max(), f"layer {layer}: values"

    o = oracle.model_from_synth(cfg, W, n)
    m.reset_kv()
    got, top = m.forward(toks[:64], 0)
    want = o.forward(toks[:64], 0)
    assert rel(got, want) <= TOL
    assert argmax_ok(top, want)
    m.close()
    o.close()
