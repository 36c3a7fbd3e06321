"""GPU parity at the full sizes of the four named workloads (the tiny one is in test_gpu_parity.py).

For each model: the same seeded weights on both sides, a 16-token prompt run as one bulk forward,
then 16 teacher-forced decode steps; then, after a KV reset, the same N(0, 1) keys and values
injected into positions [0, L-4) on both sides and 4 teacher-forced steps ending at position L-1,
with L the context length the decode is measured at (4096 for qwen3-0.6B, 8192 for llama-3-8B and
gemma3-1B, where 22 of the 26 layers only see their last 512 keys, 2048 for qwen2-7B).

qwen2-7B (Q4_0, Q/K/V bias) also runs its 2048-token prompt as one bulk forward and token by token
on the GPU: the last row's logits and every cached key and value must agree within the tolerance;
and a 64-token bulk forward is compared with the oracle's.

qwen2-7B also decodes 256 teacher-forced steps from the cache its 2048-token bulk prefill wrote and
from the cache the token-by-token prefill wrote: every step's logits must agree, so the bulk path
writes a cache that decode reads as it reads its own.

Tolerances as in test_gpu_parity.py: max|dlogit| <= 2e-3 * max|logit| per step, argmax equal where
the oracle's top-2 gap exceeds twice that; the hidden state (the residual x after the last block,
which the decode and bulk plans keep in register x) within ||dx||_inf <= 1e-3 ||x||_inf every step.
"""
import numpy as np
import pytest

import oracle
import synth
from decoder_token_step_gb300 import build as syn_build
from decoder_token_step_gb300 import syn

pytestmark = pytest.mark.gpu

TOL = 2e-3
HIDDEN_TOL = 1e-3
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


def forward_checked(m, o, cfg, toks, pos):
    """One forward on both sides: logits, argmax and the hidden state. A decode step's fused plan
    folds the epilogue's in-place rms_norm into the logits matmul, so its register x holds the
    residual after the last block (the oracle's last layer output); a bulk plan runs that norm and
    `last`, so x holds the last row after the epilogue (the oracle's x_out)."""
    got, top = m.forward(toks, pos)
    want, x_out, lx = o.forward(toks, pos, want_x=True, n_layer=cfg.n_layer)
    e = rel(got, want)
    assert e <= TOL, f"position {pos}: relative logit error {e:.3g}"
    assert argmax_ok(top, want), f"position {pos}: argmax {top} vs {int(np.argmax(want))}"
    x = m.read_register("x", cfg.n_embd)
    ref = lx[-1] if len(toks) == 1 else x_out
    ex = rel(x, ref.astype(np.float64))
    assert ex <= HIDDEN_TOL, f"position {pos}: relative hidden-state error {ex:.3g}"


def check(m, o, cfg, toks, pos0):
    for i, t in enumerate(toks):
        forward_checked(m, o, cfg, [int(t)], pos0 + i)


@pytest.mark.parametrize("name", ["qwen3_0_6b", "gemma3_1b", "qwen2_7b", "llama3_8b"])
def test_full_size_prompt_decode_and_long_context(name):
    cfg = synth.CONFIGS[name]
    L = LONG[name]
    W = synth.make_model(cfg, seed=0)
    m = gpu_model(cfg, W, L)
    o = oracle.model_from_synth(cfg, W, L)
    toks = synth.tokens(cfg, 32, seed=1)

    forward_checked(m, o, cfg, toks[:16], 0)
    check(m, o, cfg, toks[16:], 16)

    m.reset_kv()
    o.reset_kv()
    P = L - 4
    for layer in range(cfg.n_layer):
        k, v = synth.kv_fill(cfg, layer, P, seed=2)
        m.write_kv(layer, 0, k, v)
        o.write_kv(layer, 0, k, v)
    o.set_kv_len(P)
    check(m, o, cfg, synth.tokens(cfg, 4, seed=3), P)
    m.close()
    o.close()


def test_qwen2_7b_bulk_prefill_2048_matches_token_by_token_then_256_decode_steps():
    cfg = synth.CONFIGS["qwen2_7b"]
    n, steps = 2048, 256
    W = synth.make_model(cfg, seed=0)
    m = gpu_model(cfg, W, n + steps)
    toks = synth.tokens(cfg, n + steps, seed=1)

    bulk, _ = m.forward(toks[:n], 0)
    kv_bulk = [m.read_kv(layer, 0, n, cfg.n_head_kv, cfg.head_dim) for layer in range(cfg.n_layer)]
    after_bulk = [m.forward([int(toks[n + i])], n + i)[0] for i in range(steps)]
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
    # the same 256 decode steps from the token-by-token cache
    for i in range(steps):
        want, top = m.forward([int(toks[n + i])], n + i)
        want = want.astype(np.float64)
        got = after_bulk[i]
        assert rel(got, want) <= TOL, f"decode step {i} after the bulk prefill"
        assert argmax_ok(int(np.argmax(got)), want), f"decode step {i}: argmax"

    o = oracle.model_from_synth(cfg, W, n)
    m.reset_kv()
    forward_checked(m, o, cfg, toks[:64], 0)
    m.close()
    o.close()
