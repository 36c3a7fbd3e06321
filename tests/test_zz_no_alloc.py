"""The allocation-free attention entry point (syn_attention_static), through the C ABI.

It exists for callers that cannot allocate device memory when they need attention, for example
code running while a stream is captured into a CUDA graph, or a plug-in inside a host framework
that has already reserved the device memory. Its scratch lives in a fixed device array inside the
library. Its output is compared with the oracle's attention (per query head over the same keys) and
with the attention that syn_forward computes for the same query and cache, each on two calls in a
row (the shared array keeps the previous call's contents, so the second call checks that the state
a call needs is cleared). A bounded wait that gives up is reported by syn_attention_static_status.
This file is collected last.
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


@pytest.fixture(scope="module")
def L():
    syn_build.build()
    return syn.lib()


def call(L, q, kc, vc, n_head, n_head_kv, hd, max_ctx, n_ctx, window, splits, out):
    return L.syn_attention_static(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), n_head, n_head_kv, hd, max_ctx, n_ctx,
                                  window, splits, out.data_ptr(), None)


def oracle_attention(q, K, V, n_head, n_head_kv, hd, n_ctx, window):
    """Per query head h: the oracle's softmax(q_h . K_t / sqrt(hd)) V_t over the allowed keys
    lo .. pos (both included) of KV head h / (n_head / n_head_kv)."""
    G = n_head // n_head_kv
    pos = n_ctx - 1
    lo = max(0, pos - window + 1) if window > 0 else 0
    out = np.empty(n_head * hd, np.float32)
    for h in range(n_head):
        g = h // G
        out[h * hd:(h + 1) * hd] = oracle.attend(q[h * hd:(h + 1) * hd], K[g], V[g], lo, pos)
    return out


SHAPES = [(64, 8, 8), (64, 16, 2), (128, 32, 8), (128, 8, 1), (256, 4, 1), (256, 2, 2)]


@pytest.mark.parametrize("splits", [1, 7, 64])
@pytest.mark.parametrize("window", [0, 64])
@pytest.mark.parametrize("hd,n_head,n_head_kv", SHAPES)
def test_static_attention_matches_the_oracle_on_two_calls(L, hd, n_head, n_head_kv, window, splits):
    """Head sizes 64/128/256; 1, 4 and 8 query heads per KV head; global and windowed keys; 1, 7 and
    64 key slices. The second call has fewer keys than 64 slices, so some slices are empty."""
    import torch

    max_ctx = 320
    rng = np.random.default_rng(hd * 1000 + n_head * 10 + n_head_kv + window + splits)
    K = rng.standard_normal((n_head_kv, max_ctx, hd)).astype(np.float32)
    V = rng.standard_normal((n_head_kv, max_ctx, hd)).astype(np.float32)
    kc = torch.from_numpy(K).cuda()
    vc = torch.from_numpy(V).cuda()
    for n_ctx in (300, 40):
        q = rng.standard_normal(n_head * hd).astype(np.float32)
        dq = torch.from_numpy(q).cuda()
        out = torch.full((n_head * hd,), float("nan"), dtype=torch.float32, device="cuda")
        assert call(L, dq, kc, vc, n_head, n_head_kv, hd, max_ctx, n_ctx, window, splits, out) == 0
        assert L.syn_attention_static_status(None) == 0
        got = out.cpu().numpy()
        want = oracle_attention(q, K, V, n_head, n_head_kv, hd, n_ctx, window)
        err = float(np.abs(got - want).max() / np.abs(want).max())
        assert err <= HIDDEN_TOL, f"n_ctx {n_ctx}: relative error {err:.3g}"


def test_static_scratch_attention_matches_the_forward_twice(L):
    import torch

    cfg = synth.scaled(synth.CONFIGS["llama3_8b"], name="llama_small", n_layer=2, n_embd=512, n_head=8,
                       n_head_kv=2, head_dim=128, n_ff=768, n_vocab=500, wtype="f16")
    max_ctx = 320
    m = syn.Model(syn.read_archdef("llama"), synth.metadata(cfg, max_ctx), max_ctx, arch="llama")
    m.set_option("fusion", 0)  # keep the q and a registers materialised
    m.load_tensors(synth.make_model(cfg, seed=0))
    m.finalize()
    P0 = 200
    for layer in range(cfg.n_layer):
        k, v = synth.kv_fill(cfg, layer, P0, seed=2)
        m.write_kv(layer, 0, k, v)
    toks = synth.tokens(cfg, 2, seed=1)
    last = cfg.n_layer - 1
    width = cfg.n_head * cfg.head_dim
    for step in range(2):
        pos = P0 + step
        m.forward([int(toks[step])], pos)
        q = m.read_register("q", width)
        want = m.read_register("a", width)
        k, v = m.read_kv(last, 0, pos + 1, cfg.n_head_kv, cfg.head_dim)
        kc = torch.zeros((cfg.n_head_kv, max_ctx, cfg.head_dim), dtype=torch.float32, device="cuda")
        vc = torch.zeros_like(kc)
        kc[:, :pos + 1] = torch.from_numpy(k).cuda()
        vc[:, :pos + 1] = torch.from_numpy(v).cuda()
        dq = torch.from_numpy(q).cuda()
        out = torch.full((width,), float("nan"), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        assert call(L, dq, kc, vc, cfg.n_head, cfg.n_head_kv, cfg.head_dim, max_ctx, pos + 1, 0, 7, out) == 0
        assert L.syn_attention_static_status(None) == 0
        got = out.cpu().numpy()
        err = float(np.abs(got - want).max() / np.abs(want).max())
        assert err <= TOL, f"call {step}: relative error {err:.3g}"


def test_a_wait_that_gives_up_is_reported_and_the_next_call_is_valid(L):
    """With the wait bound at zero polls every bounded wait gives up at once: the kernel records the
    error and drains its copies; the status call reports it (and clears it); the device stays usable
    and the next call with the default bound is correct."""
    import torch

    hd, n_head, n_head_kv, max_ctx, n_ctx = 128, 8, 2, 512, 500
    rng = np.random.default_rng(5)
    K = rng.standard_normal((n_head_kv, max_ctx, hd)).astype(np.float32)
    V = rng.standard_normal((n_head_kv, max_ctx, hd)).astype(np.float32)
    q = rng.standard_normal(n_head * hd).astype(np.float32)
    kc, vc, dq = torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda(), torch.from_numpy(q).cuda()
    out = torch.zeros(n_head * hd, dtype=torch.float32, device="cuda")
    try:
        L.syn_debug_set_spin_limit(0)
        assert call(L, dq, kc, vc, n_head, n_head_kv, hd, max_ctx, n_ctx, 0, 4, out) == 0
        assert L.syn_attention_static_status(None) == 10       # SYN_E_CUDA: a wait gave up
    finally:
        L.syn_debug_set_spin_limit(-1)
    assert L.syn_attention_static_status(None) == 0            # read once, then cleared
    assert call(L, dq, kc, vc, n_head, n_head_kv, hd, max_ctx, n_ctx, 0, 4, out) == 0
    assert L.syn_attention_static_status(None) == 0
    want = oracle_attention(q, K, V, n_head, n_head_kv, hd, n_ctx, 0)
    got = out.cpu().numpy()
    assert float(np.abs(got - want).max() / np.abs(want).max()) <= HIDDEN_TOL


def test_static_scratch_attention_rejects_oversized_requests(L):
    import ctypes
    dummy = ctypes.c_void_p(16)  # never dereferenced: the size checks come first
    f = L.syn_attention_static
    # 64 splits x 128 heads x (256 + 4) floats is more than the 4 MiB array holds
    assert f(dummy, dummy, dummy, 128, 32, 256, 1024, 10, 0, 64, dummy, None) == 12
    assert f(dummy, dummy, dummy, 8, 2, 128, 1024, 10, 0, 65, dummy, None) == 12   # too many splits
    assert f(dummy, dummy, dummy, 8, 2, 96, 1024, 10, 0, 4, dummy, None) == 1      # unsupported head_dim


def test_static_attention_on_a_second_device_when_one_is_visible(L):
    """The kernel's shared-memory limit is set per device: a call on device 1 (after calls on device
    0 above) must run and match the oracle. Skipped where only one GPU is visible."""
    import torch

    if torch.cuda.device_count() < 2:
        pytest.skip("one GPU visible")
    hd, n_head, n_head_kv, max_ctx, n_ctx = 128, 8, 2, 256, 200
    rng = np.random.default_rng(11)
    K = rng.standard_normal((n_head_kv, max_ctx, hd)).astype(np.float32)
    V = rng.standard_normal((n_head_kv, max_ctx, hd)).astype(np.float32)
    q = rng.standard_normal(n_head * hd).astype(np.float32)
    with torch.cuda.device(1):
        kc, vc, dq = (torch.from_numpy(a).cuda() for a in (K, V, q))
        out = torch.zeros(n_head * hd, dtype=torch.float32, device="cuda")
        assert call(L, dq, kc, vc, n_head, n_head_kv, hd, max_ctx, n_ctx, 0, 7, out) == 0
        assert L.syn_attention_static_status(None) == 0
        got = out.cpu().numpy()
    want = oracle_attention(q, K, V, n_head, n_head_kv, hd, n_ctx, 0)
    assert float(np.abs(got - want).max() / np.abs(want).max()) <= HIDDEN_TOL
