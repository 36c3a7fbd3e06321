"""The allocation-free attention entry point (syn_attention_static), through the C ABI.

It exists for callers that cannot allocate device memory when they need attention, for example
code running while a stream is captured into a CUDA graph, or a plug-in inside a host framework
that has already reserved the device memory. Its scratch lives in a fixed device array inside the
library. Here its output is compared with the attention that syn_forward computes for the same
query and cache, on two calls in a row (the shared array keeps the previous call's contents, so the
second call checks that the state a call needs is cleared). This file is collected last.
"""
import ctypes

import numpy as np
import pytest

import synth
from decoder_token_step_gb300 import build as syn_build
from decoder_token_step_gb300 import syn

pytestmark = pytest.mark.gpu

TOL = 2e-3


def test_static_scratch_attention_matches_the_forward_twice():
    import torch

    syn_build.build()
    L = syn.lib()
    f = L.syn_attention_static
    P, I = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [P, P, P, I, I, I, I, I, I, I, P, P]
    f.restype = I

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
        rc = f(dq.data_ptr(), kc.data_ptr(), vc.data_ptr(), cfg.n_head, cfg.n_head_kv, cfg.head_dim, max_ctx,
               pos + 1, 0, 7, out.data_ptr(), None)
        assert rc == 0
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        err = float(np.abs(got - want).max() / np.abs(want).max())
        assert err <= TOL, f"call {step}: relative error {err:.3g}"


def test_static_scratch_attention_rejects_oversized_requests():
    syn_build.build()
    f = syn.lib().syn_attention_static
    P, I = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [P, P, P, I, I, I, I, I, I, I, P, P]
    f.restype = I
    dummy = ctypes.c_void_p(16)  # never dereferenced: the size checks come first
    # 64 splits x 128 heads x (256 + 4) floats is more than the 4 MiB array holds
    assert f(dummy, dummy, dummy, 128, 32, 256, 1024, 10, 0, 64, dummy, None) == 12
    assert f(dummy, dummy, dummy, 8, 2, 128, 1024, 10, 0, 65, dummy, None) == 12   # too many splits
    assert f(dummy, dummy, dummy, 8, 2, 96, 1024, 10, 0, 4, dummy, None) == 1      # unsupported head_dim
