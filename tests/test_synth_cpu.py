"""The seeded input generator that both sides read (CPU only).

It must give the same bytes whatever the thread count, write GGUF storage formats of the right
sizes, and draw from the stated distributions: dense weights N(0, 0.02), norm weights 1 + N(0, 0.1),
biases N(0, 0.02), Q8_0 codes uniform on [-127, 127] and Q4_0 codes uniform on 0..15, both with
f16 block scales |N(0, 0.002)|, tokens uniform on the vocabulary, injected keys and values N(0, 1).
"""
import math

import numpy as np
import pytest

import synth


def _small(wtype, **over):
    d = dict(n_layer=2, n_embd=256, n_head=4, n_head_kv=2, head_dim=64, n_ff=512, n_vocab=1000, wtype=wtype)
    d.update(over)
    return synth.scaled(synth.CONFIGS["llama3_8b"], name=f"synth_{wtype}", **d)


def test_bytes_do_not_depend_on_the_thread_count():
    cfg = _small("q8_0", n_embd=2048, n_ff=4096)   # several generator chunks per tensor
    a = synth.make_model(cfg, seed=0)
    saved = synth._POOL
    try:
        synth._POOL = synth.ThreadPoolExecutor(1)
        b = synth.make_model(cfg, seed=0)
    finally:
        synth._POOL.shutdown()
        synth._POOL = saved
    assert a.keys() == b.keys()
    for name in a:
        assert np.array_equal(a[name].data, b[name].data), name


def test_seeds_and_names_give_independent_streams():
    cfg = _small("f32")
    a, b = synth.make_model(cfg, seed=0), synth.make_model(cfg, seed=1)
    q0 = a["blk.0.attn_q.weight"].data.view(np.float32)
    assert not np.array_equal(q0, b["blk.0.attn_q.weight"].data.view(np.float32))
    assert not np.array_equal(q0[:1000], a["blk.1.attn_q.weight"].data.view(np.float32)[:1000])


@pytest.mark.parametrize("wtype", ["f32", "f16", "q8_0", "q4_0"])
def test_tensor_bytes_are_the_gguf_storage_sizes(wtype):
    cfg = _small(wtype)
    per_block = {"f32": 4 * 32, "f16": 2 * 32, "q8_0": 34, "q4_0": 18}[wtype]
    for name, t in synth.make_model(cfg).items():
        if len(t.ne) == 2:
            assert t.data.nbytes == t.n_elements // 32 * per_block, name
            assert t.dtype == synth.DTYPE_IDS[wtype]
        else:
            assert t.data.nbytes == 4 * t.n_elements and t.dtype == 0, name   # vectors are f32


def test_dense_norm_and_bias_distributions():
    cfg = _small("f32", n_embd=1024, qkv_bias=True)
    W = synth.make_model(cfg)
    w = W["blk.0.ffn_gate.weight"].data.view(np.float32).astype(np.float64)
    assert abs(w.mean()) < 2e-4 and abs(w.std() / 0.02 - 1) < 0.01
    n = np.concatenate([W[f"blk.{i}.{k}_norm.weight"].data.view(np.float32) for i in range(2) for k in ("attn", "ffn")])
    assert abs(n.mean() - 1) < 0.01 and abs(n.std() / 0.1 - 1) < 0.05
    b = np.concatenate([W[f"blk.{i}.attn_{k}.bias"].data.view(np.float32) for i in range(2) for k in "qkv"])
    assert abs(b.mean()) < 2e-3 and abs(b.std() / 0.02 - 1) < 0.1
    h = W["blk.0.attn_q.weight"]
    f16 = synth.make_weight(0, "x", "f16", h.ne).data.view(np.float16)
    assert np.array_equal(f16, synth.make_weight(0, "x", "f32", h.ne).data.view(np.float32).astype(np.float16))


def _blocks(t, size):
    return t.data.reshape(-1, size)


def test_q8_0_codes_and_scales():
    cfg = _small("q8_0", n_embd=1024, n_ff=2048)
    t = synth.make_model(cfg)["blk.0.ffn_up.weight"]
    blk = _blocks(t, 34)
    d = blk[:, :2].copy().view(np.float16).astype(np.float64).reshape(-1)
    q = blk[:, 2:].view(np.int8).astype(np.int64)
    assert q.min() == -127 and q.max() == 127                     # never -128
    counts = np.bincount(q.reshape(-1) + 127, minlength=255)
    assert counts.min() > 0.8 * counts.mean() and counts.max() < 1.2 * counts.mean()
    assert (d >= 0).all()
    assert abs(d.mean() / (0.002 * math.sqrt(2 / math.pi)) - 1) < 0.02   # mean of |N(0, s)| is s * sqrt(2/pi)


def test_q4_0_codes_and_scales():
    cfg = _small("q4_0", n_embd=1024, n_ff=2048)
    t = synth.make_model(cfg)["blk.0.ffn_down.weight"]
    blk = _blocks(t, 18)
    d = blk[:, :2].copy().view(np.float16).astype(np.float64).reshape(-1)
    codes = np.concatenate([blk[:, 2:] & 15, blk[:, 2:] >> 4]).reshape(-1)
    counts = np.bincount(codes, minlength=16)
    assert len(counts) == 16 and counts.min() > 0.95 * counts.mean() and counts.max() < 1.05 * counts.mean()
    assert (d >= 0).all() and abs(d.mean() / (0.002 * math.sqrt(2 / math.pi)) - 1) < 0.03


def test_tokens_and_injected_kv():
    cfg = _small("f32")
    tok = synth.tokens(cfg, 20000, seed=1)
    assert tok.dtype == np.int32 and tok.min() >= 0 and tok.max() < cfg.n_vocab
    assert np.array_equal(tok, synth.tokens(cfg, 20000, seed=1))
    k, v = synth.kv_fill(cfg, 0, 500, seed=2)
    assert k.shape == (cfg.n_head_kv, 500, cfg.head_dim) and v.shape == k.shape
    for x in (k, v):
        assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02
    k1, _ = synth.kv_fill(cfg, 1, 500, seed=2)
    assert not np.array_equal(k, k1)
