"""An independent float64 restatement of the decoder forward with PyTorch CPU library routines.

Used only to pin the oracle (tests/test_oracle_pins.py). It is written from the model's
definition, not from the oracle and not from an .archdef text: ``F.rms_norm`` for RMSNorm,
complex multiplication (``torch.polar``) for the rotary embedding, ``F.scaled_dot_product_attention``
with an explicit causal / sliding-window mask for attention, ``F.silu`` / ``F.gelu`` for the gates.
GGUF blocks are decoded with numpy structured dtypes.
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F

import synth


def dequant(t: "synth.Tensor") -> np.ndarray:
    """float64 matrix [ne1][ne0] (or vector) of a GGUF tensor."""
    k = t.ne[0]
    rows = t.n_elements // k
    if t.dtype == synth.GGML_F32:
        w = t.data.view(np.float32).astype(np.float64)
    elif t.dtype == synth.GGML_F16:
        w = t.data.view(np.float16).astype(np.float64)
    elif t.dtype == synth.GGML_Q8_0:
        blk = t.data.view(np.dtype([("d", "<f2"), ("q", "i1", (32,))]))
        w = (blk["d"].astype(np.float64)[:, None] * blk["q"].astype(np.float64)).reshape(-1)
    elif t.dtype == synth.GGML_Q4_0:
        blk = t.data.view(np.dtype([("d", "<f2"), ("qs", "u1", (16,))]))
        lo = (blk["qs"] & 15).astype(np.float64) - 8
        hi = (blk["qs"] >> 4).astype(np.float64) - 8
        w = (blk["d"].astype(np.float64)[:, None] * np.concatenate([lo, hi], axis=1)).reshape(-1)
    else:
        raise ValueError(t.dtype)
    return w.reshape(rows, k) if len(t.ne) > 1 else w


def _rope(x: torch.Tensor, pos: torch.Tensor, base: float, adjacent: bool) -> torch.Tensor:
    """x [n, heads, hd] rotated at positions pos [n]."""
    hd = x.shape[-1]
    freqs = base ** (-torch.arange(0, hd, 2, dtype=torch.float64) / hd)
    rot = torch.polar(torch.ones(len(pos), hd // 2, dtype=torch.float64), pos[:, None] * freqs[None])
    if adjacent:
        z = torch.view_as_complex(x.reshape(*x.shape[:-1], hd // 2, 2).contiguous())
        return torch.view_as_real(z * rot[:, None, :]).reshape(x.shape)
    z = torch.complex(x[..., : hd // 2], x[..., hd // 2:])
    z = z * rot[:, None, :]
    return torch.cat([z.real, z.imag], dim=-1)


def forward(cfg: "synth.ModelConfig", tensors, tokens, *, rope_adjacent: bool,
            window_pattern: int = 0, embed_scale: float = 0.0, act: str = "silu",
            kv_prefix=None):
    """Logits (float64) of every row for a prompt processed from position 0 (or after kv_prefix).

    kv_prefix: optional list per layer of (K, V) float64 [n_head_kv][P][hd] already in the cache.
    Returns (logits [n][V], x_final [n][H]).
    """
    W = {name: torch.from_numpy(dequant(t)) for name, t in tensors.items()}
    H, nh, nkv, hd, eps = cfg.n_embd, cfg.n_head, cfg.n_head_kv, cfg.head_dim, cfg.eps
    toks = torch.as_tensor(np.asarray(tokens, dtype=np.int64))
    n = len(toks)
    P = 0 if kv_prefix is None else kv_prefix[0][0].shape[1]
    pos = torch.arange(P, P + n, dtype=torch.float64)
    x = W["token_embd.weight"][toks]
    if embed_scale:
        x = x * torch.tensor(np.float32(embed_scale), dtype=torch.float64)
    act_fn = {"silu": F.silu, "gelu_tanh": lambda t: F.gelu(t, approximate="tanh"),
              "gelu": F.gelu}[act]
    for i in range(cfg.n_layer):
        b = f"blk.{i}."
        h = F.rms_norm(x, (H,), W[b + "attn_norm.weight"], eps)
        q = h @ W[b + "attn_q.weight"].T
        k = h @ W[b + "attn_k.weight"].T
        v = h @ W[b + "attn_v.weight"].T
        if cfg.qkv_bias:
            q, k, v = q + W[b + "attn_q.bias"], k + W[b + "attn_k.bias"], v + W[b + "attn_v.bias"]
        q, k, v = q.view(n, nh, hd), k.view(n, nkv, hd), v.view(n, nkv, hd)
        if cfg.qk_norm:
            q = F.rms_norm(q, (hd,), W[b + "attn_q_norm.weight"], eps)
            k = F.rms_norm(k, (hd,), W[b + "attn_k_norm.weight"], eps)
        q, k = _rope(q, pos, cfg.rope_base, rope_adjacent), _rope(k, pos, cfg.rope_base, rope_adjacent)
        K, V = k.transpose(0, 1), v.transpose(0, 1)  # [nkv, n, hd]
        if kv_prefix is not None:
            K = torch.cat([torch.as_tensor(kv_prefix[i][0], dtype=torch.float64), K], dim=1)
            V = torch.cat([torch.as_tensor(kv_prefix[i][1], dtype=torch.float64), V], dim=1)
        kpos = torch.arange(0, P + n, dtype=torch.float64)
        allowed = kpos[None, :] <= pos[:, None]
        glob = window_pattern and i % window_pattern == window_pattern - 1
        if cfg.sliding_window and not glob:
            allowed &= kpos[None, :] > pos[:, None] - cfg.sliding_window
        grp = nh // nkv
        a = F.scaled_dot_product_attention(q.transpose(0, 1), K.repeat_interleave(grp, 0),
                                           V.repeat_interleave(grp, 0), attn_mask=allowed,
                                           scale=1.0 / math.sqrt(hd))
        a = a.transpose(0, 1).reshape(n, nh * hd)
        o = a @ W[b + "attn_output.weight"].T
        if cfg.post_norms:
            o = F.rms_norm(o, (H,), W[b + "post_attention_norm.weight"], eps)
        x = x + o
        h = F.rms_norm(x, (H,), W[b + "ffn_norm.weight"], eps)
        g = act_fn(h @ W[b + "ffn_gate.weight"].T) * (h @ W[b + "ffn_up.weight"].T)
        d = g @ W[b + "ffn_down.weight"].T
        if cfg.post_norms:
            d = F.rms_norm(d, (H,), W[b + "post_ffw_norm.weight"], eps)
        x = x + d
    x = F.rms_norm(x, (H,), W["output_norm.weight"], eps)
    out = W["output.weight"] if "output.weight" in W else W["token_embd.weight"]
    return (x @ out.T).numpy(), x.numpy()
