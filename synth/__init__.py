"""Seeded synthetic GGUF decoders: the inputs that both the oracle and the CUDA path consume.

This module draws random numbers and lays them out in GGUF's storage formats. It holds none of
the decoder's arithmetic: no dequantisation, no matmul, no normalisation. The oracle and the
CUDA library read the *same bytes* it produces, so no random generator is re-implemented on
either side.

Shapes and value distributions follow the five workloads of the decoder token step:

* ``tiny``        qwen3-shaped, f32 weights, 2 layers, hidden 256, 4 Q / 2 KV heads of 64, FFN 512,
                  vocab 1024, untied output.
* ``qwen3_0_6b``  qwen3-shaped, f16 weights, 28 layers, hidden 1024, 16 Q / 8 KV heads of 128,
                  FFN 3072, vocab 151936, tied embeddings.
* ``llama3_8b``   llama-shaped, Q8_0 weights, 32 layers, hidden 4096, 32 Q / 8 KV heads of 128,
                  FFN 14336, vocab 128256, untied, rope base 5e5.
* ``qwen2_7b``    qwen2-shaped (Q/K/V bias), Q4_0 weights, 28 layers, hidden 3584, 28 Q / 4 KV
                  heads of 128, FFN 18944, vocab 152064, untied.
* ``gemma3_1b``   gemma3-shaped, f16 weights, 26 layers, hidden 1152, 4 Q / 1 KV heads of 256,
                  gelu_tanh FFN 6912, vocab 262144, tied, sliding window 512 on 5 of every 6 layers.

Distributions: dense weights N(0, 0.02); Q8_0 codes uniform on [-127, 127] with f16 block scales
|N(0, 0.002)|; Q4_0 codes uniform on 0..15 with the same scale law; norm weights 1 + N(0, 0.1)
(f32); biases N(0, 0.02) (f32); token ids uniform on [0, vocab).

Every tensor has its own stream, derived from (seed, tensor name, chunk index), so a tensor's bytes
do not depend on which other tensors were drawn or on the number of threads used.
"""
from __future__ import annotations

import dataclasses
import os
import zlib
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, Iterator, List, Optional, Tuple

import numpy as np

# GGUF tensor type ids (ggml_type) for the formats the library handles.
GGML_F32 = 0
GGML_F16 = 1
GGML_Q4_0 = 2
GGML_Q8_0 = 8

DTYPE_IDS = {"f32": GGML_F32, "f16": GGML_F16, "q4_0": GGML_Q4_0, "q8_0": GGML_Q8_0}
# (elements per block, bytes per block) of each GGUF storage format
BLOCK = {GGML_F32: (1, 4), GGML_F16: (1, 2), GGML_Q4_0: (32, 18), GGML_Q8_0: (32, 34)}

_CHUNK = 1 << 22  # elements per independently seeded chunk


def tensor_nbytes(dtype_id: int, n_elements: int) -> int:
    per, nb = BLOCK[dtype_id]
    assert n_elements % per == 0, "element count must be a whole number of blocks"
    return n_elements // per * nb


@dataclasses.dataclass(frozen=True)
class ModelConfig:
    name: str
    arch: str
    n_layer: int
    n_embd: int
    n_head: int
    n_head_kv: int
    head_dim: int
    n_ff: int
    n_vocab: int
    wtype: str
    tied: bool
    rope_base: float
    eps: float = 1e-6
    qkv_bias: bool = False
    qk_norm: bool = False
    post_norms: bool = False
    sliding_window: int = 0
    context_length: int = 8192

    @property
    def n_q(self) -> int:
        return self.n_head * self.head_dim

    @property
    def n_kv(self) -> int:
        return self.n_head_kv * self.head_dim


CONFIGS: Dict[str, ModelConfig] = {
    "tiny": ModelConfig("tiny", "qwen3", 2, 256, 4, 2, 64, 512, 1024, "f32", False, 1e6,
                        qk_norm=True, context_length=256),
    "qwen3_0_6b": ModelConfig("qwen3_0_6b", "qwen3", 28, 1024, 16, 8, 128, 3072, 151936, "f16",
                              True, 1e6, qk_norm=True, context_length=4096),
    "llama3_8b": ModelConfig("llama3_8b", "llama", 32, 4096, 32, 8, 128, 14336, 128256, "q8_0",
                             False, 5e5, context_length=8192),
    "qwen2_7b": ModelConfig("qwen2_7b", "qwen2", 28, 3584, 28, 4, 128, 18944, 152064, "q4_0",
                            False, 1e6, qkv_bias=True, context_length=4096),
    "gemma3_1b": ModelConfig("gemma3_1b", "gemma3", 26, 1152, 4, 1, 256, 6912, 262144, "f16",
                             True, 1e6, qk_norm=True, post_norms=True, sliding_window=512,
                             context_length=8192),
}


def scaled(cfg: ModelConfig, **over) -> ModelConfig:
    """A copy of ``cfg`` with some fields replaced (smaller cases of the same architecture)."""
    return dataclasses.replace(cfg, **over)


def metadata(cfg: ModelConfig, max_ctx: Optional[int] = None) -> Dict[str, str]:
    """GGUF metadata keys (as ``key -> text value``) that the forward reads."""
    a = cfg.arch
    md = {
        "general.architecture": a,
        f"{a}.block_count": str(cfg.n_layer),
        f"{a}.embedding_length": str(cfg.n_embd),
        f"{a}.feed_forward_length": str(cfg.n_ff),
        f"{a}.context_length": str(max_ctx or cfg.context_length),
        f"{a}.attention.head_count": str(cfg.n_head),
        f"{a}.attention.head_count_kv": str(cfg.n_head_kv),
        f"{a}.attention.key_length": str(cfg.head_dim),
        f"{a}.attention.value_length": str(cfg.head_dim),
        f"{a}.attention.layer_norm_rms_epsilon": repr(float(cfg.eps)),
        f"{a}.rope.freq_base": repr(float(cfg.rope_base)),
        f"{a}.vocab_size": str(cfg.n_vocab),
    }
    if cfg.sliding_window:
        md[f"{a}.attention.sliding_window"] = str(cfg.sliding_window)
    return md


def metadata_text(md: Dict[str, str]) -> str:
    return "".join(f"{k}={v}\n" for k, v in md.items())


@dataclasses.dataclass
class Tensor:
    """One GGUF tensor: ``ne`` in GGUF order (ne[0] is the contiguous, in-feature axis)."""
    name: str
    dtype: int
    ne: Tuple[int, ...]
    data: np.ndarray  # uint8 view of the GGUF-format bytes

    @property
    def n_elements(self) -> int:
        n = 1
        for e in self.ne:
            n *= e
        return n


def tensor_specs(cfg: ModelConfig) -> List[Tuple[str, str, Tuple[int, ...]]]:
    """(name, kind, ne) for every tensor of the model, in GGUF naming.

    kind is one of "w" (matrix in the model's storage type), "norm" (f32 1+N(0,0.1)),
    "bias" (f32 N(0,0.02)).
    """
    H, Q, KV, F, V, hd = cfg.n_embd, cfg.n_q, cfg.n_kv, cfg.n_ff, cfg.n_vocab, cfg.head_dim
    specs = [("token_embd.weight", "w", (H, V)), ("output_norm.weight", "norm", (H,))]
    if not cfg.tied:
        specs.append(("output.weight", "w", (H, V)))
    for i in range(cfg.n_layer):
        b = f"blk.{i}."
        specs += [
            (b + "attn_norm.weight", "norm", (H,)),
            (b + "attn_q.weight", "w", (H, Q)),
            (b + "attn_k.weight", "w", (H, KV)),
            (b + "attn_v.weight", "w", (H, KV)),
        ]
        if cfg.qkv_bias:
            specs += [(b + "attn_q.bias", "bias", (Q,)), (b + "attn_k.bias", "bias", (KV,)),
                      (b + "attn_v.bias", "bias", (KV,))]
        if cfg.qk_norm:
            specs += [(b + "attn_q_norm.weight", "norm", (hd,)),
                      (b + "attn_k_norm.weight", "norm", (hd,))]
        specs.append((b + "attn_output.weight", "w", (Q, H)))
        if cfg.post_norms:
            specs.append((b + "post_attention_norm.weight", "norm", (H,)))
        specs += [
            (b + "ffn_norm.weight", "norm", (H,)),
            (b + "ffn_gate.weight", "w", (H, F)),
            (b + "ffn_up.weight", "w", (H, F)),
            (b + "ffn_down.weight", "w", (F, H)),
        ]
        if cfg.post_norms:
            specs.append((b + "post_ffw_norm.weight", "norm", (H,)))
    return specs


def _gen(seed: int, name: str, chunk: int) -> np.random.Generator:
    key = zlib.crc32(name.encode())
    return np.random.Generator(np.random.SFC64(np.random.SeedSequence([seed, key, chunk])))


_POOL: Optional[ThreadPoolExecutor] = None


def _pool() -> ThreadPoolExecutor:
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max(1, min(32, os.cpu_count() or 1)))
    return _POOL


def _chunked(n: int, fill, seed: int, name: str) -> None:
    """Call fill(gen, lo, hi) for every chunk of [0, n), in parallel."""
    jobs = [(c, c * _CHUNK, min(n, (c + 1) * _CHUNK)) for c in range((n + _CHUNK - 1) // _CHUNK)]
    list(_pool().map(lambda j: fill(_gen(seed, name, j[0]), j[1], j[2]), jobs))


def normal_f32(seed: int, name: str, n: int, mean: float, std: float) -> np.ndarray:
    out = np.empty(n, np.float32)

    def fill(g, lo, hi):
        g.standard_normal(out=out[lo:hi], dtype=np.float32)
        out[lo:hi] *= np.float32(std)
        if mean:
            out[lo:hi] += np.float32(mean)
    _chunked(n, fill, seed, name)
    return out


def _int8_symmetric(seed: int, name: str, n: int) -> np.ndarray:
    """int8 codes uniform on [-127, 127]."""
    out = np.empty(n, np.int8)

    def fill(g, lo, hi):
        out[lo:hi] = g.integers(-127, 128, size=hi - lo, dtype=np.int8)
    _chunked(n, fill, seed, name + "#codes")
    return out


def _uint8_full(seed: int, name: str, n: int) -> np.ndarray:
    """bytes uniform on 0..255 (two independent uniform 4-bit codes per byte)."""
    out = np.empty(n, np.uint8)

    def fill(g, lo, hi):
        out[lo:hi] = g.integers(0, 256, size=hi - lo, dtype=np.uint8)
    _chunked(n, fill, seed, name + "#codes")
    return out


def block_scales(seed: int, name: str, n_blocks: int) -> np.ndarray:
    """f16 block scales |N(0, 0.002)|."""
    s = normal_f32(seed, name + "#scales", n_blocks, 0.0, 0.002)
    np.abs(s, out=s)
    return s.astype(np.float16)


def make_weight(seed: int, name: str, wtype: str, ne: Tuple[int, ...]) -> Tensor:
    n = int(np.prod(ne))
    dt = DTYPE_IDS[wtype]
    if dt == GGML_F32:
        raw = normal_f32(seed, name, n, 0.0, 0.02).view(np.uint8)
    elif dt == GGML_F16:
        raw = normal_f32(seed, name, n, 0.0, 0.02).astype(np.float16).view(np.uint8)
    elif dt == GGML_Q8_0:
        nb = n // 32
        blocks = np.empty((nb, 34), np.uint8)
        blocks[:, 0:2] = block_scales(seed, name, nb).view(np.uint8).reshape(nb, 2)
        blocks[:, 2:] = _int8_symmetric(seed, name, n).view(np.uint8).reshape(nb, 32)
        raw = blocks.reshape(-1)
    elif dt == GGML_Q4_0:
        nb = n // 32
        blocks = np.empty((nb, 18), np.uint8)
        blocks[:, 0:2] = block_scales(seed, name, nb).view(np.uint8).reshape(nb, 2)
        blocks[:, 2:] = _uint8_full(seed, name, nb * 16).reshape(nb, 16)
        raw = blocks.reshape(-1)
    else:
        raise ValueError(wtype)
    return Tensor(name, dt, tuple(ne), raw)


def make_tensor(cfg: ModelConfig, seed: int, name: str, kind: str, ne: Tuple[int, ...]) -> Tensor:
    if kind == "w":
        return make_weight(seed, name, cfg.wtype, ne)
    n = int(np.prod(ne))
    if kind == "norm":
        return Tensor(name, GGML_F32, ne, normal_f32(seed, name, n, 1.0, 0.1).view(np.uint8))
    if kind == "bias":
        return Tensor(name, GGML_F32, ne, normal_f32(seed, name, n, 0.0, 0.02).view(np.uint8))
    raise ValueError(kind)


def make_model(cfg: ModelConfig, seed: int = 0) -> Dict[str, Tensor]:
    """All tensors of a seeded synthetic model (weights seed 0 by convention)."""
    return {name: make_tensor(cfg, seed, name, kind, ne) for name, kind, ne in tensor_specs(cfg)}


def iter_model(cfg: ModelConfig, seed: int = 0) -> Iterator[Tensor]:
    """Like make_model, one tensor at a time (to stream a large model into a loader)."""
    for name, kind, ne in tensor_specs(cfg):
        yield make_tensor(cfg, seed, name, kind, ne)


def tokens(cfg: ModelConfig, n: int, seed: int = 1) -> np.ndarray:
    """Token ids uniform on [0, vocab) (seed 1 by convention)."""
    g = np.random.Generator(np.random.SFC64(np.random.SeedSequence([seed, 0x70CE])))
    return g.integers(0, cfg.n_vocab, size=n, dtype=np.int64).astype(np.int32)


def kv_fill(cfg: ModelConfig, layer: int, n_pos: int, seed: int = 2) -> Tuple[np.ndarray, np.ndarray]:
    """N(0,1) keys and values [n_head_kv][n_pos][head_dim] that stand in for a long prompt."""
    n = cfg.n_head_kv * n_pos * cfg.head_dim
    shape = (cfg.n_head_kv, n_pos, cfg.head_dim)
    k = normal_f32(seed, f"kv.{layer}.k", n, 0.0, 1.0).reshape(shape)
    v = normal_f32(seed, f"kv.{layer}.v", n, 0.0, 1.0).reshape(shape)
    return k, v


def weight_bytes(cfg: ModelConfig) -> int:
    """Stored bytes of all tensors (GGUF formats)."""
    tot = 0
    for name, kind, ne in tensor_specs(cfg):
        n = int(np.prod(ne))
        tot += tensor_nbytes(DTYPE_IDS[cfg.wtype], n) if kind == "w" else 4 * n
    return tot
